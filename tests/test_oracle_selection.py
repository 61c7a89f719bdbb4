"""Pins for oracle.selection (TAPS §4.1-4.2 budgeted prefix-closed subtree; TreeGraft
§3.1 path score): brute-force enumeration of every candidate on tiny pools, exhaustive
optimality over prefix-closed sets, and closed-form special cases."""
import itertools

import numpy as np
import pytest

import synth
from oracle import selection


def _all_paths(d, k):
    for depth in range(1, d + 1):
        for path in itertools.product(range(k), repeat=depth):
            yield path


def _brute(marg, ptok, budget, root_token):
    d, k = marg.shape
    cands = []
    for path in _all_paths(d, k):
        s = np.float32(1.0)
        for pos, r in enumerate(path):
            s = np.float32(s * marg[pos, r])
        cands.append((-float(s), len(path), path))
    cands.sort()
    chosen = [c[2] for c in cands[: budget - 1]]
    index = {(): 0}
    parent, token, depth, score = [-1], [root_token], [0], [np.float32(1.0)]
    for j, path in enumerate(chosen, start=1):
        index[path] = j
        parent.append(index[path[:-1]])
        token.append(int(ptok[len(path) - 1, path[-1]]))
        depth.append(len(path))
        score.append(np.float32(-[c for c in cands if c[2] == path][0][0]))
    return parent, token, depth, score


def _pool(seed, d, k, ties=False):
    g = synth.rng(seed)
    marg, ptok = synth.marginal_pool(g, d, k, 50)
    if ties:
        marg[:] = np.float32(1.0 / k)
        ptok = np.stack([np.arange(k) + 10 * r for r in range(d)]).astype(np.int32)
    return marg, ptok


@pytest.mark.parametrize("d,k", [(1, 3), (2, 2), (3, 3), (3, 2), (2, 3)])
@pytest.mark.parametrize("ties", [False, True])
def test_matches_bruteforce_every_budget(d, k, ties):
    marg, ptok = _pool(10 * d + k, d, k, ties)
    total = sum(k ** j for j in range(1, d + 1))
    for budget in range(1, total + 3):
        got = selection.select_subtree(marg, ptok, budget, 5)
        n = got["n_nodes"]
        assert n == min(budget, total + 1)
        par, tok, dep, sc = _brute(marg, ptok, budget, 5)
        assert got["parent"][:n].tolist() == par
        assert got["token"][:n].tolist() == tok
        assert got["depth"][:n].tolist() == dep
        assert got["score"][:n].tolist() == [float(x) for x in sc]
        assert (got["parent"][n:] == -1).all()


def _prefix_closed_sets(paths, size):
    pathset = set(paths)
    for combo in itertools.combinations(paths, size):
        cs = set(combo)
        if all(len(p) == 1 or p[:-1] in cs for p in cs):
            yield cs
    del pathset


def test_selected_set_maximises_expected_accepted_length():
    d, k = 3, 2
    marg, ptok = _pool(77, d, k)
    paths = list(_all_paths(d, k))
    score = {p: float(selection.path_score(marg, p)) for p in paths}
    for budget in range(2, 9):
        got = selection.select_subtree(marg, ptok, budget, 0)
        mine = sum(float(x) for x in got["score"][1:got["n_nodes"]])
        best = max(sum(score[p] for p in cs) for cs in _prefix_closed_sets(paths, budget - 1))
        assert mine >= best - 1e-12


def test_prefix_closed_and_ordered():
    marg, ptok = _pool(3, 16, 32)
    got = selection.select_subtree(marg, ptok, 1024, 1)
    n = got["n_nodes"]
    assert n == 1024
    for i in range(1, n):
        p = got["parent"][i]
        assert 0 <= p < i
        assert got["depth"][i] == got["depth"][p] + 1
        assert got["score"][i] <= got["score"][i - 1]
        path = got["paths"][i]
        assert got["paths"][p] == path[:-1]
        assert got["token"][i] == ptok[len(path) - 1, path[-1]]


def test_single_rank_pool_is_a_chain():
    marg, ptok = _pool(4, 16, 1)
    for budget in (1, 5, 17, 40):
        got = selection.select_subtree(marg, ptok, budget, 0)
        n = got["n_nodes"]
        assert n == min(budget, 17)
        assert got["parent"][:n].tolist() == list(range(-1, n - 1))
        assert got["token"][1:n].tolist() == ptok[: n - 1, 0].tolist()


def test_budget_beyond_pool_takes_whole_tree():
    marg, ptok = _pool(6, 3, 3)
    got = selection.select_subtree(marg, ptok, 100, 0)
    assert got["n_nodes"] == 1 + 3 + 9 + 27
    assert sorted(got["paths"][1:]) == sorted(_all_paths(3, 3))


# ---- cost-aware row count (TAPS §3.1 limitation 2, §3.2)
from fractions import Fraction  # noqa: E402

import synth.workloads as W  # noqa: E402


def _exact_best(scores, a, b):
    """Independent restatement with exact rationals of the 2^-40-rounded scores."""
    unit = 2 ** selection.FIX_BITS
    best, best_n, acc = None, 1, Fraction(0)
    for n in range(1, len(scores) + 1):
        if n > 1:
            acc += Fraction(round(float(np.float32(scores[n - 1])) * unit), unit)
        val = (1 + acc) / (Fraction(float(np.float32(a))) + Fraction(float(np.float32(b))) * n)
        if best is None or val > best:
            best, best_n = val, n
    return best_n


@pytest.mark.parametrize("s,a,b,expect_all", [
    (0.5, 8.0, 1.0, True),    # s*a = 4 > b*(1-s) = 0.5: every row pays
    (0.5, 0.5, 1.0, False),   # 0.25 < 0.5: the root alone is best
    (0.25, 4.0, 2.0, False),  # 1.0 < 1.5
    (0.75, 4.0, 2.0, True),   # 3.0 > 0.5
])
def test_adaptive_equal_scores_closed_form(s, a, b, expect_all):
    # (1 + (n-1)s) / (a + bn) is monotone in n, increasing iff s*a > b*(1-s)
    scores = [1.0] + [s] * 30
    n = selection.adaptive_rows(scores, a, b)
    assert n == (31 if expect_all else 1)


def test_adaptive_flat_cost_takes_everything_and_zero_base_takes_the_root():
    scores = [1.0, 0.9, 0.5, 0.3, 0.2, 0.05]
    assert selection.adaptive_rows(scores, 1.0, 2.0 ** -30) == len(scores)
    assert selection.adaptive_rows(scores, 0.0, 1.0) == 1  # average score per row only falls


def test_adaptive_matches_exact_rationals():
    g = synth.rng(77)
    for _ in range(200):
        n = int(g.integers(1, 40))
        scores = [1.0] + sorted(g.random(n - 1).astype(np.float32).tolist(), reverse=True)
        a = float(np.float32(g.uniform(0.0, 20.0)))
        b = float(np.float32(g.uniform(0.01, 2.0)))
        assert selection.adaptive_rows(scores, a, b) == _exact_best(scores, a, b)


def test_adaptive_selection_is_a_prefix():
    g = synth.rng(78)
    marg, ptok = W.pools(g, 1, 8, 6, 5000)
    full = selection.select_subtree(marg[0], ptok[0], 40, 3)
    cut = selection.select_subtree_adaptive(marg[0], ptok[0], 40, 3, 6.0, 0.25)
    n = cut["n_nodes"]
    assert 1 <= n <= full["n_nodes"]
    for key in ("parent", "token", "depth", "score"):
        assert np.array_equal(cut[key][:n], full[key][:n])
        assert np.all(cut[key][n:] == (0 if key == "score" else -1))
