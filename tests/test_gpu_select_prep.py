"""GPU parity: tv_select_subtree and tv_tree_prep against the oracle (bit-exact)."""
import numpy as np
import pytest

import synth
import synth.workloads as W
from oracle import selection, tree

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a GPU", allow_module_level=True)

import tree_speculative_decoding_masked_gb300 as tv  # noqa: E402
from gpu_util import dev, i32  # noqa: E402


def _gpu_select(marg, ptok, budget, roots):
    out = tv.select_subtree(torch.from_numpy(marg).to(dev()), i32(ptok), budget, i32(roots))
    torch.cuda.synchronize()
    return {k: v.cpu().numpy() for k, v in out.items()}


def _check_select(marg, ptok, budget, roots, got):
    for b in range(marg.shape[0]):
        ref = selection.select_subtree(marg[b], ptok[b], budget, int(roots[b]))
        assert int(got["n_nodes"][b]) == ref["n_nodes"]
        assert np.array_equal(got["parent"][b], ref["parent"])
        assert np.array_equal(got["tokens"][b], ref["token"])
        assert np.array_equal(got["depth"][b], ref["depth"])
        assert np.array_equal(got["score"][b].view(np.uint32), ref["score"].view(np.uint32))
    assert int(got["dev_status"][0]) == 0


@pytest.mark.parametrize("d,k", [(1, 3), (2, 2), (3, 3), (2, 5)])
def test_tiny_pools_every_budget(d, k):
    g = synth.rng(40 + d * 10 + k)
    marg, ptok = W.pools(g, 3, d, k, 100)
    marg[1] = np.float32(1.0 / k)  # a pool full of ties
    roots = np.array([7, 8, 9], dtype=np.int32)
    total = sum(k ** j for j in range(1, d + 1))
    for budget in range(1, total + 3):
        _check_select(marg, ptok, budget, roots, _gpu_select(marg, ptok, budget, roots))


def test_qwen3_4b_pool():
    cfg = W.WORKLOADS["qwen3_4b_layer"]
    g = synth.rng(cfg["seed"])
    marg, ptok = W.pools(g, 1, cfg["pool_d"], cfg["pool_k"], cfg["V"])
    roots = np.array([5], dtype=np.int32)
    _check_select(marg, ptok, cfg["N"], roots, _gpu_select(marg, ptok, cfg["N"], roots))


@pytest.mark.parametrize("budget", [16, 64, 256, 1024])
def test_budget_sweep_pools(budget):
    cfg = W.WORKLOADS["budget_sweep"]
    g = synth.rng(cfg["seed"])
    marg, ptok = W.pools(g, cfg["B"], cfg["pool_d"], cfg["pool_k"], cfg["V"])
    roots = np.arange(cfg["B"], dtype=np.int32)
    _check_select(marg, ptok, budget, roots, _gpu_select(marg, ptok, budget, roots))


def test_max_sizes_and_single_rank():
    g = synth.rng(77)
    marg, ptok = W.pools(g, 2, 16, 256, 1000)
    roots = np.zeros(2, dtype=np.int32)
    _check_select(marg, ptok, 4096, roots, _gpu_select(marg, ptok, 4096, roots))
    marg1, ptok1 = W.pools(g, 2, 16, 1, 1000)
    _check_select(marg1, ptok1, 40, roots, _gpu_select(marg1, ptok1, 40, roots))


@pytest.mark.parametrize("budget", [40, 300, 2000])
def test_uniform_pools_all_ties(budget):
    # every path of a given depth ties: the order falls to depth, then the rank path;
    # budget 2000 overflows the threshold expansion and exercises the exact fallback
    d, k = 16, 8
    marg = np.full((2, d, k), 0.125, dtype=np.float32)
    ptok = np.tile(np.arange(d * k, dtype=np.int32).reshape(1, d, k), (2, 1, 1))
    roots = np.array([1, 2], dtype=np.int32)
    _check_select(marg, ptok, budget, roots, _gpu_select(marg, ptok, budget, roots))


@pytest.mark.parametrize("k,budget", [(8, 500), (9, 500), (8, 1500), (12, 3000)])
def test_dyadic_pools_many_exact_ties(k, budget):
    # marginals from {1/2, 1/4, 1/8, 1/16}: products are exact powers of two, so whole
    # score classes tie across depths and rank paths; k = 8 and 9 sit on either side of
    # the chain count at which the bound's histogram switches layout
    g = synth.rng(500 + k + budget)
    d = 16
    marg = np.sort(2.0 ** -g.integers(1, 5, size=(2, d, k)), axis=2)[:, :, ::-1].astype(np.float32)
    ptok = g.integers(0, 5000, size=(2, d, k)).astype(np.int32)
    roots = np.array([3, 4], dtype=np.int32)
    _check_select(marg, ptok, budget, roots, _gpu_select(marg, ptok, budget, roots))


@pytest.mark.parametrize("budget", [200, 1200])
def test_tiny_marginals_past_the_counting_range(budget):
    # every edge scores about 2^-11, so paths of depth >= 3 fall below 2^-32, past the
    # range of the quantised-log counting bound; the larger budget needs those paths and
    # takes the one-deviation bound instead
    g = synth.rng(900 + budget)
    d, k = 16, 8
    marg = np.sort(g.uniform(2.0 ** -12, 2.0 ** -10, size=(2, d, k)), axis=2)[:, :, ::-1].astype(np.float32)
    ptok = g.integers(0, 5000, size=(2, d, k)).astype(np.int32)
    roots = np.array([5, 6], dtype=np.int32)
    _check_select(marg, ptok, budget, roots, _gpu_select(marg, ptok, budget, roots))


def test_unsorted_pool_is_flagged():
    marg = np.array([[[0.2, 0.7], [0.6, 0.4]]], dtype=np.float32)
    ptok = np.array([[[1, 2], [3, 4]]], dtype=np.int32)
    got = _gpu_select(marg, ptok, 4, np.zeros(1, dtype=np.int32))
    assert int(got["dev_status"][0]) & tv.TV_DEV_BAD_TOKEN


@pytest.mark.parametrize("n,cap,b", [(1, 1, 1), (16, 4, 2), (257, 16, 3), (1024, 16, 2), (1024, 1024, 1)])
def test_tree_prep_matches_oracle(n, cap, b):
    g = synth.rng(n + cap)
    if cap >= n:
        par = np.stack([synth.chain_parents(n)] * b)
    else:
        par, _ = W.trees(g, b, n, cap, 100)
    out = tv.tree_prep(i32(par), 37)
    torch.cuda.synchronize()
    assert int(out["dev_status"][0]) == 0
    for bb in range(b):
        assert np.array_equal(out["depth"][bb].cpu().numpy(), tree.depth(par[bb]))
        assert np.array_equal(out["pos"][bb].cpu().numpy(), tree.position_ids(par[bb], 37))
        assert np.array_equal(out["anc_mask"][bb].cpu().numpy().view(np.uint32), tree.packed_mask(par[bb]))
        off, idx = tree.child_csr(par[bb])
        assert np.array_equal(out["child_off"][bb].cpu().numpy(), off)
        assert np.array_equal(out["child_idx"][bb].cpu().numpy()[: n - 1], idx)


def test_tree_prep_flags_bad_parent():
    par = np.array([[-1, 0, 2, 1], [-1, 0, 1, 2]], dtype=np.int32)  # node 2 points to itself
    out = tv.tree_prep(i32(par), 0)
    torch.cuda.synchronize()
    assert int(out["dev_status"][0]) & tv.TV_DEV_BAD_TREE


# ---- cost-aware tree size (tv_select_subtree_adaptive), bit-exact against the oracle
@pytest.mark.parametrize("B,d,k,budget,cost", [
    (1, 16, 4, 64, (20.0, 0.25)),     # a qwen3-like pool: the cut falls inside the budget
    (3, 8, 6, 40, (6.0, 0.25)),
    (16, 16, 32, 1024, (60.0, 0.05)),  # thousands of rows: several rows per thread in the scan
    (2, 4, 3, 30, (1.0, 2.0 ** -20)),  # nearly flat cost: every available row
    (2, 6, 5, 50, (0.0, 1.0)),         # no base cost: the root alone
])
def test_adaptive_budget_matches_oracle(B, d, k, budget, cost):
    g = synth.rng(5000 + budget + k)
    marg, ptok = W.pools(g, B, d, k, 3000)
    roots = np.arange(B, dtype=np.int32) + 5
    out = tv.select_subtree(torch.from_numpy(marg).to(dev()), i32(ptok), budget, i32(roots), cost=cost)
    torch.cuda.synchronize()
    got = {kk: v.cpu().numpy() for kk, v in out.items()}
    for b in range(B):
        ref = selection.select_subtree_adaptive(marg[b], ptok[b], budget, int(roots[b]), *cost)
        assert int(got["n_nodes"][b]) == ref["n_nodes"]
        assert np.array_equal(got["parent"][b], ref["parent"])
        assert np.array_equal(got["tokens"][b], ref["token"])
        assert np.array_equal(got["depth"][b], ref["depth"])
        assert np.array_equal(got["score"][b].view(np.uint32), ref["score"].view(np.uint32))
    assert int(got["dev_status"][0]) == 0


def test_adaptive_budget_rejects_bad_costs():
    g = synth.rng(5100)
    marg, ptok = W.pools(g, 1, 4, 3, 100)
    m, p, r = torch.from_numpy(marg).to(dev()), i32(ptok), i32(np.array([1]))
    for cost in ((1.0, 0.0), (-1.0, 1.0), (float("inf"), 1.0)):
        with pytest.raises(tv.TreeVerifyError):
            tv.select_subtree(m, p, 10, r, cost=cost)


@pytest.mark.parametrize("k,budget", [(2, 100), (3, 120), (4, 127), (32, 60)])
def test_uniform_pools_small_budgets(k, budget):
    # with all paths of a depth tied, the one-deviation bound of a small budget lies far
    # below the M-th best score: for K = 2, 3 the kept set outgrows the expansion buffer
    # and the bound-raising restarts take over; for K = 4, 32 the ranking cuts a large
    # tied set down to the coarse class that holds the M-th score
    d = 16
    marg = np.full((2, d, k), np.float32(1.0 / k), dtype=np.float32)
    ptok = np.tile(np.arange(d * k, dtype=np.int32).reshape(1, d, k), (2, 1, 1))
    roots = np.array([3, 4], dtype=np.int32)
    _check_select(marg, ptok, budget, roots, _gpu_select(marg, ptok, budget, roots))
