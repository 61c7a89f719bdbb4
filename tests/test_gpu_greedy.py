"""GPU parity: tv_verify_greedy (fused vocab pass + greedy walk) and tv_vocab_stats
against the oracle.  Argmax, accepted paths and bonus tokens bit-exact; probabilities
within the stated 1e-4 (fp32 logits) / 2e-2 (bf16 logits) max-abs, and also within 1e-4
RELATIVE for both dtypes: bf16 logits are exact inputs and the pass computes in fp32, so
only fp32 rounding and the hardware exp2/log2 separate it from the fp64 oracle (a
probability of 1e-6 checked only to 2e-2 absolute would pass as zero).  lse within 1e-4
relative likewise."""
import json
import math
import os

import numpy as np
import pytest

import synth
import synth.workloads as W
from oracle import greedy, selection, vocab

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a GPU", allow_module_level=True)

import tree_speculative_decoding_masked_gb300 as tv  # noqa: E402
from gpu_util import i32, to_dev  # noqa: E402


def _run(logits, parent, tokens, bf16, workspace=None):
    out = tv.verify_greedy(to_dev(logits, bf16), i32(parent), i32(tokens), want_stats=True, workspace=workspace)
    torch.cuda.synchronize()
    return {k: v.cpu().numpy() for k, v in out.items()}


REL = 1e-4  # relative bound on lse and drafted-token probabilities, fp32 and bf16 alike


def check_rel(got, ref, what):
    """|got - ref| <= REL * |ref| elementwise, all of got finite."""
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    err = np.abs(got - ref) / np.maximum(np.abs(ref), 1e-300)
    assert np.all(np.isfinite(got)), what
    assert float(err.max(initial=0.0)) <= REL, (what, float(err.max()))


def check_lse(got, ref):
    """|got - ref| <= REL * max(1, |ref|) elementwise."""
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert np.all(np.abs(got - ref) <= REL * np.maximum(1.0, np.abs(ref))), float(np.abs(got - ref).max())


def _check(logits, parent, tokens, got, bf16):
    tol = 2e-2 if bf16 else 1e-4
    B, N, V = logits.shape
    for b in range(B):
        m, lse, am = vocab.vocab_stats(logits[b])
        assert np.array_equal(got["row_argmax"][b], am)
        assert np.max(np.abs(got["row_lse"][b] - lse)) < tol * max(1.0, np.max(np.abs(lse)))
        check_lse(got["row_lse"][b], lse)
        p = vocab.drafted_token_prob(logits[b], lse, parent[b], tokens[b])
        assert np.isnan(got["p_draft"][b][0])
        assert np.max(np.abs(got["p_draft"][b][1:] - p[1:])) < tol
        check_rel(got["p_draft"][b][1:], p[1:], "p_draft")
        acc, bonus = greedy.greedy_walk(parent[b], tokens[b], am)
        L = int(got["accept_len"][b])
        assert L == len(acc)
        assert got["accepted_nodes"][b][:L].tolist() == acc
        assert (got["accepted_nodes"][b][L:] == -1).all()
        assert int(got["bonus_token"][b]) == bonus
    assert int(got["dev_status"][0]) == 0


def test_tiny_fp32_workload():
    cfg = W.WORKLOADS["tiny_fp32"]
    g = synth.rng(cfg["seed"])
    par, tok = W.trees(g, cfg["B"], cfg["N"], cfg["depth_cap"], cfg["V"])
    x = W.planted_logits(g, par, tok, cfg["V"], False)
    _check(x, par, tok, _run(x, par, tok, False), False)


def test_qwen3_4b_layer_workload():
    cfg = W.WORKLOADS["qwen3_4b_layer"]
    g = synth.rng(cfg["seed"])
    marg, ptok = W.pools(g, 1, cfg["pool_d"], cfg["pool_k"], cfg["V"])
    sel = selection.select_subtree(marg[0], ptok[0], cfg["N"], 11)
    par = sel["parent"][None]
    tok = sel["token"][None]
    x = W.planted_logits(g, par, tok, cfg["V"], True)
    got = _run(x, par, tok, True)
    _check(x, par, tok, got, True)
    assert int(got["accept_len"][0]) >= 1  # planted at p = 0.7: a long path is expected


@pytest.mark.parametrize("bf16", [False, True])
@pytest.mark.parametrize("V", [1, 7, 1001, 8192, 40000])
def test_ragged_vocab_and_batch(bf16, V):
    g = synth.rng(V + bf16)
    B, N = 3, 37
    par, tok = W.trees(g, B, N, 6, V if V > 40 else 10**6)
    tok = tok % V
    # siblings distinct modulo V only matters for the walk's uniqueness; duplicates are
    # resolved to the lowest index on both sides
    x = W.planted_logits(g, par, tok, V, bf16, prob=0.8)
    _check(x, par, tok, _run(x, par, tok, bf16), bf16)


def test_many_rows_and_ties():
    g = synth.rng(5)
    B, N, V = 16, 1024, 512
    par, tok = W.trees(g, B, N, 16, V)
    x = np.round(synth.normal(g, (B, N, V), 1.0)).astype(np.float32)  # many exact ties
    _check(x, par, tok, _run(x, par, tok, False), False)
    _check(x, par, tok, _run(x, par, tok, True), True)


def test_golden_cases_on_gpu():
    with open(os.path.join(os.path.dirname(__file__), "golden", "greedy_cases.json")) as f:
        cases = json.load(f)["cases"]
    V = 128
    for c in cases:
        n = len(c["parent"])
        x = np.zeros((1, n, V), dtype=np.float32)
        for u, a in enumerate(c["argmax"]):
            x[0, u, a] = 5.0
        par = np.array([c["parent"]], dtype=np.int32)
        tok = np.array([c["tokens"]], dtype=np.int32)
        got = _run(x, par, tok, False)
        L = int(got["accept_len"][0])
        assert got["accepted_nodes"][0][:L].tolist() == c["accepted"], c["name"]
        assert int(got["bonus_token"][0]) == c["bonus"], c["name"]


def test_full_acceptance_chain():
    g = synth.rng(9)
    N, V = 16, 151936
    par = synth.chain_parents(N)[None]
    tok = synth.distinct_child_tokens(g, par[0], V)[None]
    x = W.planted_logits(g, par, tok, V, True, prob=1.0)
    got = _run(x, par, tok, True)
    assert int(got["accept_len"][0]) == N - 1
    _check(x, par, tok, got, True)


def test_bad_inputs_are_flagged():
    V = 64
    ws = torch.zeros(tv.verify_workspace_size(2, 4, V, torch.float32, False), dtype=torch.uint8, device="cuda")
    x = np.zeros((2, 4, V), dtype=np.float32)
    par = np.array([[-1, 0, 5, 1], [-1, 0, 1, 2]], dtype=np.int32)
    tok = np.array([[0, 1, 2, 3], [0, 1, 2, V + 3]], dtype=np.int32)
    got = _run(x, par, tok, False, ws)
    assert int(got["dev_status"][0]) & tv.TV_DEV_BAD_TREE
    assert int(got["dev_status"][0]) & tv.TV_DEV_BAD_TOKEN
    assert (got["accept_len"] == 0).all() and (got["bonus_token"] == -1).all()
    # the workspace counters must be reset: a clean call afterwards is exact
    g = synth.rng(1)
    par2, tok2 = W.trees(g, 2, 4, 3, V)
    x2 = W.planted_logits(g, par2, tok2, V, False)
    _check(x2, par2, tok2, _run(x2, par2, tok2, False, ws), False)
    _check(x2, par2, tok2, _run(x2, par2, tok2, False, ws), False)


def test_long_context_workload_all_rows():
    # the full verification shape of the long-context workload: 8 x 128 rows of 151936
    # bf16 logits, every row checked against the oracle
    cfg = W.WORKLOADS["long_context"]
    g = synth.rng(cfg["seed"])
    par, tok = W.trees(g, cfg["B"], cfg["N"], cfg["depth_cap"], cfg["V"])
    x = W.planted_logits(g, par, tok, cfg["V"], True)
    got = _run(x, par, tok, True)
    _check(x, par, tok, got, True)
    assert int(got["accept_len"].max()) >= 1


class _LazyArgmax:
    """argmax of logits row (b, u), read back from the device one row at a time and
    computed by the oracle; remembers which rows it was asked for."""

    def __init__(self, logits, b):
        self.logits, self.b, self.rows = logits, b, {}

    def row(self, u):
        if u not in self.rows:
            self.rows[u] = self.logits[self.b, u].float().cpu().numpy()
        return self.rows[u]

    def __getitem__(self, u):
        return vocab.row_stats(self.row(int(u)))[2]


def test_budget_1024_trees_beyond_2_31_elements():
    # 16 sequences x 1024 nodes x 151936 = 2.49e9 logits (more than 2^31): the flat
    # 64-bit element index and the fp32-reciprocal divisions of the pass run for real.
    # Logits are drawn on the device (N(0,2), torch's seeded generator); the first child's
    # token of each internal node is planted as 16.0 (far above any N(0,2) draw) with
    # probability 0.7.  The oracle walks every sequence reading back only the rows it
    # visits; those rows, a random sample of others and their drafted-token
    # probabilities are compared.
    cfg = W.WORKLOADS["budget_sweep"]
    B, N, V = cfg["B"], 1024, cfg["V"]
    assert B * N * V > 2**31
    g = synth.rng(cfg["seed"] + 11)
    marg, ptok = W.pools(g, B, cfg["pool_d"], cfg["pool_k"], V)
    par = np.empty((B, N), dtype=np.int32)
    tok = np.empty((B, N), dtype=np.int32)
    for b in range(B):
        sel = selection.select_subtree(marg[b], ptok[b], N, 11)
        par[b], tok[b] = sel["parent"], sel["token"]
    assert (par[:, 1:] >= 0).all()  # every budget row is filled from the 16 x 32 pool
    dev = torch.device("cuda", 0)
    x = W.device_normal((B, N, V), math.sqrt(2.0), cfg["seed"] + 12, torch.bfloat16, dev)
    fc = [synth.first_children(par[b]) for b in range(B)]
    pb, pu, pt = [], [], []
    for b in range(B):
        for u in range(N):
            if fc[b][u] >= 0 and g.random() < 0.7:
                pb.append(b), pu.append(u), pt.append(int(tok[b][fc[b][u]]))
    x[torch.tensor(pb, device=dev), torch.tensor(pu, device=dev), torch.tensor(pt, device=dev)] = 16.0
    out = tv.verify_greedy(x, i32(par), i32(tok), want_stats=True)
    torch.cuda.synchronize()
    got = {k: v.cpu().numpy() for k, v in out.items()}
    assert int(got["dev_status"][0]) == 0
    lazy = [_LazyArgmax(x, b) for b in range(B)]
    for b in range(B):
        acc, bonus = greedy.greedy_walk(par[b], tok[b], lazy[b])
        L = int(got["accept_len"][b])
        assert got["accepted_nodes"][b][:L].tolist() == acc, b
        assert (got["accepted_nodes"][b][L:] == -1).all()
        assert int(got["bonus_token"][b]) == bonus, b
    for b in range(B):  # a random sample of other rows
        for u in g.choice(N, size=6, replace=False):
            lazy[b].row(int(u))
    checked = 0
    for b in range(B):
        kids = {}
        for c in range(1, N):
            kids.setdefault(int(par[b][c]), []).append(c)
        for u, row in lazy[b].rows.items():
            _, lse_u, am_u = vocab.row_stats(row)
            assert int(got["row_argmax"][b][u]) == am_u, (b, u)
            check_lse([got["row_lse"][b][u]], [lse_u])
            for c in kids.get(u, []):
                p = math.exp(float(row[int(tok[b][c])]) - lse_u)
                check_rel([got["p_draft"][b][c]], [p], "p_draft")
                checked += 1
    assert checked >= 100
    assert int(got["accept_len"].max()) >= 2


def test_vocab_stats_matches_oracle_and_verify():
    # the vocab pass alone: row statistics and drafted-token probabilities equal the
    # oracle's, and the same numbers tv_verify_greedy reports
    g = synth.rng(21)
    B, N, V = 3, 50, 40000
    par, tok = W.trees(g, B, N, 8, V)
    x = W.planted_logits(g, par, tok, V, True)
    xd = to_dev(x, True)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    s = tv.vocab_stats(xd, i32(par), i32(tok), dev_status=st)
    v = tv.verify_greedy(xd, i32(par), i32(tok), want_stats=True)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    for key in ("row_lse", "row_argmax"):
        assert torch.equal(s[key], v[key]), key
    assert torch.equal(s["p_draft"][:, 1:], v["p_draft"][:, 1:])
    for b in range(B):
        _, lse, am = vocab.vocab_stats(x[b])
        assert np.array_equal(s["row_argmax"][b].cpu().numpy(), am)
        check_lse(s["row_lse"][b].cpu().numpy(), lse)
        p = vocab.drafted_token_prob(x[b], lse, par[b], tok[b])
        check_rel(s["p_draft"][b].cpu().numpy()[1:], p[1:], "p_draft")


@pytest.mark.parametrize("bf16", [False, True])
def test_vocab_stats_with_draft_and_temperature(bf16):
    g = synth.rng(22 + bf16)
    B, N, V, T = 2, 33, 5000, 0.7
    par, _ = W.trees(g, B, N, 6, V)
    tgt, drf, tok = W.sampling_logits(g, par, V, bf16, T)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    s = tv.vocab_stats(to_dev(tgt, bf16), i32(par), i32(tok), draft_logits=to_dev(drf, bf16), temperature=T,
                       dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    for b in range(B):
        _, lse_p, am = vocab.vocab_stats(tgt[b], T)
        _, lse_q, _ = vocab.vocab_stats(drf[b], T)
        assert np.array_equal(s["row_argmax"][b].cpu().numpy(), am)
        check_lse(s["row_lse"][b].cpu().numpy(), lse_p)
        check_lse(s["draft_row_lse"][b].cpu().numpy(), lse_q)
        p = vocab.drafted_token_prob(tgt[b], lse_p, par[b], tok[b], T)
        q = vocab.drafted_token_prob(drf[b], lse_q, par[b], tok[b], T)
        check_rel(s["p_draft"][b].cpu().numpy()[1:], p[1:], "p_draft")
        check_rel(s["q_draft"][b].cpu().numpy()[1:], q[1:], "q_draft")
        assert np.isnan(s["p_draft"][b].cpu().numpy()[0])
