"""GPU parity: tv_verify_sample against the oracle.

Decisions are compared one by one.  Wherever every random decision on the oracle's path
clears its threshold by a safe margin, accepted path and output token must be identical;
sequences whose path passes closer are counted and must stay rare.  Margins:
  * acceptance tests r < min(1, p/q): |r - alpha| > 1e-5 (the GPU forms p and q in fp32
    from fp32 log-sum-exps, alpha to a few 1e-6 relative);
  * inverse-CDF draws: the target r * sum(p) lies more than 2e-7 * sum(p) from the
    chosen bucket's edges (the GPU rounds each fp32 probability once to a multiple of
    2^-56 and sums those exactly as 64-bit integers; a common scale error of all p
    cancels between the target and the prefix sums, the per-element rounding leaves
    ~1e-9 of the total).  Drafted-token probabilities match within 1e-4 (fp32) / 2e-2
    (bf16) max-abs and within 1e-4 relative for both dtypes (exact inputs, fp32
    arithmetic).  The distribution pin (the blog's promise that sampling verification
keeps the target distribution) is re-run on the GPU with a chi-square test."""
import math

import numpy as np
import pytest
from scipy import stats

import synth
import synth.workloads as W
from oracle import sampling, vocab

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a GPU", allow_module_level=True)

import tree_speculative_decoding_masked_gb300 as tv  # noqa: E402
from gpu_util import i32, to_dev  # noqa: E402

MARGIN = {"accept": 1e-5, "icdf": 2e-7}
REL = 1e-4  # relative bound on the drafted-token probabilities p and q


def _run(tgt, drf, par, tok, bf16, T, seed, rnd, workspace=None):
    out = tv.verify_sample(to_dev(tgt, bf16), to_dev(drf, bf16), i32(par), i32(tok), temperature=T, seed=seed,
                           round=rnd, workspace=workspace)
    torch.cuda.synchronize()
    return {k: v.cpu().numpy() for k, v in out.items()}


def _compare(tgt, drf, par, tok, got, bf16, T, seed, rnd):
    tol = 2e-2 if bf16 else 1e-4
    B = par.shape[0]
    close = 0
    for b in range(B):
        _, lse_p, _ = vocab.vocab_stats(tgt[b], T)
        _, lse_q, _ = vocab.vocab_stats(drf[b], T)
        p = vocab.drafted_token_prob(tgt[b], lse_p, par[b], tok[b], T)
        q = vocab.drafted_token_prob(drf[b], lse_q, par[b], tok[b], T)
        assert np.max(np.abs(got["p_draft"][b][1:] - p[1:])) < tol
        assert np.max(np.abs(got["q_draft"][b][1:] - q[1:])) < tol
        for what, g_, r_ in (("p_draft", got["p_draft"][b][1:], p[1:]), ("q_draft", got["q_draft"][b][1:], q[1:])):
            rel = np.abs(g_.astype(np.float64) - r_) / np.maximum(np.abs(r_), 1e-300)
            assert float(rel.max(initial=0.0)) <= REL, (what, b, float(rel.max()))
        acc, out_tok, margins, _ = sampling.sampling_walk(tgt[b], drf[b], par[b], tok[b], T, seed, rnd, b)
        L = int(got["accept_len"][b])
        if any(m <= MARGIN[kind] for kind, m in margins):
            close += 1
            continue
        assert got["accepted_nodes"][b][:L].tolist() == acc, b
        assert (got["accepted_nodes"][b][L:] == -1).all()
        assert int(got["out_token"][b]) == out_tok, b
    assert int(got["dev_status"][0]) == 0
    return close


@pytest.mark.parametrize("bf16", [False, True])
@pytest.mark.parametrize("V,T", [(64, 1.0), (4096, 1.0), (5000, 0.6)])
def test_small_vocab_many_sequences(bf16, V, T):
    g = synth.rng(V + int(bf16))
    B, N = 24, 48
    par, _ = W.trees(g, B, N, 8, V)
    tgt, drf, tok = W.sampling_logits(g, par, V, bf16, T, noise=1.0)
    close = 0
    for rnd in range(3):
        got = _run(tgt, drf, par, tok, bf16, T, 1234, rnd)
        close += _compare(tgt, drf, par, tok, got, bf16, T, 1234, rnd)
    assert close <= 3


def test_sampling_workload_full_vocab():
    cfg = W.WORKLOADS["sampling"]
    g = synth.rng(cfg["seed"])
    B = 2  # two of the workload's four sequences keep host memory modest
    par, _ = W.trees(g, B, cfg["N"], cfg["depth_cap"], cfg["V"])
    tgt, drf, tok = W.sampling_logits(g, par, cfg["V"], True, cfg["temperature"])
    got = _run(tgt, drf, par, tok, True, cfg["temperature"], cfg["seed"], 0)
    assert _compare(tgt, drf, par, tok, got, True, cfg["temperature"], cfg["seed"], 0) <= 1


@pytest.mark.parametrize("bf16", [False, True])
def test_vocab_too_large_for_the_cached_rows(bf16):
    # V = 400,000: a CTA's share of a row (25,000 elements as fp32 p and q, 200 KB at 16
    # CTAs per sequence) exceeds the walk's shared-memory budget, so every pass reads the
    # rows from global memory and replays the residual recursion (the path large
    # vocabularies take); decisions must match the oracle as on the cached path
    g = synth.rng(400 + int(bf16))
    B, N, V, T = 3, 24, 400_000, 1.0
    par, _ = W.trees(g, B, N, 6, V)
    tgt, drf, tok = W.sampling_logits(g, par, V, bf16, T, noise=1.0)
    close = 0
    for rnd in range(2):
        got = _run(tgt, drf, par, tok, bf16, T, 77, rnd)
        close += _compare(tgt, drf, par, tok, got, bf16, T, 77, rnd)
    assert close <= 1


def test_identical_distributions_accept_everything():
    g = synth.rng(3)
    N, V = 12, 2048
    par = synth.chain_parents(N)[None]
    x = synth.normal(g, (1, N, V), math.sqrt(2))
    tok = synth.distinct_child_tokens(g, par[0], V)[None]
    got = _run(x, x, par, tok, False, 1.0, 5, 0)
    assert int(got["accept_len"][0]) == N - 1


@pytest.mark.parametrize("m", [1, 3])
def test_gpu_first_token_follows_target(m):
    v, n = 8, 32000  # B * N stays within the verify limit of 131072 rows
    g = synth.rng(300 + m)
    row_t = synth.normal(g, v, math.sqrt(2))
    row_d = (row_t + synth.normal(g, v, 1.0)).astype(np.float32)
    par = np.tile(np.array([-1] + [0] * m, dtype=np.int32), (n, 1))
    rows_t = np.broadcast_to(row_t, (n, m + 1, v)).copy()
    rows_d = np.broadcast_to(row_d, (n, m + 1, v)).copy()
    tok = np.stack([synth.draw_children_from_draft(g, par[0], rows_d[0], 1.0) for _ in range(n)])
    got = _run(rows_t, rows_d, par, tok, False, 1.0, 99, 0)
    first = np.where(got["accept_len"] > 0, tok[np.arange(n), np.maximum(got["accepted_nodes"][:, 0], 0)],
                     got["out_token"])
    hist = np.bincount(first, minlength=v)
    p = sampling.softmax_row(row_t, 1.0)
    chi2 = float(np.sum((hist - n * p) ** 2 / (n * p)))
    assert chi2 < stats.chi2.ppf(1 - 1e-3, df=v - 1), (chi2, hist, n * p)


def test_bad_tree_flagged_and_workspace_reusable():
    V = 32
    ws = torch.zeros(tv.verify_workspace_size(1, 3, V, torch.float32, True), dtype=torch.uint8, device="cuda")
    x = np.zeros((1, 3, V), dtype=np.float32)
    got = _run(x, x, np.array([[-1, 2, 0]], dtype=np.int32), np.array([[0, 1, 2]], dtype=np.int32), False, 1.0, 1,
               0, ws)
    assert int(got["dev_status"][0]) & tv.TV_DEV_BAD_TREE
    g = synth.rng(8)
    par, _ = W.trees(g, 1, 3, 2, V)
    tgt, drf, tok = W.sampling_logits(g, par, V, False)
    for rnd in range(2):
        got = _run(tgt, drf, par, tok, False, 1.0, 1, rnd, ws)
        _compare(tgt, drf, par, tok, got, False, 1.0, 1, rnd)
