"""GPU parity: tv_verify_greedy (fused vocab pass + greedy walk) against the oracle.
Argmax, accepted paths and bonus tokens bit-exact; probabilities within 1e-4 (fp32
logits) / 2e-2 (bf16 logits) max-abs; lse within the same bounds."""
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


def _check(logits, parent, tokens, got, bf16):
    tol = 2e-2 if bf16 else 1e-4
    B, N, V = logits.shape
    for b in range(B):
        m, lse, am = vocab.vocab_stats(logits[b])
        assert np.array_equal(got["row_argmax"][b], am)
        assert np.max(np.abs(got["row_lse"][b] - lse)) < tol * max(1.0, np.max(np.abs(lse))) * (1 if bf16 else 1)
        p = vocab.drafted_token_prob(logits[b], lse, parent[b], tokens[b])
        assert np.isnan(got["p_draft"][b][0])
        assert np.max(np.abs(got["p_draft"][b][1:] - p[1:])) < tol
        if not bf16:
            assert np.allclose(got["p_draft"][b][1:], p[1:], rtol=1e-4, atol=1e-7)
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
