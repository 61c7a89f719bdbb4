"""GPU parity for ragged batches: sequences of one call with different node counts.

TAPS §4.1 stage 3 (the selected subtree is large when the drafter is confident and small
otherwise) and §3.1 limitation 2 (verification cost grows with the node count) make the
cost-aware cut n* differ per sequence.  Rows after a sequence's last node hold parent -1
(trailing padding, as tv_select_subtree_adaptive writes them) and are inactive: the
selection's outputs go straight into tree prep, tree attention and verification in one
call.  Padding rows get no output (attention rows left as they were, NaN probabilities
and lse, argmax -1) and are never walked; an active row after a padding row is a
malformed tree.  Active rows must match the oracle exactly as in the unpadded tests."""
import numpy as np
import pytest

import synth
import synth.workloads as W
from oracle import attention, greedy, sampling, selection, tree, vocab

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a GPU", allow_module_level=True)

import tree_speculative_decoding_masked_gb300 as tv  # noqa: E402
from gpu_util import dev, host, i32, to_dev  # noqa: E402

REL = 1e-4


def _ragged_selection(B, d, K, budget, cost, V, seed):
    """Pools whose confidence differs per sequence, cut by the cost-aware selection on
    the GPU; returns the GPU's padded parent / token arrays (checked against the oracle)
    and the per-sequence node counts."""
    g = synth.rng(seed)
    marg = np.empty((B, d, K), dtype=np.float32)
    ptok = np.empty((B, d, K), dtype=np.int32)
    for b in range(B):  # sharper marginals for later sequences: larger n*
        marg[b], ptok[b] = synth.marginal_pool(g, d, K, V, std=0.5 + 1.5 * b)
    roots = np.arange(B, dtype=np.int32) + 7
    out = tv.select_subtree(torch.from_numpy(marg).to(dev()), i32(ptok), budget, i32(roots), cost=cost)
    torch.cuda.synchronize()
    par, tok = out["parent"].cpu().numpy(), out["tokens"].cpu().numpy()
    n = out["n_nodes"].cpu().numpy()
    for b in range(B):
        ref = selection.select_subtree_adaptive(marg[b], ptok[b], budget, int(roots[b]), *cost)
        assert int(n[b]) == ref["n_nodes"]
        assert np.array_equal(par[b], ref["parent"]) and np.array_equal(tok[b], ref["token"])
    return par, tok, n


@pytest.fixture(scope="module")
def ragged():
    par, tok, n = _ragged_selection(6, 12, 6, 96, (100.0, 0.5), 5000, 7100)  # n* 40..72
    assert len(set(int(x) for x in n)) >= 3, n  # the cut differs between sequences
    assert int(n.min()) < 96 and (par[np.arange(6), np.minimum(n, 95)] == -1).any()
    return par, tok, n


def test_tree_prep_on_padded_rows(ragged):
    par, _, n = ragged
    B, N = par.shape
    P = 333
    got = {k: v.cpu().numpy() for k, v in tv.tree_prep(i32(par), P).items()}
    assert int(got["dev_status"][0]) == 0
    for b in range(B):
        assert np.array_equal(got["depth"][b], tree.depth(par[b]))
        assert np.array_equal(got["pos"][b], tree.position_ids(par[b], P))
        assert np.array_equal(got["anc_mask"][b].view(np.uint32), tree.packed_mask(par[b]))
        off, idx = tree.child_csr(par[b])
        assert np.array_equal(got["child_off"][b], off)
        k = int(n[b]) - 1
        assert np.array_equal(got["child_idx"][b][:k], idx) and (got["child_idx"][b][k:] == -1).all()


@pytest.mark.parametrize("bf16,Hq,Hkv,D,P", [(True, 8, 2, 128, 300), (True, 4, 4, 64, 0), (False, 4, 1, 64, 100)])
def test_attention_on_padded_rows(ragged, bf16, Hq, Hkv, D, P):
    # tensor-core kernels (bf16) and the CUDA-core kernel (fp32): active rows within the
    # stated tolerance, padding rows of `out` untouched
    par, _, n = ragged
    B, N = par.shape
    g = synth.rng(7200 + D + P)
    q, k, v = W.qkv_host(g, B, Hq, Hkv, D, P, N, bf16)
    out = torch.full((B, Hq, N, D), 7.0, dtype=torch.bfloat16 if bf16 else torch.float32, device=dev())
    st = torch.zeros(1, dtype=torch.int32, device=dev())
    tv.tree_attention(to_dev(q, bf16), to_dev(k, bf16), to_dev(v, bf16), i32(par), P, out=out, dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    got = host(out)
    ref = attention.tree_attention(q, k, v, par, P)
    tol = 2e-2 if bf16 else 1e-4
    for b in range(B):
        a = int(n[b])
        assert np.max(np.abs(got[b, :, :a] - ref[b, :, :a])) < tol
        assert (got[b, :, a:] == 7.0).all()


@pytest.mark.parametrize("bf16", [True, False])
def test_greedy_verify_on_padded_rows(ragged, bf16):
    par, tok, n = ragged
    B, N = par.shape
    V = 5000
    g = synth.rng(7300 + bf16)
    x = np.empty((B, N, V), dtype=np.float32)
    for b in range(B):  # planted on the active tree; padding rows hold plain draws
        a = int(n[b])
        x[b] = synth.normal(g, (N, V), np.sqrt(2.0), bf16)
        x[b, :a] = synth.plant_first_child_argmax(g, x[b, :a], par[b, :a], tok[b, :a], 0.8, bf16)
    out = tv.verify_greedy(to_dev(x, bf16), i32(par), i32(tok), want_stats=True)
    torch.cuda.synchronize()
    got = {k: v.cpu().numpy() for k, v in out.items()}
    assert int(got["dev_status"][0]) == 0
    for b in range(B):
        a = int(n[b])
        _, lse, am = vocab.vocab_stats(x[b, :a])
        assert np.array_equal(got["row_argmax"][b, :a], am) and (got["row_argmax"][b, a:] == -1).all()
        assert np.all(np.abs(got["row_lse"][b, :a] - lse) <= REL * np.maximum(1.0, np.abs(lse)))
        assert np.isnan(got["row_lse"][b, a:]).all()
        p = vocab.drafted_token_prob(x[b], np.concatenate([lse, np.zeros(N - a)]), par[b], tok[b])
        assert np.isnan(got["p_draft"][b, a:]).all() and np.isnan(p[a:]).all()
        rel = np.abs(got["p_draft"][b, 1:a] - p[1:a]) / p[1:a]
        assert float(rel.max(initial=0.0)) <= REL
        acc, bonus = greedy.greedy_walk(par[b], tok[b], np.concatenate([am, np.zeros(N - a, dtype=am.dtype)]))
        L = int(got["accept_len"][b])
        assert got["accepted_nodes"][b, :L].tolist() == acc and (got["accepted_nodes"][b, L:] == -1).all()
        assert int(got["bonus_token"][b]) == bonus
        assert all(c < a for c in acc)


def test_sampling_verify_on_padded_rows(ragged):
    par, _, n = ragged
    B, N = par.shape
    V, T = 3000, 1.0
    g = synth.rng(7400)
    tgt = (synth.normal(g, (B, N, V), 1.0) * 2).astype(np.float32)
    drf = (tgt + synth.normal(g, (B, N, V), 0.5)).astype(np.float32)
    tok = np.full((B, N), -1, dtype=np.int32)
    for b in range(B):
        a = int(n[b])
        tok[b, :a] = synth.draw_children_from_draft(g, par[b, :a], drf[b, :a], T)
    out = tv.verify_sample(to_dev(tgt, False), to_dev(drf, False), i32(par), i32(tok), temperature=T, seed=11,
                           round=2)
    torch.cuda.synchronize()
    got = {k: v.cpu().numpy() for k, v in out.items()}
    assert int(got["dev_status"][0]) == 0
    compared = 0
    for b in range(B):
        a = int(n[b])
        assert np.isnan(got["p_draft"][b, a:]).all() and np.isnan(got["q_draft"][b, a:]).all()
        acc, out_tok, margins, _ = sampling.sampling_walk(tgt[b], drf[b], par[b], tok[b], T, 11, 2, b)
        if any(m <= (1e-5 if kind == "accept" else 2e-7) for kind, m in margins):
            continue
        L = int(got["accept_len"][b])
        assert got["accepted_nodes"][b, :L].tolist() == acc and int(got["out_token"][b]) == out_tok
        compared += 1
    assert compared >= B - 1


def test_active_row_after_padding_is_flagged():
    # sequence 0: 20 active rows, padding, then an active row 30 (parent 3); sequence 1
    # is a valid padded tree.  40 rows keep G * N above 64: the bf16 case runs on the
    # tensor-core kernels, the fp32 one on the CUDA-core kernel.
    N, V, P = 40, 64, 40
    g = synth.rng(7500)
    par = np.full((2, N), -1, dtype=np.int32)
    par[0, :20] = synth.random_parents(g, 20, 6)
    par[0, 30] = 3
    par[1, :25] = synth.random_parents(g, 25, 6)
    tok = np.zeros((2, N), dtype=np.int32)
    tok[:, 1:] = np.arange(1, N)
    st = torch.zeros(1, dtype=torch.int32, device=dev())
    tv.tree_prep(i32(par), P, dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) & tv.TV_DEV_BAD_TREE
    for bf16, Hq, Hkv, D in ((True, 8, 2, 128), (False, 4, 1, 64)):
        q, k, v = W.qkv_host(g, 2, Hq, Hkv, D, P, N, bf16)
        st.zero_()
        tv.tree_attention(to_dev(q, bf16), to_dev(k, bf16), to_dev(v, bf16), i32(par), P, dev_status=st)
        torch.cuda.synchronize()
        assert int(st.item()) & tv.TV_DEV_BAD_TREE
    x = synth.normal(g, (2, N, V), 1.0)
    st.zero_()
    tv.verify_greedy(to_dev(x, False), i32(par), i32(tok), dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) & tv.TV_DEV_BAD_TREE
    st.zero_()
    tv.verify_sample(to_dev(x, False), to_dev(x, False), i32(par), i32(tok), temperature=1.0, seed=1, round=0,
                     dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) & tv.TV_DEV_BAD_TREE
