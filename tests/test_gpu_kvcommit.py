"""GPU parity: tv_commit_accepted_kv against oracle.kvcommit (bit-exact: a pure copy).
Accepted paths come from the oracle's greedy walk on planted logits, so they are real
root paths; cases cover bf16 and fp32 caches, several heads, D in {64, 128, 256}, empty
and full-depth paths, a ragged batch, and a malformed path that must only raise the
device status bit."""
import numpy as np
import pytest

import synth
import synth.workloads as W
from oracle import greedy, kvcommit, tree, vocab

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a GPU", allow_module_level=True)

import tree_speculative_decoding_masked_gb300 as tv  # noqa: E402
from gpu_util import host, i32, to_dev  # noqa: E402


def _paths(g, parent, tokens, V):
    """Accepted paths of the oracle's greedy walk on planted logits."""
    logits = W.planted_logits(g, parent, tokens, V, False)
    B, N = parent.shape
    acc = np.full((B, N), -1, dtype=np.int32)
    alen = np.zeros(B, dtype=np.int32)
    for b in range(B):
        _, _, am = vocab.vocab_stats(logits[b])
        path, _ = greedy.greedy_walk(parent[b], tokens[b], am)
        acc[b, :len(path)] = path
        alen[b] = len(path)
    return acc, alen


@pytest.mark.parametrize("B,Hkv,D,P,N,bf16,extra", [
    (1, 8, 128, 2048, 64, True, 0),
    (3, 2, 64, 17, 40, False, 5),
    (4, 1, 256, 0, 16, True, 3),
    (2, 4, 128, 300, 200, True, 0),
])
def test_commit_matches_oracle(B, Hkv, D, P, N, bf16, extra):
    g = synth.rng(4100 + N)
    parent, tokens = W.trees(g, B, N, 16, 1000)
    acc, alen = _paths(g, parent, tokens, 1000)
    S = P + N + extra
    k = synth.normal(g, (B, Hkv, S, D), bf16=bf16)
    v = synth.normal(g, (B, Hkv, S, D), bf16=bf16)
    kd, vd = to_dev(k, bf16), to_dev(v, bf16)
    st = torch.zeros(1, dtype=torch.int32, device=kd.device)
    tv.commit_accepted_kv(kd, vd, i32(acc), i32(alen), P, dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    k_ref, v_ref = kvcommit.commit_accepted(k, v, parent, acc, alen, P)
    assert np.array_equal(host(kd), k_ref)
    assert np.array_equal(host(vd), v_ref)


def test_empty_and_deepest_paths():
    g = synth.rng(4200)
    N, P, D = 20, 9, 64
    chain = np.array([[-1] + list(range(N - 1)), [-1] + [0] * (N - 1)], dtype=np.int32)
    acc = np.full((2, N), -1, dtype=np.int32)
    acc[0, :N - 1] = np.arange(1, N)  # the whole chain is accepted
    alen = np.array([N - 1, 0], dtype=np.int32)
    k = synth.normal(g, (2, 2, P + N, D))
    v = synth.normal(g, (2, 2, P + N, D))
    kd, vd = to_dev(k, False), to_dev(v, False)
    tv.commit_accepted_kv(kd, vd, i32(acc), i32(alen), P)
    torch.cuda.synchronize()
    k_ref, v_ref = kvcommit.commit_accepted(k, v, chain, acc, alen, P)
    assert np.array_equal(host(kd), k_ref) and np.array_equal(host(vd), v_ref)


def test_malformed_path_sets_status():
    g = synth.rng(4300)
    N, P, D = 8, 4, 64
    acc = np.array([[3, 2, -1, -1, -1, -1, -1, -1]], dtype=np.int32)  # not increasing
    k = synth.normal(g, (1, 1, P + N, D))
    kd, vd = to_dev(k, False), to_dev(k.copy(), False)
    st = torch.zeros(1, dtype=torch.int32, device=kd.device)
    tv.commit_accepted_kv(kd, vd, i32(acc), i32(np.array([2])), P, dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) & tv.TV_DEV_BAD_TREE


def test_host_validation():
    kd = torch.zeros(1, 1, 10, 62, dtype=torch.float32, device="cuda")  # 248-byte rows: not 16-byte multiples
    acc = torch.zeros(1, 4, dtype=torch.int32, device="cuda")
    with pytest.raises(tv.TreeVerifyError):
        tv.commit_accepted_kv(kd, kd.clone(), acc, torch.zeros(1, dtype=torch.int32, device="cuda"), 2)
