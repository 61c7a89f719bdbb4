"""tv_verify_greedy_static: the greedy verification entry point for callers that cannot
allocate device memory when they call the library (its scratch is a fixed array inside
the library).  It must give the same results as tv_verify_greedy, on consecutive calls
that reuse the shared array, whether it runs first in a fresh process or after other
tests.  This file is collected last on purpose."""
import math

import numpy as np
import pytest

import synth
import synth.workloads as W

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a GPU", allow_module_level=True)

import tree_speculative_decoding_masked_gb300 as tv  # noqa: E402
from gpu_util import i32, to_dev  # noqa: E402


def _case(seed, B, N, V, bf16):
    g = synth.rng(seed)
    par, tok = W.trees(g, B, N, 8, V)
    x = W.planted_logits(g, par, tok, V, bf16)
    return to_dev(x, bf16), i32(par), i32(tok)


@pytest.mark.parametrize("bf16", [True, False])
def test_static_matches_workspace_entry_point_twice(bf16):
    cases = [_case(11, 2, 64, 151936 if bf16 else 4096, bf16), _case(12, 3, 37, 50000, bf16)]
    for logits, par, tok in cases:  # two calls in a row on different problems
        st = torch.zeros(1, dtype=torch.int32, device="cuda")
        a = tv.verify_greedy_static(logits, par, tok, want_stats=True, dev_status=st)
        b = tv.verify_greedy(logits, par, tok, want_stats=True)
        torch.cuda.synchronize()
        assert int(st.item()) == 0
        for key in ("accepted_nodes", "accept_len", "bonus_token", "row_argmax"):
            assert torch.equal(a[key], b[key]), key
        tol = 2e-2 if bf16 else 1e-4
        pa, pb = a["p_draft"][:, 1:], b["p_draft"][:, 1:]
        assert float((pa - pb).abs().max()) <= tol
        assert float((a["row_lse"] - b["row_lse"]).abs().max()) <= tol


STATIC_BYTES = 4 << 20  # the fixed array's size, as the header states


def test_static_rejects_problems_beyond_its_array():
    B, N, V = 128, 1024, 1  # 131072 rows: ~9.4 MB of scratch, more than the fixed array holds
    assert tv.verify_workspace_size(B, N, V, torch.bfloat16, False) > STATIC_BYTES
    logits = torch.zeros(B, N, V, dtype=torch.bfloat16, device="cuda")
    par = torch.from_numpy(np.tile(synth.chain_parents(N), (B, 1))).cuda()
    tok = torch.zeros(B, N, dtype=torch.int32, device="cuda")
    with pytest.raises(tv.TreeVerifyError) as ei:
        tv.verify_greedy_static(logits, par, tok)
    assert ei.value.status == -4


def test_static_capacity_boundary():
    # the largest batch of 64-node trees whose scratch fits the array runs and matches
    # tv_verify_greedy bit for bit; one more sequence is refused
    N, V = 64, 64
    fits = [B for B in range(1, 2048) if tv.verify_workspace_size(B, N, V, torch.float32, False) <= STATIC_BYTES]
    B = max(fits)
    assert tv.verify_workspace_size(B + 1, N, V, torch.float32, False) > STATIC_BYTES
    assert 50000 <= B * N <= 60000  # about 72 bytes per row
    logits, par, tok = _case(13, B, N, V, False)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    a = tv.verify_greedy_static(logits, par, tok, want_stats=True, dev_status=st)
    b = tv.verify_greedy(logits, par, tok, want_stats=True)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    for key in ("accepted_nodes", "accept_len", "bonus_token", "row_argmax"):
        assert torch.equal(a[key], b[key]), key
    assert float((a["row_lse"] - b["row_lse"]).abs().max()) <= 1e-4
    logits, par, tok = _case(14, B + 1, N, V, False)
    with pytest.raises(tv.TreeVerifyError) as ei:
        tv.verify_greedy_static(logits, par, tok)
    assert ei.value.status == -4
