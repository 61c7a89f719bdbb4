"""GPU failure detection without a GPU fault: a bounded in-kernel wait that nothing
completes gives up, reports TV_DEV_TIMEOUT through the device status word, and the CUDA
context stays usable for the next call."""
import numpy as np
import pytest

import synth
import synth.workloads as W
from oracle import attention

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a GPU", allow_module_level=True)

import tree_speculative_decoding_masked_gb300 as tv  # noqa: E402
from gpu_util import dev, host, i32, to_dev  # noqa: E402


def test_bounded_wait_gives_up_and_reports():
    st = torch.zeros(1, dtype=torch.int32, device=dev())
    tv.selftest_bounded_wait(2000, st)  # 2 ms on a phase that never completes
    torch.cuda.synchronize()
    assert int(st.item()) & tv.TV_DEV_TIMEOUT


def test_context_usable_after_a_timeout():
    st = torch.zeros(1, dtype=torch.int32, device=dev())
    tv.selftest_bounded_wait(1000, st)
    torch.cuda.synchronize()
    assert int(st.item()) & tv.TV_DEV_TIMEOUT
    # a tensor-core attention call right after it runs normally with a clean status
    B, Hq, Hkv, D, P, N = 1, 8, 2, 128, 300, 40
    g = synth.rng(41)
    par, _ = W.trees(g, B, N, 5, 100)
    q, k, v = W.qkv_host(g, B, Hq, Hkv, D, P, N, True)
    st2 = torch.zeros(1, dtype=torch.int32, device=dev())
    out = tv.tree_attention(to_dev(q, True), to_dev(k, True), to_dev(v, True), i32(par), P, dev_status=st2)
    torch.cuda.synchronize()
    assert int(st2.item()) == 0
    assert np.max(np.abs(host(out) - attention.tree_attention(q, k, v, par, P))) < 2e-2


def test_selftest_argument_checks():
    st = torch.zeros(1, dtype=torch.int32, device=dev())
    with pytest.raises(Exception):
        tv.selftest_bounded_wait(0, st)
