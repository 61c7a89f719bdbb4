"""GPU parity: tv_frontier_topw and tv_expand_children against oracle.frontier.
Frontier positions and child tokens bit-exact (integer decisions taken on the raw
scores / logits on both sides); p and s within 2e-5 relative (the GPU's softmax
normaliser is an fp32 sum of ex2.approx terms, the oracle's an fp64 sum)."""
import numpy as np
import pytest

import synth
from oracle import frontier

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a GPU", allow_module_level=True)

import tree_speculative_decoding_masked_gb300 as tv  # noqa: E402
from gpu_util import dev, host, i32, to_dev  # noqa: E402


@pytest.mark.parametrize("B,C,W", [(1, 64, 8), (4, 300, 16), (3, 4096, 64), (2, 7, 7)])
def test_frontier_topw(B, C, W):
    g = synth.rng(6000 + C)
    sc = np.round(g.random((B, C)), 2).astype(np.float32)  # coarse: many ties
    cnt = g.integers(1, C + 1, size=B).astype(np.int32)
    cnt[0] = C
    got = host(tv.frontier_topw(torch.from_numpy(sc).to(dev()), i32(cnt), W))
    for b in range(B):
        ref = frontier.frontier_topw(sc[b], int(cnt[b]), W)
        assert got[b, :len(ref)].tolist() == ref
        assert np.all(got[b, len(ref):] == -1)


def _check_children(x, ps, m, temperature, bf16):
    got = tv.expand_children(to_dev(x, bf16), torch.from_numpy(ps).to(dev()), m, temperature=temperature)
    torch.cuda.synchronize()
    tok, p, s = (host(got[k]) for k in ("token", "p", "score"))
    assert int(got["dev_status"].item()) == 0
    for r in range(x.shape[0]):
        rt, rp, rs = frontier.attach_children(x[r], ps[r], m, temperature)
        k = len(rt)
        assert tok[r, :k].tolist() == rt.tolist()
        np.testing.assert_allclose(p[r, :k], rp, rtol=2e-5, atol=1e-12)
        np.testing.assert_allclose(s[r, :k], rs, rtol=2e-5, atol=1e-12)
        assert np.all(tok[r, k:] == -1) and np.all(p[r, k:] == 0)


@pytest.mark.parametrize("R,V,m,T,bf16", [
    (8, 151936, 8, 1.0, True),   # one TreeGraft step: 8 frontier rows over a Qwen-size vocabulary
    (3, 151936, 32, 0.7, True),
    (5, 1001, 13, 1.3, False),   # rows not 16-byte aligned: scalar loads
    (2, 5000, 1, 1.0, False),
    (4, 5, 8, 1.0, False),       # m > V
])
def test_expand_children(R, V, m, T, bf16):
    g = synth.rng(6100 + V + m)
    x = synth.normal(g, (R, V), std=2.0, bf16=bf16)
    # planted exact ties among the largest values, to exercise the token-order rule
    for r in range(R):
        top = int(np.argmax(x[r]))
        j = (top + 7) % V
        x[r, j] = x[r, top]
    ps = np.round(g.random(R), 3).astype(np.float32)
    _check_children(x, ps, m, T, bf16)


def test_expand_host_validation():
    x = torch.zeros(2, 100, dtype=torch.float32, device="cuda")
    ps = torch.ones(2, dtype=torch.float32, device="cuda")
    with pytest.raises(tv.TreeVerifyError):
        tv.expand_children(x, ps, 33)
    with pytest.raises(tv.TreeVerifyError):
        tv.expand_children(x, ps, 4, temperature=0.0)
