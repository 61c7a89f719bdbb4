"""GPU parity: tv_prune_tree against oracle.prune (bit-exact: integer decisions on the
same fp32 confidences)."""
import numpy as np
import pytest

import synth
import synth.workloads as W
from oracle import prune

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a GPU", allow_module_level=True)

import tree_speculative_decoding_masked_gb300 as tv  # noqa: E402
from gpu_util import dev, host, i32  # noqa: E402


@pytest.mark.parametrize("B,N,depth_cap,cap,lim", [
    (4, 64, 16, 2, 4),
    (3, 256, 16, 3, 8),
    (2, 1024, 16, 1, 12),
    (2, 1024, 1024, 4, 100),  # deep random trees: long ancestor walks
    (5, 17, 4, 8, 10),        # nothing to prune
    (2, 1, 1, 1, 1),          # the root alone
])
def test_prune_matches_oracle(B, N, depth_cap, cap, lim):
    g = synth.rng(7000 + N + cap)
    parent, _ = W.trees(g, B, N, depth_cap, 1000)
    conf = np.round(g.random((B, N)), 2).astype(np.float32)  # coarse: ties among siblings
    out = tv.prune_tree(i32(parent), torch.from_numpy(conf).to(dev()), cap, lim)
    torch.cuda.synchronize()
    got = {k: host(v) for k, v in out.items()}
    assert int(got["dev_status"][0]) == 0
    for b in range(B):
        ref = prune.prune_tree(parent[b], conf[b], cap, lim)
        assert int(got["n_kept"][b]) == ref["n_kept"]
        assert int(got["new_root"][b]) == ref["root"]
        assert got["old_to_new"][b].tolist() == ref["old_to_new"].tolist()
        n = ref["n_kept"]
        assert got["new_parent"][b, :n].tolist() == ref["new_parent"].tolist()
        assert np.all(got["new_parent"][b, n:] == -1)


def test_malformed_tree_sets_status():
    parent = np.array([[-1, 0, 3, 1]], dtype=np.int32)  # node 2's parent comes after it
    out = tv.prune_tree(i32(parent), torch.ones(1, 4, device=dev()), 2, 2)
    torch.cuda.synchronize()
    assert int(out["dev_status"].item()) & tv.TV_DEV_BAD_TREE
    assert int(out["n_kept"].item()) == 0
