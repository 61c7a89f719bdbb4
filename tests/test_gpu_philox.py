"""GPU parity of the sampling walk's generator: the device Philox4x32-10 words equal the
oracle's (which the published known-answer vectors pin) bit for bit over 10^6 random
counters and several keys, and the walk's uniforms follow from the documented counter
layout."""
import numpy as np
import pytest

from oracle import philox

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a GPU", allow_module_level=True)

import tree_speculative_decoding_masked_gb300 as tv  # noqa: E402
from gpu_util import dev  # noqa: E402


@pytest.mark.parametrize("seed", [0, 1005, 0xDEADBEEFCAFEF00D])
def test_device_words_match_oracle(seed):
    g = np.random.default_rng(77 + (seed & 0xFFFF))
    ctr = g.integers(0, 2**32, size=(1_000_000, 4), dtype=np.uint64).astype(np.uint32)
    ref = philox.philox4x32_10(ctr, philox.seed_key(seed))
    got = tv.philox4x32_10(seed, torch.from_numpy(ctr.view(np.int32)).to(dev()))
    assert np.array_equal(got.cpu().numpy().view(np.uint32), ref)


def test_walk_counter_layout_and_uniform():
    seed = 1003
    draws = [(r, b, u, k, kind) for r in (0, 1, 7) for b in (0, 3) for u in (0, 5, 255) for k in (0, 1, 4)
             for kind in (0, 1)]
    ctr = np.array([philox.counter(*d[:3], d[3], d[4]) for d in draws], dtype=np.uint32)
    words = tv.philox4x32_10(seed, torch.from_numpy(ctr.view(np.int32)).to(dev())).cpu().numpy().view(np.uint32)
    for (r, b, u, k, kind), w in zip(draws, words):
        assert (int(w[0]) >> 8) * (1.0 / 16777216.0) == philox.uniform(seed, r, b, u, k, kind)


def test_empty_and_argument_checks():
    ctr = torch.zeros((0, 4), dtype=torch.int32, device=dev())
    assert tv.philox4x32_10(1, ctr).shape == (0, 4)
