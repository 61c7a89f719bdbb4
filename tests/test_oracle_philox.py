"""Pins for oracle.philox: the known-answer vectors published with Philox4x32-10
(Random123 distribution, kat_vectors) and basic properties of the uniform map."""
import numpy as np

from oracle import philox

KAT = [
    ((0x00000000, 0x00000000, 0x00000000, 0x00000000), (0x00000000, 0x00000000),
     (0x6627E8D5, 0xE169C58D, 0xBC57AC4C, 0x9B00DBD8)),
    ((0xFFFFFFFF, 0xFFFFFFFF, 0xFFFFFFFF, 0xFFFFFFFF), (0xFFFFFFFF, 0xFFFFFFFF),
     (0x408F276D, 0x41C83B0E, 0xA20BC7C6, 0x6D5451FD)),
    ((0x243F6A88, 0x85A308D3, 0x13198A2E, 0x03707344), (0xA4093822, 0x299F31D0),
     (0xD16CFE09, 0x94FDCCEB, 0x5001E420, 0x24126EA1)),
]


def test_known_answers():
    for ctr, key, out in KAT:
        got = philox.philox4x32_10(np.array(ctr, dtype=np.uint32), key)
        assert [int(x) for x in got] == list(out)


def test_vectorised_matches_scalar():
    ctrs = np.array([[i, 2 * i + 1, 7, i ^ 0x55] for i in range(50)], dtype=np.uint32)
    key = (0x12345678, 0x9ABCDEF0)
    allv = philox.philox4x32_10(ctrs, key)
    for i in range(50):
        assert np.array_equal(allv[i], philox.philox4x32_10(ctrs[i], key))


def test_uniform_range_and_resolution():
    us = [philox.uniform(2024, r, 0, 0, 1, 0) for r in range(2000)]
    assert min(us) >= 0.0 and max(us) < 1.0
    assert all(u * 16777216.0 == int(u * 16777216.0) for u in us)
    assert abs(np.mean(us) - 0.5) < 0.03
