"""The identity behind the sampling walk's exact sums, checked on every float in [0, 1].

The walk adds probabilities as integers in units of 2^-56 so that a cluster's total does
not depend on the order of the additions; each term x in [0, 1] becomes round(x * 2^56)
(nearest, ties to even).  The kernel forms it from two 32-bit conversions: t = x * 2^24
and its integer part h = floor(t) are exact in fp32, so x * 2^56 = h * 2^32 + (t - h) *
2^32 where only the second term needs rounding.  A C program (gcc) runs the same steps
in fp32 on all 1,065,353,217 floats in [0, 1] and compares with the rounding of the
exact product in double precision.  (Host logic: no GPU needed.)"""
import os
import shutil
import subprocess
import tempfile

import pytest

SRC = r"""
#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <string.h>
static float bitsf(uint32_t u) { float x; memcpy(&x, &u, 4); return x; }
int main(void) {
  unsigned long long bad = 0, n = 0;
  uint32_t one;
  float f1 = 1.0f;
  memcpy(&one, &f1, 4);
  for (uint32_t u = 0; u <= one; ++u) {
    const float x = bitsf(u);
    volatile float t = x * 16777216.0f;
    volatile float h = floorf(t);
    volatile float r = t - h;
    volatile float s = r * 4294967296.0f;
    const unsigned long long got = ((unsigned long long)(uint32_t)h << 32) + (uint32_t)nearbyintf(s);
    const unsigned long long want = (unsigned long long)nearbyint((double)x * 72057594037927936.0);
    bad += got != want;
    ++n;
  }
  printf("%llu %llu\n", n, bad);
  return 0;
}
"""


def test_split_fixed_point_conversion_is_exact_on_all_floats_in_unit_interval():
    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.skip("gcc not available")
    with tempfile.TemporaryDirectory() as d:
        src, exe = os.path.join(d, "fix.c"), os.path.join(d, "fix")
        with open(src, "w") as f:
            f.write(SRC)
        subprocess.run([gcc, "-O2", "-std=c99", "-ffp-contract=off", "-fno-fast-math", src, "-o", exe, "-lm"],
                       check=True)
        out = subprocess.run([exe], check=True, capture_output=True, text=True).stdout.split()
    n, bad = int(out[0]), int(out[1])
    assert n == 1065353217 and bad == 0
