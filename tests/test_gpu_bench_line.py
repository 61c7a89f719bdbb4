"""The bench's own line on a GPU: one run of `bench.py` on the small fp32 workload and
one on the qwen3-layer workload (a tensor-core roofline), checked for every key the
measurement contract asks for and for values that follow from each other."""
import json
import math
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a GPU", allow_module_level=True)

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _line(workload):
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--workload", workload, "--steps", "20",
                          "--warmup", "3", "--no-cpu-baseline"], cwd=ROOT, capture_output=True, text=True,
                         timeout=900, check=True).stdout
    lines = [ln for ln in out.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, out
    return json.loads(lines[0])


@pytest.mark.parametrize("workload", ["tiny_fp32", "qwen3_4b_layer"])
def test_bench_line_carries_the_contract(workload):
    d = _line(workload)
    for k in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better", "scaling",
              "vs_baseline", "dtype", "data", "config", "roofline", "e2e", "gpu_launches", "clocks"):
        assert k in d, k
    assert d["n_gpus"] == 1 and d["steps"] == 20 and d["warmup"] == 3 and d["higher_is_better"] is True
    assert d["config"]["workload"] == workload and d["data"] == "synthetic"
    assert d["dtype"] == ("f32" if workload == "tiny_fp32" else "bf16")
    # value is nodes per second of the timed steps
    assert d["value"] > 0 and math.isclose(d["value"], d["config"]["B"] * d["config"]["N"] / (d["ms_per_step"] * 1e-3),
                                           rel_tol=1e-6)
    r = d["roofline"]
    for k in ("bound", "achieved", "peak", "unit", "frac", "traffic"):
        assert k in r, k
    assert r["bound"] in ("hbm", "tensor") and r["peak"] > 0 and math.isclose(r["frac"], r["achieved"] / r["peak"])
    e = d["e2e"]
    assert e["value"] > 0 and e["unit"] == d["unit"] and e["h2d_bytes_per_step"] > 0 and e["d2h_bytes_per_step"] > 0
    assert d["gpu_launches"] > 0
    c = d["clocks"]
    assert "sm_mhz" in c and "sm_max_mhz" in c and isinstance(c["reasons"], list)
