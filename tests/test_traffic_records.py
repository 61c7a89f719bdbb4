"""The DRAM-traffic records behind the bench line's roofline.traffic (CPU only).

profiles/traffic.json holds, per kernel and workload, the dram__bytes_read.sum +
dram__bytes_write.sum of one ncu launch, stamped with a hash of the kernel's source file.
The bench reports that figure only while the source still hashes to the stamp (a changed
kernel reads as "no capture"), and a record must be the capture of a launch that moved
about the kernel's algorithmic bytes: a far larger figure would be re-reads the line
hides, a far smaller one a capture of another launch."""
import hashlib
import json
import os

import bench
import synth.workloads as W

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _algorithmic_bytes(kernel, workload):
    cfg = W.WORKLOADS[workload]
    B, Hq, Hkv, D, P, N = cfg["B"], cfg["Hq"], cfg["Hkv"], cfg["D"], cfg["P"], cfg["N"]
    if kernel.startswith("attn_"):  # K and V of prefix + tree once, Q read and O written once (bf16)
        return 2 * B * Hkv * (P + N) * D * 2 + 2 * B * Hq * N * D * 2
    if kernel.startswith("vocab_pass"):  # the bf16 target logits once
        return B * N * cfg["V"] * 2
    raise AssertionError(kernel)


def test_records_are_consistent_captures():
    with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
        records = json.load(f)
    assert records
    for kernel, ent in records.items():
        assert os.path.exists(os.path.join(ROOT, "tree_speculative_decoding_masked_gb300", "csrc", ent["source"]))
        assert len(ent["source_sha256_16"]) == 16
        for workload, w in ent["workloads"].items():
            assert w["bytes_per_launch"] == w["read"] + w["write"], (kernel, workload)
            ratio = w["bytes_per_launch"] / _algorithmic_bytes(kernel, workload)
            assert 0.9 < ratio < 1.1, (kernel, workload, ratio)
            assert os.path.exists(os.path.join(ROOT, w["capture"])), w["capture"]


def test_traffic_reported_only_for_the_captured_source(tmp_path, monkeypatch):
    csrc = tmp_path / "tree_speculative_decoding_masked_gb300" / "csrc"
    csrc.mkdir(parents=True)
    (tmp_path / "profiles").mkdir()
    src = csrc / "k.cu"
    src.write_text("__global__ void k() {}\n")
    stamp = hashlib.sha256(src.read_bytes()).hexdigest()[:16]
    rec = {"k": {"source": "k.cu", "source_sha256_16": stamp,
                 "workloads": {"long_context": {"bytes_per_launch": 1234, "read": 1200, "write": 34}}}}
    (tmp_path / "profiles" / "traffic.json").write_text(json.dumps(rec))
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.kernel_traffic("k", "long_context") == 1234
    assert bench.kernel_traffic("k", "sampling") is None      # no capture of that workload
    assert bench.kernel_traffic("other", "long_context") is None
    src.write_text("__global__ void k() { /* changed */ }\n")  # the kernel changed since
    assert bench.kernel_traffic("k", "long_context") is None
    (tmp_path / "profiles" / "traffic.json").unlink()
    assert bench.kernel_traffic("k", "long_context") is None
