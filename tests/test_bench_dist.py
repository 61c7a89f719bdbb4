"""Host logic of bench.py's multi-rank launch, on CPU with the gloo backend and two ranks:
rendezvous, the barrier around the timed region, the max-over-ranks time, and the
reference arm's rank-0-only rule.  The GPU path itself runs replicas only (no data-path
collective), so these are the only cross-rank steps."""
import json
import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench
    import torch.distributed as dist
    r, w = bench.dist_init("gloo")
    bench.barrier(w)
    # each rank reports a different time; every rank must see the largest
    slowest = bench.max_over_ranks(1.5 + rank, w, device="cpu")
    bench.barrier(w)
    with open(os.path.join(out_dir, f"rank{rank}.json"), "w") as f:
        json.dump({"rank": r, "world": w, "env": list(bench.dist_env()), "max": slowest}, f)
    dist.destroy_process_group()


def test_two_rank_barrier_and_max_over_ranks(tmp_path):
    world = 2
    mp.start_processes(_rank_main, args=(world, _free_port(), str(tmp_path)), nprocs=world, join=True,
                       start_method="spawn")
    res = [json.load(open(tmp_path / f"rank{r}.json")) for r in range(world)]
    for r, x in enumerate(res):
        assert x["rank"] == r and x["world"] == world
        assert x["env"] == [r, world, r]
        assert x["max"] == pytest.approx(1.5 + world - 1)


def test_single_rank_needs_no_process_group(monkeypatch):
    sys.path.insert(0, ROOT)
    import bench
    for k in ("RANK", "WORLD_SIZE", "LOCAL_RANK"):
        monkeypatch.delenv(k, raising=False)
    assert bench.dist_env() == (0, 1, 0)
    assert bench.dist_init("gloo") == (0, 1)
    bench.barrier(1)
    assert bench.max_over_ranks(3.25, 1) == 3.25


def test_reference_arm_runs_on_rank_zero_only(monkeypatch, capsys):
    sys.path.insert(0, ROOT)
    import bench
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    args = bench.parse_args(["--impl", "reference", "--gpus", "2", "--steps", "1", "--warmup", "0"])
    bench.run_reference(args)  # a non-zero rank returns without work or output
    assert capsys.readouterr().out == ""


def test_defaults_are_one_gpu_and_the_headline_workload():
    sys.path.insert(0, ROOT)
    import bench
    a = bench.parse_args([])
    assert a.gpus == 1 and a.impl == "ours" and a.warmup >= 3
    assert a.workload == bench.DEFAULT_WORKLOAD


@pytest.mark.parametrize("workload", [None, "tiny_fp32", "budget_sweep"])
def test_reference_arm_prints_one_complete_json_line(monkeypatch, capsys, workload):
    # The oracle arm's line carries every key of the bench contract, with its own value
    # repeated as cpu_baseline and e2e and no host<->device bytes.
    sys.path.insert(0, ROOT)
    import bench
    for k in ("RANK", "WORLD_SIZE", "LOCAL_RANK"):
        monkeypatch.delenv(k, raising=False)
    argv = ["--impl", "reference", "--steps", "2", "--warmup", "0"]
    if workload:
        argv += ["--workload", workload]
    bench.run_reference(bench.parse_args(argv))
    lines = [l for l in capsys.readouterr().out.splitlines() if l.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["impl"] == "reference" and d["n_gpus"] == 1 and d["steps"] == 2 and d["warmup"] == 0
    assert d["value"] > 0 and d["ms_per_step"] > 0 and d["higher_is_better"] is True
    assert d["config"]["workload"] == (workload or bench.DEFAULT_WORKLOAD)
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["sample"] and cb["value"] == d["value"]
    assert cb["unit"] == d["unit"]
    e = d["e2e"]
    assert e["value"] == d["value"] and e["unit"] == d["unit"]
    assert e["h2d_bytes_per_step"] == 0 and e["d2h_bytes_per_step"] == 0


def test_clock_sampler_reads_clocks_and_throttle_reasons(tmp_path, monkeypatch):
    # A stand-in nvidia-smi on PATH prints three samples and then idles like the real
    # looping query; the sampler must report the median SM clock, the largest maximum
    # clock and every throttle reason seen Active in any sample.
    sys.path.insert(0, ROOT)
    import bench
    fake = tmp_path / "nvidia-smi"
    fake.write_text("#!/bin/sh\n"
                    "printf '0, 2070, 2070, 700.5, Active, Not Active, Not Active, Not Active, Not Active\\n'\n"
                    "printf '0, 1980, 2070, 720.0, Active, Active, Not Active, Not Active, Active\\n'\n"
                    "printf '0, 2070, 2070, 710.0, Not Active, Not Active, Not Active, Not Active, Not Active\\n'\n"
                    "exec sleep 30\n")
    fake.chmod(0o755)
    monkeypatch.setenv("PATH", str(tmp_path) + os.pathsep + os.environ.get("PATH", ""))
    s = bench.ClockSampler("0")
    s.start()
    c = s.stop()
    assert c["sm_mhz"] == 2070.0 and c["sm_max_mhz"] == 2070.0
    assert c["reasons"] == ["hw_slowdown", "sw_power_cap"]
    assert c["samples"] == 3 and c["power_w_max"] == 720.0


def test_clock_sampler_without_nvidia_smi(tmp_path, monkeypatch):
    sys.path.insert(0, ROOT)
    import bench
    monkeypatch.setenv("PATH", str(tmp_path))
    s = bench.ClockSampler("0")
    s.start()
    assert s.tmp is None  # the sample file is not left behind
    assert s.stop()["reasons"] == ["nvidia-smi unavailable"]


def test_cpu_baseline_runs_the_oracle_on_every_host_core():
    # The GPU arm's cpu_baseline leg: a subprocess (started before any GPU work) times the
    # oracle with one single-threaded process per host core, then on one core.
    sys.path.insert(0, ROOT)
    import bench
    cb = bench.run_oracle_subprocess(0.5, "tiny_fp32")
    assert cb["kind"] == "oracle" and cb["unit"] == bench.UNIT and cb["value"] > 0
    assert cb["cores"] == bench.host_cores()
    assert cb["single_core"]["cores"] == 1 and cb["single_core"]["value"] > 0
    assert "one per host core" in cb["sample"]
