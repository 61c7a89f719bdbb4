#!/usr/bin/env python3
"""Throughput of one tree-verification round on GB300.

A step = one pass of the hot path over one batch of seeded synthetic input:
    tv_select_subtree (pool -> tree)  ->  tv_tree_attention  ||  tv_verify_greedy
(the sampling workload runs tv_verify_sample instead of the greedy verify).
Metric: verified tree nodes per second = B * N / step time.  The default workload is
long_context (B=8, prefix 32768, 128-node trees, V=151936): the largest one that fits a
single GPU.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

Timing: W untimed warm-up steps, then exactly K steps bracketed by a barrier and a device
synchronise on both sides, timed with CUDA events on the launching stream.  Steps are
CUDA-graph replays; the inputs rotate over enough copies that their total exceeds twice
the L2, so no step reads its inputs from L2.  Under torchrun every rank runs its own
replica (the path shards by independent sequences; there is no data-path collective),
the max time over ranks is used and rank 0 prints one JSON line.

The line's roofline is that of the dominant kernel (algorithmic bytes or FLOPs per
launch over its CUDA-event time, against MEASURED_PEAKS.json); "e2e" repeats the step
through the Python API with the round's inputs copied in from pinned host memory and the
outcome copied back; "cpu_baseline" is the CPU oracle on every host core.

``--impl reference`` times the CPU oracle on the host cores instead (rank 0 only).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

# BLAS / OpenMP pool sizes of the oracle processes: one thread each (one process per core)
ORACLE_THREAD_VARS = ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS", "NUMEXPR_NUM_THREADS")
if __name__ == "__main__" and ("--impl=reference" in sys.argv[1:] or any(
        a == "--impl" and b == "reference" for a, b in zip(sys.argv[1:], sys.argv[2:]))):
    for _var in ORACLE_THREAD_VARS:  # before NumPy is first imported
        os.environ[_var] = "1"

METRIC = "verified tree nodes/sec (attn+accept) and achieved HBM GB/s vs GB300 peak"
UNIT = "nodes/s"
DEFAULT_WORKLOAD = "long_context"  # the largest workload that fits one GPU


def parse_args(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=60000)
    ap.add_argument("--warmup", type=int, default=200)
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--budget", type=int, default=None,
                    help="rows per tree for pool workloads (default: the workload's largest budget)")
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--oracle-worker", type=float, default=None, help=argparse.SUPPRESS)
    return ap.parse_args(argv)


# ------------------------------------------------------------------------------------
# distributed plumbing (timing only: barrier and max over ranks)


def dist_env():
    return int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")), int(
        os.environ.get("LOCAL_RANK", "0"))


def dist_init(backend):
    rank, world, _ = dist_env()
    if world > 1:
        import torch.distributed as dist
        if not dist.is_initialized():
            dist.init_process_group(backend=backend)
    return rank, world


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int, device=None) -> float:
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ------------------------------------------------------------------------------------
# oracle sample (CPU baseline and the reference arm), run on every host core
#
# One oracle unit is a fixed slice of the verification of sequence 0 of the workload: the
# float64 attention row of one (node, head) pair; the unit that completes a node's heads
# also takes that node's vocab row, and the unit that completes the tree also runs the
# subtree selection and the acceptance walk.  A unit counts as 1/Hq of a verified node.
# The inputs are built once, stored as float64 .npy files and memory-mapped by a pool of
# spawned worker processes (one per core the process may run on), each single-threaded.


def host_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def oracle_inputs(workload: str, dirpath: str) -> dict:
    """Build sequence 0 of ``workload`` for the oracle (oracle selection + the bench's
    synthetic recipe) and store it under ``dirpath``; returns the metadata."""
    import numpy as np

    import synth
    import synth.workloads as W
    from oracle import selection, vocab

    cfg = W.WORKLOADS[workload]
    g = synth.rng(cfg["seed"])
    Hq, Hkv, D, P, V = cfg["Hq"], cfg["Hkv"], cfg["D"], cfg["P"], cfg["V"]
    arrays = {}
    if "pool_d" in cfg:
        N = cfg.get("N") or max(cfg["budgets"])
        marg, ptok = W.pools(g, 1, cfg["pool_d"], cfg["pool_k"], V)
        sel = selection.select_subtree(marg[0], ptok[0], N, 11)
        par, tok = sel["parent"][None], sel["token"][None]
        arrays["marg"], arrays["ptok"] = marg, ptok
    else:
        N = cfg["N"]
        par, tok = W.trees(g, 1, N, cfg["depth_cap"], V)
    bf16 = cfg["bf16"]
    if cfg["mode"] == "sample":
        tgt, drf, tok = W.sampling_logits(g, par, V, bf16, cfg["temperature"])
        arrays["draft"] = drf
    else:
        tgt = W.planted_logits(g, par, tok, V, bf16)
        _, _, argmax_all = vocab.vocab_stats(tgt[0])  # set-up: lets the walk run every tree
        arrays["argmax"] = argmax_all
    arrays["logits"] = tgt
    q, k, v = W.qkv_host(g, 1, Hq, Hkv, D, P, N, bf16)
    arrays.update(q=q.astype(np.float64), k=k.astype(np.float64), v=v.astype(np.float64), par=par, tok=tok)
    for name, arr in arrays.items():
        np.save(os.path.join(dirpath, name + ".npy"), arr)
    meta = {"workload": workload, "N": int(N), "Hq": Hq, "P": P, "V": V, "mode": cfg["mode"],
            "temperature": cfg.get("temperature", 1.0), "pool": "pool_d" in cfg}
    with open(os.path.join(dirpath, "meta.json"), "w") as f:
        json.dump(meta, f)
    return meta


def oracle_sample_desc(meta: dict) -> str:
    N, Hq = meta["N"], meta["Hq"]
    return (f"{meta['workload']}, sequence 0 (N={N}, Hq={Hq}, P={meta['P']}, V={meta['V']}): one oracle unit = "
            f"the float64 attention row of one (node, head) pair; every {Hq}th unit adds that node's vocab row, "
            f"every {N * Hq}th unit the subtree selection and acceptance walk; a unit counts as 1/{Hq} node")


_ORACLE = {}  # per-process state of an oracle worker


def oracle_worker_init(dirpath: str):
    """Memory-map the stored inputs and build the unit function (pool initializer)."""
    import numpy as np

    from oracle import attention, greedy, sampling, selection, vocab

    with open(os.path.join(dirpath, "meta.json")) as f:
        meta = json.load(f)
    A = {name[:-4]: np.load(os.path.join(dirpath, name), mmap_mode="r")
         for name in os.listdir(dirpath) if name.endswith(".npy")}
    N, Hq, P = meta["N"], meta["Hq"], meta["P"]
    par, tok = np.asarray(A["par"]), np.asarray(A["tok"])

    def unit(i):
        node = (i // Hq) % N
        head = i % Hq
        attention.tree_attention(A["q"], A["k"], A["v"], par, P, nodes=[node], heads=[head])
        if head == Hq - 1:
            vocab.row_stats(A["logits"][0][node])
            if node == N - 1:
                if meta["pool"]:
                    selection.select_subtree(A["marg"][0], A["ptok"][0], N, 11)
                if meta["mode"] == "sample":
                    sampling.sampling_walk(A["logits"][0], A["draft"][0], par[0], tok[0], meta["temperature"], 1, i, 0)
                else:
                    greedy.greedy_walk(par[0], tok[0], A["argmax"])
        return 1.0 / Hq

    _ORACLE["unit"] = unit
    _ORACLE["meta"] = meta


def oracle_run_units(job):
    """Run units start, start + stride, ... (count of them); returns (nodes, seconds)."""
    start, count, stride = job
    unit = _ORACLE["unit"]
    t0 = time.perf_counter()
    nodes = 0.0
    for j in range(count):
        nodes += unit(start + j * stride)
    return nodes, time.perf_counter() - t0


def oracle_run_for(job):
    """Run units start, start + stride, ... for ``seconds``; returns (nodes, units, seconds)."""
    start, stride, seconds = job
    unit = _ORACLE["unit"]
    t0 = time.perf_counter()
    nodes, i = 0.0, 0
    while True:
        nodes += unit(start + i * stride)
        i += 1
        if time.perf_counter() - t0 >= seconds:
            break
    return nodes, i, time.perf_counter() - t0


def oracle_pool(dirpath: str, cores: int):
    import multiprocessing as mp
    for var in ORACLE_THREAD_VARS:  # spawned workers inherit one-thread BLAS pools
        os.environ[var] = "1"
    return mp.get_context("spawn").Pool(cores, initializer=oracle_worker_init, initargs=(dirpath,))


def oracle_worker(budget_s: float, workload: str):
    """CPU baseline: the oracle on every host core for ``budget_s`` seconds of wall time
    (each worker runs its own interleaved units), then on one core for a quarter of it."""
    cores = host_cores()
    with tempfile.TemporaryDirectory() as d:
        meta = oracle_inputs(workload, d)
        with oracle_pool(d, cores) as pool:
            pool.map(oracle_run_units, [(k, 1, cores) for k in range(cores)])  # warm every worker
            res = pool.map(oracle_run_for, [(k, cores, budget_s) for k in range(cores)])
        nodes = sum(r[0] for r in res)
        units = sum(r[1] for r in res)
        wall = max(r[2] for r in res)
        oracle_worker_init(d)
        n1, u1, t1 = oracle_run_for((0, 1, max(2.0, budget_s / 4)))
    print(json.dumps({"value": nodes / wall, "units": units, "seconds": wall, "cores": cores,
                      "single_core_value": n1 / t1, "single_core_units": u1, "single_core_seconds": t1,
                      "sample": oracle_sample_desc(meta)}))


def run_oracle_subprocess(budget_s: float, workload: str) -> dict:
    env = dict(os.environ)
    for var in ORACLE_THREAD_VARS:
        env[var] = "1"
    env.pop("RANK", None)
    env.pop("WORLD_SIZE", None)
    res = subprocess.run([sys.executable, os.path.abspath(__file__), "--oracle-worker", str(budget_s), "--workload",
                          workload], capture_output=True, text=True, env=env, timeout=1800)
    if res.returncode != 0:
        raise RuntimeError("oracle worker failed:\n" + res.stderr[-2000:])
    out = json.loads(res.stdout.strip().splitlines()[-1])
    return {"value": out["value"], "unit": UNIT, "cores": out["cores"], "kind": "oracle",
            "sample": out["sample"] + f"; {out['units']} units in {out['seconds']:.1f} s over {out['cores']} "
                      f"single-threaded NumPy processes (one per host core)",
            "single_core": {"value": out["single_core_value"], "unit": UNIT, "cores": 1,
                            "sample": f"{out['single_core_units']} units in {out['single_core_seconds']:.1f} s "
                                      f"in one process"}}


def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return
    import synth.workloads as W
    cfg = W.WORKLOADS[args.workload]
    cores = host_cores()
    with tempfile.TemporaryDirectory() as d:
        meta = oracle_inputs(args.workload, d)
        with oracle_pool(d, cores) as pool:
            # a step = the same number of units on every worker, sized so that the whole
            # run takes about two minutes (at most 0.25 s per step)
            probe = pool.map(oracle_run_units, [(k, 2, cores) for k in range(cores)])
            per_unit = max(1e-6, max(t for _, t in probe) / 2)
            step_s = min(0.25, max(0.002, 120.0 / max(1, args.steps + args.warmup)))
            per_worker = max(1, int(round(step_s / per_unit)))
            base = [2 * cores]

            def step():
                jobs = [(base[0] + k, per_worker, cores) for k in range(cores)]
                base[0] += cores * per_worker
                return sum(n for n, _ in pool.map(oracle_run_units, jobs))

            for _ in range(args.warmup):
                step()
            nodes = 0.0
            t0 = time.perf_counter()
            for _ in range(args.steps):
                nodes += step()
            dt = time.perf_counter() - t0
    value = nodes / dt
    sample = (oracle_sample_desc(meta) + f"; a step = {per_worker} units on each of {cores} single-threaded NumPy "
              f"processes (one per host core), {args.steps} steps timed in {dt:.2f} s")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt * 1e3 / max(1, args.steps),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": workload_config(args.workload, cfg),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------------------------
# GPU arm


def workload_config(name, cfg):
    keys = ("B", "Hq", "Hkv", "D", "P", "N", "V", "mode")
    c = {"workload": name}
    c.update({k: cfg[k] for k in keys if k in cfg})
    if "pool_d" in cfg:
        c["pool"] = f"{cfg['pool_d']}x{cfg['pool_k']}"
        c.setdefault("N", cfg.get("N"))
    c["dtype"] = "bf16" if cfg["bf16"] else "f32"
    return c


class ClockSampler:
    """nvidia-smi clock / throttle sampling during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str):
        self.gpu_id = gpu_id
        self.proc = None
        self.tmp = None

    def start(self):
        try:
            self.tmp = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                                          "-i", self.gpu_id, "-lms", "50"], stdout=self.tmp,
                                         stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
            if self.tmp is not None:  # no sampler: drop the empty sample file
                self.tmp.close()
                os.unlink(self.tmp.name)
                self.tmp = None
        time.sleep(0.3)

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.1)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.tmp.flush()
        self.tmp.seek(0)
        lines = [ln.strip() for ln in self.tmp.read().splitlines() if ln.strip()]
        self.tmp.close()
        os.unlink(self.tmp.name)
        sms, maxs, reasons, power = [], [], set(), []
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sms.append(float(parts[1]))
                maxs.append(float(parts[2]))
                power.append(float(parts[3]))
            except ValueError:
                continue
            for nm, val in zip(names, parts[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(nm)
        return {"sm_mhz": statistics.median(sms) if sms else None, "sm_max_mhz": max(maxs) if maxs else None,
                "reasons": sorted(reasons), "samples": len(sms), "power_w_max": max(power) if power else None}


def gpu_identifier(torch, device_index):
    try:
        uuid = str(torch.cuda.get_device_properties(device_index).uuid)
        if uuid:
            return uuid if uuid.startswith("GPU-") else "GPU-" + uuid
    except Exception:
        pass
    vis = os.environ.get("CUDA_VISIBLE_DEVICES")
    if vis:
        return vis.split(",")[device_index]
    return str(device_index)


def measured_peaks():
    """(HBM GB/s, bf16 dense TFLOP/s burst, 'measured' | 'fallback')."""
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return d.get("hbm_gbs"), d.get("bf16_tflops"), "measured"
    return 6800.0, 1900.0, "fallback"


def sustained_bf16_peak():
    """bf16 dense TFLOP/s of a seconds-long GEMM loop under the power cap, or None."""
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            return json.load(f).get("bf16_tflops_sustained")
    return 1700.0


def kernel_traffic(kernel: str, workload: str):
    """DRAM bytes per launch of ``kernel`` on ``workload`` from the committed ncu summary,
    if it was taken on the current kernel source; else None."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        d = json.load(f)
    ent = d.get(kernel)
    if not ent or workload not in ent.get("workloads", {}):
        return None
    src = os.path.join(ROOT, "tree_speculative_decoding_masked_gb300", "csrc", ent["source"])
    h = hashlib.sha256(open(src, "rb").read()).hexdigest()[:16]
    return ent["workloads"][workload]["bytes_per_launch"] if h == ent["source_sha256_16"] else None


def roofline_entry(kernel, bytes_per_launch, flops_per_launch, seconds, workload):
    """Roofline of one kernel: HBM-bound unless its arithmetic intensity is above the
    ridge point of the measured peaks, then bf16 tensor-bound."""
    hbm, tflops, kind = measured_peaks()
    tensor = flops_per_launch > 0 and flops_per_launch / bytes_per_launch > tflops * 1e12 / (hbm * 1e9)
    if tensor:
        achieved, peak, unit = flops_per_launch / seconds / 1e12, tflops, "TFLOP/s"
    else:
        achieved, peak, unit = bytes_per_launch / seconds / 1e9, hbm, "GB/s"
    out = {"bound": "tensor" if tensor else "hbm", "kernel": kernel, "achieved": achieved, "peak": peak,
           "unit": unit, "frac": achieved / peak, "peak_kind": kind,
           "traffic": kernel_traffic(kernel, workload), "algorithmic_bytes_per_launch": bytes_per_launch,
           "algorithmic_flops_per_launch": flops_per_launch}
    sus = sustained_bf16_peak() if tensor else None
    if sus:  # the kernel's timing loop runs long enough to sit at the power cap
        out["frac_of_sustained_peak"] = achieved / sus
    return out


def run_ours(args):
    import numpy as np
    import torch

    import synth
    import synth.workloads as W
    import tree_speculative_decoding_masked_gb300 as tv

    rank, world, local = dist_env()
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU (the library has no CPU path)")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    cpu_base = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        # before any GPU work: the oracle runs in its own processes, one per host core
        cpu_base = run_oracle_subprocess(10.0, args.workload)
    rank, world = dist_init("nccl")
    tv.load_library()

    cfg = W.WORKLOADS[args.workload]
    bf16 = cfg["bf16"]
    tdt = torch.bfloat16 if bf16 else torch.float32
    B, Hq, Hkv, D, P, V = cfg["B"], cfg["Hq"], cfg["Hkv"], cfg["D"], cfg["P"], cfg["V"]
    sampling_mode = cfg["mode"] == "sample"
    g = synth.rng(cfg["seed"] + rank)

    def to_dev(x):
        if bf16:
            bits = synth.bf16_bits(x)
            return torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(dev)
        return torch.from_numpy(x).to(dev)

    # ---- inputs (one set on the host; device copies rotate)
    use_pool = "pool_d" in cfg
    if use_pool:
        N = args.budget or cfg.get("N") or max(cfg["budgets"])
        marg, ptok = W.pools(g, B, cfg["pool_d"], cfg["pool_k"], V)
        marg_d, ptok_d = torch.from_numpy(marg).to(dev), torch.from_numpy(ptok).to(dev)
        root_d = torch.full((B,), 11, dtype=torch.int32, device=dev)
        sel = tv.select_subtree(marg_d, ptok_d, N, root_d)
        torch.cuda.synchronize()
        par = sel["parent"].cpu().numpy()
        tok = sel["tokens"].cpu().numpy()
    else:
        N = cfg["N"]
        par, tok = W.trees(g, B, N, cfg["depth_cap"], V)
    if sampling_mode:
        tgt, drf, tok = W.sampling_logits(g, par, V, bf16, cfg["temperature"])
    else:
        tgt = W.planted_logits(g, par, tok, V, bf16)
        drf = None
    q, k, v = W.qkv_host(g, B, Hq, Hkv, D, P, N, bf16)
    host = {"q": q, "k": k, "v": v, "logits": tgt}
    if drf is not None:
        host["draft"] = drf
    if use_pool:
        host["marg"], host["ptok"] = marg, ptok

    elt = 2 if bf16 else 4
    bytes_attn = (B * Hkv * (P + N) * D * 2 + 2 * B * Hq * N * D) * elt
    bytes_vocab = B * N * V * elt * (2 if sampling_mode else 1)
    bytes_set = bytes_attn + bytes_vocab
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    n_sets = max(2, -(-2 * l2 // bytes_set))
    base = {kk: to_dev(vv) if kk in ("q", "k", "v", "logits", "draft") else torch.from_numpy(vv).to(dev)
            for kk, vv in host.items()}
    sets = [base] + [{kk: t.clone() for kk, t in base.items()} for _ in range(n_sets - 1)]
    par_d = torch.from_numpy(par.astype(np.int32)).to(dev)
    tok_d = torch.from_numpy(tok.astype(np.int32)).to(dev)
    for s in sets:
        s["out"] = torch.empty(B, Hq, N, D, dtype=tdt, device=dev)
        s["root"] = torch.full((B,), 11, dtype=torch.int32, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    ws_attn = torch.zeros(max(256, tv.tree_attention_workspace_size(B, Hq, Hkv, D, P, N, tdt)), dtype=torch.uint8,
                          device=dev)
    ws_ver = torch.zeros(tv.verify_workspace_size(B, N, V, tdt, sampling_mode), dtype=torch.uint8, device=dev)
    sel_out = {"parent": par_d.clone(), "tokens": tok_d.clone(),
               "depth": torch.empty(B, N, dtype=torch.int32, device=dev),
               "score": torch.empty(B, N, dtype=torch.float32, device=dev),
               "n_nodes": torch.empty(B, dtype=torch.int32, device=dev)}
    ver_out = {"accepted_nodes": torch.empty(B, N, dtype=torch.int32, device=dev),
               "accept_len": torch.empty(B, dtype=torch.int32, device=dev),
               "bonus_token": torch.empty(B, dtype=torch.int32, device=dev),
               "out_token": torch.empty(B, dtype=torch.int32, device=dev),
               "p_draft": torch.empty(B, N, dtype=torch.float32, device=dev),
               "q_draft": torch.empty(B, N, dtype=torch.float32, device=dev)}

    def k_select(s):
        if use_pool:
            tv.select_subtree(s["marg"], s["ptok"], N, s["root"], dev_status=status, out=sel_out)

    def k_attn(s):
        tv.tree_attention(s["q"], s["k"], s["v"], sel_out["parent"], P, out=s["out"], workspace=ws_attn,
                          dev_status=status)

    def k_verify(s, rnd=0):
        if sampling_mode:
            tv.verify_sample(s["logits"], s["draft"], sel_out["parent"], sel_out["tokens"],
                             temperature=cfg["temperature"], seed=cfg["seed"], round=rnd, workspace=ws_ver,
                             dev_status=status, out=ver_out)
        else:
            tv.verify_greedy(s["logits"], sel_out["parent"], sel_out["tokens"], workspace=ws_ver, dev_status=status,
                             out=ver_out)

    vocab_out = {"row_lse": torch.empty(B, N, dtype=torch.float32, device=dev),
                 "row_argmax": torch.empty(B, N, dtype=torch.int32, device=dev),
                 "p_draft": torch.empty(B, N, dtype=torch.float32, device=dev),
                 "draft_row_lse": torch.empty(B, N, dtype=torch.float32, device=dev),
                 "q_draft": torch.empty(B, N, dtype=torch.float32, device=dev)}

    def k_vocab(s):
        # the vocab pass alone (the first kernel of either verify call)
        tv.vocab_stats(s["logits"], sel_out["parent"], sel_out["tokens"], draft_logits=s.get("draft"),
                       temperature=cfg.get("temperature", 1.0), workspace=ws_ver, dev_status=status, out=vocab_out)

    # cost line for the cost-aware selection: step time against tree rows, fitted to this
    # bench's own budget_sweep runs (attention + verify, B=16): ~38 us + 3.09 us per row
    cost_line = (38.0, 3.09)
    sel_ad_out = {kk: torch.empty_like(t) for kk, t in sel_out.items()}

    def k_select_adaptive(s):
        if use_pool:
            tv.select_subtree(s["marg"], s["ptok"], N, s["root"], dev_status=status, out=sel_ad_out, cost=cost_line)

    Wm = (N + 31) // 32
    prep_out = {"depth": torch.empty(B, N, dtype=torch.int32, device=dev),
                "pos": torch.empty(B, N, dtype=torch.int32, device=dev),
                "anc_mask": torch.empty(B, N, Wm, dtype=torch.int32, device=dev),
                "child_off": torch.empty(B, N + 1, dtype=torch.int32, device=dev),
                "child_idx": torch.empty(B, N, dtype=torch.int32, device=dev)}

    def k_prep(s):
        tv.tree_prep(sel_out["parent"], P, dev_status=status, out=prep_out)

    # one TreeGraft-style expansion step: 8 frontier rows per sequence, top-8 children each;
    # the first rows of the set's logits stand in for the drafter's next-token rows
    exp_rows = min(B * 8, B * N)
    exp_m = 8
    exp_ps = torch.full((exp_rows,), 0.5, dtype=torch.float32, device=dev)
    exp_ws = torch.zeros(tv.expand_workspace_size(exp_rows, V, exp_m), dtype=torch.uint8, device=dev)
    exp_out = {"token": torch.empty(exp_rows, exp_m, dtype=torch.int32, device=dev),
               "p": torch.empty(exp_rows, exp_m, dtype=torch.float32, device=dev),
               "score": torch.empty(exp_rows, exp_m, dtype=torch.float32, device=dev)}

    def k_expand(s):
        tv.expand_children(s["logits"].view(B * N, V)[:exp_rows], exp_ps, exp_m, workspace=exp_ws,
                           dev_status=status, out=exp_out)

    # PTD width / depth control on the step's tree: at most 2 children per node, 8 levels
    prune_conf = sel_out["score"] if use_pool else torch.ones(B, N, dtype=torch.float32, device=dev)
    prune_out = {"old_to_new": torch.empty(B, N, dtype=torch.int32, device=dev),
                 "new_parent": torch.empty(B, N, dtype=torch.int32, device=dev),
                 "n_kept": torch.empty(B, dtype=torch.int32, device=dev),
                 "new_root": torch.empty(B, dtype=torch.int32, device=dev)}

    def k_prune(s):
        tv.prune_tree(sel_out["parent"], prune_conf, 2, 8, dev_status=status, out=prune_out)

    def k_commit(s):
        # keep the accepted path's KV rows (timed in the breakdown, not part of the step)
        tv.commit_accepted_kv(s["k"], s["v"], ver_out["accepted_nodes"], ver_out["accept_len"], P, dev_status=status)

    side = torch.cuda.Stream(device=dev)
    order = {"verify_on_main": False}

    def step(s):
        # selection feeds both; tree attention and the vocab pass are independent of each
        # other and run concurrently (fork after selection, join before the next step).
        # The kernel on selection's own stream starts its CTAs while selection finishes
        # (programmatic dependent launch); the other one waits for an event.
        first, second = (k_verify, k_attn) if order["verify_on_main"] else (k_attn, k_verify)
        k_select(s)
        fork = torch.cuda.Event()
        fork.record()
        side.wait_event(fork)
        first(s)
        with torch.cuda.stream(side):
            second(s)
            join = torch.cuda.Event()
            join.record()
        torch.cuda.current_stream().wait_event(join)

    launches_per_step = (1 if use_pool else 0) + 1 + (2 if sampling_mode else 1)

    stream = torch.cuda.Stream(device=dev)
    with torch.cuda.stream(stream):
        for i in range(max(3, args.warmup)):
            step(sets[i % n_sets])
    torch.cuda.synchronize()
    if int(status.item()) != 0:
        raise SystemExit(f"device status {int(status.item())} after warm-up")

    def capture(fn):
        gph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gph, stream=stream):
            fn()
        return gph

    # attention and the vocab pass run concurrently; pick the SM shares that give the
    # fastest step (the whole device for both, or disjoint parts so both grids are
    # resident together)
    n_sm = torch.cuda.get_device_properties(dev).multi_processor_count
    parts = [(0, 0)] + [(v, n_sm - v) for v in (n_sm // 4, n_sm // 3, 5 * n_sm // 12, n_sm // 2,
                                                   7 * n_sm // 12, 2 * n_sm // 3)]
    if bf16:
        # when the whole-device attention grid leaves SMs free, give exactly those to verify
        tv.set_sm_partition(0, 0)
        kern, spl = tv.tree_attention_plan(B, Hq, Hkv, D, P, N, tdt)
        G = Hq // Hkv
        nt = (128 // G) // 8 * 8
        mtiles = -(-N // nt)
        ctas = B * Hkv * (-(-mtiles // 2) if kern >= 2 else mtiles) * spl
        if kern in (1, 2, 3, 5) and ctas < n_sm:  # the persistent grid (4) fills the device
            parts.append((n_sm - ctas, ctas))
    candidates = [(part, vm) for part in parts for vm in (False, True)]
    trial, trial_reps = {}, {}
    # two rounds over the candidates, keeping each one's faster round, so that a noisy
    # round does not decide the configuration
    for cand in candidates + candidates:
        tv.set_sm_partition(*cand[0])
        order["verify_on_main"] = cand[1]
        with torch.cuda.stream(stream):
            g_try = capture(lambda: [step(s) for s in sets])
            for _ in range(3):
                g_try.replay()
        torch.cuda.synchronize()
        ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        reps = trial_reps.get(cand)
        if reps is None:  # about 0.25 s of replays per round, from the first round's pace
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            with torch.cuda.stream(stream):
                g_try.replay()
            e1.record(stream)
            torch.cuda.synchronize()
            reps = trial_reps[cand] = int(min(max(3, 2000 // n_sets), max(3, 250.0 / max(e0.elapsed_time(e1), 1e-3))))
        ev0.record(stream)
        with torch.cuda.stream(stream):
            for _ in range(reps):
                g_try.replay()
        ev1.record(stream)
        torch.cuda.synchronize()
        trial[cand] = min(trial.get(cand, float("inf")), ev0.elapsed_time(ev1) / reps)
        del g_try
    sm_partition, verify_on_main = min(trial, key=trial.get)
    tv.set_sm_partition(*sm_partition)
    order["verify_on_main"] = verify_on_main

    with torch.cuda.stream(stream):
        g_all = capture(lambda: [step(s) for s in sets])          # one step per input set
        g_one = [capture(lambda s=s: step(s)) for s in sets]
    # one graph per kernel family covering every input set (launch overhead amortised the
    # same way as in the step graph), each kernel alone on the whole device: the SM split
    # above is for running attention and verify side by side
    tv.set_sm_partition(0, 0)
    with torch.cuda.stream(stream):
        fam_graphs = {"attention": capture(lambda: [k_attn(s) for s in sets]),
                      "verify": capture(lambda: [k_verify(s) for s in sets]),
                      "vocab": capture(lambda: [k_vocab(s) for s in sets]),
                      "commit": capture(lambda: [k_commit(s) for s in sets]),
                      "tree_prep": capture(lambda: [k_prep(s) for s in sets]),
                      "expand": capture(lambda: [k_expand(s) for s in sets]),
                      "prune": capture(lambda: [k_prune(s) for s in sets])}
        if use_pool:
            fam_graphs["select"] = capture(lambda: [k_select(s) for s in sets])
            fam_graphs["select_adaptive"] = capture(lambda: [k_select_adaptive(s) for s in sets])
    torch.cuda.synchronize()
    tv.set_sm_partition(*sm_partition)

    def timed(fn, reps):
        ev0 = torch.cuda.Event(enable_timing=True)
        ev1 = torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        barrier(world)
        torch.cuda.synchronize()
        ev0.record(stream)
        fn(reps)
        ev1.record(stream)
        torch.cuda.synchronize()
        barrier(world)
        return ev0.elapsed_time(ev1)  # ms

    def run_steps(k):
        with torch.cuda.stream(stream):
            full, rest = divmod(k, n_sets)
            for _ in range(full):
                g_all.replay()
            for i in range(rest):
                g_one[i].replay()

    # warm the graphs, then the timed region
    run_steps(min(args.steps, 4 * n_sets))
    sampler = ClockSampler(gpu_identifier(torch, local))
    if rank == 0:
        sampler.start()
    ms = timed(run_steps, args.steps)
    clocks = sampler.stop() if rank == 0 else None
    ms = max_over_ranks(ms, world, dev)
    ms_per_step = ms / args.steps
    value = world * B * N / (ms_per_step / 1e3)
    if int(status.item()) != 0:
        raise SystemExit(f"device status {int(status.item())} after the timed region")

    # ---- per-kernel breakdown (one family at a time, every input set per graph replay)
    fam_reps = max(1, min(args.steps, 20000) // n_sets)

    def fam(name):
        def f(k):
            with torch.cuda.stream(stream):
                for _ in range(k):
                    fam_graphs[name].replay()
        return f

    br = {name: timed(fam(name), fam_reps) * 1e3 / (fam_reps * n_sets) for name in fam_graphs}
    if sampling_mode:
        br["walk"] = br["verify"] - br["vocab"]  # the sampling walk kernel after the vocab pass
    expand_bytes = exp_rows * V * elt
    commit_bytes = int(ver_out["accept_len"].sum().item()) * Hkv * D * elt * 2 * 2  # K and V rows, read + write
    # algorithmic attention FLOPs: QK^T and PV over each node's visible keys only, the
    # prefix plus its |pi(i)| = depth + 1 tree keys; the dense bound counts every
    # (node, key) pair of the prefix and the tree block, as the tile kernels compute them
    depth = np.zeros((B, N), dtype=np.int64)
    for i in range(1, N):
        depth[:, i] = depth[np.arange(B), par[:, i]] + 1
    visible = int(B * N * P + (depth + 1).sum())
    flops_alg = 4 * Hq * D * visible
    flops_dense = 4 * B * Hq * N * (P + N) * D
    tv.set_sm_partition(0, 0)  # the plan of the attention family, timed on the whole device
    attn_kernel, attn_splits = tv.tree_attention_plan(B, Hq, Hkv, D, P, N, tdt)
    tv.set_sm_partition(*sm_partition)
    attn_name = ("attn_simt_kernel", "attn_tc_kernel", "attn_pair_kernel", "attn_pair2_kernel",
                 "attn_stream_kernel", "attn_pair2_kernel")[attn_kernel]
    rooflines = {
        attn_name: roofline_entry(attn_name, bytes_attn, flops_alg if bf16 else 0, br["attention"] * 1e-6,
                                  args.workload),
        "vocab_pass_tma_kernel": roofline_entry("vocab_pass_tma_kernel", bytes_vocab, 0, br["vocab"] * 1e-6,
                                                args.workload),
    }
    rooflines[attn_name]["dense_flops_per_launch"] = flops_dense
    rooflines["vocab_pass_tma_kernel"]["timed"] = "tv_vocab_stats alone (the vocab pass without a walk)"
    dom = attn_name if br["attention"] >= br["vocab"] else "vocab_pass_tma_kernel"
    roofline = rooflines[dom]

    # ---- end to end through the public API with host buffers (pinned), copies timed.
    # A decoding loop keeps the committed prefix KV cache (rows 0..P-1) on the device
    # across rounds; what a round brings is the tree's queries, the tree's own K/V rows
    # (written into cache rows P..P+N-1), the target (and draft) logits and the
    # candidate pool.  Those are copied in from pinned host memory every step, and the
    # accept outcome is copied back.
    # Two device input sets alternate: the copies of round i + 1 run on a copy stream while
    # round i computes (each round's copies finish before its compute starts, and a set
    # is refilled only after the round that read it has finished).
    round_in = {"q": (host["q"], lambda d: d["q"]),
                "k_tree": (np.ascontiguousarray(host["k"][:, :, P:P + N]), lambda d: d["k"][:, :, P:P + N]),
                "v_tree": (np.ascontiguousarray(host["v"][:, :, P:P + N]), lambda d: d["v"][:, :, P:P + N]),
                "logits": (host["logits"], lambda d: d["logits"])}
    if "draft" in host:
        round_in["draft"] = (host["draft"], lambda d: d["draft"])
    if use_pool:
        round_in["marg"] = (host["marg"], lambda d: d["marg"])
        round_in["ptok"] = (host["ptok"], lambda d: d["ptok"])
    pinned = {kk: ((to_dev(vv) if kk not in ("marg", "ptok") else torch.from_numpy(vv)).cpu().pin_memory(), where)
              for kk, (vv, where) in round_in.items()}
    res_host = [{kk: torch.empty_like(ver_out[kk], device="cpu").pin_memory()
                 for kk in (("accepted_nodes", "accept_len", "out_token") if sampling_mode else
                            ("accepted_nodes", "accept_len", "bonus_token"))} for _ in range(2)]
    h2d = sum(t.numel() * t.element_size() for t, _ in pinned.values())
    d2h = sum(t.numel() * t.element_size() for t in res_host[0].values())
    dsts = sets[:2] if n_sets >= 2 else [sets[0], {kk: t.clone() for kk, t in sets[0].items()}]
    dst_views = [{kk: where(d) for kk, (_, where) in pinned.items()} for d in dsts]
    e2e_steps = max(20, min(2000, args.steps // 20))
    copy_stream = torch.cuda.Stream(device=dev)

    def copies_in(j):
        for kk, (t, _) in pinned.items():
            dst_views[j][kk].copy_(t, non_blocking=True)

    def copies_out(j):
        for kk, t in res_host[j].items():
            t.copy_(ver_out[kk], non_blocking=True)

    def e2e(k):
        # copy stream: inputs of round i into set i % 2; compute stream: round i, then its
        # outcome back to the host
        done = [None, None]
        ready = torch.cuda.Event()
        copy_stream.wait_stream(stream)  # after the timed region's start event
        with torch.cuda.stream(copy_stream):
            copies_in(0)
            ready.record()
        for i in range(k):
            j = i % 2
            stream.wait_event(ready)
            if i + 1 < k:
                with torch.cuda.stream(copy_stream):
                    if done[1 - j] is not None:
                        copy_stream.wait_event(done[1 - j])
                    copies_in(1 - j)
                    ready = torch.cuda.Event()
                    ready.record()
            with torch.cuda.stream(stream):
                step(dsts[j])
                copies_out(j)
                ev = torch.cuda.Event()
                ev.record()
                done[j] = ev
        stream.wait_stream(copy_stream)

    def copies_only(k):
        with torch.cuda.stream(stream):
            for i in range(k):
                copies_in(i % 2)
                copies_out(i % 2)

    e2e(3)
    ms_e2e = max_over_ranks(timed(e2e, e2e_steps), world, dev)
    e2e_value = world * B * N / (ms_e2e / e2e_steps / 1e3)
    copies_only(2)
    ms_copy = timed(copies_only, e2e_steps) / e2e_steps

    # pinned host <-> device copy ceiling: one 256 MiB copy each way, best of three
    probe_bytes = 1 << 28
    hbuf = torch.empty(probe_bytes, dtype=torch.uint8).pin_memory()
    dbuf = torch.empty(probe_bytes, dtype=torch.uint8, device=dev)
    best = {"h2d": float("inf"), "d2h": float("inf")}
    for _ in range(3):
        for way in ("h2d", "d2h"):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            with torch.cuda.stream(stream):
                (dbuf.copy_(hbuf, non_blocking=True) if way == "h2d" else hbuf.copy_(dbuf, non_blocking=True))
            e1.record(stream)
            torch.cuda.synchronize()
            best[way] = min(best[way], e0.elapsed_time(e1))
    del hbuf, dbuf

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16" if bf16 else "f32", "data": "synthetic",
            "config": dict(workload_config(args.workload, cfg), N=N,
                           l2=f"inputs rotate over {n_sets} device copies, {n_sets * bytes_set / 1e6:.0f} MB "
                              f"> 2 x L2 ({l2 / 1e6:.0f} MB)",
                           step=("select_subtree, then " if use_pool else "given trees: ") + "tree_attention || " +
                                ("verify_sample" if sampling_mode else "verify_greedy") +
                                " (two streams; " + ("verify" if verify_on_main else "attention") +
                                (" on selection's stream with programmatic dependent launch)" if use_pool
                                 else " on the main stream)"),
                           parallelism=f"replicas x{world}",
                           sm_partition={"verify": sm_partition[0] or n_sm, "attention": sm_partition[1] or n_sm},
                           sm_partition_trials_us={
                               f"verify {v or n_sm} / attention {a or n_sm}, {'verify' if vm else 'attention'} "
                               f"on main": round(t * 1e3 / n_sets, 2) for ((v, a), vm), t in sorted(trial.items())},
                           attention_kernel=attn_name, attention_kv_splits=attn_splits),
            "path_gbs": bytes_set / (ms_per_step * 1e-3) / 1e9,
            "breakdown_us": br,
            "commit_bytes_per_launch": commit_bytes,
            "expand": {"rows": exp_rows, "m": exp_m, "bytes_per_launch": expand_bytes,
                       "gbs": expand_bytes / (br["expand"] * 1e-6) / 1e9},
            "roofline": roofline,
            "rooflines": rooflines,
            "cpu_baseline": cpu_base,
            "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                    "steps": e2e_steps, "ms_per_step": ms_e2e / e2e_steps,
                    "copied": "per round: " + ", ".join(pinned) + "; the prefix KV cache rows 0..P-1 stay on the "
                              "device across rounds; the next round's copies overlap this round's compute "
                              "(two device input sets)",
                    "copy_ms_per_step": ms_copy, "h2d_gbs": h2d / (ms_copy * 1e-3) / 1e9,
                    "copy_probe_gbs": {w: probe_bytes / (best[w] * 1e-3) / 1e9 for w in best}},
            "gpu_launches": launches_per_step * args.steps,
            "clocks": clocks,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def main(argv=None):
    args = parse_args(argv)
    if args.oracle_worker is not None:
        oracle_worker(args.oracle_worker, args.workload)
        return
    if args.impl == "reference":
        run_reference(args)
        return
    run_ours(args)


if __name__ == "__main__":
    main()
