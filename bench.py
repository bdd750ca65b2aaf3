"""Benchmark: µs per fused LM-head + Gumbel-max decode sample step on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--batch B] [--impl reference]

One step is one pass of the whole hot path over one batch: the fused Stage 1 (LM-head GEMM on
the tensor cores, transform, Philox noise, per-tile argmax; the [B, V] logits never reach
memory) and Stage 2 (per-row reduction of the tile candidates), both through the C ABI
``lms_lmhead_sample``.  The workload is the Qwen3-8B-shaped decode batch (D = 4096,
V = 151936, bf16 W ~ N(0, 0.02), H RMS-normalised N(0, 1), T = 0.7, per-row seeds, positions =
step), B = 64 by default: W (1.24 GB) is far larger than L2, so no flush is needed between steps.

Prints one JSON line.  `value` is µs per step (lower is better), `roofline` the achieved HBM
bandwidth of the step against the measured copy bandwidth, `e2e` the same metric with the
step's inputs copied from pinned host memory and the tokens copied back inside the timed
region, `cpu_baseline` the CPU oracle on a bounded slice of the same workload.  With
``--impl reference`` the CPU oracle itself is timed as the reference arm.
Multi-GPU (torchrun): every rank runs an independent replica; rank 0 prints the max over ranks.
"""
from __future__ import annotations

import argparse
import csv
import hashlib
import io
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "µs per decode sample step & achieved HBM GB/s vs peak, fused LM-head+Gumbel"
UNIT = "us/step"
TC_SOURCES = ["lm_head_gumbel_lmhead_gb300/csrc/lmhead_tc.cu",
              "lm_head_gumbel_lmhead_gb300/csrc/lms_device.cuh"]


def kernel_source_hash() -> str:
    h = hashlib.sha256()
    for p in TC_SOURCES:
        with open(os.path.join(ROOT, p), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def measured_peaks() -> dict:
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return {"hbm_gbs": float(d["hbm_gbs"]), "bf16_tflops": float(d["bf16_tflops"]),
                "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "source": "fallback"}


def recorded_traffic():
    """DRAM bytes per launch of the fused kernel from the committed ncu summary, if it was taken
    on the current kernel source (else None)."""
    p = os.path.join(ROOT, "profiles", "lmhead_tc_traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        d = json.load(f)
    if d.get("kernel_source_hash") != kernel_source_hash():
        return None
    return d


def algorithmic_bytes(B: int, D: int, V: int, n_tiles: int) -> int:
    """Bytes the method must move per step: W once, H once, the Stage-1 candidates written and
    read back, the per-row parameters (T, seed, position) and the tokens."""
    return V * D * 2 + B * D * 2 + 2 * B * n_tiles * 8 + B * 20 + B * 8


# ------------------------------------------------------------------------------------------
# distributed plumbing (replicas only; every rank runs the whole step on its own GPU)
# ------------------------------------------------------------------------------------------
def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    return int(os.environ.get("RANK", "0")), ws, int(os.environ.get("LOCAL_RANK", "0"))


def init_dist(backend: str):
    import torch.distributed as dist
    rank, ws, _ = dist_env()
    if ws > 1 and not dist.is_initialized():
        dist.init_process_group(backend=backend)
    return rank, ws


def barrier():
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized():
        dist.barrier()


def max_over_ranks(x: float, device=None) -> float:
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()):
        return x
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ------------------------------------------------------------------------------------------
# clocks during the timed region
# ------------------------------------------------------------------------------------------
class ClockSampler:
    FIELDS = ["timestamp", "clocks.sm", "clocks.max.sm", "power.draw",
              "clocks_event_reasons.hw_slowdown", "clocks_event_reasons.hw_thermal_slowdown",
              "clocks_event_reasons.sw_thermal_slowdown", "clocks_event_reasons.sw_power_cap"]

    def __init__(self, gpu_index: int):
        self.proc = None
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(gpu_index), "--query-gpu=" + ",".join(self.FIELDS),
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self, t0: float, t1: float) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        rows = []
        for r in csv.reader(io.StringIO(out)):
            if len(r) < len(self.FIELDS):
                continue
            try:
                ts = time.mktime(time.strptime(r[0].strip().split(".")[0], "%Y/%m/%d %H:%M:%S"))
                rows.append((ts, float(r[1]), float(r[2]), [x.strip() for x in r[4:8]]))
            except ValueError:
                continue
        inside = [x for x in rows if t0 - 1 <= x[0] <= t1 + 1]
        window = "timed" if inside else "warmup+timed"
        use = inside or rows
        if not use:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for x in use for i, v in enumerate(x[3]) if v == "Active"})
        return {"sm_mhz": statistics.median(x[1] for x in use), "sm_max_mhz": max(x[2] for x in use),
                "reasons": reasons, "samples": len(use), "window": window}


# ------------------------------------------------------------------------------------------
# the CPU oracle timed on a bounded slice (cpu_baseline leg and --impl reference)
# ------------------------------------------------------------------------------------------
def oracle_sample_time(w, v_slice: int, threads: int):
    """Seconds for the oracle's fused path on all B rows over the first v_slice vocabulary
    rows; scaled linearly to the full vocabulary by the caller."""
    import oracle
    W = w.W[:v_slice].contiguous()
    t0 = time.perf_counter()
    oracle.lmhead_sample(w.H, W, temperature=w.temperature.double().numpy(), seeds=w.seeds.numpy(),
                         positions=w.positions.numpy(), tile_v=128, threads=threads)
    return time.perf_counter() - t0


def cpu_baseline(w, target_s: float = 10.0):
    import oracle  # noqa: F401  (test infrastructure: CPU baseline only)
    threads = os.cpu_count() or 1
    v = 1024
    t = oracle_sample_time(w, v, threads)
    v2 = int(min(w.V, max(v, v * target_s / max(t, 1e-3))))
    v2 = max(128, v2 // 128 * 128)
    t2 = oracle_sample_time(w, v2, threads)
    us = t2 / v2 * w.V * 1e6
    return {"value": us, "unit": UNIT, "cores": threads, "kind": "oracle",
            "sample": f"B={w.B} rows x first {v2} of {w.V} vocabulary rows (D={w.D}), fp64 GEMM + "
                      f"Philox noise + argmax, {t2:.1f} s wall, scaled linearly to the full vocabulary"}


def run_reference(args):
    rank, ws = init_dist("gloo")
    if rank != 0:
        return
    from lm_head_gumbel_lmhead_gb300 import workloads
    w = workloads.qwen3_8b(args.batch, D=args.D, V=args.V)
    threads = os.cpu_count() or 1
    v_slice = args.ref_vslice
    for _ in range(args.warmup):
        oracle_sample_time(w, min(v_slice, 512), threads)
    times = [oracle_sample_time(w, v_slice, threads) for _ in range(args.steps)]
    us = statistics.mean(times) / v_slice * w.V * 1e6
    line = {"impl": "reference", "metric": METRIC, "value": us, "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": us / 1e3,
            "higher_is_better": False, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic",
            "config": {"workload": w.name, "B": w.B, "D": w.D, "V": w.V, "noise": "fp32",
                       "parallelism": "replicas"},
            "cpu_baseline": {"value": us, "unit": UNIT, "cores": threads, "kind": "oracle",
                             "sample": f"each step: B={w.B} rows x first {v_slice} of {w.V} "
                                       f"vocabulary rows, scaled linearly to the full vocabulary"},
            "e2e": {"value": us, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------------------------------
# the GPU arm
# ------------------------------------------------------------------------------------------
def run_gpu(args):
    import torch

    import lm_head_gumbel_lmhead_gb300 as lms
    from lm_head_gumbel_lmhead_gb300 import workloads

    rank, ws = init_dist("nccl")
    _, _, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    B, D, V = args.batch, args.D, args.V
    w = workloads.qwen3_8b(B, D=D, V=V)
    H, W = w.H.to(dev), w.W.to(dev)
    T, seeds = w.temperature.to(dev), w.seeds.to(dev)
    n_steps = args.warmup + args.steps
    # positions = step: one row of positions per step, made before timing
    pos_all = torch.arange(n_steps, dtype=torch.int64, device=dev)[:, None].expand(n_steps, B).contiguous()
    tv, nt, ws_bytes, path = lms.tile_info(lms.OP_LMHEAD, B, D, V)
    workspace = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
    out = torch.empty(B, dtype=torch.int64, device=dev)
    stream = torch.cuda.current_stream(dev)
    launches_per_step = (1 + (B - 1) // 256 if path == lms.PATH_TCGEN05 else 1) + 1

    def step(i):
        lms.lmhead_sample(H, W, temperature=T, seeds=seeds, positions=pos_all[i], out=out,
                          workspace=workspace)

    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize(dev)
    sampler = ClockSampler(local) if rank == 0 else None
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps + 1)]
    barrier()
    torch.cuda.synchronize(dev)
    t0 = time.time()
    ev[0].record(stream)
    for k in range(args.steps):
        step(args.warmup + k)
        ev[k + 1].record(stream)
    torch.cuda.synchronize(dev)
    t1 = time.time()
    barrier()
    per_step_ms = [ev[k].elapsed_time(ev[k + 1]) for k in range(args.steps)]
    total_ms = ev[0].elapsed_time(ev[args.steps])
    clocks = sampler.stop(t0, t1) if sampler else None
    ms_per_step = max_over_ranks(total_ms / args.steps, dev)
    us = ms_per_step * 1e3

    # e2e: the step's inputs from pinned host memory, the tokens back to pinned host memory
    H_h = w.H.pin_memory()
    T_h, seeds_h = w.temperature.pin_memory(), w.seeds.pin_memory()
    pos_h = pos_all.cpu().pin_memory()
    out_h = torch.empty(B, dtype=torch.int64).pin_memory()
    H_d, T_d, s_d = torch.empty_like(H), torch.empty_like(T), torch.empty_like(seeds)
    p_d = torch.empty(B, dtype=torch.int64, device=dev)

    def e2e_step(i):
        H_d.copy_(H_h, non_blocking=True)
        T_d.copy_(T_h, non_blocking=True)
        s_d.copy_(seeds_h, non_blocking=True)
        p_d.copy_(pos_h[i], non_blocking=True)
        lms.lmhead_sample(H_d, W, temperature=T_d, seeds=s_d, positions=p_d, out=out,
                          workspace=workspace)
        out_h.copy_(out, non_blocking=True)

    for i in range(args.warmup):
        e2e_step(i)
    torch.cuda.synchronize(dev)
    barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for k in range(args.steps):
        e2e_step(args.warmup + k)
    e1.record(stream)
    torch.cuda.synchronize(dev)
    barrier()
    e2e_us = max_over_ranks(e0.elapsed_time(e1) / args.steps, dev) * 1e3
    h2d = B * D * 2 + B * 4 + B * 8 + B * 8
    d2h = B * 8

    if rank != 0:
        return
    peaks = measured_peaks()
    alg = algorithmic_bytes(B, D, V, nt)
    achieved = alg / (us * 1e-6) / 1e9
    traffic = recorded_traffic()
    roofline = {"bound": "hbm", "achieved": round(achieved, 1), "peak": peaks["hbm_gbs"],
                "unit": "GB/s", "frac": round(achieved / peaks["hbm_gbs"], 4),
                "traffic": traffic["dram_bytes_per_launch"] if traffic else None,
                "peak_source": peaks["source"] + " (MEASURED_PEAKS.json hbm_gbs, burst copy)",
                "kernel": "lmhead_tc_kernel + stage2_kernel (one step, CUDA events)",
                "algorithmic_bytes": alg}
    line = {"metric": METRIC, "value": round(us, 2), "unit": UNIT, "n_gpus": ws,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_per_step, 5),
            "higher_is_better": False, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic",
            "config": {"workload": w.name, "B": B, "D": D, "V": V, "noise": "fp32",
                       "path": {1: "gemv", 2: "tcgen05"}[path], "tile_v": tv,
                       "l2": "inputs larger than L2 (W is %.2f GB), no flush" % (V * D * 2 / 1e9),
                       "parallelism": "replicas" if ws > 1 else "single-gpu"},
            "hbm_gbs": round(achieved, 1), "samples_per_s": round(B / (us * 1e-6), 1),
            "p50_us": round(statistics.median(per_step_ms) * 1e3, 2),
            "p10_us": round(sorted(per_step_ms)[len(per_step_ms) // 10] * 1e3, 2),
            "p90_us": round(sorted(per_step_ms)[(len(per_step_ms) * 9) // 10] * 1e3, 2),
            "roofline": roofline, "clocks": clocks,
            "e2e": {"value": round(e2e_us, 2), "unit": UNIT, "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h},
            "gpu_launches": launches_per_step * args.steps}
    if not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(w, args.cpu_seconds)
    print(json.dumps(line), flush=True)


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=25)
    ap.add_argument("--batch", type=int, default=64)
    ap.add_argument("--D", type=int, default=4096)
    ap.add_argument("--V", type=int, default=151936)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--ref-vslice", type=int, default=4096)
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.impl == "reference":
        run_reference(args)
    else:
        run_gpu(args)


if __name__ == "__main__":
    main()
