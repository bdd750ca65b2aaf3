"""Benchmark: µs per fused LM-head + Gumbel-max decode sample step on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--batch B]
                    [--impl reference]

One step is one pass of the whole hot path over one batch. For the fused workloads that means the
fused Stage 1 and then Stage 2, both through the C ABI ``lms_lmhead_sample``:

- Stage 1 runs the LM-head GEMM on the tensor cores, applies the transform, draws the Philox
  noise and takes the per-tile argmax. The [B, V] logits never reach memory.
- Stage 2 reduces each row's tile candidates to one token.

Workloads (synthetic, seeded; the shapes of the FlashSampling page's measurements):

- ``qwen3-8b`` (default; B = 64): D = 4096, V = 151936. W is bf16 ~ N(0, 0.02) and H is
  RMS-normalised N(0, 1). Noise is fp32, T = 0.7 with per-row seeds, and positions = step.
- ``llama3-hetero`` (B = 64): D = 4096, V = 128256. Rows mix T ~ U[0.3, 1.2] with 8 greedy
  rows. It adds an fp32 bias and a 90% -inf mask on half the rows.
- ``large-vocab`` (B in 128/256/512): D = 8192, V = 262144, wide noise.
- ``logits``: ``lms_sample_from_logits`` over materialised N(0, 4) logits, V = 131072.
- ``noise``: ``lms_philox_fill_noise`` of Gumbel noise, B x V float32.
- ``qwen3-8b-fp8``: the Qwen3-8B shape through ``lms_lmhead_sample_fp8``. W is offline-quantised
  to E4M3 with per-row scales, and H is quantised per row on the GPU each step (W8A8).
- ``filtered``: ``lms_sample_from_logits_filtered`` with top-k 50 and top-p 0.9 at T = 0.7 over
  bf16 logits, V = 131072 (the Megatron-LM PR's filter settings).
- ``qwen3-8b-mxfp4``: the Qwen3-8B shape through ``lms_lmhead_sample_mxfp4``. W is offline-quantised
  to MXFP4 (E2M1 codes with one UE8M0 scale per block of 32), H stays bf16 (W4A16).
- ``qwen3-8b-topk``: the Qwen3-8B shape through ``lms_lmhead_sample_topk`` (Gumbel-top-k: k
  draws without replacement per row, k = ``--topk``, default 8).
- ``verify``: ``lms_verify_from_logits`` (speculative-decoding verification) over bf16 target
  [B, k+1, V] and draft [B, k, V] logits, V = 128256 (the spec-decode-ops page's latency
  vocabulary), k = ``--spec-k`` (default 4), T = 0.8, draft tokens drawn from the draft.

The fused workloads stream W of 1.05–4.3 GB, larger than L2, so they need no flush. The
materialised-logits workloads write a 256 MB buffer between timed steps whenever their inputs are
under 512 MB (``--l2-flush auto``), and time each step's own events.

The script prints one JSON line:

- `value`: µs per step (lower is better).
- `roofline`: the step's algorithmic bytes (or flops, where the tensor floor dominates) over its
  event time, against ``MEASURED_PEAKS.json``.
- `e2e`: the same metric with the step's inputs copied from pinned host memory and the tokens
  copied back, inside the timed region.
- `cpu_baseline`: the CPU oracle on a bounded slice of the same workload.

With ``--impl reference`` the CPU oracle itself is timed as the reference arm. Under torchrun every
rank runs an independent replica, and rank 0 prints the max over ranks.
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
              "lm_head_gumbel_lmhead_gb300/csrc/tcgen05_common.cuh",
              "lm_head_gumbel_lmhead_gb300/csrc/lms_device.cuh"]
# the Stage-1 kernel of each fused workload and its sources: the single-group kernel, the row-group
# kernel (race workloads above 256 rows) and the MXFP4 kernel
STAGE1_SOURCES = {
    "tc": TC_SOURCES,
    "rows": ["lm_head_gumbel_lmhead_gb300/csrc/lmhead_tc_rows.cu",
             "lm_head_gumbel_lmhead_gb300/csrc/tcgen05_common.cuh",
             "lm_head_gumbel_lmhead_gb300/csrc/lms_device.cuh"],
    "mx": ["lm_head_gumbel_lmhead_gb300/csrc/lmhead_mx.cu",
           "lm_head_gumbel_lmhead_gb300/csrc/tcgen05_common.cuh",
           "lm_head_gumbel_lmhead_gb300/csrc/lms_device.cuh"],
}
FUSED = ("qwen3-8b", "llama3-hetero", "large-vocab", "qwen3-8b-fp8", "qwen3-8b-topk", "qwen3-8b-mxfp4")


def stage1_kind(workload: str, B: int) -> str:
    if workload == "qwen3-8b-mxfp4":
        return "mx"
    if workload in ("qwen3-8b", "llama3-hetero", "large-vocab") and B > 256:
        return "rows"
    return "tc"


def kernel_source_hash(kind: str = "tc") -> str:
    h = hashlib.sha256()
    for p in STAGE1_SOURCES[kind]:
        with open(os.path.join(ROOT, p), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def measured_peaks() -> dict:
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return {"hbm_gbs": float(d["hbm_gbs"]), "bf16_tflops": float(d["bf16_tflops"]),
                "bf16_tflops_sustained": float(d.get("bf16_tflops_sustained", d["bf16_tflops"])),
                "sm_max_mhz": float(d.get("sm_max_mhz", 2070.0)), "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
            "sm_max_mhz": 2070.0, "source": "fallback"}


def recorded_traffic(workload: str, B: int):
    """DRAM bytes per launch of the fused Stage-1 kernel from the committed ncu summary, if it was
    taken for this workload on the current sources of that kernel (else None)."""
    p = os.path.join(ROOT, "profiles", "lmhead_tc_traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        d = json.load(f)
    rec = d.get(f"{workload}/B={B}")
    if rec is None or rec.get("kernel_source_hash") != kernel_source_hash(stage1_kind(workload, B)):
        return None
    return rec


ALU_SOURCES = {"logits": ["lm_head_gumbel_lmhead_gb300/csrc/logits_sample.cu",
                          "lm_head_gumbel_lmhead_gb300/csrc/stage2.cu",
                          "lm_head_gumbel_lmhead_gb300/csrc/lms_device.cuh"],
               "noise": ["lm_head_gumbel_lmhead_gb300/csrc/noise_fill.cu",
                         "lm_head_gumbel_lmhead_gb300/csrc/lms_device.cuh"]}


def alu_source_hash(workload: str) -> str:
    h = hashlib.sha256()
    for p in ALU_SOURCES[workload]:
        with open(os.path.join(ROOT, p), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def recorded_instructions(key: str, workload: str):
    """Warp instructions per step of an ALU-bound workload from the committed ncu record, if it
    was taken on the current kernel sources (else None)."""
    p = os.path.join(ROOT, "profiles", "alu_instructions.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        d = json.load(f)
    rec = d.get(key)
    if rec is None or rec.get("source_hash") != alu_source_hash(workload):
        return None
    return rec


def algorithmic_bytes(B: int, D: int, V: int, n_tiles: int, bias: bool = False,
                      mask: bool = False) -> int:
    """Bytes the fused method must move per step: W once, H once, the Stage-1 candidates written
    and read back, the per-row parameters (T, seed, position), the tokens, and the optional bias
    and mask rows."""
    b = V * D * 2 + B * D * 2 + 2 * B * n_tiles * 8 + B * 20 + B * 8
    if bias:
        b += B * V * 4
    if mask:
        b += B * ((V + 31) // 32) * 4
    return b


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
    """nvidia-smi sampling the SM clock, its maximum, power and the throttle reasons every 50 ms,
    read on a thread as the lines arrive (each stamped with the host time it came in).  Started
    before the workload is set up; the caller waits for the first sample before it times."""
    FIELDS = ["clocks.sm", "clocks.max.sm", "power.draw",
              "clocks_event_reasons.hw_slowdown", "clocks_event_reasons.hw_thermal_slowdown",
              "clocks_event_reasons.sw_thermal_slowdown", "clocks_event_reasons.sw_power_cap"]
    NAMES = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]

    def __init__(self, gpu_index: int):
        import threading
        self.rows = []
        self.first = threading.Event()
        self.proc = None
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(gpu_index), "--query-gpu=" + ",".join(self.FIELDS),
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True, bufsize=1)
        except (OSError, FileNotFoundError):
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            r = [x.strip() for x in line.split(",")]
            if len(r) < len(self.FIELDS):
                continue
            try:
                self.rows.append((time.time(), float(r[0]), float(r[1]), r[3:7]))
            except ValueError:
                continue
            self.first.set()

    def wait_first(self, timeout_s: float = 15.0):
        if self.proc is not None:
            self.first.wait(timeout_s)

    def stop(self, t0: float, t1: float) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            self.proc.wait()
        self.thread.join(timeout=5)
        rows = list(self.rows)
        # samples that came in during the timed region (a line arrives within one period of its
        # sample); a short region may hold none, then those within a second of it
        use = [x for x in rows if t0 <= x[0] <= t1 + 0.05]
        window = "timed"
        if not use:
            use = [x for x in rows if t0 - 1.0 <= x[0] <= t1 + 1.0]
            window = "within 1 s of the timed region (the region is shorter than the sampling period)"
        if not use:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
        reasons = sorted({self.NAMES[i] for x in use for i, v in enumerate(x[3]) if v == "Active"})
        return {"sm_mhz": statistics.median(x[1] for x in use), "sm_max_mhz": max(x[2] for x in use),
                "reasons": reasons, "samples": len(use), "window": window}


# ------------------------------------------------------------------------------------------
# workloads
# ------------------------------------------------------------------------------------------
def make_workload(name: str, B: int, D: int, V: int):
    from lm_head_gumbel_lmhead_gb300 import workloads
    if name in ("qwen3-8b", "qwen3-8b-fp8", "qwen3-8b-topk", "qwen3-8b-mxfp4"):
        return workloads.qwen3_8b(B, D=D or 4096, V=V or 151936)
    if name == "llama3-hetero":
        return workloads.llama3_hetero(B, D=D or 4096, V=V or 128256)
    if name == "large-vocab":
        return workloads.large_vocab(B, D=D or 8192, V=V or 262144)
    raise ValueError(name)


def default_batch(name: str) -> int:
    return {"large-vocab": 256, "logits": 64, "noise": 64, "filtered": 64, "verify": 64}.get(name, 64)


# ------------------------------------------------------------------------------------------
# the CPU oracle timed on a bounded slice (cpu_baseline leg and --impl reference)
# ------------------------------------------------------------------------------------------
def _orc_kw(w, v_slice):
    mask = None if w.mask is None else w.mask.numpy().view("uint32")
    bias = None if w.bias is None else w.bias[:, :v_slice].double().numpy()
    if mask is not None:
        mask = mask[:, : (v_slice + 31) // 32]
    return dict(temperature=w.temperature.double().numpy(), seeds=w.seeds.numpy(),
                positions=w.positions.numpy(), bias=bias, mask=mask, base_seed=w.base_seed,
                offset=w.offset, wide=w.noise_mode == 1)


def oracle_sample_time(w, v_slice: int, threads: int):
    """Seconds for the oracle's fused path on all B rows over the first v_slice vocabulary
    rows; scaled linearly to the full vocabulary by the caller."""
    import oracle
    W = w.W[:v_slice].contiguous()
    t0 = time.perf_counter()
    oracle.lmhead_sample(w.H, W, tile_v=128, threads=threads, **_orc_kw(w, v_slice))
    return time.perf_counter() - t0


def oracle_logits_time(logits, v_slice: int, threads: int):
    import oracle
    import numpy as np
    B = logits.shape[0]
    y = logits[:, :v_slice].double().numpy()
    t0 = time.perf_counter()
    oracle.sample_from_logits(y, temperature=np.full(B, 0.7), seeds=np.arange(B) + 1000,
                              positions=np.zeros(B, np.int64), threads=threads)
    return time.perf_counter() - t0


def oracle_verify_time(tgt, dft, tokens, rows: int):
    """Seconds for the oracle's verification of the first `rows` batch rows (full vocabulary)."""
    import numpy as np
    import oracle
    t = tgt[:rows].double().numpy()
    d = dft[:rows].double().numpy()
    x = tokens[:rows].numpy()
    t0 = time.perf_counter()
    oracle.verify_from_logits(t, d, x, temperature=np.full(rows, 0.8), seeds=np.arange(rows) + 1000,
                              positions=np.zeros(rows, np.int64))
    return time.perf_counter() - t0


def _scaled_oracle_us(w, threads: int, target_s: float):
    """(us per full step, vocabulary rows timed, seconds) for the oracle's fused path on all B
    rows: the first v rows of the vocabulary, v sized for about target_s seconds (the whole
    vocabulary when it fits), scaled linearly to the full vocabulary."""
    v = min(1024, w.V)
    t = oracle_sample_time(w, v, threads)
    v2 = int(min(w.V, max(v, v * target_s / max(t, 1e-3))))
    v2 = w.V if v2 >= w.V else max(128, v2 // 128 * 128)
    t2 = oracle_sample_time(w, v2, threads)
    return t2 / v2 * w.V * 1e6, v2, t2


def cpu_baseline(w, target_s: float = 10.0):
    """The oracle on the host cores: all threads (the headline figure) and one thread, on a
    bounded vocabulary slice of this workload, plus the small workloads it runs in full."""
    import oracle  # noqa: F401  (test infrastructure: CPU baseline only)
    from lm_head_gumbel_lmhead_gb300 import workloads
    threads = os.cpu_count() or 1
    us, v2, t2 = _scaled_oracle_us(w, threads, target_s)
    us1, v1, t1 = _scaled_oracle_us(w, 1, target_s / 4)
    full = {}
    for name, wl in (("tiny B=4 D=512 V=8192", workloads.tiny()),
                     ("qwen3-8b B=1", workloads.qwen3_8b(1)),
                     ("qwen3-8b B=8", workloads.qwen3_8b(8))):
        if wl.D != w.D and name.startswith("qwen"):
            continue
        full[name] = {"us_per_step_all_threads": round(oracle_sample_time(wl, wl.V, threads) * 1e6, 1)}
    return {"value": us, "unit": UNIT, "cores": threads, "kind": "oracle",
            "sample": f"B={w.B} rows x first {v2} of {w.V} vocabulary rows (D={w.D}), fp64 GEMM + "
                      f"Philox noise + argmax, {t2:.1f} s wall on {threads} threads"
                      + ("" if v2 == w.V else ", scaled linearly to the full vocabulary"),
            "single_thread": {"value": us1, "unit": UNIT, "cores": 1,
                              "sample": f"B={w.B} rows x first {v1} of {w.V} vocabulary rows, "
                                        f"{t1:.1f} s wall, scaled linearly to the full vocabulary"},
            "full_workloads": full}


def run_reference(args):
    rank, ws = init_dist("gloo")
    if rank != 0:
        return
    if args.workload not in FUSED:
        print(json.dumps({"impl": "reference", "unavailable":
                          f"the reference arm times the oracle's fused path; workload {args.workload} has none"}))
        return
    w = make_workload(args.workload, args.batch, args.D, args.V)
    threads = os.cpu_count() or 1
    # each step runs the whole workload when all steps fit in the budget, else the first v_slice
    # vocabulary rows, scaled linearly (the slice and its measured time are in the line)
    probe_v = min(2048, w.V)
    probe = oracle_sample_time(w, probe_v, threads)
    est_full = probe / probe_v * w.V
    v_slice = w.V
    if est_full * args.steps > args.ref_budget_s:
        v_slice = int(w.V * args.ref_budget_s / (est_full * args.steps))
        v_slice = max(128, min(w.V, v_slice // 128 * 128))
    for _ in range(args.warmup):
        oracle_sample_time(w, min(v_slice, 512), threads)
    times = [oracle_sample_time(w, v_slice, threads) for _ in range(args.steps)]
    step_s = statistics.mean(times)
    us = step_s / v_slice * w.V * 1e6
    config = {"workload": w.name, "B": w.B, "D": w.D, "V": w.V,
              "noise": "wide53" if w.noise_mode else "fp32", "tile_v": 128,
              "parallelism": "replicas" if ws > 1 else "single-gpu"}
    sample = (f"each step: B={w.B} rows x all {w.V} vocabulary rows" if v_slice == w.V else
              f"each step: B={w.B} rows x first {v_slice} of {w.V} vocabulary rows, scaled linearly "
              f"to the full vocabulary")
    line = {"impl": "reference", "metric": METRIC, "value": us, "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": us / 1e3,
            "higher_is_better": False, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": config,
            "measured_seconds_per_step": step_s, "vocab_rows_per_step": v_slice,
            "extrapolated_from_v": None if v_slice == w.V else v_slice,
            "cpu_baseline": {"value": us, "unit": UNIT, "cores": threads, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": us, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------------------------------
# the GPU arm
# ------------------------------------------------------------------------------------------
def _time_steps(step, n_warm, n_steps, dev, stream, first_index=0, flush=None):
    import torch
    for i in range(n_warm):
        step(first_index + i)
    torch.cuda.synchronize(dev)
    if flush is not None:
        # L2 flushed before every timed step, outside its own pair of events
        e0 = [torch.cuda.Event(enable_timing=True) for _ in range(n_steps)]
        e1 = [torch.cuda.Event(enable_timing=True) for _ in range(n_steps)]
        barrier()
        torch.cuda.synchronize(dev)
        t0 = time.time()
        for k in range(n_steps):
            flush()
            e0[k].record(stream)
            step(first_index + n_warm + k)
            e1[k].record(stream)
        torch.cuda.synchronize(dev)
        t1 = time.time()
        barrier()
        per_ms = [e0[k].elapsed_time(e1[k]) for k in range(n_steps)]
        return statistics.mean(per_ms), per_ms, t0, t1
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(n_steps + 1)]
    barrier()
    torch.cuda.synchronize(dev)
    t0 = time.time()
    ev[0].record(stream)
    for k in range(n_steps):
        step(first_index + n_warm + k)
        ev[k + 1].record(stream)
    torch.cuda.synchronize(dev)
    t1 = time.time()
    barrier()
    per_ms = [ev[k].elapsed_time(ev[k + 1]) for k in range(n_steps)]
    return ev[0].elapsed_time(ev[n_steps]) / n_steps, per_ms, t0, t1


def run_gpu(args):
    import torch

    import lm_head_gumbel_lmhead_gb300 as lms
    from lm_head_gumbel_lmhead_gb300 import workloads

    rank, ws = init_dist("nccl")
    _, _, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    stream = torch.cuda.current_stream(dev)
    n_steps = args.warmup + args.steps
    peaks = measured_peaks()
    B = args.batch
    extra = {}
    # the clock sampler starts before the workload is set up, so that it runs by the time the
    # timed region starts, and keeps sampling through the e2e phase
    sampler = ClockSampler(local) if rank == 0 else None
    alu_key = None                                 # key of the ALU-bound workloads' ncu record

    if args.workload in FUSED:
        w = make_workload(args.workload, B, args.D, args.V)
        D, V = w.D, w.V
        H, W = w.H.to(dev), w.W.to(dev)
        T, seeds = w.temperature.to(dev), w.seeds.to(dev)
        bias = None if w.bias is None else w.bias.to(dev)
        mask = None if w.mask is None else w.mask.to(dev)
        # positions advance with the step: one row per step, made before timing
        pos_all = (w.positions[None, :] + torch.arange(n_steps)[:, None]).contiguous().to(dev)
        fp8 = args.workload == "qwen3-8b-fp8"
        mx = args.workload == "qwen3-8b-mxfp4"
        topk = args.topk if args.workload == "qwen3-8b-topk" else 0
        tv, nt, ws_bytes, path = lms.tile_info(lms.OP_LMHEAD_FP8 if fp8 else lms.OP_LMHEAD, B, D, V)
        if topk:
            ws_bytes = lms.lib().lms_workspace_bytes_topk(B, V, topk)
        workspace = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
        out = torch.empty((B, topk) if topk else (B,), dtype=torch.int64, device=dev)
        scores_k = torch.empty(B, topk, dtype=torch.float32, device=dev) if topk else None
        wide = w.noise_mode == 1
        kw = dict(temperature=T, seeds=seeds, bias=bias, mask=mask, base_seed=w.base_seed,
                  offset=w.offset, wide=wide, out=out, workspace=workspace)
        path_req = {"auto": lms.PATH_AUTO, "gemv": lms.PATH_GEMV, "tcgen05": lms.PATH_TCGEN05}[args.path]
        if path_req != lms.PATH_AUTO:
            if fp8 or topk or mx:
                raise SystemExit("--path applies to the bf16 race workloads")
            path = path_req
        launches_per_step = (1 + (B - 1) // 256 if path == lms.PATH_TCGEN05 else 1) + 1
        if fp8:
            W8_h, wsc_h = workloads.quantize_weight_e4m3(w.W)
            W8, wsc = W8_h.to(dev), wsc_h.to(dev)
            W = None                               # the bf16 copy is not needed on the device
            launches_per_step += 1                 # the activation quantisation

            def step(i):
                lms.lmhead_sample_fp8(H, W8, wsc, positions=pos_all[i], **kw)
        elif mx:
            W4_h, S4_h = workloads.quantize_weight_mxfp4(w.W)
            Wt = lms.mxfp4_pack(W4_h.to(dev), S4_h.to(dev))      # the one-time tiling
            W = None                               # the bf16 copy is not needed on the device

            def step(i):
                lms.lmhead_sample_mxfp4(H, Wt, V, positions=pos_all[i], **kw)
        elif topk:
            def step(i):
                lms.lmhead_sample_topk(H, W, topk, positions=pos_all[i], scores=scores_k, **kw)
        else:
            def step(i):
                lms.lmhead_sample(H, W, positions=pos_all[i], path=path, **kw)

        alg = algorithmic_bytes(B, D, V, nt, bias is not None, mask is not None)
        if fp8:
            # W at one byte per weight plus its row scales; H read once, its E4M3 copy written
            # and read once
            alg = alg - V * D * 2 + V * D + V * 4 + 2 * B * D
        if mx:
            # W at half a byte per weight plus one scale byte per block of 32
            alg = alg - V * D * 2 + V * D // 2 + V * D // 32
        if topk:
            # the tiles' ordered k-lists written and read instead of one candidate each, and k
            # indices and scores per row out
            alg = alg - 2 * B * nt * 8 - B * 8 + 2 * B * nt * topk * 8 + B * topk * 12
        flops = 2 * B * V * D
        config = {"workload": w.name + (" fp8-e4m3 W8A8" if fp8 else "") + (" mxfp4 W4A16" if mx else "") +
                  (f" Gumbel-top-{topk}" if topk else ""), "B": B, "D": D, "V": V,
                  "noise": "wide53" if wide else "fp32",
                  "path": {1: "gemv", 2: "tcgen05"}[path], "tile_v": tv,
                  "l2": "inputs larger than L2 (W is %.2f GB), no flush" % (V * D * (1 if fp8 else 0.53125 if mx else 2) / 1e9)}
        kernel = ("quantize_rows_e4m3_kernel + " if fp8 else "") + \
            ("lmhead_tc_kernel (top-k epilogue) + stage2_topk_row (stage2_topk_part + stage2_topk_final above "
             "1024 lists a row)" if topk else
             "lmhead_mx_kernel + stage2_kernel" if mx else
             "lmhead_tc_rows_kernel (row groups) + stage2_kernel" if path == 2 and B > 256 else
             "lmhead_tc_kernel + stage2_kernel") + " (one step, CUDA events)"
    elif args.workload == "logits":
        V = args.V or 131072
        D = 0
        dt = torch.bfloat16 if args.logits_dtype == "bf16" else torch.float32
        logits = workloads.logits_normal(B, V, std=2.0, seed=5, dtype=dt).to(dev)
        T = torch.full((B,), 0.7, device=dev)
        seeds = 1000 + torch.arange(B, dtype=torch.int64, device=dev)
        pos_all = torch.arange(n_steps, dtype=torch.int64)[:, None].expand(n_steps, B).contiguous().to(dev)
        tv, nt, ws_bytes, _ = lms.tile_info(lms.OP_LOGITS, B, 0, V, args.tile_v)
        workspace = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
        out = torch.empty(B, dtype=torch.int64, device=dev)
        launches_per_step = 2

        def step(i):
            lms.sample_from_logits(logits, temperature=T, seeds=seeds, positions=pos_all[i], out=out,
                                   workspace=workspace, tile_v=args.tile_v)

        alg = B * V * logits.element_size() + 2 * B * nt * 8 + B * 28
        flops = 0
        config = {"workload": f"sample_from_logits B={B} V={V} {args.logits_dtype} logits ~ N(0, 4)",
                  "B": B, "V": V, "noise": "fp32", "tile_v": tv,
                  "l2": "inputs %s L2 (%.0f MB)" % ("larger than" if alg > 130e6 else "within", alg / 1e6)}
        kernel = "logits_stage1_kernel + stage2_kernel (one step, CUDA events)"
        alu_key = f"logits/B={B}/V={V}/{args.logits_dtype}"
    elif args.workload == "filtered":
        V = args.V or 131072
        D = 0
        logits = workloads.logits_normal(B, V, std=2.0, seed=6, dtype=torch.bfloat16).to(dev)
        T = torch.full((B,), 0.7, device=dev)
        seeds = 1000 + torch.arange(B, dtype=torch.int64, device=dev)
        top_k = torch.full((B,), 50, dtype=torch.int32, device=dev)
        top_p = torch.full((B,), 0.9, device=dev)
        pos_all = torch.arange(n_steps, dtype=torch.int64)[:, None].expand(n_steps, B).contiguous().to(dev)
        out = torch.empty(B, dtype=torch.int64, device=dev)
        launches_per_step = 1

        def step(i):
            lms.sample_from_logits_filtered(logits, temperature=T, seeds=seeds, positions=pos_all[i],
                                            top_k=top_k, top_p=top_p, out=out)

        alg = B * V * 2 + B * 44
        flops = 0
        config = {"workload": f"filtered sample_from_logits top-k 50 top-p 0.9 T 0.7 B={B} V={V} bf16",
                  "B": B, "V": V, "noise": "fp32",
                  "l2": "inputs %s L2 (%.0f MB)" % ("larger than" if alg > 130e6 else "within", alg / 1e6)}
        kernel = "filtered_race_kernel (one launch per step)"
    elif args.workload == "verify":
        V = args.V or 128256
        D = 0
        k = args.spec_k
        dt = torch.bfloat16 if args.logits_dtype == "bf16" else torch.float32
        tgt_h, dft_h = workloads.spec_logits(B, k, V, seed=7, dtype=dt)
        tgt, dft = tgt_h.to(dev), dft_h.to(dev)
        T = torch.full((B,), 0.8, device=dev)
        seeds = 1000 + torch.arange(B, dtype=torch.int64, device=dev)
        # positions advance by k + 1 per step; draft tokens drawn from the draft at T (setup)
        pos_all = (torch.arange(n_steps, dtype=torch.int64)[:, None] * (k + 1)).expand(n_steps, B) \
            .contiguous().to(dev)
        gen = torch.Generator(device=dev).manual_seed(5)
        pd = torch.softmax(dft.float() / 0.8, dim=-1).reshape(B * k, V)
        tokens = torch.multinomial(pd, 1, generator=gen).reshape(B, k).contiguous()
        del pd
        ws_bytes = lms.lib().lms_workspace_bytes_verify(B, k, V)
        workspace = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
        acc = torch.empty(B, dtype=torch.int64, device=dev)
        out = torch.empty(B, k + 1, dtype=torch.int64, device=dev)
        launches_per_step = 4

        def step(i):
            lms.verify_from_logits(tgt, dft, tokens, temperature=T, seeds=seeds, positions=pos_all[i],
                                   accept_len=acc, out=out, workspace=workspace)

        esz = tgt.element_size()
        # every logit read once; draft tokens and row parameters in; accept_len and k + 1 tokens out
        alg = (2 * k + 1) * B * V * esz + B * k * 8 + B * 20 + B * (k + 2) * 8
        flops = 0
        config = {"workload": f"verify_from_logits B={B} k={k} V={V} {args.logits_dtype} logits, "
                              f"draft corr 0.8, T 0.8", "B": B, "k": k, "V": V, "noise": "fp32"}
        kernel = "verify_partials + verify_decide + verify_race + verify_finalize (one step, CUDA events)"
    elif args.workload == "noise":
        V = args.V or 151936
        D = 0
        seeds = 1000 + torch.arange(B, dtype=torch.int64, device=dev)
        pos_all = torch.arange(n_steps, dtype=torch.int64)[:, None].expand(n_steps, B).contiguous().to(dev)
        g = torch.empty(B, V, dtype=torch.float32, device=dev)
        launches_per_step = 1

        def step(i):
            lms.philox_fill_noise(B, V, kind="gumbel", seeds=seeds, positions=pos_all[i], out=g)

        alg = B * V * 4 + B * 16
        flops = 0
        config = {"workload": f"philox_fill_noise gumbel B={B} V={V}", "B": B, "V": V,
                  "noise": "fp32", "l2": "output %.0f MB" % (alg / 1e6)}
        kernel = "noise_fill_kernel (one launch per step)"
        alu_key = f"noise/B={B}/V={V}"
    else:
        raise SystemExit(f"unknown workload {args.workload}")

    flush = None
    if args.workload not in FUSED and (args.l2_flush == "on" or (args.l2_flush == "auto" and alg < 512e6)):
        flush_buf = torch.empty(256 << 20, dtype=torch.uint8, device=dev)

        def flush():
            flush_buf.fill_(1)
        config["l2"] = "inputs %.0f MB; a 256 MB buffer written between timed steps" % (alg / 1e6)
    elif "l2" not in config:
        config["l2"] = "inputs %.0f MB, larger than L2, no flush" % (alg / 1e6)
    if sampler is not None:
        sampler.wait_first()
    avg_ms, per_ms, t0, t1 = _time_steps(step, args.warmup, args.steps, dev, stream, flush=flush)
    ms_per_step = max_over_ranks(avg_ms, dev)
    us = ms_per_step * 1e3

    e2e = None
    if args.workload in FUSED:
        # e2e: the step's per-request inputs from pinned host memory, the tokens back to pinned
        # host memory; W is a resident weight.  The inputs of a step (H, T, seeds, positions and
        # the optional bias and mask) sit in one pinned staging block and go over in one copy.
        # The copies run on two copy streams, one per direction, so that step i+1's inputs go
        # over while step i's kernels run and step i's tokens come back while step i+1's run.
        # Device inputs and outputs are double-buffered; events order every reuse.
        host = {"H": w.H, "T": w.temperature, "seeds": w.seeds, "positions": w.positions}
        if w.bias is not None:
            host["bias"] = w.bias
        if w.mask is not None:
            host["mask"] = w.mask
        offs, total = {}, 0
        for k, v in host.items():
            offs[k] = total
            total += (v.numel() * v.element_size() + 255) // 256 * 256
        ring = 4
        stage = [torch.empty(total, dtype=torch.uint8).pin_memory() for _ in range(ring)]

        def view(buf, k):
            v = host[k]
            n = v.numel() * v.element_size()
            return buf[offs[k]:offs[k] + n].view(v.dtype).view(v.shape)

        for blk in stage:
            for k, v in host.items():
                view(blk, k).copy_(v)
        h2d_stream = torch.cuda.Stream(dev)
        d2h_stream = torch.cuda.Stream(dev)
        h2d_done = [torch.cuda.Event() for _ in range(ring)]      # pinned block i % ring read
        dblk = [torch.empty(total, dtype=torch.uint8, device=dev) for _ in range(2)]
        devb = [{k: view(b, k) for k in host} for b in dblk]
        outs = [torch.empty_like(out) for _ in range(2)]
        ready = [torch.cuda.Event() for _ in range(2)]            # inputs of the slot landed
        computed = [torch.cuda.Event() for _ in range(2)]         # the slot's kernels finished
        fetched = [torch.cuda.Event() for _ in range(2)]          # the slot's tokens are back
        pos_np = pos_all.cpu().numpy()
        pos_stage = [view(blk, "positions").numpy() for blk in stage]
        out_h = [torch.empty(tuple(out.shape), dtype=torch.int64).pin_memory() for _ in range(ring)]
        for ev in computed + fetched:
            ev.record(stream)
        # one C-ABI call per device slot, marshalled once: a step changes the slot's contents
        # (its inputs arrive by copy), never its addresses
        calls = []
        for slot in range(2):
            b = devb[slot]
            ekw = dict(temperature=b["T"], seeds=b["seeds"], positions=b["positions"],
                       bias=b.get("bias"), mask=b.get("mask"), base_seed=w.base_seed,
                       offset=w.offset, wide=wide, out=outs[slot], workspace=workspace,
                       stream=stream)
            if fp8:
                calls.append(lms.prepare_lmhead_sample_fp8(b["H"], W8, wsc, **ekw))
            elif mx:
                calls.append(lms.prepare_lmhead_sample_mxfp4(b["H"], Wt, V, **ekw))
            elif topk:
                calls.append(lms.prepare_lmhead_sample_topk(b["H"], W, topk, scores=scores_k, **ekw))
            else:
                calls.append(lms.prepare_lmhead_sample(b["H"], W, path=path, **ekw))

        def e2e_step(i):
            j, slot = i % ring, i % 2
            h2d_done[j].synchronize()              # the copy that last read this block is done
            pos_stage[j][:] = pos_np[i]
            torch.cuda.set_stream(h2d_stream)
            h2d_stream.wait_event(computed[slot])       # step i-2's kernels read this slot
            dblk[slot].copy_(stage[j], non_blocking=True)
            h2d_done[j].record(h2d_stream)
            ready[slot].record(h2d_stream)
            torch.cuda.set_stream(stream)
            stream.wait_event(ready[slot])
            stream.wait_event(fetched[slot])       # step i-2's tokens have left this slot
            calls[slot]()
            computed[slot].record(stream)
            torch.cuda.set_stream(d2h_stream)
            d2h_stream.wait_event(computed[slot])
            out_h[j].copy_(outs[slot], non_blocking=True)
            fetched[slot].record(d2h_stream)
            torch.cuda.set_stream(stream)

        def e2e_time(n_warm, n_steps):
            for i in range(n_warm):
                e2e_step(i)
            torch.cuda.synchronize(dev)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            barrier()
            torch.cuda.synchronize(dev)
            e0.record(stream)
            h0 = time.perf_counter()
            for k in range(n_steps):
                e2e_step(n_warm + k)
            host_us = (time.perf_counter() - h0) / n_steps * 1e6
            stream.wait_event(fetched[(n_warm + n_steps - 1) % 2])   # the last tokens are back
            e1.record(stream)
            torch.cuda.synchronize(dev)
            barrier()
            return e0.elapsed_time(e1) / n_steps, host_us

        e2e_ms, e2e_host_us = e2e_time(args.warmup, args.steps)
        e2e = {"value": round(max_over_ranks(e2e_ms, dev) * 1e3, 2), "unit": UNIT,
               "h2d_bytes_per_step": total,
               "d2h_bytes_per_step": out.numel() * 8,
               "copies": "pinned host <-> device on one copy stream per direction, overlapped with "
                         "the neighbouring steps' kernels",
               "host_us_per_step": round(e2e_host_us, 2)}

    clocks = sampler.stop(t0, t1) if sampler else None
    if rank != 0:
        return
    achieved_gbs = alg / (us * 1e-6) / 1e9
    # a contraction takes the peak of its own input type: E4M3 runs at twice the bf16 rate
    # (nominal 4.5 vs 2.25 PFLOP/s dense), applied to the measured bf16 figure
    fp8_run = args.workload == "qwen3-8b-fp8"
    tensor_peak = peaks["bf16_tflops"] * (2.0 if fp8_run else 1.0)
    t_hbm = alg / (peaks["hbm_gbs"] * 1e9)
    t_tensor = flops / (tensor_peak * 1e12) if flops else 0.0
    if t_tensor > t_hbm:
        tf = flops / (us * 1e-6) / 1e12
        roofline = {"bound": "tensor", "achieved": round(tf, 1), "peak": round(tensor_peak, 1),
                    "unit": "TFLOP/s", "frac": round(tf / tensor_peak, 4),
                    "peak_source": peaks["source"] + (" (MEASURED_PEAKS.json bf16_tflops x 2, the nominal "
                                                      "fp8/bf16 ratio)" if fp8_run else
                                                      " (MEASURED_PEAKS.json bf16_tflops, burst cuBLAS)"),
                    "algorithmic_flops": flops}
    else:
        roofline = {"bound": "hbm", "achieved": round(achieved_gbs, 1), "peak": peaks["hbm_gbs"],
                    "unit": "GB/s", "frac": round(achieved_gbs / peaks["hbm_gbs"], 4),
                    "peak_source": peaks["source"] + " (MEASURED_PEAKS.json hbm_gbs, burst copy)",
                    "algorithmic_bytes": alg}
    traffic = recorded_traffic(args.workload, B) if args.workload in FUSED else None
    roofline["traffic"] = traffic["dram_bytes_per_launch"] if traffic else None
    inst = recorded_instructions(alu_key, args.workload) if alu_key else None
    if inst is not None:
        # Philox and the noise transform bound these kernels: the roofline is the SMs' issue
        # rate (4 warp schedulers per SM, one warp instruction each per clock, at the maximum
        # SM clock), against the step's warp instructions counted by ncu
        sms = torch.cuda.get_device_properties(dev).multi_processor_count
        issue_peak = sms * 4 * peaks["sm_max_mhz"] * 1e6 / 1e9
        achieved_gi = inst["warp_inst_per_step"] / (us * 1e-6) / 1e9
        roofline = {"bound": "alu", "achieved": round(achieved_gi, 1), "peak": round(issue_peak, 1),
                    "unit": "Gwarp-inst/s", "frac": round(achieved_gi / issue_peak, 4),
                    "peak_source": f"derived: {sms} SMs x 4 warp schedulers x 1 warp instruction per "
                                   f"clock x {peaks['sm_max_mhz']:.0f} MHz",
                    "warp_inst_per_step": inst["warp_inst_per_step"],
                    "hbm": {"achieved": round(achieved_gbs, 1), "peak": peaks["hbm_gbs"], "unit": "GB/s",
                            "frac": round(achieved_gbs / peaks["hbm_gbs"], 4), "algorithmic_bytes": alg},
                    "traffic": inst.get("dram_bytes_per_step")}
    roofline["kernel"] = kernel
    line = {"metric": METRIC, "value": round(us, 2), "unit": UNIT, "n_gpus": ws,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_per_step, 5),
            "higher_is_better": False, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic",
            "config": dict(config, parallelism="replicas" if ws > 1 else "single-gpu"),
            "hbm_gbs": round(achieved_gbs, 1), "samples_per_s": round(B / (us * 1e-6), 1),
            "p50_us": round(statistics.median(per_ms) * 1e3, 2),
            "p10_us": round(sorted(per_ms)[len(per_ms) // 10] * 1e3, 2),
            "p90_us": round(sorted(per_ms)[(len(per_ms) * 9) // 10] * 1e3, 2),
            "roofline": roofline, "clocks": clocks,
            "gpu_launches": launches_per_step * args.steps}
    if flops:
        line["tflops"] = round(flops / (us * 1e-6) / 1e12, 1)
    if e2e is not None:
        line["e2e"] = e2e
    if not args.no_cpu_baseline:
        if args.workload in ("qwen3-8b", "llama3-hetero", "large-vocab"):
            line["cpu_baseline"] = cpu_baseline(w, args.cpu_seconds)
        elif args.workload == "logits":
            threads = os.cpu_count() or 1
            vs = min(V, 16384)
            t = oracle_logits_time(logits.cpu(), vs, threads)
            line["cpu_baseline"] = {"value": t / vs * V * 1e6, "unit": UNIT, "cores": threads,
                                    "kind": "oracle",
                                    "sample": f"B={B} rows x first {vs} of {V} logits, scaled linearly"}
        elif args.workload == "verify":
            rows = 1
            t = oracle_verify_time(tgt_h, dft_h, tokens.cpu(), rows)
            rows = int(max(1, min(B, args.cpu_seconds / max(t, 1e-3))))
            t = oracle_verify_time(tgt_h, dft_h, tokens.cpu(), rows)
            line["cpu_baseline"] = {"value": t / rows * B * 1e6, "unit": UNIT, "cores": 1,
                                    "kind": "oracle",
                                    "sample": f"{rows} of {B} batch rows (k={k}, full V={V}), "
                                              f"{t:.1f} s wall, numpy fp64 on one thread, scaled linearly"}
    line.update(extra)
    print(json.dumps(line), flush=True)


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=25)
    ap.add_argument("--workload", default="qwen3-8b",
                    choices=list(FUSED) + ["logits", "noise", "filtered", "verify"])
    ap.add_argument("--batch", type=int, default=0)
    ap.add_argument("--topk", type=int, default=8, help="k of the qwen3-8b-topk workload")
    ap.add_argument("--path", choices=["auto", "gemv", "tcgen05"], default="auto",
                    help="Stage-1 path of the bf16 fused race workloads")
    ap.add_argument("--tile-v", type=int, default=0,
                    help="tile width of the logits workload (0 = the library's choice)")
    ap.add_argument("--spec-k", type=int, default=4, help="draft length k of the verify workload")
    ap.add_argument("--l2-flush", choices=["auto", "on", "off"], default="auto")
    ap.add_argument("--D", type=int, default=0)
    ap.add_argument("--V", type=int, default=0)
    ap.add_argument("--logits-dtype", choices=["fp32", "bf16"], default="bf16")
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--ref-budget-s", type=float, default=120.0,
                    help="seconds of oracle time the reference arm's timed steps may take")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.batch <= 0:
        args.batch = default_batch(args.workload)
    if args.impl == "reference":
        run_reference(args)
    else:
        run_gpu(args)


if __name__ == "__main__":
    main()
