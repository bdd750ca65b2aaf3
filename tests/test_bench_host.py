"""Host-side logic of bench.py: the max-over-ranks reduction across replicas (gloo, world size
2, CPU), the reference arm's JSON line, the algorithmic byte count, and the rule that recorded ncu
counters are used only on the kernel sources they were taken on."""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE="2", LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench
    import torch.distributed as dist
    bench.init_dist("gloo")
    v = bench.max_over_ranks(10.0 + 5 * rank)
    bench.barrier()
    q.put((rank, v))
    dist.destroy_process_group()


def test_max_over_ranks_gloo_world2():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    ps = [ctx.Process(target=_worker, args=(r, port, q)) for r in range(2)]
    for p in ps:
        p.start()
    res = dict(q.get(timeout=120) for _ in ps)
    for p in ps:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert res == {0: 15.0, 1: 15.0}


def _reference_line(*extra):
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "2", "--warmup", "3", "--batch", "4", "--D", "256", "--V", "4096",
                        *extra], capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    return json.loads(r.stdout.strip().splitlines()[-1])


def test_reference_arm_prints_contract_line():
    line = _reference_line()
    assert line["impl"] == "reference" and line["unit"] == "us/step" and line["value"] > 0
    assert line["higher_is_better"] is False
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["value"] == line["value"]
    assert line["e2e"]["h2d_bytes_per_step"] == 0
    # the GPU arm's config keys for a single-GPU run; a small workload runs in full each step
    assert line["config"]["parallelism"] == "single-gpu" and line["config"]["tile_v"] == 128
    assert line["vocab_rows_per_step"] == 4096 and line["extrapolated_from_v"] is None
    assert abs(line["measured_seconds_per_step"] * 1e6 - line["value"]) <= 1e-6 * line["value"] + 100


def test_reference_arm_states_its_slice_when_the_budget_is_short():
    line = _reference_line("--ref-budget-s", "0.000001")
    assert line["extrapolated_from_v"] == line["vocab_rows_per_step"] == 128
    per_row = line["measured_seconds_per_step"] / 128
    assert abs(per_row * 4096 * 1e6 - line["value"]) <= 1e-3 * line["value"]


def test_algorithmic_bytes_qwen_b64():
    sys.path.insert(0, ROOT)
    import bench
    b = bench.algorithmic_bytes(64, 4096, 151936, 1187)
    assert b == 151936 * 4096 * 2 + 64 * 4096 * 2 + 2 * 64 * 1187 * 8 + 64 * 28
    assert abs(b / 1e9 - 1.2464) < 1e-3


def test_recorded_counters_follow_the_kernel_sources(tmp_path, monkeypatch):
    # ncu records (DRAM bytes of the fused kernel, warp instructions of the ALU-bound workloads) are
    # used only while they were taken on the current kernel sources
    sys.path.insert(0, ROOT)
    import bench
    rec = bench.recorded_traffic("qwen3-8b", 64)
    assert rec is not None and rec["kernel_source_hash"] == bench.kernel_source_hash()
    assert rec["dram_bytes_per_launch"] == rec["dram_bytes_read"] + rec["dram_bytes_write"]
    assert bench.recorded_traffic("qwen3-8b", 3) is None
    for key, wl in (("logits/B=64/V=131072/bf16", "logits"), ("noise/B=64/V=151936", "noise")):
        r = bench.recorded_instructions(key, wl)
        assert r is not None and r["warp_inst_per_step"] == sum(k["warp_inst"] for k in r["kernels"].values())
    # a changed source invalidates the records
    fake = tmp_path / "noise_fill.cu"
    fake.write_text("// another kernel\n")
    monkeypatch.setitem(bench.ALU_SOURCES, "noise", [str(fake)])
    assert bench.recorded_instructions("noise/B=64/V=151936", "noise") is None


def test_traffic_records_follow_their_own_stage1_kernel():
    # each fused workload's DRAM record is tied to the sources of the Stage-1 kernel that runs it:
    # the MXFP4 kernel, the row-group kernel above 256 rows (race workloads), else the single-group one
    sys.path.insert(0, ROOT)
    import bench
    assert bench.stage1_kind("qwen3-8b-mxfp4", 1) == "mx"
    assert bench.stage1_kind("qwen3-8b", 512) == "rows" and bench.stage1_kind("large-vocab", 512) == "rows"
    assert bench.stage1_kind("qwen3-8b", 256) == "tc" and bench.stage1_kind("qwen3-8b-topk", 512) == "tc"
    assert bench.stage1_kind("qwen3-8b-fp8", 512) == "tc"
    for workload, B, kind in (("qwen3-8b-mxfp4", 1, "mx"), ("qwen3-8b-mxfp4", 64, "mx"),
                              ("large-vocab", 512, "rows")):
        rec = bench.recorded_traffic(workload, B)
        assert rec is not None and rec["kernel_source_hash"] == bench.kernel_source_hash(kind), (workload, B)
        assert rec["dram_bytes_per_launch"] == rec["dram_bytes_read"] + rec["dram_bytes_write"]
    # the three kernels' hashes differ (a record cannot pass for another kernel's)
    assert len({bench.kernel_source_hash(k) for k in ("tc", "rows", "mx")}) == 3
