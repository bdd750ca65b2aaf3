"""The fused LM-head + Gumbel-max path on the GPU against the oracle.

  * every output (indices, statuses, all Stage-1 candidates) on the tiny workload and on ragged
    shapes (B not a multiple of 16, V not a multiple of 128, D not a multiple of 64, batches
    above 256 rows) for both the CUDA-core GEMV path and the tcgen05 path;
  * every row at full size (Qwen3-8B shape at B = 1, 8, 64, 256; the Llama-3 heterogeneous
    batch; the large-vocabulary shape with wide noise at B = 128), and rows on both sides of
    every 256-row launch boundary at B = 512, in the configuration the benchmark times, with
    every Stage-1 candidate of those rows compared;
  * seeded rows invariant to batch position; repeat calls bit-equal;
  * a device-side wait that runs out of time reports row status 3 and leaves the context usable.
"""
import numpy as np
import pytest
import torch

import lm_head_gumbel_lmhead_gb300 as lms
import oracle
from lm_head_gumbel_lmhead_gb300 import workloads
from parity import check_rows, check_tiles

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda")


def to_dev(w):
    d = dict(H=w.H.to(DEV), W=w.W.to(DEV), temperature=w.temperature.to(DEV),
             seeds=w.seeds.to(DEV), positions=w.positions.to(DEV),
             bias=None if w.bias is None else w.bias.to(DEV),
             mask=None if w.mask is None else w.mask.to(DEV))
    return d


def run_fused(w, d, path=lms.PATH_AUTO, **extra):
    B, D, V = w.B, w.D, w.V
    tv, nt, ws_bytes, _ = lms.tile_info(lms.OP_LMHEAD, B, D, V)
    ws = torch.full((ws_bytes,), 0xEE, dtype=torch.uint8, device=DEV)
    status = torch.full((B,), -7, dtype=torch.int32, device=DEV)
    out = lms.lmhead_sample(d["H"], d["W"], temperature=d["temperature"], seeds=d["seeds"],
                            positions=d["positions"], bias=d["bias"], mask=d["mask"],
                            base_seed=w.base_seed, offset=w.offset, wide=w.noise_mode == 1,
                            path=path, workspace=ws, row_status=status, **extra)
    torch.cuda.synchronize()
    cs, ci = lms.split_workspace(ws, B, nt)
    return out.cpu().numpy(), status.cpu().numpy(), cs.cpu().numpy(), ci.cpu().numpy()


def orc_kw(w):
    return dict(temperature=w.temperature.double().numpy(), seeds=w.seeds.numpy(),
                positions=w.positions.numpy(),
                bias=None if w.bias is None else w.bias.double().numpy(),
                mask=None if w.mask is None else w.mask.numpy().view(np.uint32),
                base_seed=w.base_seed, offset=w.offset, wide=w.noise_mode == 1)


def full_parity(w, path):
    d = to_dev(w)
    out, st, cs, ci = run_fused(w, d, path)
    orc = oracle.lmhead_sample(w.H, w.W, tile_v=128, want_scores=True, **orc_kw(w))
    score_of = lambda i, v: orc.scores[i, v]
    near = check_rows(out, st, orc, score_of)
    check_tiles(cs, ci, orc, score_of)
    return near


@pytest.mark.parametrize("path", [lms.PATH_GEMV, lms.PATH_TCGEN05])
def test_tiny_workload_every_output(path):
    full_parity(workloads.tiny(), path)


def _ragged(B, D, V, seed, wide=False, features=True):
    g = torch.Generator().manual_seed(seed)
    H = (torch.randn(B, D, generator=g)).to(torch.bfloat16)
    W = (torch.randn(V, D, generator=g) / D ** 0.5).to(torch.bfloat16)
    T = 0.3 + torch.rand(B, generator=g)
    seeds = 100 + torch.arange(B, dtype=torch.int64)
    bias = mask = None
    if features:
        T[::5] = 0.0
        if B > 3:
            T[3] = -2.0
        seeds[1::4] = -1
        bias = torch.randn(B, V, generator=g) * 0.3
        allowed = torch.rand(B, V, generator=g) < 0.5
        allowed[B // 2:] = True
        if B > 2:
            allowed[2] = False
        mask = workloads.pack_allow_bits(allowed)
    return workloads.Workload(f"ragged B={B} D={D} V={V}", B, D, V, H, W, T, seeds,
                              torch.arange(B, dtype=torch.int64) * 3 + 1, bias, mask,
                              1 if wide else 0, base_seed=321, offset=6)


@pytest.mark.parametrize("B,D,V", [(1, 64, 1000), (2, 200, 8229), (5, 512, 3000), (8, 1024, 4097)])
def test_gemv_ragged(B, D, V):
    full_parity(_ragged(B, D, V, seed=B + D), lms.PATH_GEMV)


@pytest.mark.parametrize("B,D,V,wide", [(1, 64, 1000, False), (3, 200, 8229, True),
                                        (17, 512, 3000, False), (40, 1024, 4097, True),
                                        (130, 256, 2000, False), (256, 128, 1500, True),
                                        (300, 192, 1300, False)])
def test_tcgen05_ragged(B, D, V, wide):
    full_parity(_ragged(B, D, V, seed=B * 7 + D, wide=wide), lms.PATH_TCGEN05)


@pytest.mark.parametrize("B,D,V,wide,features", [(700, 128, 1300, False, True),
                                                 (1100, 64, 2100, True, True),
                                                 (520, 96, 1500, False, False)])
def test_tcgen05_batches_above_256(B, D, V, wide, features):
    # above 256 rows the tcgen05 path runs row-group launches of up to 1024 rows (groups of 256
    # whose CTAs share each tile of W): one launch of 3 groups (700), one of 4 groups and a 76-row
    # single-group launch (1100), one of 3 groups with an 8-row last group (520)
    full_parity(_ragged(B, D, V, seed=B + V, wide=wide, features=features), lms.PATH_TCGEN05)


def test_row_group_timeout_poisons_its_group_only():
    # CTA 0 serves row group 0; its withheld first load runs out, so every row of group 0 (one
    # tile of each is CTA 0's) reports status 3 and the other group's rows are sampled as usual
    w = _ragged(300, 128, 3000, seed=23, features=False)
    d = to_dev(w)
    out, st, _, ci = run_fused(w, d, lms.PATH_TCGEN05, timeout_ms=20,
                               debug_flags=lms.DEBUG_WITHHOLD_FIRST_LOAD)
    assert (st[:256] == lms.ROW_DEVICE_TIMEOUT).all() and (out[:256] == -1).all()
    assert (st[256:] != lms.ROW_DEVICE_TIMEOUT).all()
    # the next call on the same context is correct
    full_parity(w, lms.PATH_TCGEN05)


def test_tcgen05_without_optional_inputs():
    full_parity(_ragged(33, 256, 2500, seed=5, features=False), lms.PATH_TCGEN05)


@pytest.mark.parametrize("wide", [False, True])
def test_tcgen05_plain_launch_greedy_invalid_and_ragged(wide):
    # no bias and no mask: the plain epilogue, with greedy, invalid and unseeded rows and a last
    # vocabulary tile that ends inside an 8-row chunk (V = 2500 = 19 * 128 + 68)
    w = _ragged(37, 256, 2500, seed=9, wide=wide)
    w = workloads.Workload(w.name, w.B, w.D, w.V, w.H, w.W, w.temperature, w.seeds, w.positions,
                           None, None, w.noise_mode, base_seed=w.base_seed, offset=w.offset)
    full_parity(w, lms.PATH_TCGEN05)


def sampled_parity(w, rows, path=lms.PATH_AUTO):
    d = to_dev(w)
    out, st, cs, ci = run_fused(w, d, path)
    rows = np.asarray(rows)
    orc = oracle.lmhead_sample_rows(w.H, w.W, rows, tile_v=128, **orc_kw(w))

    def score_of(i, v):
        kw = orc_kw(w)
        return float(oracle.lmhead_scores_at(w.H, w.W, [rows[i]], [v], **kw)[0])
    near = check_rows(out[rows], st[rows], orc, score_of, rows=rows)
    check_tiles(cs[rows], ci[rows], orc, score_of)
    # properties every row satisfies
    assert ((st == 0) | (st == 1) | (st == 2)).all()
    assert ((out >= 0) & (out < w.V) | (out == -1)).all()
    return out, st, near


@pytest.fixture(scope="module")
def qwen_w():
    return workloads.qwen3_8b(256, step=3)


@pytest.mark.parametrize("B", [1, 8, 64, 256])
def test_qwen3_8b_shape_every_row(qwen_w, B):
    w = qwen_w
    sub = workloads.Workload(w.name, B, w.D, w.V, w.H[:B].contiguous(), w.W, w.temperature[:B],
                             w.seeds[:B], w.positions[:B], None, None, w.noise_mode)
    out, st, _ = sampled_parity(sub, range(B))
    assert (st == 0).all()


def test_qwen3_8b_shape_paths_agree_at_small_batch(qwen_w):
    w = qwen_w
    sub = workloads.Workload(w.name, 2, w.D, w.V, w.H[:2].contiguous(), w.W, w.temperature[:2],
                             w.seeds[:2], w.positions[:2], None, None, w.noise_mode)
    d = to_dev(sub)
    a = run_fused(sub, d, lms.PATH_GEMV)[0]
    b = run_fused(sub, d, lms.PATH_TCGEN05)[0]
    if not np.array_equal(a, b):
        # only a near-tie may separate the two accumulation orders
        sampled_parity(sub, [0, 1], lms.PATH_GEMV)
        sampled_parity(sub, [0, 1], lms.PATH_TCGEN05)


def test_llama3_hetero_every_row():
    w = workloads.llama3_hetero()
    out, st, _ = sampled_parity(w, range(w.B))
    assert (st == 0).all()


def test_large_vocab_wide_noise_every_row_b128():
    w = workloads.large_vocab(128)
    sampled_parity(w, range(128))


def test_large_vocab_wide_noise_b512_launch_boundaries():
    # one row-group launch of two groups of 256 rows: rows on both sides of the group boundary and
    # at both ends
    w = workloads.large_vocab(512)
    rows = list(range(0, 8)) + list(range(248, 264)) + list(range(504, 512))
    sampled_parity(w, rows)


def test_seeded_rows_batch_position_invariant_tcgen05():
    w = _ragged(48, 256, 3000, seed=11, features=True)
    d = to_dev(w)
    full = run_fused(w, d, lms.PATH_TCGEN05)[0]
    perm = torch.randperm(w.B, generator=torch.Generator().manual_seed(1))
    pw = workloads.Workload(w.name, w.B, w.D, w.V, w.H[perm].contiguous(), w.W, w.temperature[perm],
                            w.seeds[perm], w.positions[perm], w.bias[perm].contiguous(),
                            w.mask[perm].contiguous(), w.noise_mode, w.base_seed, w.offset)
    pout = run_fused(pw, to_dev(pw), lms.PATH_TCGEN05)[0]
    seeded = (w.seeds[perm] >= 0).numpy()
    assert np.array_equal(pout[seeded], full[perm.numpy()][seeded])
    again = run_fused(w, d, lms.PATH_TCGEN05)[0]
    assert np.array_equal(again, full)


def test_timeout_reports_status_and_context_survives():
    w = _ragged(20, 256, 4000, seed=13, features=False)
    d = to_dev(w)
    out, st, _, ci = run_fused(w, d, lms.PATH_TCGEN05, timeout_ms=20,
                               debug_flags=lms.DEBUG_WITHHOLD_FIRST_LOAD)
    assert (st == lms.ROW_DEVICE_TIMEOUT).all() and (out == -1).all()
    assert (ci == -2).any()
    # the next call on the same context is correct
    full_parity(w, lms.PATH_TCGEN05)


# ---- the CTA-pair tcgen05 path (cta_group::2, M = 256) ----
@pytest.mark.parametrize("B,D,V,wide", [(1, 64, 1000, False), (17, 200, 1300, True),
                                        (40, 512, 3000, False), (128, 256, 2000, True)])
def test_tcgen05_pair_ragged(B, D, V, wide):
    full_parity(_ragged(B, D, V, seed=B * 5 + D, wide=wide), lms.PATH_TCGEN05_PAIR)


@pytest.mark.parametrize("B,D,V,wide", [(256, 128, 1500, True), (300, 192, 1300, False)])
def test_tcgen05_pair_ragged_wide_batches(B, D, V, wide):
    full_parity(_ragged(B, D, V, seed=B * 5 + D, wide=wide), lms.PATH_TCGEN05_PAIR)


def test_tcgen05_pair_matches_single_cta_path():
    # same accumulation (fp32, same K order per 128-row tile): bit-equal tokens and candidates
    w = _ragged(96, 512, 5000, seed=21, features=True)
    d = to_dev(w)
    a = run_fused(w, d, lms.PATH_TCGEN05)
    b = run_fused(w, d, lms.PATH_TCGEN05_PAIR)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])
    assert np.array_equal(a[3], b[3])


def test_tcgen05_pair_timeout_reports_status():
    w = _ragged(20, 256, 4000, seed=13, features=False)
    d = to_dev(w)
    out, st, _, ci = run_fused(w, d, lms.PATH_TCGEN05_PAIR, timeout_ms=20,
                               debug_flags=lms.DEBUG_WITHHOLD_FIRST_LOAD)
    assert (st == lms.ROW_DEVICE_TIMEOUT).all() and (out == -1).all()
    full_parity(w, lms.PATH_TCGEN05_PAIR)


@pytest.mark.parametrize("B", [64, 256])
def test_qwen3_8b_shape_pair_sampled_rows(qwen_w, B):
    w = qwen_w
    sub = workloads.Workload(w.name, B, w.D, w.V, w.H[:B].contiguous(), w.W, w.temperature[:B],
                             w.seeds[:B], w.positions[:B], None, None, w.noise_mode)
    out, st, _ = sampled_parity(sub, [0, B // 2, B - 1], lms.PATH_TCGEN05_PAIR)
    assert (st == 0).all()
