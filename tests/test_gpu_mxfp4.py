"""The fused path with MXFP4 weights (W4A16) on the GPU against the oracle.

  * every output (indices, statuses, every Stage-1 candidate) on ragged shapes: B not a multiple
    of 16, V not a multiple of 128, D = 96 (the last 64-element K chunk half out of range), more
    than 256 rows, with bias, masks, greedy, invalid and unseeded rows, in both noise modes;
  * weights from the offline quantiser (realistic block scales) and random codes with block
    scales spread over 2^-27 .. 2^27;
  * every row at the Qwen3-8B shape (D = 4096, V = 151936) at B = 64;
  * a device-side wait that runs out of time reports row status 3, and the context survives;
  * the packer (lms_mxfp4_pack) writes exactly the tiled layout the header states (including the
    word layout that moves each sign next to its bf16 high byte), checked against this file's own
    re-tiling on the host, with ragged V and D and scale rows with a stride.
The parity rule is tests/parity.py's: the oracle decodes the same codes and scales exactly in
fp64, the kernel rebuilds them as exact bf16 values and accumulates in fp32.
"""
import numpy as np
import pytest
import torch

import lm_head_gumbel_lmhead_gb300 as lms
import oracle
from lm_head_gumbel_lmhead_gb300 import workloads
from parity import check_rows, check_tiles
from test_gpu_lmhead import _ragged, orc_kw

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda")


def random_mx(V, D, seed, lo=110, hi=135):
    rng = np.random.default_rng(seed)
    codes = rng.integers(0, 16, (V, D)).astype(np.uint8)
    W4 = (codes[:, 0::2] | (codes[:, 1::2] << 4)).astype(np.uint8)
    S = torch.from_numpy(rng.integers(lo, hi, (D // 32, V)).astype(np.uint8))
    return torch.from_numpy(W4), S


def run_mx(w, W4, S, **extra):
    B, D, V = w.B, w.D, w.V
    tv, nt, ws_bytes, _ = lms.tile_info(lms.OP_LMHEAD, B, D, V)
    ws = torch.full((ws_bytes,), 0xEE, dtype=torch.uint8, device=DEV)
    status = torch.full((B,), -7, dtype=torch.int32, device=DEV)
    Wt = lms.mxfp4_pack(W4.to(DEV), S.to(DEV))
    out = lms.lmhead_sample_mxfp4(
        w.H.to(DEV), Wt, V, temperature=w.temperature.to(DEV), seeds=w.seeds.to(DEV),
        positions=w.positions.to(DEV), bias=None if w.bias is None else w.bias.to(DEV),
        mask=None if w.mask is None else w.mask.to(DEV), base_seed=w.base_seed, offset=w.offset,
        wide=w.noise_mode == 1, workspace=ws, row_status=status, **extra)
    torch.cuda.synchronize()
    cs, ci = lms.split_workspace(ws, B, nt)
    return out.cpu().numpy(), status.cpu().numpy(), cs.cpu().numpy(), ci.cpu().numpy()


def mx_parity(w, W4, S, rows=None):
    """Compare the GPU's outputs with the oracle's for the given rows (all when None): the fused
    oracle's result, checked equal to the plain race over the oracle's fp64 logits of the whole
    batch, whose scores serve the near-tie rule."""
    out, st, cs, ci = run_mx(w, W4, S)
    kw = orc_kw(w)
    y = oracle.lmhead_logits_mxfp4(w.H, W4.numpy(), S.numpy())
    full = oracle.sample_from_logits(y, tile_v=128, want_scores=True, **kw)
    rows = np.arange(w.B) if rows is None else np.asarray(rows)
    fused = oracle.lmhead_sample_mxfp4(w.H, W4.numpy(), S.numpy(), rows=rows, tile_v=128, **kw)
    assert np.array_equal(fused.out, full.out[rows]) and np.array_equal(fused.tile_idx, full.tile_idx[rows])
    score_of = lambda i, v: full.scores[rows[i], v]
    near = check_rows(out[rows], st[rows], fused, score_of, rows=rows)
    check_tiles(cs[rows], ci[rows], fused, score_of)
    return out, st, near


def _case(B, D, V, seed, wide, features=True):
    return _ragged(B, D, V, seed=seed, wide=wide, features=features)


@pytest.mark.parametrize("B,D,V,wide", [(1, 64, 1000, False), (3, 96, 8229, True),
                                        (17, 512, 3000, False), (40, 1024, 4097, True),
                                        (130, 256, 2000, False), (256, 128, 1500, True),
                                        (300, 192, 1300, False)])
def test_mxfp4_ragged_every_output(B, D, V, wide):
    w = _case(B, D, V, seed=B * 13 + D, wide=wide)
    W4, S = random_mx(V, D, seed=B + V)
    mx_parity(w, W4, S)


@pytest.mark.parametrize("wide", [False, True])
def test_mxfp4_plain_launch_greedy_invalid_unseeded(wide):
    # no bias and no mask (the plain epilogue), with greedy, invalid and unseeded rows
    w = _ragged(37, 256, 2500, seed=41, wide=wide)
    w = workloads.Workload(w.name, w.B, w.D, w.V, w.H, w.W, w.temperature, w.seeds, w.positions,
                           None, None, w.noise_mode, base_seed=w.base_seed, offset=w.offset)
    mx_parity(w, *random_mx(w.V, w.D, seed=43))


def test_mxfp4_quantised_weights_and_wide_scales():
    w = _case(24, 512, 5000, seed=51, wide=False, features=False)
    W4q, Sq = workloads.quantize_weight_mxfp4(w.W)
    mx_parity(w, W4q, Sq)
    W4, S = random_mx(w.V, w.D, seed=52, lo=100, hi=155)
    mx_parity(w, W4, S)


def test_mxfp4_qwen3_8b_shape_every_row():
    w = workloads.qwen3_8b(64, step=5)
    W4, S = workloads.quantize_weight_mxfp4(w.W)
    out, st, _ = mx_parity(w, W4, S, rows=range(64))
    assert (st == 0).all()


def test_mxfp4_timeout_reports_status_and_context_survives():
    w = _case(20, 256, 4000, seed=61, wide=False, features=False)
    W4, S = random_mx(w.V, w.D, seed=62)
    out, st, _, ci = run_mx(w, W4, S, timeout_ms=20, debug_flags=lms.DEBUG_WITHHOLD_FIRST_LOAD)
    assert (st == lms.ROW_DEVICE_TIMEOUT).all() and (out == -1).all()
    assert (ci == -2).any()
    mx_parity(w, W4, S)


def tiled_words(codes):
    """The header's word layout for elements e0..e7 of each group of eight (codes [..., 8], values
    0..15): magnitude bits of e_k at bits 4k..4k+2, sign of e_k at bit 8k+7 (k < 4) or 8(k-4)+3
    (k >= 4); returned as little-endian bytes [..., 4]."""
    codes = codes.astype(np.uint64)
    word = np.zeros(codes.shape[:-1], np.uint64)
    for k in range(8):
        word |= (codes[..., k] & 7) << np.uint64(4 * k)
        word |= (codes[..., k] >> np.uint64(3)) << np.uint64(8 * k + 7 if k < 4 else 8 * (k - 4) + 3)
    return np.stack([(word >> np.uint64(8 * i)) & np.uint64(0xFF) for i in range(4)], -1).astype(np.uint8)


def retile_on_host(W4, S, V, D):
    """This file's own writing of the tiled format, from the header's statement: block (t, c) of
    4352 bytes at (t * ceil(D/64) + c) * 4352: row r's 32 code bytes at 32 r (elements 64 c ..
    64 c + 63 as eight words of eight, zero past D), then the scale codes of blocks 2c and 2c + 1
    (row r at 4096 + r and 4096 + 128 + r); zero past V."""
    W4, S = W4.numpy(), S.numpy()
    nt, nk = -(-V // 128), -(-D // 64)
    codes = np.zeros((nt * 128, nk * 64), np.uint8)            # logical codes, zero padded
    codes[:V, 0:D:2] = W4[:, :D // 2] & 0xF
    codes[:V, 1:D:2] = W4[:, :D // 2] >> 4
    words = tiled_words(codes.reshape(nt * 128, nk * 8, 8)).reshape(nt * 128, nk, 32)
    out = np.zeros(nt * nk * 4352, np.uint8)
    for t in range(nt):
        for c in range(nk):
            base = (t * nk + c) * 4352
            out[base: base + 4096] = words[128 * t: 128 * t + 128, c].reshape(-1)
            for r in range(128):
                v = 128 * t + r
                if v >= V:
                    continue
                for k in range(2):
                    if 2 * c + k < D // 32:
                        out[base + 4096 + 128 * k + r] = S[2 * c + k, v]
    return out


@pytest.mark.parametrize("V,D", [(300, 96), (129, 64), (1000, 256)])
def test_mxfp4_pack_writes_the_stated_layout(V, D):
    W4, S = random_mx(V, D, seed=V + D)
    S_strided = torch.zeros(D // 32, V + 9, dtype=torch.uint8, device=DEV)[:, :V]   # a row stride != V
    S_strided.copy_(S.to(DEV))
    Wt = lms.mxfp4_pack(W4.to(DEV), S_strided)
    assert Wt.numel() == lms.lib().lms_mxfp4_tiled_bytes(V, D)
    assert np.array_equal(Wt.cpu().numpy(), retile_on_host(W4, S, V, D))
