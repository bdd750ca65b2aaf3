"""Pins of the oracle's MXFP4 weights (W4A16: E2M1 elements, one UE8M0 scale per block of 32
along K; the Open Compute Project Microscaling format), the low-precision input the FlashSampling
page names ("Limitations", "Future directions") for the memory-bound regime.

  * E2M1 decode against a hand table of all 16 codes (sign bit, 2 exponent bits with bias 1,
    1 mantissa bit: 0, 0.5, 1, 1.5, 2, 3, 4, 6 and their negatives);
  * UE8M0 decode against torch's float8_e8m0fnu for all 256 codes;
  * E2M1 encode: round-trips every value, takes the even mantissa at every midpoint, saturates,
    and equals a brute-force nearest search over the hand table on random values;
  * the packed layout: a matrix packed by this file's own packer (written from the layout
    statement: element d in the low nibble of byte d/2 when d is even, the high nibble when odd;
    scale of block d/32 of row v at S[d/32][v]) decodes entry by entry to the dense matrix;
  * fp64 logits equal numpy's matmul of bf16 H and the dense decoded W (1e-12), a one-hot H
    reproduces a decoded row exactly, and the fused race over MXFP4 equals the plain race over
    those logits bit for bit;
  * the workload quantiser (input preparation) keeps every weight within half a grid step.
"""
import numpy as np
import pytest
import torch

import oracle
from lm_head_gumbel_lmhead_gb300 import workloads

# E2M1 code -> value, written out from the format's definition
E2M1_TABLE = {0: 0.0, 1: 0.5, 2: 1.0, 3: 1.5, 4: 2.0, 5: 3.0, 6: 4.0, 7: 6.0,
              8: -0.0, 9: -0.5, 10: -1.0, 11: -1.5, 12: -2.0, 13: -3.0, 14: -4.0, 15: -6.0}


def test_e2m1_decode_hand_table():
    got = oracle.e2m1_decode(np.arange(16))
    for c, v in E2M1_TABLE.items():
        assert got[c] == v and np.signbit(got[c]) == np.signbit(v), (c, got[c], v)


def test_ue8m0_decode_matches_torch():
    codes = torch.arange(256, dtype=torch.uint8)
    ref = codes.view(torch.float8_e8m0fnu).to(torch.float64).numpy()
    got = oracle.ue8m0_decode(codes.numpy())
    assert np.isnan(got[255]) and np.isnan(ref[255])
    assert np.array_equal(got[:255], ref[:255])
    assert got[127] == 1.0 and got[0] == 2.0 ** -127 and got[254] == 2.0 ** 127


def test_e2m1_encode_round_trip_midpoints_saturation():
    for c, v in E2M1_TABLE.items():
        assert oracle.e2m1_encode(v) == c
    mags = sorted(set(abs(v) for v in E2M1_TABLE.values()))
    for lo, hi in zip(mags[:-1], mags[1:]):
        mid = (lo + hi) / 2
        code = int(oracle.e2m1_encode(mid))
        assert code & 1 == 0 and abs(E2M1_TABLE[code]) in (lo, hi), (mid, code)
        assert oracle.e2m1_encode(-mid) == (code | 8)
    assert oracle.e2m1_encode(100.0) == 7 and oracle.e2m1_encode(-7.0) == 15
    rng = np.random.default_rng(2)
    x = rng.normal(0, 3, 2000)
    vals = np.array([E2M1_TABLE[c] for c in range(16)])
    got = oracle.e2m1_encode(x)
    for xi, c in zip(x, got):
        d = np.abs(vals - xi)
        assert d[c] == d.min(), (xi, c)


def pack(codes, scale_codes):
    """This file's own packer: codes [V, D] (0..15) -> W4 [V, D/2]; scale codes [V, D/32] ->
    S [D/32, V]."""
    V, D = codes.shape
    W4 = np.zeros((V, D // 2), np.uint8)
    for d in range(D):
        if d % 2 == 0:
            W4[:, d // 2] |= codes[:, d].astype(np.uint8)
        else:
            W4[:, d // 2] |= (codes[:, d].astype(np.uint8) << 4)
    return W4, np.ascontiguousarray(scale_codes.T.astype(np.uint8))


def dense(codes, scale_codes):
    V, D = codes.shape
    vals = np.vectorize(E2M1_TABLE.get)(codes).astype(np.float64)
    return vals * np.repeat(2.0 ** (scale_codes.astype(np.float64) - 127), 32, axis=1)


def _random_mx(V, D, seed):
    rng = np.random.default_rng(seed)
    codes = rng.integers(0, 16, (V, D))
    scales = rng.integers(110, 135, (V, D // 32))
    return codes, scales


def test_packed_layout_decodes_entry_by_entry():
    codes, scales = _random_mx(5, 96, 1)
    W4, S = pack(codes, scales)
    Wd = dense(codes, scales)
    for v in range(5):
        for d in range(96):
            assert oracle.mxfp4_weight(W4, S, v, d) == Wd[v, d], (v, d)


def test_logits_match_numpy_and_one_hot_rows():
    codes, scales = _random_mx(300, 128, 3)
    W4, S = pack(codes, scales)
    Wd = dense(codes, scales)
    g = torch.Generator().manual_seed(4)
    H = torch.randn(7, 128, generator=g).to(torch.bfloat16)
    y = oracle.lmhead_logits_mxfp4(H, W4, S)
    ref = H.double().numpy() @ Wd.T
    assert np.allclose(y, ref, rtol=1e-12, atol=1e-12)
    one = torch.zeros(2, 128, dtype=torch.bfloat16)
    one[0, 5] = 1.0
    one[1, 127] = 1.0
    y1 = oracle.lmhead_logits_mxfp4(one, W4, S)
    assert np.array_equal(y1[0], Wd[:, 5]) and np.array_equal(y1[1], Wd[:, 127])
    rows = oracle.lmhead_logits_mxfp4(H, W4, S, rows=[6, 2])
    assert np.array_equal(rows, y[[6, 2]])


@pytest.mark.parametrize("wide", [False, True])
def test_fused_race_equals_race_over_its_logits(wide):
    codes, scales = _random_mx(1000, 64, 5)
    W4, S = pack(codes, scales)
    g = torch.Generator().manual_seed(6)
    B = 9
    H = torch.randn(B, 64, generator=g).to(torch.bfloat16)
    T = np.full(B, 0.8)
    T[2] = 0.0
    T[5] = -1.0
    seeds = np.arange(B, dtype=np.int64) + 40
    seeds[1::3] = -1
    pos = np.arange(B, dtype=np.int64) * 7
    kw = dict(temperature=T, seeds=seeds, positions=pos, base_seed=3, offset=4, wide=wide)
    fused = oracle.lmhead_sample_mxfp4(H, W4, S, tile_v=128, **kw)
    plain = oracle.sample_from_logits(oracle.lmhead_logits_mxfp4(H, W4, S), tile_v=128, **kw)
    assert np.array_equal(fused.out, plain.out) and np.array_equal(fused.status, plain.status)
    assert np.array_equal(fused.tile_idx, plain.tile_idx)
    assert np.array_equal(fused.tile_max, plain.tile_max)
    sub = oracle.lmhead_sample_mxfp4(H, W4, S, rows=[4, 0], tile_v=128, **kw)
    assert np.array_equal(sub.out, fused.out[[4, 0]])


def test_workload_quantiser_keeps_weights_within_half_a_step():
    g = torch.Generator().manual_seed(8)
    W = (torch.randn(64, 256, generator=g) * 0.02).to(torch.bfloat16)
    W[3, :32] = 0.0                                   # an all-zero block
    W4, S = workloads.quantize_weight_mxfp4(W)
    assert W4.shape == (64, 128) and S.shape == (8, 64)
    W4n, Sn = W4.numpy(), S.numpy()
    w = W.double().numpy()
    for v in range(64):
        for blk in range(8):
            scale = 2.0 ** (int(Sn[blk, v]) - 127)
            block = w[v, 32 * blk: 32 * blk + 32]
            deq = np.array([oracle.mxfp4_weight(W4n, Sn, v, 32 * blk + i) for i in range(32)])
            amax = np.abs(block).max()
            assert np.abs(block).max() <= 6 * scale or amax == 0.0
            # the grid step near x is at most 2 * scale (between 4 and 6); rounding to nearest
            assert np.all(np.abs(deq - block) <= np.maximum(scale, 2 * scale * (np.abs(block) > 4 * scale)) / 2 + 1e-30)
            if amax > 0:
                assert amax > 3 * scale or scale == 2.0 ** -127      # the smallest scale that fits
