"""Pins for the oracle's FP8 (E4M3) path: the codec against torch's float8_e4m3fn conversion run
on the CPU (a library routine), the power-of-two row quantiser against its definition's
extremes, and the FP8 logits against numpy's matmul of the decoded operands."""
import numpy as np
import pytest
import torch

import oracle


def torch_e4m3(x):
    return torch.from_numpy(np.asarray(x, np.float64)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def test_decode_all_codes_matches_torch():
    codes = np.arange(256, dtype=np.uint8)
    ours = oracle.e4m3_decode(codes)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).double().numpy()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan) and nan.sum() == 2
    assert np.array_equal(ours[~nan], ref[~nan])
    assert ours[0x7E] == 448.0 and ours[0x01] == 2.0 ** -9


def test_encode_matches_torch_on_grids_ties_and_subnormals():
    codes = np.arange(0x7F, dtype=np.uint8)
    vals = oracle.e4m3_decode(codes)
    mids = (vals[:-1] + vals[1:]) / 2                        # exact ties between neighbours
    rng = np.random.default_rng(0)
    x = np.concatenate([vals, mids, -mids, np.linspace(-448, 448, 4001),
                        rng.standard_normal(4000) * 2.0 ** rng.integers(-12, 8, 4000),
                        np.linspace(0, 2.0 ** -5, 513)])
    assert np.array_equal(oracle.e4m3_encode(x), torch_e4m3(x))
    # ties go to the even code
    assert oracle.e4m3_encode(np.array([mids[10]]))[0] % 2 == 0


def test_quantize_rows_power_of_two_scale():
    rng = np.random.default_rng(1)
    H = torch.from_numpy((rng.standard_normal((6, 300)) * np.array([[1e-3], [1], [7], [300], [1e5], [0]])).astype(np.float32)).to(torch.bfloat16)
    q, e = oracle.quantize_rows_e4m3(H)
    h = H.double().numpy()
    for b in range(6):
        amax = np.abs(h[b]).max()
        if amax == 0:                                        # zeros keep their sign bit
            assert e[b] == 0 and np.array_equal(q[b], torch_e4m3(h[b]))
            continue
        assert amax * 2.0 ** -int(e[b]) <= 448 < amax * 2.0 ** -(int(e[b]) - 1)
        assert np.array_equal(q[b], torch_e4m3(h[b] * 2.0 ** -int(e[b])))


def test_fp8_logits_match_numpy_and_race_consistent():
    rng = np.random.default_rng(2)
    B, D, V = 5, 96, 400
    H = torch.from_numpy(rng.standard_normal((B, D)).astype(np.float32)).to(torch.bfloat16)
    W8 = torch_e4m3(rng.standard_normal((V, D)) * 3)
    w_scale = rng.uniform(0.001, 0.01, V)
    q, e = oracle.quantize_rows_e4m3(H)
    y = oracle.lmhead_logits_fp8(q, e, W8, w_scale)
    ref = (oracle.e4m3_decode(q) * 2.0 ** e[:, None]) @ oracle.e4m3_decode(W8).T * w_scale[None, :]
    assert np.allclose(y, ref, rtol=1e-12, atol=1e-12)
    T = np.full(B, 0.8)
    seeds = np.arange(B) + 3
    r = oracle.lmhead_sample_fp8(H, W8, w_scale, temperature=T, seeds=seeds, positions=seeds)
    r2 = oracle.sample_from_logits(y, temperature=T, seeds=seeds, positions=seeds, tile_v=128)
    assert (r.out == r2.out).all() and np.array_equal(r.tile_max, r2.tile_max)
    sub = oracle.lmhead_sample_fp8(H, W8, w_scale, rows=[4, 1], temperature=T, seeds=seeds, positions=seeds)
    assert list(sub.out) == [r.out[4], r.out[1]]
