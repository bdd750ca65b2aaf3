"""Pins for the oracle's race: the sampled law, the tail, tiles, greedy, the GEMM, invariance.

  * Gumbel-max = softmax (FlashSampling page, "Gumbel-Max trick"): chi-square of the empirical
    histogram over a 16-token row against softmax, as the Megatron-LM PR's test does ("Tests":
    1M draws, 15 dof, below the 1e-6 quantile), with bias added before the temperature
    (sampling-kernel guide, reasoning step 4) and masked tokens at zero mass.
  * The tail rate on rows [0, -D, ..., -D] against the closed form (V-1) r / (1 + (V-1) r)
    (Megatron-LM PR, "Problem"), inside the two-sided 1e-6 Poisson interval ("Tests").
  * Path exactness (FlashSampling "core method": argmax decomposes over vocabulary tiles):
    brute force over every tile width on tiny rows with ties, against numpy's argmax.
  * Greedy (T == 0) against numpy's argmax (smallest index on ties; guide step 3).
  * The fp64 GEMM against numpy's matmul; one-hot H reproduces rows of W exactly.
  * Seeded rows are batch-position invariant (Megatron-LM PR, "Tests").
"""
import math

import numpy as np
import pytest
import torch
from scipy import stats

import oracle
from lm_head_gumbel_lmhead_gb300 import workloads


def softmax(x):
    x = np.asarray(x, np.float64)
    m = np.max(x[np.isfinite(x)])
    e = np.where(np.isfinite(x), np.exp(x - m), 0.0)
    return e / e.sum()


def chi2_stat(counts, probs):
    keep = probs > 0
    exp = probs[keep] * counts.sum()
    return float(((counts[keep] - exp) ** 2 / exp).sum()), int(keep.sum()) - 1


ROW16 = np.array([1.2, -0.3, 0.0, 2.1, -1.7, 0.4, 0.9, -2.5, 1.6, -0.8, 0.05, 1.1, -1.2, 0.7,
                  -0.1, 0.3])


@pytest.mark.parametrize("wide", [False, True])
@pytest.mark.parametrize("seeded", [True, False])
def test_chi_square_16_token_row_matches_softmax(golden, wide, seeded):
    page = golden["chi_square"]
    n = page["draws"]
    kw = dict(seeds=np.full(n, 1234), positions=np.arange(n)) if seeded else \
        dict(base_seed=1234, offset=3)
    r = oracle.sample_from_logits(ROW16, B=n, temperature=np.full(n, 1.0), wide=wide, **kw)
    assert (r.status == 0).all()
    counts = np.bincount(r.out, minlength=16).astype(np.float64)
    stat, dof = chi2_stat(counts, softmax(ROW16))
    assert dof == page["dof"]
    thr = stats.chi2.isf(1e-6, dof)
    assert round(thr, 1) == page["threshold_printed"]
    assert stat < thr


def test_chi_square_with_bias_temperature_and_mask():
    n = 1_000_000
    T = 0.6
    bias = np.linspace(-1.0, 1.0, 16)[::-1].copy()
    allowed = np.ones(16, bool)
    allowed[[2, 5, 11, 14]] = False
    mask = workloads.pack_allow_bits(torch.from_numpy(allowed)[None]).numpy().view(np.uint32)[0]
    r = oracle.sample_from_logits(ROW16, B=n, temperature=np.full(n, T), bias=bias, mask=mask,
                                  seeds=np.full(n, 77), positions=np.arange(n), wide=True)
    counts = np.bincount(r.out, minlength=16).astype(np.float64)
    assert counts[~allowed].sum() == 0                        # masked tokens: zero mass
    law = softmax(np.where(allowed, (ROW16 + bias) / T, -np.inf))
    stat, dof = chi2_stat(counts, law)
    assert dof == 11 and stat < stats.chi2.isf(1e-6, dof)
    # the test has power against the wrong transform order (bias after temperature)
    wrong = softmax(np.where(allowed, ROW16 / T + bias, -np.inf))
    assert chi2_stat(counts, wrong)[0] > 100 * stats.chi2.isf(1e-6, dof)


def poisson_interval(mu, alpha=1e-6):
    return stats.poisson.ppf(alpha / 2, mu), stats.poisson.isf(alpha / 2, mu)


def tail_expected(V, r, draws):
    p = (V - 1) * r / (1 + (V - 1) * r)
    return draws * p


@pytest.mark.parametrize("wide", [False, True])
@pytest.mark.parametrize("seeded", [True, False])
def test_tail_rate_matches_closed_form_small_vocab(wide, seeded):
    # V = 2048, r = 1e-6 (13.8 nats below the top, inside both modes' range): ~204 misses
    V, r, n = 2048, 1e-6, 100_000
    row = workloads.tail_row(V, r).numpy()
    kw = dict(seeds=np.full(n, 1234), positions=np.arange(n)) if seeded else \
        dict(base_seed=1234, offset=0)
    res = oracle.sample_from_logits(row, B=n, wide=wide, **kw)
    misses = int((res.out != 0).sum())
    lo, hi = poisson_interval(tail_expected(V, r, n))
    assert lo <= misses <= hi, (misses, lo, hi)


def test_fp32_noise_cannot_reach_beyond_its_range_but_wide_can():
    # Closed form on the extremes: in fp32 mode the largest possible gap g_other - g_top is
    # log(E_max / E_min) = log(17.33 / 2.98e-8) = 20.18 nats, so a row whose runner-up sits 21
    # nats below the top can never miss; in wide mode the gap reaches 40.3 nats.
    def gap(wide):
        e_max = -math.log(oracle.uniform(0, 0, wide))
        e_min = -math.log(oracle.uniform(0xFFFFFFFF, 0xFFFFFFFF, wide))
        return math.log(e_max) - math.log(e_min)
    assert 20.0 < gap(False) < 21.0
    assert 40.0 < gap(True) < 41.0


def test_tile_decomposition_brute_force():
    rng = np.random.default_rng(5)
    for V in list(range(1, 9)) + [13, 33]:
        for trial in range(6):
            y = rng.integers(-2, 3, size=V).astype(np.float64)     # many ties
            B = 3
            T = np.array([0.0, 1.0, 0.5])
            seeds = np.array([3, 4, -1])
            full = oracle.sample_from_logits(y, B=B, temperature=T, seeds=seeds,
                                             positions=np.array([trial] * B), base_seed=9,
                                             want_scores=True)
            for b in range(B):
                assert full.out[b] == int(np.argmax(full.scores[b]))
                assert full.top1[b] == full.scores[b].max()
            for tile in range(1, V + 1):
                r = oracle.sample_from_logits(y, B=B, temperature=T, seeds=seeds,
                                              positions=np.array([trial] * B), base_seed=9,
                                              tile_v=tile)
                for b in range(B):
                    t_star = int(np.argmax(r.tile_max[b]))           # smallest tile on ties
                    assert r.tile_idx[b, t_star] == full.out[b]
                    for t in range(r.tile_max.shape[1]):
                        seg = full.scores[b, t * tile:(t + 1) * tile]
                        assert r.tile_max[b, t] == seg.max()
                        assert r.tile_idx[b, t] == t * tile + int(np.argmax(seg))


def test_greedy_is_plain_argmax_with_bias_and_mask():
    rng = np.random.default_rng(6)
    B, V = 8, 1000
    y = rng.integers(-5, 5, size=(B, V)).astype(np.float64)
    bias = rng.integers(-2, 2, size=(B, V)).astype(np.float64)
    allowed = rng.random((B, V)) < 0.3
    mask = workloads.pack_allow_bits(torch.from_numpy(allowed)).numpy().view(np.uint32)
    for off in (0, 1):
        r = oracle.sample_from_logits(y, temperature=np.zeros(B), bias=bias, mask=mask,
                                      seeds=np.arange(B) + off, positions=np.arange(B), offset=off)
        ref = np.argmax(np.where(allowed, y + bias, -np.inf), axis=1)
        assert (r.out == ref).all() and (r.status == 0).all()


def test_edge_rows_all_masked_invalid_temperature_nan():
    V = 70
    y = np.zeros((5, V))
    y[3, :] = np.nan
    y[4, 10] = np.inf
    allowed = np.ones((5, V), bool)
    allowed[0] = False
    mask = workloads.pack_allow_bits(torch.from_numpy(allowed)).numpy().view(np.uint32)
    T = np.array([1.0, -1.0, np.nan, 1.0, 1.0])
    r = oracle.sample_from_logits(y, temperature=T, mask=mask, base_seed=1)
    assert list(r.out[:4]) == [-1, -1, -1, -1]
    assert list(r.status) == [1, 2, 2, 1, 0]
    assert r.out[4] == 10


def test_gemm_matches_numpy_and_one_hot():
    rng = np.random.default_rng(7)
    B, D, V = 5, 96, 300
    H = torch.from_numpy(rng.standard_normal((B, D)).astype(np.float32)).to(torch.bfloat16)
    W = torch.from_numpy(rng.standard_normal((V, D)).astype(np.float32)).to(torch.bfloat16)
    y = oracle.lmhead_logits(H, W)
    ref = H.double().numpy() @ W.double().numpy().T
    assert np.allclose(y, ref, rtol=0, atol=1e-12)
    one = torch.zeros(B, D, dtype=torch.bfloat16)
    for b in range(B):
        one[b, 7 * b] = 1.0
    y1 = oracle.lmhead_logits(one, W)
    for b in range(B):
        assert (y1[b] == W[:, 7 * b].double().numpy()).all()


def test_lmhead_sample_equals_race_over_its_logits_and_scores_at():
    w = workloads.tiny()
    H, W = w.H, w.W
    r = oracle.lmhead_sample(H, W, temperature=w.temperature.numpy(), seeds=w.seeds.numpy(),
                             positions=w.positions.numpy(), tile_v=128, want_scores=True)
    y = oracle.lmhead_logits(H, W)
    r2 = oracle.sample_from_logits(y, temperature=w.temperature.numpy(), seeds=w.seeds.numpy(),
                                   positions=w.positions.numpy(), tile_v=128)
    assert (r.out == r2.out).all() and (r.tile_idx == r2.tile_idx).all()
    rows = np.repeat(np.arange(w.B), 3)
    cols = np.array([0, 8191, 4000] * w.B)
    s = oracle.lmhead_scores_at(H, W, rows, cols, temperature=w.temperature.numpy(),
                                seeds=w.seeds.numpy(), positions=w.positions.numpy())
    assert np.allclose(s, r.scores[rows, cols], rtol=0, atol=1e-12)


def test_seeded_rows_are_batch_position_invariant():
    rng = np.random.default_rng(8)
    B, V = 6, 3000
    y = rng.standard_normal((B, V)) * 3
    T = np.full(B, 0.7)
    seeds = np.array([11, 12, -1, 13, -1, 14])
    pos = np.array([100, 5, 0, 2**35, 0, 9])
    for wide in (False, True):
        full = oracle.sample_from_logits(y, temperature=T, seeds=seeds, positions=pos, wide=wide,
                                         base_seed=3, offset=4)
        perm = np.array([5, 2, 0, 4, 3, 1])
        pr = oracle.sample_from_logits(y[perm], temperature=T[perm], seeds=seeds[perm],
                                       positions=pos[perm], wide=wide, base_seed=3, offset=4)
        for i, b in enumerate(perm):
            if seeds[b] >= 0:
                assert pr.out[i] == full.out[b]
                single = oracle.sample_from_logits(y[b:b + 1], temperature=T[b:b + 1],
                                                   seeds=seeds[b:b + 1], positions=pos[b:b + 1],
                                                   wide=wide)
                assert single.out[0] == full.out[b]
        again = oracle.sample_from_logits(y, temperature=T, seeds=seeds, positions=pos, wide=wide,
                                          base_seed=3, offset=4)
        assert (again.out == full.out).all()
    # unseeded rows: the offset changes the draw (advanced every step)
    outs = {int(oracle.sample_from_logits(np.zeros(V), B=1, base_seed=3, offset=o).out[0])
            for o in range(8)}
    assert len(outs) > 4


def test_row_subset_equals_full_batch():
    rng = np.random.default_rng(10)
    B, D, V = 9, 64, 700
    H = torch.from_numpy(rng.standard_normal((B, D)).astype(np.float32)).to(torch.bfloat16)
    W = torch.from_numpy(rng.standard_normal((V, D)).astype(np.float32)).to(torch.bfloat16)
    T = rng.uniform(0.3, 1.2, B); T[2] = 0.0
    seeds = np.arange(B) + 50; seeds[[1, 5]] = -1
    pos = np.arange(B) * 3
    bias = rng.standard_normal((B, V))
    allowed = rng.random((B, V)) < 0.5
    mask = workloads.pack_allow_bits(torch.from_numpy(allowed)).numpy().view(np.uint32)
    kw = dict(temperature=T, seeds=seeds, positions=pos, bias=bias, mask=mask, base_seed=8,
              offset=2, wide=True)
    full = oracle.lmhead_sample(H, W, tile_v=128, **kw)
    rows = np.array([7, 1, 5, 2])
    sub = oracle.lmhead_sample_rows(H, W, rows, tile_v=128, **kw)
    assert (sub.out == full.out[rows]).all()
    assert (sub.status == full.status[rows]).all()
    assert (sub.tile_idx == full.tile_idx[rows]).all()
    assert np.array_equal(sub.tile_max, full.tile_max[rows])
