"""Pins for the oracle's uniform -> exponential -> Gumbel noise.

What the pages fix (Megatron-LM PR 8370):
  * "The change": two Philox words give the 52-bit midpoint uniform (k + 1/2)/2^52 and the
    exponential noise then lies in [1.1e-16, 36.7] with no endpoint clamp;
  * "Problem": a float32 uniform keeps 24 bits near 1 and caps the noise ratio near e^20.
Mathematics fixes the rest: E = -log U is Exp(1) (mean 1, variance 1) and g = -log E is
Gumbel(0, 1) (mean = Euler-Mascheroni constant, variance pi^2/6); U is uniform on (0, 1).
"""
import math

import numpy as np
import pytest
from scipy import stats

import oracle

EULER_GAMMA = 0.5772156649015329


def _E(w0, w1, wide):
    return -math.log(oracle.uniform(w0, w1, wide))


def test_wide_noise_range_matches_page(golden):
    page = golden["wide_noise_range"]
    e_max = _E(0, 0, True)                      # k = 0
    e_min = _E(0xFFFFFFFF, 0xFFFFFFFF, True)    # k = 2^52 - 1
    assert e_max == pytest.approx(53 * math.log(2), rel=1e-15)
    assert f"{e_max:.1f}" == f"{page['E_max_printed']:.1f}"
    assert f"{e_min:.1e}" == f"{page['E_min_printed']:.1e}"
    # the representable tail: log(E_max / E_min) is about 40 nats
    assert round(math.log(e_max / e_min) / 10) * 10 == page["tail_nats_printed"]


def test_fp32_noise_tail_caps_near_e20(golden):
    page = golden["fp32_noise_tail"]
    e_max = _E(0, 0, False)
    e_min = _E(0xFFFFFFFF, 0, False)
    assert e_max == pytest.approx(25 * math.log(2), rel=1e-15)
    assert e_min == pytest.approx(2.0 ** -25, rel=1e-7)
    assert round(math.log(e_max / e_min)) == page["max_log_ratio_printed"]
    # the low 8 bits of word 0 and all of word 1 are unused in fp32 mode
    assert oracle.uniform(0x12345600, 0xABCDEF, False) == oracle.uniform(0x123456FF, 0, False)


def test_uniform_is_midpoint_of_its_cell_and_inside_unit_interval():
    for wide, m in [(False, 24), (True, 52)]:
        lo = oracle.uniform(0, 0, wide)
        hi = oracle.uniform(0xFFFFFFFF, 0xFFFFFFFF, wide)
        assert lo == 2.0 ** -(m + 1) and hi == 1 - 2.0 ** -(m + 1)
        assert 0.0 < lo < hi < 1.0
    # wide: word 1 carries the high bits
    assert oracle.uniform(0, 0x80000000, True) == 0.5 + 2.0 ** -53
    assert oracle.uniform(0, 0x80000000, False) == oracle.uniform(0, 0, False)


@pytest.fixture(scope="module")
def noise_draws():
    B, V = 64, 16384          # 2^20 draws per mode
    res = {}
    for wide in (False, True):
        seeds = np.arange(B, dtype=np.int64) * 7 + 1
        seeds[::3] = -1       # mix seeded and unseeded rows
        _, u, E, g = oracle.noise(B, V, seeds, np.arange(B, dtype=np.int64) * 11, 99, 5, wide)
        res[wide] = (u.ravel(), E.ravel(), g.ravel())
    return res


@pytest.mark.parametrize("wide", [False, True])
def test_uniform_is_uniform(noise_draws, wide):
    u, _, _ = noise_draws[wide]
    assert stats.kstest(u, "uniform").pvalue > 1e-4
    assert abs(u.mean() - 0.5) < 5 * math.sqrt(1 / 12 / u.size)


@pytest.mark.parametrize("wide", [False, True])
def test_exponential_and_gumbel_moments(noise_draws, wide):
    _, E, g = noise_draws[wide]
    n = E.size
    assert abs(E.mean() - 1.0) < 5 / math.sqrt(n)
    assert abs(E.var() - 1.0) < 5 * math.sqrt(8 / n)
    assert abs(g.mean() - EULER_GAMMA) < 5 * math.sqrt(math.pi ** 2 / 6 / n)
    assert abs(g.var() - math.pi ** 2 / 6) < 0.02
    assert stats.kstest(E, "expon").pvalue > 1e-4
    assert stats.kstest(g, "gumbel_r").pvalue > 1e-4


def test_noise_is_consistent_with_words():
    B, V = 3, 257
    seeds = np.array([5, -1, 2**40], np.int64)
    pos = np.array([0, 0, 2**33 + 1], np.int64)
    for wide in (False, True):
        words, u, E, g = oracle.noise(B, V, seeds, pos, 77, 3, wide)
        for b, v in [(0, 0), (1, 100), (2, 256), (0, 3), (1, 5)]:
            lo, hi = oracle.entry_words(words[b, v], v, wide)
            assert u[b, v] == oracle.uniform(int(lo), int(hi), wide)
            assert E[b, v] == -math.log(u[b, v])
            assert g[b, v] == -math.log(E[b, v])


@pytest.mark.parametrize("wide", [False, True])
def test_each_call_serves_consecutive_entries_without_dropping_words(wide):
    # fp32 noise: entries 4n..4n+3 share call n and use its four words once each; wide noise:
    # entries 2n, 2n+1 share call n and use words (0, 1) and (2, 3).  The call is Philox at
    # counter word 0 = n with the row's key -- the same (seed, position, v) keying for every v.
    B, V = 2, 64
    seeds = np.array([11, -1], np.int64)
    pos = np.array([2**35 + 7, 0], np.int64)
    words, u, _, _ = oracle.noise(B, V, seeds, pos, 5, 9, wide)
    per = 2 if wide else 4
    for b in range(B):
        for n in range(V // per):
            group = words[b, per * n: per * (n + 1)]
            assert (group == group[0]).all()
            used = []
            for v in range(per * n, per * (n + 1)):
                lo, hi = oracle.entry_words(words[b, v], v, wide)
                used += [int(lo)] + ([int(hi)] if wide else [])
            assert sorted(used) == sorted(int(x) for x in group[0])
        # the call itself: Philox4x32-10 at counter (n, pos lo, pos hi, 0) with key = seed
        if seeds[b] >= 0:
            n = 3
            ctr = np.array([[n, pos[b] & 0xFFFFFFFF, pos[b] >> 32, 0]], np.uint64).astype(np.uint32)
            key = np.array([[seeds[b] & 0xFFFFFFFF, seeds[b] >> 32]], np.uint64).astype(np.uint32)
            assert (oracle.philox4x32(ctr, key)[0] == words[b, per * n]).all()
        # neighbouring entries get different uniforms
        assert len(set(u[b].tolist())) == V
