"""GPU noise generator against the oracle: Philox words bit-exact, the uniform bit-exact, E and g
within the fp32 bound; replay under contention; single-row launches equal batched ones
(Megatron-LM PR 8370, "Tests": the noise replays bit-exactly under side-stream contention and
single-row launches equal batched ones; the noise range)."""
import math

import numpy as np
import pytest
import torch

import lm_head_gumbel_lmhead_gb300 as lms
import oracle

pytestmark = pytest.mark.gpu

# fp32 noise error bound (derivation in the design notes): E to a few ulp relative, g to
# ~4e-7 + 3 ulp of |g|.
E_RTOL = 2.0 ** -20
G_ATOL, G_RTOL = 2e-6, 1e-6


def _u32(t):
    return t.cpu().numpy().view(np.uint32)


@pytest.fixture(scope="module")
def rows():
    B = 37
    seeds = np.arange(B, dtype=np.int64) * 1_000_003 + 5
    seeds[::4] = -1
    seeds[5] = 2**40 + 17
    pos = np.arange(B, dtype=np.int64) * 977
    pos[6] = 2**33 + 3
    return B, seeds, pos


@pytest.mark.parametrize("wide", [False, True])
def test_words_uniform_noise_match_oracle(rows, wide):
    B, seeds, pos = rows
    V = 3001
    dev = torch.device("cuda")
    sd, pd = torch.from_numpy(seeds).to(dev), torch.from_numpy(pos).to(dev)
    kw = dict(wide=wide, seeds=sd, positions=pd, base_seed=0xABCDEF0123, offset=2**32 + 9)
    words = lms.philox_fill_noise(B, V, kind="words", **kw)
    u = lms.philox_fill_noise(B, V, kind="uniform", **kw)
    E = lms.philox_fill_noise(B, V, kind="exponential", **kw)
    g = lms.philox_fill_noise(B, V, kind="gumbel", **kw)
    ow, ou, oE, og = oracle.noise(B, V, seeds, pos, 0xABCDEF0123, 2**32 + 9, wide)
    assert np.array_equal(_u32(words), ow)
    assert np.array_equal(u.cpu().numpy(), ou)
    Eg = E.cpu().numpy().astype(np.float64)
    assert np.all(np.abs(Eg - oE) <= E_RTOL * oE)
    gg = g.cpu().numpy().astype(np.float64)
    assert np.all(np.abs(gg - og) <= G_ATOL + G_RTOL * np.abs(og))


@pytest.mark.parametrize("wide", [False, True])
def test_noise_extremes_keep_the_tail(wide):
    # 2^26 draws: the largest and smallest u of the grid, computed from the GPU's (bit-exact)
    # words by the oracle, against the GPU's E -- the far tail E -> 0 keeps relative precision.
    B, V = 64, 1 << 20
    dev = torch.device("cuda")
    kw = dict(wide=wide, base_seed=77, offset=1)
    E = lms.philox_fill_noise(B, V, kind="exponential", **kw)
    flat = E.view(-1)
    idx = torch.cat([torch.topk(flat, 16).indices, torch.topk(-flat, 16).indices]).cpu().numpy()
    words = lms.philox_fill_noise(B, V, kind="words", **kw).view(-1, 4)[torch.from_numpy(idx).to(dev)]
    w = _u32(words)
    lo, hi = oracle.entry_words(w, idx % V, wide)
    ref = np.array([-math.log(oracle.uniform(int(a), int(b), wide)) for a, b in zip(lo, hi)])
    got = flat[torch.from_numpy(idx).to(dev)].cpu().numpy().astype(np.float64)
    assert np.all(np.abs(got - ref) <= E_RTOL * ref)
    lo_bound = 2.0 ** -53 if wide else 2.0 ** -25
    hi_bound = (53 if wide else 25) * math.log(2)
    assert got.min() >= lo_bound * (1 - 1e-6) and got.max() <= hi_bound * (1 + 1e-6)
    if not wide:
        # with 2^26 draws the fp32 extremes are reached within a few cells of 2^-24
        assert got.min() < 3 * 2.0 ** -24


@pytest.mark.parametrize("wide", [False, True])
def test_noise_dense_grid_matches_oracle(wide):
    # 2^22 entries, every one against the oracle's fp64 E and g: covers both evaluations of E
    # (from u, and from the exact complement c below 3/8) and the switch between them.
    B, V = 16, 1 << 18
    seeds = np.arange(B, dtype=np.int64) * 7919 + 3
    seeds[::3] = -1
    pos = np.arange(B, dtype=np.int64) * 11 + 2**31
    dev = torch.device("cuda")
    kw = dict(wide=wide, seeds=torch.from_numpy(seeds).to(dev), positions=torch.from_numpy(pos).to(dev),
              base_seed=99, offset=5)
    E = lms.philox_fill_noise(B, V, kind="exponential", **kw).cpu().numpy().astype(np.float64)
    g = lms.philox_fill_noise(B, V, kind="gumbel", **kw).cpu().numpy().astype(np.float64)
    _, ou, oE, og = oracle.noise(B, V, seeds, pos, 99, 5, wide)
    rel = np.abs(E - oE) / oE
    assert rel.max() <= E_RTOL, (rel.max(), ou.reshape(-1)[rel.argmax()])
    assert np.all(np.abs(g - og) <= G_ATOL + G_RTOL * np.abs(og))
    # both evaluations were exercised: u <= 5/8 and u > 5/8 each hold about their share
    frac_c = np.mean(ou > 5 / 8)
    assert 0.35 < frac_c < 0.40


def test_replay_under_contention_and_single_row_equals_batched(rows):
    B, seeds, pos = rows
    V = 50_000
    dev = torch.device("cuda")
    sd, pd = torch.from_numpy(seeds).to(dev), torch.from_numpy(pos).to(dev)
    ref = lms.philox_fill_noise(B, V, kind="words", wide=True, seeds=sd, positions=pd, base_seed=3)
    side = torch.cuda.Stream()
    a = torch.randn(4096, 4096, device=dev)
    with torch.cuda.stream(side):
        for _ in range(20):
            a = a @ a
            a = a / a.norm()
    again = lms.philox_fill_noise(B, V, kind="words", wide=True, seeds=sd, positions=pd, base_seed=3)
    torch.cuda.synchronize()
    assert torch.equal(ref, again)
    for b in np.nonzero(seeds >= 0)[0][:6]:
        one = lms.philox_fill_noise(1, V, kind="words", wide=True, seeds=sd[b:b + 1],
                                    positions=pd[b:b + 1], base_seed=3)
        assert torch.equal(one[0], ref[b])
    # the fp32 stream: entry v takes the top 24 bits of word v & 3 of its call
    w32 = _u32(lms.philox_fill_noise(B, V, kind="words", wide=False, seeds=sd, positions=pd, base_seed=3))
    u32 = lms.philox_fill_noise(B, V, kind="uniform", wide=False, seeds=sd, positions=pd, base_seed=3)
    lo, _ = oracle.entry_words(w32, np.arange(V)[None, :].repeat(B, 0), False)
    assert np.array_equal(u32.cpu().numpy(), (np.floor(lo.astype(np.float64) / 256) * 2 + 1) * 2.0 ** -25)


@pytest.mark.parametrize("wide", [False, True])
@pytest.mark.parametrize("kind", ["exponential", "gumbel"])
def test_unaligned_output_buffer_matches_aligned(wide, kind):
    # the entry point takes any 4-byte aligned buffer: one offset by 4 bytes (scalar stores)
    # holds the same values as an aligned one (16- or 8-byte stores), for V a multiple of 4 and not
    B = 5
    for V in (4096, 1001):
        ref = lms.philox_fill_noise(B, V, kind=kind, wide=wide, base_seed=11, offset=3)
        raw = torch.empty(B * V + 1, dtype=torch.float32, device="cuda")
        off = raw[1:].view(B, V)
        assert off.data_ptr() % 16 == 4
        lms.philox_fill_noise(B, V, kind=kind, wide=wide, base_seed=11, offset=3, out=off)
        assert torch.equal(off, ref)
