"""The noise layout that include/lms.h states ("Exact definitions") reproduces the oracle's noise.

A caller who replays the noise from the header alone (the Megatron-LM PR's "Tests" section
expects seeded noise to replay bit-exactly) must get the oracle's words and uniforms.  The
formula below is written out from the header's text, not imported: key and counter of call n,
the call and word(s) an entry takes, and the midpoint uniform.  The only routine borrowed is the
raw Philox4x32-10 call, which tests/test_oracle_philox.py pins against Triton's own Philox.
The test also checks that the header still states this layout, so that the two cannot drift
apart silently.
"""
import os
import re

import numpy as np
import pytest

import oracle

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
M32 = 0xFFFFFFFF


def _header_text():
    text = open(os.path.join(ROOT, "include", "lms.h")).read()
    text = re.sub(r"\n\s*\*(?!/)", "\n", text)       # comment continuation markers
    return re.sub(r"\s+", " ", text)


def test_header_states_the_packed_layout():
    h = _header_text()
    for phrase in ("counter (n, pos lo32, pos hi32, 0)",
                   "(n, offset lo32, offset hi32, 0x80000000 | b)",
                   "entry v takes word w[v & 3] of call n = v >> 2",
                   "entry v takes lo = w[2 (v & 1)] and hi = w[2 (v & 1) + 1] of call n = v >> 1",
                   "k = w >> 8", "u = (k + 1/2) / 2^24",
                   "k = ((hi << 32) | lo) >> 12", "u = (k + 1/2) / 2^52"):
        assert phrase in h, phrase


def _key_and_counter(b, n, seed, pos, base_seed, offset):
    """Key and counter of call n of row b, as the header states them."""
    if seed >= 0:
        return (seed & M32, (seed >> 32) & M32), (n, pos & M32, (pos >> 32) & M32, 0)
    return ((base_seed & M32, (base_seed >> 32) & M32),
            (n, offset & M32, (offset >> 32) & M32, 0x80000000 | b))


def _entry(b, v, seed, pos, base_seed, offset, wide):
    """(the call's four words, u) of entry v of row b from the header's formula."""
    n = v >> 1 if wide else v >> 2
    key, ctr = _key_and_counter(b, n, seed, pos, base_seed, offset)
    w = [int(x) for x in oracle.philox4x32([ctr], [key])[0]]
    if wide:
        lo, hi = w[2 * (v & 1)], w[2 * (v & 1) + 1]
        k = ((hi << 32) | lo) >> 12
        u = (k + 0.5) / 2.0 ** 52
    else:
        k = w[v & 3] >> 8
        u = (k + 0.5) / 2.0 ** 24
    return w, u


@pytest.mark.parametrize("wide", [False, True])
def test_header_formula_reproduces_the_oracle_noise(wide):
    B, V = 5, 1031
    seeds = np.array([1234, -1, 2 ** 40 + 7, 0, -5], np.int64)
    positions = np.array([0, 17, 2 ** 33 + 3, 99, 4], np.int64)
    base_seed, offset = 2 ** 35 + 11, 2 ** 32 + 9
    words, u, _, _ = oracle.noise(B, V, seeds, positions, base_seed, offset, wide)
    rng = np.random.default_rng(3)
    vs = sorted(set([0, 1, 2, 3, 4, 5, 6, 7, V - 1, V - 2, V - 3]) |
                set(int(x) for x in rng.integers(0, V, 24)))
    for b in range(B):
        for v in vs:
            w, uh = _entry(b, v, int(seeds[b]), int(positions[b]), base_seed, offset, wide)
            assert [int(x) for x in words[b, v]] == w, (b, v)
            assert u[b, v] == uh, (b, v, u[b, v], uh)


def test_entries_of_one_call_share_its_words_and_use_distinct_ones():
    # fp32 noise: entries 4n..4n+3 take the four different words of call n; wide noise: entries
    # 2n and 2n+1 take its two halves.  No word is dropped.
    for wide, per in ((False, 4), (True, 2)):
        words, u, _, _ = oracle.noise(1, 16, np.array([77]), np.array([5]), 0, 0, wide)
        for n in range(16 // per):
            block = words[0, per * n: per * (n + 1)]
            assert (block == block[0]).all()
            assert len(set(u[0, per * n: per * (n + 1)].tolist())) == per
