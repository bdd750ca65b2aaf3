"""Pins for the oracle's Gumbel-top-k (k draws without replacement).

The FlashSampling page ("Limitations", "Future directions") names the top-k extension of the
Gumbel-max race: the k largest perturbed scores, in order, are k draws without replacement from
the softmax.  Pins, none of which re-types the oracle's selection:

- the ordered-pair law of the first two draws is the Plackett-Luce (successive sampling) law
  p_i p_j / (1 - p_i), by chi-square over 400k draws;
- k = 1 equals the race's own argmax (a C loop, not a sort);
- indices and scores equal a numpy recomputation from the pinned noise grid;
- greedy rows give numpy's stable descending argsort;
- rows with fewer finite scores than k end in -1; all-masked and invalid rows keep the race's
  statuses;
- the two-stage split is exact: per-tile top-k lists merged give the global top-k, for every tile
  width on rows full of ties;
- seeded rows are invariant to their batch position.
"""
import numpy as np
import pytest
from scipy import stats

import oracle

P5 = np.array([0.4, 0.25, 0.2, 0.1, 0.05])


def test_ordered_pairs_follow_plackett_luce():
    n = 400_000
    idx, val, st = oracle.gumbel_topk(np.log(P5), 2, B=n, seeds=np.full(n, 17),
                                      positions=np.arange(n))
    assert (st == 0).all() and (idx[:, 0] != idx[:, 1]).all() and (val[:, 0] >= val[:, 1]).all()
    counts = np.zeros((5, 5))
    np.add.at(counts, (idx[:, 0], idx[:, 1]), 1)
    law = P5[:, None] * P5[None, :] / (1.0 - P5[:, None])
    np.fill_diagonal(law, 0.0)
    assert abs(law.sum() - 1.0) < 1e-12
    off = ~np.eye(5, dtype=bool)
    exp = law[off] * n
    stat = ((counts[off] - exp) ** 2 / exp).sum()
    assert stat < stats.chi2.isf(1e-6, off.sum() - 1), stat
    assert counts[np.eye(5, dtype=bool)].sum() == 0


def test_first_draw_is_the_race_and_k1_equals_it():
    rng = np.random.default_rng(3)
    B, V = 40, 3000
    y = rng.standard_normal((B, V)) * 2
    T = rng.uniform(0.3, 1.5, B)
    T[[0, 7]] = 0.0
    seeds = np.arange(B) * 5 + 1
    seeds[::4] = -1
    kw = dict(temperature=T, seeds=seeds, positions=np.arange(B) + 9, base_seed=3, offset=11)
    race = oracle.sample_from_logits(y, **kw)
    for k in (1, 8):
        idx, val, st = oracle.gumbel_topk(y, k, **kw)
        assert np.array_equal(idx[:, 0], race.out) and np.array_equal(st, race.status)
        assert np.array_equal(val[:, 0], race.top1)
        if k > 1:
            assert np.array_equal(val[:, 1], race.top2)


@pytest.mark.parametrize("wide", [False, True])
def test_matches_numpy_from_the_noise_grid(wide):
    rng = np.random.default_rng(5)
    B, V, k = 6, 777, 16
    y = rng.standard_normal((B, V))
    T = np.array([0.5, 1.0, 2.0, 0.8, 1.3, 0.7])
    seeds = np.array([1, 2, -1, 4, 5, -1])
    pos = np.arange(B) * 3
    idx, val, _ = oracle.gumbel_topk(y, k, temperature=T, seeds=seeds, positions=pos,
                                     base_seed=21, offset=8, wide=wide)
    _, _, _, g = oracle.noise(B, V, seeds, pos, 21, 8, wide)
    s = y / T[:, None] + g
    for b in range(B):
        ref = np.lexsort((np.arange(V), -s[b]))[:k]
        assert np.array_equal(idx[b], ref)
        assert np.allclose(val[b], s[b][ref], rtol=0, atol=1e-12)
        assert len(set(idx[b])) == k and (np.diff(val[b]) <= 0).all()


def test_greedy_rows_are_the_deterministic_top_k():
    rng = np.random.default_rng(6)
    y = np.round(rng.standard_normal((4, 500)) * 3) / 2          # ties
    idx, val, st = oracle.gumbel_topk(y, 12, temperature=np.zeros(4))
    for b in range(4):
        ref = np.argsort(-y[b], kind="stable")[:12]
        assert np.array_equal(idx[b], ref) and np.array_equal(val[b], y[b][ref])
    assert (st == 0).all()


def test_short_masked_and_invalid_rows():
    V, k = 64, 5
    y = np.zeros((3, V))
    allowed = np.zeros((3, V), bool)
    allowed[0, [3, 40, 63]] = True                               # three tokens left
    allowed[2] = True
    words = np.zeros((3, 2), np.uint32)
    for b in range(3):
        for v in np.nonzero(allowed[b])[0]:
            words[b, v // 32] |= np.uint32(1) << np.uint32(v % 32)
    T = np.array([1.0, 1.0, -1.0])
    idx, val, st = oracle.gumbel_topk(y, k, temperature=T, seeds=np.arange(3), positions=np.arange(3),
                                      mask=words)
    assert sorted(idx[0, :3]) == [3, 40, 63] and (idx[0, 3:] == -1).all() and (val[0, 3:] == -np.inf).all()
    assert st[0] == 0
    assert st[1] == 1 and (idx[1] == -1).all()                   # nothing allowed
    assert st[2] == 2 and (idx[2] == -1).all()                   # invalid temperature


def test_per_tile_lists_merged_give_the_global_top_k():
    rng = np.random.default_rng(8)
    B, V, k = 5, 301, 7
    s = np.round(rng.standard_normal((B, V)) * 2) / 4            # many ties across tiles
    s[1, 100:] = -np.inf
    s[3] = 0.0                                                   # everything tied
    want_i, want_v = oracle.topk_from_scores(s, k)
    for tile_v in (1, 7, 64, 128, 300, 301, 512):
        ti, tv = oracle.tile_topk_from_scores(s, k, tile_v)
        flat_i, flat_v = ti.reshape(B, -1), tv.reshape(B, -1)
        merged = np.full((B, V), -np.inf)
        for b in range(B):
            ok = flat_i[b] >= 0
            merged[b, flat_i[b][ok]] = flat_v[b][ok]
        got_i, got_v = oracle.topk_from_scores(merged, k)
        assert np.array_equal(got_i, want_i) and np.array_equal(got_v, want_v), tile_v


def test_seeded_rows_are_batch_position_invariant():
    rng = np.random.default_rng(9)
    B, V = 12, 1000
    y = rng.standard_normal((B, V))
    seeds = np.arange(B) + 100
    pos = np.arange(B) * 7
    T = np.full(B, 0.9)
    idx, _, _ = oracle.gumbel_topk(y, 10, temperature=T, seeds=seeds, positions=pos)
    perm = rng.permutation(B)
    idx_p, _, _ = oracle.gumbel_topk(y[perm], 10, temperature=T[perm], seeds=seeds[perm],
                                     positions=pos[perm])
    assert np.array_equal(idx_p, idx[perm])
