"""Pins for the oracle's filtered race (top-k -> top-p -> min-p, then the Gumbel race).

spec-decode-ops, "Semantics", and the sampling-kernel guide (reasoning steps 6-8, "Correctness
requirements") fix the following:

- top-k keeps the k most likely tokens;
- top-p keeps the smallest sorted prefix whose probability mass, normalised over the top-k prefix,
  reaches top_p, the crossing token included;
- min-p keeps p >= min_p * p_max;
- every filter keeps at least one token;
- the draw is the softmax renormalised over what is kept.

Each expected kept set below is worked out by hand from probabilities chosen so that the set is
evident. The sampled law is checked by chi-square against the renormalised softmax.
"""
import math

import numpy as np
import pytest
from scipy import stats

import oracle

# probabilities 0.5, 0.3, 0.15, 0.05 (T = 1): logits are their logs
P4 = np.array([0.5, 0.3, 0.15, 0.05])
Y4 = np.log(P4)
N = 200_000


def draws(y, **kw):
    out, status, kept = oracle.sample_filtered(y, B=N, seeds=np.full(N, 99), positions=np.arange(N),
                                               **{k: (np.full(N, v) if np.isscalar(v) else v)
                                                  for k, v in kw.items()})
    assert (status == 0).all()
    return out, kept


def chi2_ok(out, law):
    counts = np.bincount(out, minlength=len(law)).astype(float)
    keep = law > 0
    assert counts[~keep].sum() == 0, "a filtered-out token was drawn"
    exp = law[keep] / law[keep].sum() * len(out)
    stat = ((counts[keep] - exp) ** 2 / exp).sum()
    return stat < stats.chi2.isf(1e-6, max(1, keep.sum() - 1))


@pytest.mark.parametrize("kw,kept_set", [
    (dict(top_k=2), [0, 1]),
    (dict(top_k=3), [0, 1, 2]),
    (dict(top_p=0.7), [0, 1]),              # mass 0.5, 0.8: the crossing token (1) is kept
    (dict(top_p=0.79), [0, 1]),
    (dict(top_p=0.81), [0, 1, 2]),
    (dict(top_p=0.1), [0]),                 # always at least the top token
    (dict(min_p=0.25), [0, 1, 2]),          # p >= 0.125
    (dict(min_p=0.55), [0, 1]),             # p >= 0.275
    (dict(min_p=0.99), [0]),
    (dict(top_k=3, top_p=0.9), [0, 1, 2]),  # over the top-3: 0.526, 0.842, 1.0
    (dict(top_k=3, top_p=0.8), [0, 1]),
    (dict(top_k=3, min_p=0.5), [0, 1]),
])
def test_kept_sets_and_law(kw, kept_set):
    out, kept = draws(Y4, **kw)
    assert (kept == len(kept_set)).all()
    law = np.zeros(4)
    law[kept_set] = P4[kept_set]
    assert chi2_ok(out, law)


def test_ties_at_the_top_k_boundary_keep_the_smallest_indices():
    y = np.array([1.0, 1.0, 1.0, 0.0])
    out, kept = draws(y, top_k=2)
    assert set(np.unique(out)) == {0, 1}
    assert chi2_ok(out, np.array([0.5, 0.5, 0.0, 0.0]))
    out, _ = draws(y, min_p=1.0)            # t_i - t_max >= log(1): the three tied tokens
    assert chi2_ok(out, np.array([1 / 3, 1 / 3, 1 / 3, 0.0]))


def test_no_filter_equals_the_plain_race():
    rng = np.random.default_rng(3)
    y = rng.standard_normal((50, 300)) * 2
    T = rng.uniform(0.4, 1.3, 50)
    seeds = np.arange(50) + 7
    seeds[::3] = -1
    plain = oracle.sample_from_logits(y, temperature=T, seeds=seeds, positions=np.arange(50),
                                      base_seed=5, offset=2, wide=True)
    out, status, kept = oracle.sample_filtered(y, temperature=T, seeds=seeds,
                                               positions=np.arange(50), base_seed=5, offset=2,
                                               wide=True, top_k=np.zeros(50), top_p=np.ones(50),
                                               min_p=np.zeros(50))
    assert (out == plain.out).all() and (kept == 300).all()


def test_greedy_rows_ignore_filters_and_masks_apply():
    y = np.array([[0.1, 3.0, 2.9, -1.0]] * 3)
    T = np.array([0.0, 0.0, 1.0])
    mask = np.array([0b1111, 0b1101, 0b1101], np.uint32)[:, None]   # rows 1, 2: token 1 masked
    out, status, kept = oracle.sample_filtered(y, temperature=T, mask=mask, top_k=np.array([1, 2, 1]),
                                               top_p=np.array([0.5, 0.5, 0.5]), base_seed=1)
    assert list(out) == [1, 2, 2] and (status == 0).all()


def test_top_p_without_top_k_uses_the_k_max_prefix():
    # 3000 equal tokens, top_p = 0.9 with k_max = 1024: the prefix is cut at k_max first, so the
    # kept set is 922 tokens (0.9 of the 1024 renormalised) rather than 2700
    y = np.zeros(3000)
    _, _, kept = oracle.sample_filtered(y, B=2, top_p=np.full(2, 0.9), k_max=1024)
    assert (kept == math.ceil(0.9 * 1024 - 1e-9)).all()
