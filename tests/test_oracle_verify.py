"""Pins for the oracle's speculative-decoding verification (spec-decode-ops "verify").

The laws come from the rejection-sampling construction itself, not from the oracle's code:

- with each draft token drawn from the draft distribution, the first emitted token follows the
  target distribution exactly, and the first acceptance happens with probability
  sum_v min(p_t(v), p_d(v)) (the page's "Measured behavior" checks both);
- given a rejection at position 0, the emitted token follows max(p_t - p_d, 0) renormalised;
- with fixed logits and independent draft draws, the accept length m in {0..k} has the law
  P(m) = (prod_{i<m} a_i) (1 - a_m) for m < k and prod a_i for m = k, a_i the acceptance rates;
- a fully accepted row's bonus token is the plain race's draw at that absolute position (the
  C race, not the verifier's numpy code);
- greedy rows accept while the draft token is the target argmax; invalid and masked rows keep the
  race's statuses; seeded rows are invariant to their batch position.
"""
import numpy as np
import pytest
from scipy import stats

import oracle


def softmax(z):
    e = np.exp(z - z.max(axis=-1, keepdims=True))
    return e / e.sum(axis=-1, keepdims=True)


def draft_draws(pd, n, rng):
    """n draft tokens per position from pd [k, V] (numpy's generator; independent of Philox)."""
    k, V = pd.shape
    return np.stack([rng.choice(V, size=n, p=pd[i]) for i in range(k)], axis=1)


def chi2_ok(counts, law):
    keep = law > 0
    assert counts[~keep].sum() == 0
    exp = law[keep] / law[keep].sum() * counts.sum()
    stat = ((counts[keep] - exp) ** 2 / exp).sum()
    return stat < stats.chi2.isf(1e-6, max(1, keep.sum() - 1)), stat


PT = np.log(np.array([0.35, 0.25, 0.2, 0.1, 0.06, 0.04]))
PD = np.log(np.array([0.1, 0.4, 0.1, 0.25, 0.1, 0.05]))     # a deliberately mismatched draft


def test_first_token_is_the_target_law_and_acceptance_rate():
    rng = np.random.default_rng(1)
    n, V = 120_000, 6
    pt, pd = softmax(PT), softmax(PD)
    x = draft_draws(pd[None], n, rng)
    tgt = np.broadcast_to(np.stack([PT, PT]), (n, 2, V))
    dft = np.broadcast_to(PD[None], (n, 1, V))
    acc, out, st = oracle.verify_from_logits(tgt, dft, x, seeds=np.arange(n) + 5,
                                             positions=np.zeros(n, np.int64))
    assert (st == 0).all()
    ok, stat = chi2_ok(np.bincount(out[:, 0], minlength=V).astype(float), pt)
    assert ok, stat
    alpha = np.minimum(pt, pd).sum()
    rate = (acc == 1).mean()
    assert abs(rate - alpha) < 5 * np.sqrt(alpha * (1 - alpha) / n), (rate, alpha)
    # given a rejection, the residual law
    r = np.maximum(pt - pd, 0.0)
    ok, stat = chi2_ok(np.bincount(out[acc == 0, 0], minlength=V).astype(float), r / r.sum())
    assert ok, stat


def test_accept_length_law_k4():
    rng = np.random.default_rng(2)
    n, V, k = 50_000, 6, 4
    shifts = [0.0, 0.6, 1.2, 0.3]
    tl = np.stack([PT + 0.2 * i for i in range(k + 1)])
    dl = np.stack([PD * (1 + shifts[i]) for i in range(k)])
    pt, pd = softmax(tl), softmax(dl)
    x = draft_draws(pd, n, rng)
    acc, out, st = oracle.verify_from_logits(np.broadcast_to(tl, (n, k + 1, V)),
                                             np.broadcast_to(dl, (n, k, V)), x,
                                             seeds=np.arange(n), positions=np.arange(n) * 7)
    a = np.minimum(pt[:k], pd).sum(axis=1)
    law = np.array([np.prod(a[:m]) * (1 - a[m]) for m in range(k)] + [np.prod(a)])
    ok, stat = chi2_ok(np.bincount(acc, minlength=k + 1).astype(float), law)
    assert ok, stat
    # emitted prefixes are the draft tokens; the next token is set; nothing after it
    for m in range(k + 1):
        rows = acc == m
        assert np.array_equal(out[rows, :m], x[rows, :m])
        assert (out[rows, m] >= 0).all() and (out[rows, m + 1:] == -1).all()


@pytest.mark.parametrize("wide", [False, True])
def test_bonus_token_is_the_plain_race_at_its_position(wide):
    rng = np.random.default_rng(3)
    B, k, V = 16, 3, 500
    tl = rng.standard_normal((B, k + 1, V))
    dl = tl[:, :k].copy()                     # the draft equals the target: always accepted
    T = rng.uniform(0.5, 1.5, B)
    x = np.array([[int(np.argmax(tl[b, i])) for i in range(k)] for b in range(B)])
    seeds = np.arange(B) + 40
    pos = np.arange(B) * 11
    acc, out, st = oracle.verify_from_logits(tl, dl, x, temperature=T, seeds=seeds, positions=pos,
                                             wide=wide)
    assert (acc == k).all() and np.array_equal(out[:, :k], x)
    race = oracle.sample_from_logits(tl[:, k], temperature=T, seeds=seeds, positions=pos + k,
                                     wide=wide)
    assert np.array_equal(out[:, k], race.out)


def test_greedy_invalid_and_masked_rows():
    rng = np.random.default_rng(4)
    B, k, V = 5, 3, 50
    tl = rng.standard_normal((B, k + 1, V))
    dl = rng.standard_normal((B, k, V))
    x = np.array([[int(np.argmax(tl[b, i])) for i in range(k)] for b in range(B)])
    x[1, 1] = (x[1, 1] + 1) % V                # row 1: the second draft token is not the argmax
    tl[3, 0] = -np.inf                          # row 3: nothing finite at position 0
    T = np.array([0.0, 0.0, -1.0, 1.0, np.nan])
    acc, out, st = oracle.verify_from_logits(tl, dl, x, temperature=T, seeds=np.arange(B),
                                             positions=np.arange(B))
    assert acc[0] == k and np.array_equal(out[0, :k], x[0]) and out[0, k] == np.argmax(tl[0, k])
    assert acc[1] == 1 and out[1, 1] == np.argmax(tl[1, 1]) and (out[1, 2:] == -1).all()
    assert st[2] == 2 and st[4] == 2 and (out[2] == -1).all()
    assert st[3] == 1 and (out[3] == -1).all()
    # nothing finite at the drawn position after an accepted prefix: no token at all
    tl2 = tl[:2].copy()
    tl2[:, 1] = -np.inf
    tl2[1, 1, 7] = np.nan
    acc2, out2, st2 = oracle.verify_from_logits(tl2, tl2[:, :k], x[:2, :], temperature=[0.0, 1.0],
                                                seeds=[1, 2], positions=[0, 0])
    assert (st2 == 1).all() and (acc2 == 0).all() and (out2 == -1).all()


def test_seeded_rows_are_batch_position_invariant():
    rng = np.random.default_rng(5)
    B, k, V = 10, 2, 40
    tl = rng.standard_normal((B, k + 1, V))
    dl = tl[:, :k] + rng.standard_normal((B, k, V))
    x = rng.integers(0, V, (B, k))
    seeds, pos = np.arange(B) + 3, np.arange(B) * 5
    acc, out, _ = oracle.verify_from_logits(tl, dl, x, seeds=seeds, positions=pos)
    perm = rng.permutation(B)
    acc_p, out_p, _ = oracle.verify_from_logits(tl[perm], dl[perm], x[perm], seeds=seeds[perm],
                                                positions=pos[perm])
    assert np.array_equal(acc_p, acc[perm]) and np.array_equal(out_p, out[perm])
