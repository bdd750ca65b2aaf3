"""Speculative-decoding verification (spec-decode-ops "verify") on the GPU against the oracle,
and the laws of the rejection-sampling construction measured on the GPU's own draws.

Parity, per row: statuses equal; accept lengths and emitted tokens equal, with two exceptions the
arithmetic allows (counted, and bounded by the tests that use them):
  * an acceptance test whose oracle margin |u p_d - p_t| is below MARGIN: the kernels form
    p = exp(y / T - log Z) in fp32 (about 1e-6 absolute error against the oracle's fp64), so the
    two sides may decide it either way; the row is then compared up to that position;
  * the final draw on a near-tie row: the GPU's token must score (by the oracle) within its error
    interval of the oracle's top score.  The interval is the race's NEAR_TIE, widened for a
    residual entry by the fp32 cancellation in p_t - p_d (relative error ~ eps (p_t + p_d) / r).
Laws (the "Measured behavior" of the spec-decode-ops page): the first emitted token follows the
target distribution with a deliberately mismatched draft; the acceptance rate is
sum_v min(p_t, p_d); the k = 4 accept-length law is P(m) = prod_{i<m} a_i (1 - a_m).
Also: a fully accepted row's bonus token is sample_from_logits' token at position pos + k, bit for
bit; a rejection with a zero residual falls back to the target's own race, bit for bit.
"""
import numpy as np
import pytest
import torch
from scipy import stats

import lm_head_gumbel_lmhead_gb300 as lms
import oracle
from parity import NEAR_TIE
from parity import _add as count_parity

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda")
MARGIN = 1e-5


def _softmax_rows(z):
    z = np.where(np.isnan(z), -np.inf, z)
    m = z.max(axis=-1, keepdims=True)
    e = np.exp(z - np.where(np.isfinite(m), m, 0.0))
    s = e.sum(axis=-1, keepdims=True)
    return np.divide(e, s, out=np.zeros_like(e), where=s > 0)


def draw_tokens(dl, T, rng):
    """Draft tokens from the draft's own distribution at temperature T (numpy's generator)."""
    B, k, V = dl.shape
    x = np.zeros((B, k), np.int64)
    for b in range(B):
        Tb = T[b] if T[b] > 0 else 1.0
        p = _softmax_rows(dl[b] / Tb)
        for i in range(k):
            x[b, i] = rng.choice(V, p=p[i]) if p[i].sum() > 0 else 0
    return x


def _rounded(z, dtype):
    """The values the kernels see: z rounded to dtype, back in fp64."""
    return torch.from_numpy(z).to(dtype).double().numpy()


def make_case(B, k, V, seed, features=True, dtype=torch.float32):
    rng = np.random.default_rng(seed)
    tl = _rounded(rng.standard_normal((B, k + 1, V)) * 2.0, dtype)
    spread = rng.uniform(0.05, 1.5, B)
    dl = _rounded(tl[:, :k] + rng.standard_normal((B, k, V)) * spread[:, None, None], dtype)
    T = rng.uniform(0.5, 1.5, B)
    seeds = (np.arange(B) * 13 + 5).astype(np.int64)
    seeds[::4] = -1                                  # unseeded rows
    pos = (np.arange(B) * 977).astype(np.int64)
    x = draw_tokens(dl, T, rng)
    if features and B >= 12:
        T[0] = 0.0                                   # greedy: accepts the argmax prefix
        x[0] = np.argmax(tl[0, :k], axis=-1)
        x[0, k - 1] = (x[0, k - 1] + 1) % V
        T[1] = -1.0                                  # invalid
        T[2] = np.nan                                # invalid
        x[3, 0] = -1                                 # not a vocabulary entry
        x[4, k - 1] = V
        tl[5, 0] = -np.inf                           # nothing finite: status 1
        dl[6] = tl[6, :k]                            # the draft is the target
        x[6] = np.argmax(tl[6, :k], axis=-1)
        dl[7, 0] = -np.inf                           # the draft has nothing finite at 0
        tl[8, :, ::7] = np.nan                       # NaN entries count as -inf
        dl[8, :, ::5] = np.nan
        tl[9, :, : V // 2] = -np.inf                 # half the target's vocabulary masked
        T[10] = 0.0                                  # greedy, first draft token not the argmax
        x[10, 0] = (np.argmax(tl[10, 0]) + 3) % V
        dl[11] = tl[11, :k] + 5.0                    # the same distribution, shifted logits
    return tl, dl, x, T, seeds, pos


def run_gpu(tl, dl, x, T, seeds, pos, dtype, wide, base_seed=7, offset=3):
    t = torch.from_numpy(tl).to(dtype).to(DEV)
    d = torch.from_numpy(dl).to(dtype).to(DEV)
    st = torch.full((tl.shape[0],), -7, dtype=torch.int32, device=DEV)
    acc, out = lms.verify_from_logits(
        t, d, torch.from_numpy(x).to(DEV), temperature=torch.from_numpy(T.astype(np.float32)).to(DEV),
        seeds=torch.from_numpy(seeds).to(DEV), positions=torch.from_numpy(pos).to(DEV),
        base_seed=base_seed, offset=offset, wide=wide, row_status=st)
    torch.cuda.synchronize()
    return (acc.cpu().numpy(), out.cpu().numpy(), st.cpu().numpy(),
            t.cpu().double().numpy(), d.cpu().double().numpy())


def run_oracle(t64, d64, x, T, seeds, pos, wide, base_seed=7, offset=3):
    return oracle.verify_from_logits(t64, d64, x, temperature=T.astype(np.float32).astype(np.float64),
                                     seeds=seeds, positions=pos, base_seed=base_seed, offset=offset,
                                     wide=wide, want_detail=True)


def _draw_tolerance(t64, d64, T, b, j, k):
    """Per-entry error interval of the final draw's scores (see the module docstring)."""
    V = t64.shape[-1]
    if j >= k or not T[b] > 0:
        return np.full(V, NEAR_TIE)
    pt = _softmax_rows(t64[b, j] / T[b])
    pd = _softmax_rows(d64[b, j] / T[b])
    r = pt - pd
    with np.errstate(divide="ignore", invalid="ignore"):
        rel = np.where(r > 0, 1e-6 * (pt + pd) / r, 0.0)
    return NEAR_TIE + rel


def check_verify(g, o, t64, d64, T, k):
    g_acc, g_out, g_st = g
    o_acc, o_out, o_st, margin, top2, scores = o
    assert np.array_equal(g_st, o_st), (np.nonzero(g_st != o_st)[0][:8], g_st[g_st != o_st][:8],
                                        o_st[g_st != o_st][:8])
    near_accept = near_draw = 0
    for b in range(g_acc.shape[0]):
        if o_st[b] != 0:
            assert g_acc[b] == 0 and (g_out[b] == -1).all(), (b, g_acc[b], g_out[b])
            continue
        jg, jo = int(g_acc[b]), int(o_acc[b])
        if jg != jo:
            i = min(jg, jo)
            assert abs(margin[b, i]) < MARGIN, f"row {b}: accept {jg} vs oracle {jo}, margin {margin[b, i]}"
            assert np.array_equal(g_out[b, :i], o_out[b, :i])
            near_accept += 1
            continue
        assert np.array_equal(g_out[b, :jg], o_out[b, :jg]), (b, g_out[b], o_out[b])
        assert (g_out[b, jg + 1:] == -1).all(), (b, g_out[b])
        a, ao = int(g_out[b, jg]), int(o_out[b, jg])
        if a != ao:
            assert 0 <= a < t64.shape[-1], (b, a)
            tol = _draw_tolerance(t64, d64, T, b, jg, k)
            assert scores[b, a] + tol[a] >= np.max(scores[b] - tol), (
                f"row {b}: gpu {a} ({scores[b, a]:.6f}) oracle {ao} ({top2[b, 0]:.6f}), "
                f"not within the error interval")
            near_draw += 1
    count_parity(rows=g_acc.shape[0], accept_tests_near_margin=near_accept,
                 draws_index_differs_within_error=near_draw)
    return near_accept, near_draw


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("wide", [False, True])
@pytest.mark.parametrize("B,k,V", [(12, 1, 1000), (16, 3, 5003), (24, 5, 8192), (13, 8, 4097)])
def test_parity_mixed_rows(dtype, wide, B, k, V):
    case = make_case(B, k, V, seed=B * 31 + k * 7 + V, dtype=dtype)
    tl, dl, x, T, seeds, pos = case
    g_acc, g_out, g_st, t64, d64 = run_gpu(*case, dtype, wide)
    o = run_oracle(t64, d64, x, T, seeds, pos, wide)
    near = check_verify((g_acc, g_out, g_st), o, t64, d64, T, k)
    assert sum(near) <= 2, near
    assert list(g_st[[1, 2, 5]]) == [2, 2, 1]
    assert g_acc[0] == k - 1 and g_acc[10] == 0 and g_acc[3] == 0
    assert g_acc[6] == k                              # the draft is the target: all accepted
    assert g_acc[4] <= k - 1


def test_k32_and_single_row():
    case = make_case(3, 32, 1500, seed=99, features=False)
    g_acc, g_out, g_st, t64, d64 = run_gpu(*case, torch.float32, False)
    o = run_oracle(t64, d64, *case[2:], False)
    assert sum(check_verify((g_acc, g_out, g_st), o, t64, d64, case[3], 32)) <= 1
    case = make_case(1, 2, 70, seed=5, features=False)
    g_acc, g_out, g_st, t64, d64 = run_gpu(*case, torch.float32, True)
    o = run_oracle(t64, d64, *case[2:], True)
    assert sum(check_verify((g_acc, g_out, g_st), o, t64, d64, case[3], 2)) == 0


def test_llama3_vocab_bf16():
    """V = 128256 (the page's latency vocabulary), k = 4, bf16 logits, every row checked."""
    B, k, V = 12, 4, 128256
    case = make_case(B, k, V, seed=2024, dtype=torch.bfloat16)
    g_acc, g_out, g_st, t64, d64 = run_gpu(*case, torch.bfloat16, False)
    o = run_oracle(t64, d64, *case[2:], False)
    near = check_verify((g_acc, g_out, g_st), o, t64, d64, case[3], k)
    assert sum(near) <= 1, near


def _chi2_ok(counts, law):
    keep = law > 0
    assert counts[~keep].sum() == 0
    exp = law[keep] / law[keep].sum() * counts.sum()
    stat = ((counts[keep] - exp) ** 2 / exp).sum()
    return stat < stats.chi2.isf(1e-6, max(1, keep.sum() - 1)), stat


PT = np.log(np.array([0.35, 0.25, 0.2, 0.1, 0.06, 0.04]))
PD = np.log(np.array([0.1, 0.4, 0.1, 0.25, 0.1, 0.05]))     # a deliberately mismatched draft


@pytest.mark.parametrize("seeded", [True, False])
def test_first_token_law_and_acceptance_rate(seeded):
    """The first emitted token follows p_t; acceptance happens with probability sum min(p_t, p_d);
    given a rejection, the token follows the residual (about 2e6 trials)."""
    n, V = 1 << 21, 6
    pt, pd = _softmax_rows(PT), _softmax_rows(PD)
    g = torch.Generator(device=DEV).manual_seed(11 if seeded else 12)
    x = torch.multinomial(torch.from_numpy(pd).float().to(DEV), n, replacement=True, generator=g)
    tgt = torch.from_numpy(np.stack([PT, PT])).float().to(DEV).expand(n, 2, V).contiguous()
    dft = torch.from_numpy(PD).float().to(DEV).expand(n, 1, V).contiguous()
    kw = dict(seeds=torch.arange(n, device=DEV) + 17, positions=torch.zeros(n, dtype=torch.int64, device=DEV)) \
        if seeded else dict(base_seed=4242, offset=9)
    acc, out = lms.verify_from_logits(tgt, dft, x[:, None].contiguous(), **kw)
    acc, out = acc.cpu().numpy(), out.cpu().numpy()
    first = out[:, 0]
    ok, stat = _chi2_ok(np.bincount(first, minlength=V).astype(float), pt)
    assert ok, stat
    tvd = 0.5 * np.abs(np.bincount(first, minlength=V) / n - pt).sum()
    assert tvd < 3e-3, tvd
    alpha = np.minimum(pt, pd).sum()
    rate = (acc == 1).mean()
    assert abs(rate - alpha) < 5 * np.sqrt(alpha * (1 - alpha) / n), (rate, alpha)
    r = np.maximum(pt - pd, 0.0)
    ok, stat = _chi2_ok(np.bincount(first[acc == 0], minlength=V).astype(float), r / r.sum())
    assert ok, stat


def test_accept_length_law_k4():
    n, V, k = 1 << 20, 6, 4
    shifts = [0.0, 0.6, 1.2, 0.3]
    tl = np.stack([PT + 0.2 * i for i in range(k + 1)])
    dl = np.stack([PD * (1 + shifts[i]) for i in range(k)])
    pt, pd = _softmax_rows(tl), _softmax_rows(dl)
    g = torch.Generator(device=DEV).manual_seed(3)
    x = torch.stack([torch.multinomial(torch.from_numpy(pd[i]).float().to(DEV), n, replacement=True,
                                       generator=g) for i in range(k)], dim=1).contiguous()
    tgt = torch.from_numpy(tl).float().to(DEV).expand(n, k + 1, V).contiguous()
    dft = torch.from_numpy(dl).float().to(DEV).expand(n, k, V).contiguous()
    acc, out = lms.verify_from_logits(tgt, dft, x, seeds=torch.arange(n, device=DEV),
                                      positions=torch.arange(n, device=DEV) * 7)
    acc, out, x = acc.cpu().numpy(), out.cpu().numpy(), x.cpu().numpy()
    a = np.minimum(pt[:k], pd).sum(axis=1)
    law = np.array([np.prod(a[:m]) * (1 - a[m]) for m in range(k)] + [np.prod(a)])
    counts = np.bincount(acc, minlength=k + 1).astype(float)
    ok, stat = _chi2_ok(counts, law)
    assert ok, stat
    assert np.abs(counts / n - law).max() < 2e-3
    for m in range(k + 1):
        rows = acc == m
        assert np.array_equal(out[rows, :m], x[rows, :m])
        assert (out[rows, m] >= 0).all() and (out[rows, m + 1:] == -1).all()


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("wide", [False, True])
def test_bonus_and_zero_residual_are_the_plain_race(dtype, wide):
    """A fully accepted row draws its bonus token exactly as sample_from_logits draws at position
    pos + k (seeded rows) or at row index b (k + 1) + k (unseeded rows); a rejection whose residual
    is zero everywhere (the draft equals the target) draws the target's race at that position."""
    B, k, V = 48, 3, 20000
    rng = np.random.default_rng(8)
    tl = torch.from_numpy(rng.standard_normal((B, k + 1, V)) * 2.0).to(dtype).to(DEV)
    dl = tl[:, :k].contiguous()
    x = tl[:, :k].float().argmax(dim=-1)
    x[B // 2:, 0] = V + 5                                  # rejected at 0, residual zero
    T = torch.from_numpy(rng.uniform(0.4, 1.4, B)).float().to(DEV)
    seeds = torch.arange(B, device=DEV) * 3 + 1
    seeds[::3] = -1
    pos = torch.arange(B, device=DEV) * 101
    acc, out = lms.verify_from_logits(tl, dl, x, temperature=T, seeds=seeds, positions=pos,
                                      base_seed=77, offset=2, wide=wide)
    acc, out = acc.cpu(), out.cpu()
    assert (acc[: B // 2] == k).all() and (acc[B // 2:] == 0).all()
    flat = tl.reshape(B * (k + 1), V)
    Tr = T.repeat_interleave(k + 1)
    sr = seeds.repeat_interleave(k + 1)
    pr = pos.repeat_interleave(k + 1) + torch.arange(k + 1, device=DEV).repeat(B)
    race = lms.sample_from_logits(flat, temperature=Tr, seeds=sr, positions=pr, base_seed=77,
                                  offset=2, wide=wide).cpu().reshape(B, k + 1)
    assert torch.equal(out[: B // 2, k], race[: B // 2, k])
    assert torch.equal(out[B // 2:, 0], race[B // 2:, 0])
    assert (out[B // 2:, 1:] == -1).all()


def test_greedy_rows_are_exact():
    B, k, V = 40, 4, 30000
    rng = np.random.default_rng(9)
    tl = torch.from_numpy(rng.standard_normal((B, k + 1, V))).float().to(DEV)
    dl = torch.from_numpy(rng.standard_normal((B, k, V))).float().to(DEV)
    am = tl.argmax(dim=-1)
    x = am[:, :k].clone()
    stop = torch.from_numpy(rng.integers(0, k + 1, B)).to(DEV)
    for b in range(B):
        if stop[b] < k:
            x[b, stop[b]] = (x[b, stop[b]] + 1) % V
    acc, out = lms.verify_from_logits(tl, dl, x, temperature=torch.zeros(B, device=DEV))
    assert torch.equal(acc, stop)
    for b in range(B):
        m = int(stop[b])
        assert torch.equal(out[b, :m], x[b, :m]) and int(out[b, m]) == int(am[b, m])
        assert (out[b, m + 1:] == -1).all()


def test_deterministic_and_offset_changes_draws():
    case = make_case(64, 4, 3000, seed=31, features=False)
    a1 = run_gpu(*case, torch.float32, False)
    a2 = run_gpu(*case, torch.float32, False)
    assert np.array_equal(a1[0], a2[0]) and np.array_equal(a1[1], a2[1])
    tl, dl, x, T, seeds, pos = case
    b = run_gpu(tl, dl, x, T, np.full_like(seeds, -1), pos, torch.float32, False, offset=3)
    c = run_gpu(tl, dl, x, T, np.full_like(seeds, -1), pos, torch.float32, False, offset=4)
    assert not np.array_equal(b[1], c[1])


def test_workspace_reuse_and_stream():
    """Caller-owned workspace and outputs on a side stream; a second call reuses them."""
    case = make_case(20, 3, 2500, seed=41, features=False)
    tl, dl, x, T, seeds, pos = case
    t = torch.from_numpy(tl).float().to(DEV)
    d = torch.from_numpy(dl).float().to(DEV)
    ws = torch.empty(lms.lib().lms_workspace_bytes_verify(20, 3, 2500), dtype=torch.uint8, device=DEV)
    acc = torch.empty(20, dtype=torch.int64, device=DEV)
    out = torch.empty(20, 4, dtype=torch.int64, device=DEV)
    s = torch.cuda.Stream()
    kw = dict(temperature=torch.from_numpy(T).float().to(DEV), seeds=torch.from_numpy(seeds).to(DEV),
              positions=torch.from_numpy(pos).to(DEV), base_seed=7, offset=3, accept_len=acc, out=out,
              workspace=ws)
    xd = torch.from_numpy(x).to(DEV)
    torch.cuda.synchronize()
    with torch.cuda.stream(s):
        lms.verify_from_logits(t, d, xd, stream=s, **kw)
    s.synchronize()
    first = (acc.cpu().clone(), out.cpu().clone())
    lms.verify_from_logits(t, d, xd, **kw)
    torch.cuda.synchronize()
    assert torch.equal(first[0], acc.cpu()) and torch.equal(first[1], out.cpu())
    g = run_gpu(*case, torch.float32, False)
    assert np.array_equal(g[0], first[0].numpy()) and np.array_equal(g[1], first[1].numpy())
