"""The filtered race (top-k -> top-p -> min-p, then the Gumbel race) on the GPU.

Parity against the oracle works as follows:

- Tokens and statuses are equal row by row.
- The top-p cut (a prefix sum) and the min-p cut are floating-point decisions: fp32 in the kernel,
  fp64 in the oracle. A row whose cut moves when the oracle shifts top_p by 1e-5 or scales min_p by
  1 +- 1e-5 may take either of the resulting tokens. Such rows are counted.
- So may rows whose two best kept perturbed scores are within 1e-3 (the near-tie rule).

It also checks the sampled law against the renormalised softmax (chi-square). Finally, it checks
the Megatron-LM PR's batch-position invariance case ("Tests": no filter, top-p 0.9 and top-k 50 at
T 0.7): seeded draws are bit-equal across repeated calls, single-row calls and a permuted batch.
"""
import numpy as np
import pytest
import torch
from scipy import stats

import lm_head_gumbel_lmhead_gb300 as lms
import oracle
from lm_head_gumbel_lmhead_gb300 import workloads
from parity import _add as count_parity

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda")
EPS = 1e-5


def _gpu(logits, B=None, **kw):
    d = {}
    for k, v in kw.items():
        if isinstance(v, np.ndarray):
            t = torch.from_numpy(np.ascontiguousarray(v))
            if k in ("temperature", "top_p", "min_p", "bias"):
                t = t.float()
            elif k == "top_k":
                t = t.to(torch.int32)
            elif k == "mask":
                t = t.view(torch.int32) if t.dtype == torch.int32 else torch.from_numpy(v.view(np.int32))
            v = t.to(DEV)
        d[k] = v
    Bn = B if B is not None else logits.shape[0]
    st = torch.full((Bn,), -5, dtype=torch.int32, device=DEV)
    out = lms.sample_from_logits_filtered(logits, B=B, row_status=st, **d)
    torch.cuda.synchronize()
    return out.cpu().numpy(), st.cpu().numpy()


def _orc(y, **kw):
    o = dict(kw)
    if o.get("mask") is not None:
        o["mask"] = np.asarray(o["mask"]).view(np.uint32)
    return o


def check_filtered(gpu_out, gpu_st, y, B=None, **kw):
    kw_o = _orc(y, **kw)
    out, st, kept, t1, t2 = oracle.sample_filtered(y, B=B, want_top2=True, **kw_o)
    assert np.array_equal(gpu_st, st), (np.nonzero(gpu_st != st)[0][:5], gpu_st[gpu_st != st][:5], st[gpu_st != st][:5])
    bad = np.nonzero(gpu_out != out)[0]
    count_parity(rows=gpu_out.shape[0])
    if bad.size == 0:
        return 0
    alts = [oracle.sample_filtered(y, B=B, p_shift=ps, minp_scale=ms, **kw_o)[0]
            for ps, ms in [(EPS, 1.0), (-EPS, 1.0), (0.0, 1 + EPS), (0.0, 1 - EPS)]]
    accepted = 0
    for i in bad:
        if any(a[i] == gpu_out[i] for a in alts) or (t1[i] - t2[i] < 1e-3):
            accepted += 1
        else:
            raise AssertionError(f"row {i}: gpu {gpu_out[i]} oracle {out[i]} kept {kept[i]} "
                                 f"alternatives {[a[i] for a in alts]} top-two gap {t1[i] - t2[i]:.3e}")
    count_parity(rows_index_differs_filter_boundary_or_near_tie=accepted)
    return accepted


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("wide", [False, True])
def test_parity_mixed_filters(dtype, wide):
    rng = np.random.default_rng(7)
    B, V = 48, 5003
    logits = workloads.logits_normal(B, V, std=2.0, seed=4, dtype=dtype)
    y = logits.double().numpy()
    T = rng.uniform(0.4, 1.4, B).astype(np.float32)
    T[[0, 13]] = 0.0
    T[5] = -1.0
    top_k = rng.choice([0, 1, 5, 50, 1024, 2000, 7000], B).astype(np.int32)
    top_p = rng.choice([1.0, 0.5, 0.9, 0.99, 0.2], B).astype(np.float32)
    min_p = rng.choice([0.0, 0.0, 0.05, 0.3], B).astype(np.float32)
    seeds = (np.arange(B) * 13 + 1).astype(np.int64)
    seeds[::5] = -1
    pos = np.arange(B, dtype=np.int64) * 3
    bias = (rng.standard_normal((B, V)) * 0.3).astype(np.float32)
    allowed = rng.random((B, V)) < 0.6
    allowed[B // 2:] = True
    allowed[9] = False                   # no token left: status 1
    mask = workloads.pack_allow_bits(torch.from_numpy(allowed)).numpy()
    kw = dict(temperature=T, top_k=top_k, top_p=top_p, min_p=min_p, seeds=seeds, positions=pos,
              bias=bias, mask=mask, base_seed=11, offset=4, wide=wide)
    g_out, g_st = _gpu(logits.to(DEV), **kw)
    kw_o = dict(kw, temperature=T.astype(np.float64), top_p=top_p.astype(np.float64),
                min_p=min_p.astype(np.float64), bias=bias.astype(np.float64))
    check_filtered(g_out, g_st, y, **kw_o)
    assert g_st[5] == 2 and g_st[9] == 1


def test_broadcast_row_and_ties():
    V = 3000
    row = torch.zeros(V)
    row[::7] = 1.0                        # 429 tied maxima
    B = 64
    seeds = np.arange(B, dtype=np.int64)
    top_k = np.full(B, 100, np.int32)     # keeps the 100 smallest-index maxima
    g_out, g_st = _gpu(row.to(DEV), B=B, top_k=top_k, seeds=seeds, positions=seeds)
    check_filtered(g_out, g_st, row.double().numpy(), B=B, top_k=top_k, seeds=seeds, positions=seeds)
    assert (g_out % 7 == 0).all() and (g_out <= 7 * 99).all()


P4 = np.array([0.5, 0.3, 0.15, 0.05])


@pytest.mark.parametrize("kw,kept", [(dict(top_k=2), [0, 1]), (dict(top_p=0.7), [0, 1]),
                                     (dict(min_p=0.25), [0, 1, 2]),
                                     (dict(top_k=3, top_p=0.8), [0, 1])])
def test_law_on_gpu(kw, kept):
    n = 1_000_000
    row = torch.from_numpy(np.log(P4).astype(np.float32)).to(DEV)
    args = {k: (np.full(n, v, np.int32) if k == "top_k" else np.full(n, v, np.float32)) for k, v in kw.items()}
    out, st = _gpu(row, B=n, seeds=np.full(n, 5, np.int64), positions=np.arange(n, dtype=np.int64), **args)
    assert (st == 0).all()
    counts = np.bincount(out, minlength=4).astype(float)
    law = np.zeros(4)
    law[kept] = P4[kept]
    assert counts[law == 0].sum() == 0
    exp = law[law > 0] / law.sum() * n
    stat = ((counts[law > 0] - exp) ** 2 / exp).sum()
    assert stat < stats.chi2.isf(1e-6, max(1, len(kept) - 1))


@pytest.mark.parametrize("filters", [dict(), dict(top_p=0.9), dict(top_k=50)])
def test_batch_position_invariance_with_filters_full_vocab(filters):
    B, V = 24, 131072
    logits = workloads.logits_normal(B, V, std=2.0, seed=8, dtype=torch.bfloat16).to(DEV)
    T = torch.full((B,), 0.7, device=DEV)
    seeds = 500 + torch.arange(B, dtype=torch.int64, device=DEV)
    seeds[2::4] = -1
    pos = torch.arange(B, dtype=torch.int64, device=DEV) + 100
    fk = {}
    if "top_p" in filters:
        fk["top_p"] = torch.full((B,), filters["top_p"], device=DEV)
    if "top_k" in filters:
        fk["top_k"] = torch.full((B,), filters["top_k"], dtype=torch.int32, device=DEV)
    run = lambda lg, t, s, p, f: lms.sample_from_logits_filtered(lg, temperature=t, seeds=s, positions=p,
                                                                 base_seed=3, **f)
    full = run(logits, T, seeds, pos, fk)
    again = run(logits, T, seeds, pos, fk)
    assert torch.equal(full, again)
    perm = torch.randperm(B, generator=torch.Generator().manual_seed(2)).to(DEV)
    pr = run(logits[perm].contiguous(), T[perm].contiguous(), seeds[perm].contiguous(),
             pos[perm].contiguous(), {k: v[perm].contiguous() for k, v in fk.items()})
    seeded = seeds[perm] >= 0
    assert torch.equal(pr[seeded], full[perm][seeded])
    for b in (0, 5, 11):
        one = run(logits[b:b + 1], T[b:b + 1], seeds[b:b + 1], pos[b:b + 1],
                  {k: v[b:b + 1] for k, v in fk.items()})
        assert one.item() == full[b].item()
    # and the oracle agrees on a few rows
    y = logits[:4].double().cpu().numpy()
    args = dict(temperature=np.full(4, 0.7), seeds=seeds[:4].cpu().numpy(), positions=pos[:4].cpu().numpy(),
                base_seed=3)
    if "top_p" in filters:
        args["top_p"] = np.full(4, filters["top_p"])
    if "top_k" in filters:
        args["top_k"] = np.full(4, filters["top_k"], np.int32)
    check_filtered(full[:4].cpu().numpy(), np.zeros(4, np.int32), y, **args)


@pytest.mark.parametrize("dtype,wide", [(torch.float32, False), (torch.bfloat16, True)])
def test_parity_multi_cta_rows_with_ties_across_slices(dtype, wide):
    """Rows long enough to span several CTAs of a cluster, with logits on a coarse grid so that
    the k-th value is shared by entries in different slices (the index cut at K)."""
    rng = np.random.default_rng(17)
    B, V = 6, 50_000
    y = np.round(rng.standard_normal((B, V)) * 8.0) / 4.0          # many exact ties
    logits = torch.from_numpy(y.astype(np.float32)).to(dtype)
    yd = logits.double().numpy()
    T = np.array([1.0, 0.5, 0.8, 1.25, 0.7, 2.0], np.float32)
    top_k = np.array([37, 500, 1000, 0, 3, 1024], np.int32)
    top_p = np.array([1.0, 0.9, 1.0, 0.95, 0.5, 0.3], np.float32)
    min_p = np.array([0.0, 0.0, 0.1, 0.0, 0.0, 0.02], np.float32)
    seeds = np.arange(B, dtype=np.int64) + 77
    pos = np.arange(B, dtype=np.int64) * 5
    allowed = rng.random((B, V)) < 0.9
    allowed[:3] = True
    mask = workloads.pack_allow_bits(torch.from_numpy(allowed)).numpy()
    kw = dict(temperature=T, top_k=top_k, top_p=top_p, min_p=min_p, seeds=seeds, positions=pos,
              mask=mask, base_seed=5, offset=9, wide=wide)
    for rep in range(3):                                              # several positions
        kw["positions"] = pos + 1000 * rep
        g_out, g_st = _gpu(logits.to(DEV), **kw)
        kw_o = dict(kw, temperature=T.astype(np.float64), top_p=top_p.astype(np.float64),
                    min_p=min_p.astype(np.float64))
        check_filtered(g_out, g_st, yd, **kw_o)


@pytest.mark.parametrize("filters", [dict(top_k=50), dict(top_k=50, top_p=0.9), dict(top_p=0.5)])
def test_tail_row_keeps_smallest_indices_at_the_cut(filters):
    """The Megatron-LM PR's tail row [0, -D, ..., -D] (V = 131072): every entry but the first ties
    at the k-th value, so the kept set is {0} and the smallest tied indices."""
    V, B = 131072, 32
    row = workloads.tail_row(V, 0.999)
    seeds = np.arange(B, dtype=np.int64)
    kw = {k: np.full(B, v, np.int32 if k == "top_k" else np.float32) for k, v in filters.items()}
    g_out, g_st = _gpu(row.to(DEV), B=B, seeds=seeds, positions=seeds, **kw)
    check_filtered(g_out, g_st, row.double().numpy(), B=B, seeds=seeds, positions=seeds,
                   **{k: (v.astype(np.float64) if v.dtype == np.float32 else v) for k, v in kw.items()})
    k = filters.get("top_k", 1024)
    assert (g_st == 0).all() and (g_out < k).all()


def test_parity_rows_beyond_the_shared_memory_slice():
    """V = 800000: a slice no longer fits in shared memory, so keys are recomputed from global
    memory on every pass."""
    rng = np.random.default_rng(23)
    B, V = 3, 800_000
    logits = workloads.logits_normal(B, V, std=2.0, seed=12, dtype=torch.float32)
    y = logits.double().numpy()
    T = np.array([0.9, 1.0, 0.6], np.float32)
    top_k = np.array([100, 0, 1024], np.int32)
    top_p = np.array([0.95, 0.8, 1.0], np.float32)
    seeds = np.array([1, -1, 3], np.int64)
    pos = np.array([4, 5, 6], np.int64)
    kw = dict(temperature=T, top_k=top_k, top_p=top_p, seeds=seeds, positions=pos, base_seed=2)
    g_out, g_st = _gpu(logits.to(DEV), **kw)
    check_filtered(g_out, g_st, y, **dict(kw, temperature=T.astype(np.float64),
                                          top_p=top_p.astype(np.float64)))


@pytest.mark.parametrize("wide", [False, True])
def test_parity_outliers_and_bf16_ties(wide):
    """Rows that leave the near window (an outlier maximum, so fewer than k entries lie within two
    octaves of it) and bf16 rows whose ties make the boundary bin hold many equal keys."""
    B, V = 6, 40_000
    logits = workloads.logits_normal(B, V, std=2.0, seed=31, dtype=torch.float32)
    logits[0, 777] = 60.0                        # one outlier, top-k 50: the full-width select
    logits[1, [5, 30000, 39999]] = torch.tensor([45.0, 44.0, 46.0])
    logits = logits.to(torch.bfloat16)           # bf16: about a thousand distinct values per row
    y = logits.double().numpy()
    T = np.array([1.0, 0.8, 0.7, 1.3, 0.9, 0.6], np.float32)
    top_k = np.array([50, 0, 1024, 700, 1000, 200], np.int32)
    top_p = np.array([1.0, 0.9, 0.95, 0.8, 1.0, 0.99], np.float32)
    min_p = np.array([0.0, 0.0, 0.0, 0.05, 0.01, 0.0], np.float32)
    seeds = np.arange(B, dtype=np.int64) + 900
    for rep in range(3):
        pos = np.arange(B, dtype=np.int64) + 50 * rep
        kw = dict(temperature=T, top_k=top_k, top_p=top_p, min_p=min_p, seeds=seeds, positions=pos,
                  wide=wide)
        g_out, g_st = _gpu(logits.to(DEV), **kw)
        check_filtered(g_out, g_st, y, **dict(kw, temperature=T.astype(np.float64),
                                              top_p=top_p.astype(np.float64),
                                              min_p=min_p.astype(np.float64)))
        assert g_out[0] == 777
