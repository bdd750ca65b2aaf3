"""Gumbel-top-k of the fused path (k draws without replacement) on the GPU against the oracle.

Parity: statuses equal; each row's finite count equal; the GPU's r-th index either equals the
oracle's r-th or scores (by the oracle) within 1e-3 of the oracle's r-th score (a near-tie swap,
counted); indices distinct; GPU scores within 2e-4 (1 + |s|) of the oracle's scores of the same
indices.  Also: entry 0 is lmhead_sample's token bit for bit; the law of ordered pairs is
Plackett-Luce; a bounded wait that runs out gives status 3 and the context stays usable.
"""
import numpy as np
import pytest
import torch
from scipy import stats

import lm_head_gumbel_lmhead_gb300 as lms
import oracle
from lm_head_gumbel_lmhead_gb300 import workloads
from parity import _add as count_parity
from test_gpu_lmhead import _ragged, orc_kw, to_dev

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda")


def run_topk(w, d, k, **extra):
    status = torch.full((w.B,), -7, dtype=torch.int32, device=DEV)
    idx, val = lms.lmhead_sample_topk(d["H"], d["W"], k, temperature=d["temperature"], seeds=d["seeds"],
                                      positions=d["positions"], bias=d["bias"], mask=d["mask"],
                                      base_seed=w.base_seed, offset=w.offset, wide=w.noise_mode == 1,
                                      row_status=status, **extra)
    torch.cuda.synchronize()
    return idx.cpu().numpy(), val.cpu().numpy(), status.cpu().numpy()


def check_topk(g_idx, g_val, g_st, o_idx, o_val, o_st, o_scores):
    assert np.array_equal(g_st, o_st), (np.nonzero(g_st != o_st)[0][:5], g_st[g_st != o_st][:5])
    near = 0
    for b in range(g_idx.shape[0]):
        gi, oi = g_idx[b], o_idx[b]
        if o_st[b] != 0:
            assert (gi == -1).all(), (b, gi)
            continue
        assert np.array_equal(gi >= 0, oi >= 0), (b, gi, oi)
        m = int((oi >= 0).sum())
        assert len(set(gi[:m].tolist())) == m, (b, gi)
        for r in range(m):
            if gi[r] != oi[r]:
                gap = abs(o_scores[b, gi[r]] - o_val[b, r])
                assert gap < 1e-3, f"row {b} rank {r}: gpu {gi[r]} oracle {oi[r]} score gap {gap:.3e}"
                near += 1
        os_ = o_scores[b, gi[:m]]
        assert np.all(np.abs(g_val[b, :m] - os_) <= 2e-4 * (1 + np.abs(os_))), (b, g_val[b, :m], os_)
        assert np.all(g_val[b, m:] == -np.inf)
    count_parity(rows=g_idx.shape[0], ranks_index_differs_near_tie=near)
    return near


def full_topk_parity(w, k):
    d = to_dev(w)
    g_idx, g_val, g_st = run_topk(w, d, k)
    o_idx, o_val, o_st, o_scores = oracle.lmhead_gumbel_topk(w.H, w.W, k, **orc_kw(w))
    return check_topk(g_idx, g_val, g_st, o_idx, o_val, o_st, o_scores)


@pytest.mark.parametrize("B,D,V,wide,k", [(1, 64, 1000, False, 1), (3, 200, 8229, True, 4),
                                          (17, 512, 3000, False, 16), (40, 1024, 4097, True, 7),
                                          (130, 256, 2000, False, 5), (300, 192, 1300, True, 16)])
def test_topk_ragged(B, D, V, wide, k):
    # greedy, invalid, unseeded and all-masked rows, bias and masks; B = 300 takes two launches
    full_topk_parity(_ragged(B, D, V, seed=B * 11 + D, wide=wide), k)


def test_topk_many_lists_split_stage2():
    # 160 rows at k = 16 keep one list per tile and quadrant (running lists would not fit in shared
    # memory), and 313 tiles give 1252 lists a row: more than one Stage-2 CTA takes, so each row is
    # split over several CTAs whose part lists the final kernel merges
    full_topk_parity(_ragged(160, 64, 40000, seed=29, wide=False), 16)


@pytest.mark.parametrize("wide,k", [(False, 8), (True, 16)])
def test_topk_plain_launch_greedy_invalid_and_ragged(wide, k):
    # no bias and no mask (the plain epilogue), with greedy, invalid and unseeded rows and a
    # last vocabulary tile that ends inside an 8-row chunk (V = 2500 = 19 * 128 + 68); entry 0
    # is the plain race's token
    w = _ragged(37, 256, 2500, seed=19, wide=wide)
    w = workloads.Workload(w.name, w.B, w.D, w.V, w.H, w.W, w.temperature, w.seeds, w.positions,
                           None, None, w.noise_mode, base_seed=w.base_seed, offset=w.offset)
    full_topk_parity(w, k)
    d = to_dev(w)
    g_idx, _, g_st = run_topk(w, d, k)
    race = lms.lmhead_sample(d["H"], d["W"], temperature=d["temperature"], seeds=d["seeds"],
                             positions=d["positions"], base_seed=w.base_seed, offset=w.offset,
                             wide=wide)
    torch.cuda.synchronize()
    assert np.array_equal(g_idx[:, 0], race.cpu().numpy())


@pytest.mark.parametrize("wide", [False, True])
def test_topk_tiny_every_output(wide):
    w = workloads.tiny()
    w.noise_mode = 1 if wide else 0
    full_topk_parity(w, 16)


@pytest.mark.parametrize("k", [1, 8, 16])
def test_first_draw_is_the_race_token(k):
    w = _ragged(64, 512, 5000, seed=41)
    d = to_dev(w)
    g_idx, _, g_st = run_topk(w, d, k)
    st = torch.full((w.B,), -7, dtype=torch.int32, device=DEV)
    race = lms.lmhead_sample(d["H"], d["W"], temperature=d["temperature"], seeds=d["seeds"],
                             positions=d["positions"], bias=d["bias"], mask=d["mask"],
                             base_seed=w.base_seed, offset=w.offset, row_status=st)
    torch.cuda.synchronize()
    assert np.array_equal(g_idx[:, 0], race.cpu().numpy()) and np.array_equal(g_st, st.cpu().numpy())


def test_short_rows_end_in_minus_one():
    B, D, V, k = 4, 128, 2000, 8
    w = _ragged(B, D, V, seed=3, features=False)
    allowed = torch.ones(B, V, dtype=torch.bool)
    allowed[1] = False
    allowed[1, [5, 700, 1999]] = True            # three tokens left
    allowed[3] = False                           # none left
    w.mask = workloads.pack_allow_bits(allowed)
    d = to_dev(w)
    g_idx, g_val, g_st = run_topk(w, d, k)
    assert sorted(g_idx[1, :3].tolist()) == [5, 700, 1999] and (g_idx[1, 3:] == -1).all()
    assert (g_val[1, 3:] == -np.inf).all() and g_st[1] == 0
    assert g_st[3] == 1 and (g_idx[3] == -1).all()
    full_topk_parity(w, k)


def test_topk_qwen3_8b_shape_every_row():
    w = workloads.qwen3_8b(64)
    d = to_dev(w)
    k = 8
    g_idx, g_val, g_st = run_topk(w, d, k)
    rows = np.arange(64)
    o_idx, o_val, o_st, o_scores = oracle.lmhead_gumbel_topk(w.H, w.W, k, rows=rows, **orc_kw(w))
    check_topk(g_idx[rows], g_val[rows], g_st[rows], o_idx, o_val, o_st, o_scores)
    assert (g_st == 0).all()


def test_ordered_pairs_follow_plackett_luce_on_gpu():
    # logits = bf16(log p) through the GEMM: H = e_0, W[v][0] = log p_v
    p = np.array([0.4, 0.25, 0.2, 0.1, 0.05])
    V, D = 5, 64
    Wt = torch.zeros(V, D)
    Wt[:, 0] = torch.from_numpy(np.log(p)).float()
    W = Wt.to(torch.bfloat16)
    y = W[:, 0].double().numpy()
    q = np.exp(y) / np.exp(y).sum()             # the law of the rounded logits
    n_call, calls = 50_000, 8
    H = torch.zeros(n_call, D, dtype=torch.bfloat16)
    H[:, 0] = 1.0
    Hd, Wd = H.to(DEV), W.to(DEV)
    counts = np.zeros((V, V))
    for c in range(calls):
        seeds = (torch.arange(n_call, dtype=torch.int64) + c * n_call).to(DEV)
        pos = torch.full((n_call,), c, dtype=torch.int64, device=DEV)
        idx, _ = lms.lmhead_sample_topk(Hd, Wd, 2, seeds=seeds, positions=pos, want_scores=False)
        i = idx.cpu().numpy()
        assert (i[:, 0] != i[:, 1]).all() and (i >= 0).all()
        np.add.at(counts, (i[:, 0], i[:, 1]), 1)
    law = q[:, None] * q[None, :] / (1.0 - q[:, None])
    off = ~np.eye(V, dtype=bool)
    exp = law[off] * n_call * calls
    stat = ((counts[off] - exp) ** 2 / exp).sum()
    assert stat < stats.chi2.isf(1e-6, off.sum() - 1), stat


def test_topk_timeout_reports_status_and_context_survives():
    w = _ragged(20, 256, 4000, seed=13, features=False)
    d = to_dev(w)
    g_idx, g_val, g_st = run_topk(w, d, 4, timeout_ms=20, debug_flags=lms.DEBUG_WITHHOLD_FIRST_LOAD)
    assert (g_st == lms.ROW_DEVICE_TIMEOUT).all() and (g_idx == -1).all()
    full_topk_parity(w, 4)


def test_topk_host_validation():
    w = _ragged(4, 64, 300, seed=1, features=False)
    d = to_dev(w)
    for k in (0, lms.TOPK_MAX + 1):
        with pytest.raises(lms.LmsError):
            lms.lmhead_sample_topk(d["H"], d["W"], k)
