"""The fused path with FP8 (E4M3) inputs on the GPU against the oracle: the per-row activation
quantisation bit-exact, then every output (tokens, statuses, all Stage-1 candidates) on ragged
shapes and every row at the Qwen3-8B shape."""
import numpy as np
import pytest
import torch

import lm_head_gumbel_lmhead_gb300 as lms
import oracle
from lm_head_gumbel_lmhead_gb300 import workloads
from parity import check_rows, check_tiles

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda")


def _case(B, D, V, seed, wide=False, features=True):
    g = torch.Generator().manual_seed(seed)
    H = (torch.randn(B, D, generator=g) * 2).to(torch.bfloat16)
    H[B // 3] *= 1e-3
    W = (torch.randn(V, D, generator=g) / D ** 0.5).to(torch.bfloat16)
    W8, ws = workloads.quantize_weight_e4m3(W)
    T = 0.3 + torch.rand(B, generator=g)
    seeds = 100 + torch.arange(B, dtype=torch.int64)
    bias = mask = None
    if features:
        T[::5] = 0.0
        seeds[1::4] = -1
        bias = torch.randn(B, V, generator=g) * 0.3
        allowed = torch.rand(B, V, generator=g) < 0.5
        allowed[B // 2:] = True
        mask = workloads.pack_allow_bits(allowed)
    return dict(B=B, D=D, V=V, H=H, W8=W8, ws=ws, T=T, seeds=seeds,
                pos=torch.arange(B, dtype=torch.int64) * 5, bias=bias, mask=mask, wide=wide)


def run(c, **extra):
    B, D, V = c["B"], c["D"], c["V"]
    tv, nt, ws_bytes, _ = lms.tile_info(lms.OP_LMHEAD_FP8, B, D, V)
    wsp = torch.full((ws_bytes,), 0xEE, dtype=torch.uint8, device=DEV)
    st = torch.full((B,), -7, dtype=torch.int32, device=DEV)
    out = lms.lmhead_sample_fp8(c["H"].to(DEV), c["W8"].to(DEV), c["ws"].to(DEV),
                                temperature=c["T"].to(DEV), seeds=c["seeds"].to(DEV),
                                positions=c["pos"].to(DEV),
                                bias=None if c["bias"] is None else c["bias"].to(DEV),
                                mask=None if c["mask"] is None else c["mask"].to(DEV),
                                base_seed=5, offset=3, wide=c["wide"], workspace=wsp, row_status=st,
                                **extra)
    torch.cuda.synchronize()
    cs, ci, q, e = lms.split_workspace_fp8(wsp, B, D, nt)
    return (out.cpu().numpy(), st.cpu().numpy(), cs.cpu().numpy(), ci.cpu().numpy(),
            q.cpu().numpy()[:, :D], e.cpu().numpy())


def orc_kw(c):
    return dict(temperature=c["T"].double().numpy(), seeds=c["seeds"].numpy(),
                positions=c["pos"].numpy(),
                bias=None if c["bias"] is None else c["bias"].double().numpy(),
                mask=None if c["mask"] is None else c["mask"].numpy().view(np.uint32),
                base_seed=5, offset=3, wide=c["wide"])


@pytest.mark.parametrize("B,D,V,wide", [(1, 128, 1000, False), (4, 512, 8192, False),
                                        (17, 256, 3001, True), (64, 1024, 4097, False),
                                        (130, 384, 1500, True), (300, 128, 1300, False)])
def test_fp8_every_output(B, D, V, wide):
    c = _case(B, D, V, seed=B + D + V, wide=wide)
    out, st, cs, ci, q, e = run(c)
    oq, oe = oracle.quantize_rows_e4m3(c["H"])
    assert np.array_equal(e, oe) and np.array_equal(q, oq)
    orc = oracle.lmhead_sample_fp8(c["H"], c["W8"].numpy(), c["ws"].double().numpy(), **orc_kw(c))
    # scores of any (b, v) for near-tie checks: the race over the oracle's fp8 logits
    y = oracle.lmhead_logits_fp8(oq, oe, c["W8"].numpy(), c["ws"].double().numpy())
    full = oracle.sample_from_logits(y, want_scores=True, tile_v=128, **orc_kw(c))
    assert (full.out == orc.out).all()
    score_of = lambda i, v: full.scores[i, v]
    check_rows(out, st, orc, score_of)
    check_tiles(cs, ci, orc, score_of)


def test_fp8_qwen3_8b_shape_every_row():
    w = workloads.qwen3_8b(64, step=2)
    W8, ws = workloads.quantize_weight_e4m3(w.W)
    c = dict(B=64, D=w.D, V=w.V, H=w.H, W8=W8, ws=ws, T=w.temperature, seeds=w.seeds,
             pos=w.positions, bias=None, mask=None, wide=False)
    out, st, cs, ci, q, e = run(c)
    oq, oe = oracle.quantize_rows_e4m3(w.H)
    assert np.array_equal(e, oe) and np.array_equal(q, oq)
    rows = np.arange(64)
    orc = oracle.lmhead_sample_fp8(w.H, W8.numpy(), ws.double().numpy(), rows=rows, **orc_kw(c))
    # every row's full scores
    y = oracle.lmhead_logits_fp8(oq, oe, W8.numpy(), ws.double().numpy(), rows=rows)
    kw = orc_kw(c)
    full = oracle.sample_from_logits(y, temperature=kw["temperature"][rows], seeds=kw["seeds"][rows],
                                     positions=kw["positions"][rows], want_scores=True, tile_v=128)
    assert (full.out == orc.out).all()
    score_of = lambda i, v: full.scores[i, v]
    check_rows(out[rows], st[rows], orc, score_of, rows=rows)
    check_tiles(cs[rows], ci[rows], orc, score_of)
    assert (st == 0).all()


def test_fp8_timeout_reports_status():
    c = _case(20, 256, 4000, seed=3, features=False)
    out, st, _, _, _, _ = run(c, timeout_ms=20, debug_flags=lms.DEBUG_WITHHOLD_FIRST_LOAD)
    assert (st == lms.ROW_DEVICE_TIMEOUT).all() and (out == -1).all()
