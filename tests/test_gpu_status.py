"""lms_read_status on the GPU: the status word that every workspace-taking call leaves at the head
of its workspace, for callers that pass no row_status buffer.

For each entry point the word must equal the set of the call's non-zero row statuses (read from
a row_status buffer of a twin call), a clean call must clear what the previous call left, and a
device-side wait that runs out of time must make lms_read_status return LMS_ERR_TIMEOUT.  The
row conditions are the pages': a row without a finite score (FlashSampling "Limitations") and an
invalid temperature (the sampling-kernel guide's review checklist).
"""
import numpy as np
import pytest
import torch

import lm_head_gumbel_lmhead_gb300 as lms
from test_gpu_lmhead import _ragged, to_dev

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda")


def _bits(status):
    return sum(1 << int(s) for s in set(np.asarray(status).tolist()) if s != 0)


def _ws(n):
    # every byte set: the call itself must clear the status word
    return torch.full((n,), 0xFF, dtype=torch.uint8, device=DEV)


def _fused_kw(w, d):
    return dict(temperature=d["temperature"], seeds=d["seeds"], positions=d["positions"],
                bias=d["bias"], mask=d["mask"], base_seed=w.base_seed, offset=w.offset,
                wide=w.noise_mode == 1)


def test_fused_status_word_clean_call_and_timeout():
    w = _ragged(40, 256, 3000, seed=17)          # rows with status 1 (all masked) and 2 (T < 0)
    d = to_dev(w)
    ws = _ws(lms.workspace_bytes(lms.OP_LMHEAD, w.B, w.D, w.V))
    st = torch.full((w.B,), -7, dtype=torch.int32, device=DEV)
    lms.lmhead_sample(d["H"], d["W"], row_status=st, workspace=ws, **_fused_kw(w, d))
    expect = _bits(st.cpu().numpy())
    assert expect == (1 << 1) | (1 << 2)
    lms.lmhead_sample(d["H"], d["W"], workspace=ws, **_fused_kw(w, d))
    assert lms.read_status(ws) == (lms.LMS_OK, expect)
    clean = _ragged(40, 256, 3000, seed=17, features=False)
    dc = to_dev(clean)
    lms.lmhead_sample(dc["H"], dc["W"], workspace=ws, **_fused_kw(clean, dc))
    assert lms.read_status(ws) == (lms.LMS_OK, 0)
    # a bounded wait that runs out (the first CTA withholds its first load)
    lms.lmhead_sample(dc["H"], dc["W"], workspace=ws, timeout_ms=20,
                      debug_flags=lms.DEBUG_WITHHOLD_FIRST_LOAD, **_fused_kw(clean, dc))
    status, bits = lms.read_status(ws)
    assert status == lms.LMS_ERR_TIMEOUT and bits == 1 << 3
    # the context stays usable and the next call clears the word again
    lms.lmhead_sample(dc["H"], dc["W"], workspace=ws, **_fused_kw(clean, dc))
    assert lms.read_status(ws) == (lms.LMS_OK, 0)


def test_fused_status_word_above_256_rows():
    # several Stage-1 launches: only the first clears the word, every row's Stage 2 reports
    w = _ragged(300, 64, 1300, seed=23)
    d = to_dev(w)
    ws = _ws(lms.workspace_bytes(lms.OP_LMHEAD, w.B, w.D, w.V))
    st = torch.full((w.B,), -7, dtype=torch.int32, device=DEV)
    lms.lmhead_sample(d["H"], d["W"], row_status=st, workspace=ws, **_fused_kw(w, d))
    expect = _bits(st.cpu().numpy())
    assert lms.read_status(ws) == (lms.LMS_OK, expect) and expect != 0


def test_logits_status_word():
    B, V = 12, 5000
    logits = torch.randn(B, V, device=DEV)
    T = torch.full((B,), 0.8, device=DEV)
    T[4] = float("nan")
    logits[7] = float("-inf")
    ws = _ws(lms.workspace_bytes(lms.OP_LOGITS, B, 0, V))
    st = torch.full((B,), -7, dtype=torch.int32, device=DEV)
    lms.sample_from_logits(logits, temperature=T, workspace=ws, row_status=st)
    expect = _bits(st.cpu().numpy())
    assert expect == (1 << 1) | (1 << 2)
    lms.sample_from_logits(logits, temperature=T, workspace=ws)
    assert lms.read_status(ws) == (lms.LMS_OK, expect)
    lms.sample_from_logits(logits[:3].contiguous(), temperature=T[:3].contiguous(), workspace=ws)
    assert lms.read_status(ws) == (lms.LMS_OK, 0)


def test_topk_status_word_and_timeout():
    w = _ragged(40, 256, 3000, seed=29)
    d = to_dev(w)
    k = 4
    ws = _ws(lms.lib().lms_workspace_bytes_topk(w.B, w.V, k))
    st = torch.full((w.B,), -7, dtype=torch.int32, device=DEV)
    lms.lmhead_sample_topk(d["H"], d["W"], k, row_status=st, workspace=ws, **_fused_kw(w, d))
    expect = _bits(st.cpu().numpy())
    assert expect != 0
    lms.lmhead_sample_topk(d["H"], d["W"], k, workspace=ws, **_fused_kw(w, d))
    assert lms.read_status(ws) == (lms.LMS_OK, expect)
    lms.lmhead_sample_topk(d["H"], d["W"], k, workspace=ws, timeout_ms=20,
                           debug_flags=lms.DEBUG_WITHHOLD_FIRST_LOAD, **_fused_kw(w, d))
    status, bits = lms.read_status(ws)
    assert status == lms.LMS_ERR_TIMEOUT and bits & (1 << 3)


def test_verify_status_word():
    B, k, V = 6, 3, 2000
    t = torch.randn(B, k + 1, V, device=DEV)
    dft = (t[:, :k] + 0.3 * torch.randn(B, k, V, device=DEV)).contiguous()
    x = dft.argmax(dim=-1).contiguous()
    T = torch.full((B,), 0.9, device=DEV)
    T[2] = -1.0                                   # status 2
    t[4, 0] = float("-inf")                       # nothing finite at position 0: status 1
    ws = _ws(lms.lib().lms_workspace_bytes_verify(B, k, V))
    st = torch.full((B,), -7, dtype=torch.int32, device=DEV)
    lms.verify_from_logits(t, dft, x, temperature=T, workspace=ws, row_status=st)
    expect = _bits(st.cpu().numpy())
    assert expect & (1 << 2)
    lms.verify_from_logits(t, dft, x, temperature=T, workspace=ws)
    assert lms.read_status(ws) == (lms.LMS_OK, expect)
