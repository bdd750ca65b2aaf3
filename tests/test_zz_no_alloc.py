"""The allocation-free fused entry point, lms_lmhead_sample_noalloc, through the C ABI.

It serves callers that cannot allocate device memory (for instance code running inside an
allocator or a memory-pool callback): its Stage-1 scratch is the library's fixed device
array instead of a caller workspace.  Its tokens and row statuses must equal those of
lms_lmhead_sample on the same inputs, call after call (the array keeps the previous call's
candidates, which the next call must overwrite), and calls that would not fit the array must be
refused on the host.  This file is collected last so that a failure here cannot hide any other
test; it also passes on its own in a fresh process.
"""
import ctypes

import numpy as np
import pytest
import torch

import lm_head_gumbel_lmhead_gb300 as lms
from lm_head_gumbel_lmhead_gb300 import workloads

DEV = torch.device("cuda") if torch.cuda.is_available() else None


def _lib():
    from lm_head_gumbel_lmhead_gb300 import build
    build.build()
    return lms.lib()


def _params(w, d, wide, status):
    return lms._params(w.B, d["H"].device, d["T"], d["seeds"], d["pos"], d["bias"], d["mask"], w.base_seed,
                       w.offset, wide, 0, lms.PATH_AUTO, status, 0, 0)


def _case(B, D, V, seed):
    g = torch.Generator().manual_seed(seed)
    H = torch.randn(B, D, generator=g).to(torch.bfloat16)
    W = (torch.randn(V, D, generator=g) / D ** 0.5).to(torch.bfloat16)
    T = 0.4 + torch.rand(B, generator=g)
    T[::7] = 0.0
    seeds = 500 + torch.arange(B, dtype=torch.int64)
    seeds[2::5] = -1
    bias = torch.randn(B, V, generator=g) * 0.2
    allowed = torch.rand(B, V, generator=g) < 0.7
    return workloads.Workload("noalloc", B, D, V, H, W, T, seeds,
                              torch.arange(B, dtype=torch.int64), bias,
                              workloads.pack_allow_bits(allowed), 0, base_seed=9, offset=1)


def _run_both(L, w, positions, wide):
    d = dict(H=w.H.to(DEV), W=w.W.to(DEV), T=w.temperature.to(DEV), seeds=w.seeds.to(DEV),
             pos=positions.to(DEV), bias=w.bias.to(DEV), mask=w.mask.to(DEV))
    st_ref = torch.full((w.B,), -9, dtype=torch.int32, device=DEV)
    st_new = torch.full((w.B,), -9, dtype=torch.int32, device=DEV)
    out_ref = torch.full((w.B,), -5, dtype=torch.int64, device=DEV)
    out_new = torch.full((w.B,), -5, dtype=torch.int64, device=DEV)
    ws = torch.empty(lms.workspace_bytes(lms.OP_LMHEAD, w.B, w.D, w.V), dtype=torch.uint8, device=DEV)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    p_ref = _params(w, d, wide, st_ref)
    rc = L.lms_lmhead_sample(ctypes.c_void_p(d["H"].data_ptr()), w.D, ctypes.c_void_p(d["W"].data_ptr()),
                             w.D, w.B, w.D, w.V, ctypes.byref(p_ref), ctypes.c_void_p(out_ref.data_ptr()),
                             ctypes.c_void_p(ws.data_ptr()), ws.numel(), stream)
    assert rc == 0, L.lms_last_error()
    p_new = _params(w, d, wide, st_new)
    rc = L.lms_lmhead_sample_noalloc(ctypes.c_void_p(d["H"].data_ptr()), w.D,
                                     ctypes.c_void_p(d["W"].data_ptr()), w.D, w.B, w.D, w.V,
                                     ctypes.byref(p_new), ctypes.c_void_p(out_new.data_ptr()), stream)
    assert rc == 0, L.lms_last_error()
    torch.cuda.synchronize()
    return out_ref.cpu().numpy(), st_ref.cpu().numpy(), out_new.cpu().numpy(), st_new.cpu().numpy()


@pytest.mark.gpu
def test_noalloc_matches_workspace_entry_point_on_consecutive_calls():
    L = _lib()
    w = _case(37, 256, 5000, seed=3)
    for call, (positions, wide) in enumerate([(torch.arange(w.B) * 2, False),
                                              (torch.arange(w.B) * 2 + 1, True)]):
        out_ref, st_ref, out_new, st_new = _run_both(L, w, positions.to(torch.int64), wide)
        # same kernels, same inputs: the tokens are identical, not merely within the near-tie rule
        assert np.array_equal(st_new, st_ref), call
        assert np.array_equal(out_new, out_ref), call
        assert (st_ref >= 0).all() and (out_ref[st_ref == 0] >= 0).all()
    # a smaller call after a larger one reads only candidates it wrote itself
    w2 = _case(3, 128, 700, seed=4)
    out_ref, st_ref, out_new, st_new = _run_both(L, w2, torch.arange(3, dtype=torch.int64), False)
    assert np.array_equal(out_new, out_ref) and np.array_equal(st_new, st_ref)


@pytest.mark.gpu
def test_noalloc_fills_its_scratch_across_launches():
    # B * ceil(V / 128) = 512 * 1024 = 524288 candidates: the whole array, written by one row-group
    # Stage-1 launch of two groups of 256 rows (the second group from candidate offset 256 * 1024);
    # then a smaller call
    L = _lib()
    w = _case(512, 64, 131072, seed=5)
    out_ref, st_ref, out_new, st_new = _run_both(L, w, torch.arange(w.B, dtype=torch.int64) * 3, True)
    assert np.array_equal(st_new, st_ref) and np.array_equal(out_new, out_ref)
    assert (st_ref >= 0).all()
    w2 = _case(5, 64, 3000, seed=6)
    out_ref, st_ref, out_new, st_new = _run_both(L, w2, torch.arange(5, dtype=torch.int64), False)
    assert np.array_equal(out_new, out_ref) and np.array_equal(st_new, st_ref)


def test_noalloc_refuses_calls_beyond_its_scratch():
    L = _lib()
    p = lms.SampleParams()
    fake = ctypes.c_void_p(0x100000)   # never dereferenced: the call is refused on the host
    # B * ceil(V / 128) = 442 * 1187 > 524288 candidates
    rc = L.lms_lmhead_sample_noalloc(fake, 4096, fake, 4096, 442, 4096, 151936, ctypes.byref(p),
                                     fake, None)
    assert rc == lms.LMS_ERR_WORKSPACE
    assert b"static scratch" in L.lms_last_error()
    # one candidate more than the array holds: 513 * 1024 = 525312
    rc = L.lms_lmhead_sample_noalloc(fake, 64, fake, 64, 513, 64, 131072, ctypes.byref(p), fake, None)
    assert rc == lms.LMS_ERR_WORKSPACE
    # invalid sizes get the regular entry point's checks
    assert L.lms_lmhead_sample_noalloc(fake, 64, fake, 64, 0, 64, 100, ctypes.byref(p), fake,
                                       None) == lms.LMS_ERR_INVALID_ARG
