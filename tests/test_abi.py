"""The C ABI without a GPU: the library loads, exports every function include/lms.h declares,
and rejects bad arguments on the host before anything is launched."""
import ctypes
import os
import re

import pytest

import lm_head_gumbel_lmhead_gb300 as lms

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    text = open(os.path.join(ROOT, "include", "lms.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(lms_[a-z0-9_]+)\s*\(", text)))


@pytest.fixture(scope="module")
def L():
    from lm_head_gumbel_lmhead_gb300 import build
    build.build()
    return lms.lib()


def test_every_declared_function_is_exported(L):
    names = _declared()
    assert "lms_lmhead_sample" in names and "lms_sample_from_logits" in names
    assert "lms_philox_fill_noise" in names
    for n in names:
        assert hasattr(L, n), f"{n} declared in lms.h but not exported"


def test_version_and_empty_error(L):
    assert lms.version().startswith("lms")


def test_params_struct_matches_header_size(L):
    # pointers/int64 x9, 4 x int32, pointer, 2 x uint32 = 72 + 16 + 8 + 8
    assert ctypes.sizeof(lms.SampleParams) == 104


def test_tile_info(L):
    tv, nt, ws, path = lms.tile_info(lms.OP_LMHEAD, 64, 4096, 151936)
    assert tv == 128 and nt == 1187 and path == lms.PATH_TCGEN05
    cand = 64 * 1187 * 4
    # the 256-byte status block, then scores and indices at 256-byte boundaries
    assert ws == 256 + 2 * ((cand + 255) // 256 * 256)
    assert lms.tile_info(lms.OP_LMHEAD, 1, 4096, 151936)[3] == lms.PATH_TCGEN05
    tv, nt, _, _ = lms.tile_info(lms.OP_LOGITS, 8192, 0, 131072)
    assert tv == 8192 and nt == 16
    tv, nt, _, _ = lms.tile_info(lms.OP_LOGITS, 1, 0, 131072)
    assert tv == 1024 and nt == 128
    tv, nt, _, _ = lms.tile_info(lms.OP_LOGITS, 8, 0, 131072)
    assert tv == 2048 and nt == 64
    assert lms.tile_info(lms.OP_LOGITS, 3, 0, 1000, 256)[:2] == (256, 4)
    assert lms.workspace_bytes(lms.OP_LMHEAD, 0, 4096, 100) == 0


@pytest.mark.parametrize("args,status", [
    ((lms.OP_LMHEAD, 0, 64, 100, 0), lms.LMS_ERR_INVALID_ARG),
    ((lms.OP_LMHEAD, 4, 0, 100, 0), lms.LMS_ERR_INVALID_ARG),
    ((lms.OP_LMHEAD, 4, 64, 2**31, 0), lms.LMS_ERR_INVALID_ARG),
    ((lms.OP_LMHEAD, 4, 64, 100, 64), lms.LMS_ERR_UNSUPPORTED),
    ((lms.OP_LOGITS, 4, 0, 100, 300), lms.LMS_ERR_UNSUPPORTED),
    ((lms.OP_LOGITS, 4, 0, 100, 128), lms.LMS_ERR_UNSUPPORTED),
    ((7, 4, 0, 100, 0), lms.LMS_ERR_INVALID_ARG),
])
def test_tile_info_rejects(L, args, status):
    with pytest.raises(lms.LmsError) as e:
        lms.tile_info(*args)
    assert e.value.status == status


def _params(**kw):
    p = lms.SampleParams()
    for k, v in kw.items():
        setattr(p, k, v)
    return p


FAKE = ctypes.c_void_p(0x100000)   # a 16-byte aligned non-null address; never dereferenced


@pytest.mark.parametrize("kw,call_kw,status", [
    (dict(), dict(H=None), lms.LMS_ERR_INVALID_ARG),
    (dict(noise_mode=5), dict(), lms.LMS_ERR_INVALID_ARG),
    (dict(seeds=0x1000), dict(), lms.LMS_ERR_INVALID_ARG),           # seeds without positions
    (dict(reserved=1), dict(), lms.LMS_ERR_INVALID_ARG),
    (dict(debug_flags=8), dict(), lms.LMS_ERR_INVALID_ARG),
    (dict(bias=0x1000, ld_bias=10), dict(), lms.LMS_ERR_INVALID_ARG),
    (dict(), dict(D=60), lms.LMS_ERR_UNSUPPORTED),                    # D % 8 != 0
    (dict(), dict(ldh=70), lms.LMS_ERR_UNSUPPORTED),
    (dict(), dict(H=ctypes.c_void_p(0x100008)), lms.LMS_ERR_UNSUPPORTED),
    (dict(), dict(ws_bytes=16), lms.LMS_ERR_WORKSPACE),
    (dict(path=lms.PATH_GEMV), dict(B=9), lms.LMS_ERR_UNSUPPORTED),
    (dict(path=9), dict(), lms.LMS_ERR_INVALID_ARG),
])
def test_lmhead_host_validation(L, kw, call_kw, status):
    c = dict(H=FAKE, ldh=64, W=FAKE, ldw=64, B=4, D=64, V=1000, out=FAKE, ws=FAKE, ws_bytes=1 << 20)
    c.update(call_kw)
    p = _params(**kw)
    st = L.lms_lmhead_sample(c["H"], c["ldh"], c["W"], c["ldw"], c["B"], c["D"], c["V"],
                             ctypes.byref(p), c["out"], c["ws"], c["ws_bytes"], None)
    assert st == status, L.lms_last_error()
    assert L.lms_last_error()


def test_logits_and_noise_host_validation(L):
    p = _params()
    assert L.lms_sample_from_logits(FAKE, 7, 0, 4, 100, ctypes.byref(p), FAKE, FAKE, 1 << 20, None) == lms.LMS_ERR_INVALID_ARG
    assert L.lms_sample_from_logits(FAKE, 0, 50, 4, 100, ctypes.byref(p), FAKE, FAKE, 1 << 20, None) == lms.LMS_ERR_INVALID_ARG
    assert L.lms_sample_from_logits(FAKE, 0, 0, 4, 100, ctypes.byref(p), FAKE, FAKE, 8, None) == lms.LMS_ERR_WORKSPACE
    p2 = _params(debug_flags=1)
    assert L.lms_sample_from_logits(FAKE, 0, 0, 4, 100, ctypes.byref(p2), FAKE, FAKE, 1 << 20, None) == lms.LMS_ERR_INVALID_ARG
    assert L.lms_philox_fill_noise(None, 0, 0, 4, 100, None, None, 0, 0, None) == lms.LMS_ERR_INVALID_ARG
    assert L.lms_philox_fill_noise(FAKE, 9, 0, 4, 100, None, None, 0, 0, None) == lms.LMS_ERR_INVALID_ARG
    assert L.lms_philox_fill_noise(FAKE, 0, 0, 0, 100, None, None, 0, 0, None) == lms.LMS_ERR_INVALID_ARG
    assert L.lms_philox_fill_noise(ctypes.c_void_p(0x100008), 0, 0, 4, 100, None, None, 0, 0, None) == lms.LMS_ERR_UNSUPPORTED


def test_verify_host_validation(L):
    def call(p=None, dtype=0, ld=1000, B=4, k=3, V=1000, ws_bytes=1 << 24, tokens=FAKE):
        p = _params() if p is None else p
        return L.lms_verify_from_logits(FAKE, FAKE, dtype, ld, B, k, V, tokens, ctypes.byref(p),
                                        FAKE, FAKE, FAKE, ws_bytes, None)
    assert call(dtype=5) == lms.LMS_ERR_INVALID_ARG
    assert call(k=0) == lms.LMS_ERR_INVALID_ARG
    assert call(k=lms.VERIFY_MAX_K + 1) == lms.LMS_ERR_INVALID_ARG
    assert call(ld=999) == lms.LMS_ERR_INVALID_ARG
    assert call(B=0) == lms.LMS_ERR_INVALID_ARG
    assert call(tokens=None) == lms.LMS_ERR_INVALID_ARG
    assert call(p=_params(bias=0x1000, ld_bias=1000)) == lms.LMS_ERR_INVALID_ARG
    assert call(p=_params(allow_mask=0x1000, ld_mask=32)) == lms.LMS_ERR_INVALID_ARG
    assert call(p=_params(path=lms.PATH_GEMV)) == lms.LMS_ERR_INVALID_ARG
    assert call(p=_params(seeds=0x1000)) == lms.LMS_ERR_INVALID_ARG     # seeds without positions
    need = L.lms_workspace_bytes_verify(4, 3, 1000)
    r256 = lambda x: -(-x // 256) * 256
    assert need > 0 and call(ws_bytes=need - 1) == lms.LMS_ERR_WORKSPACE
    assert L.lms_workspace_bytes_verify(4, 0, 1000) == 0
    assert L.lms_workspace_bytes_verify(4, 3, 2**31) == 0
    # partials of 2k+1 rows per batch row (three arrays), decisions, two candidates per chunk
    # (sized for fp32 logits: one partial per warp over chunks of 8192 entries, 16-byte row
    # decisions, race candidates over chunks of 4096), and a per-row completion counter, after
    # the 256-byte status block every workspace starts with
    assert need == 256 + 3 * r256(4 * 7 * 8 * 4) + 256 + 2 * 256 + 256
    big = L.lms_workspace_bytes_verify(64, 4, 151936)
    nc, ncr = -(-151936 // 8192), -(-151936 // 4096)
    r256 = lambda x: -(-x // 256) * 256
    assert big == 256 + 3 * r256(64 * 9 * nc * 8 * 4) + r256(64 * 16) + 2 * r256(64 * ncr * 8) + r256(64 * 4)


def test_topk_fp8_filtered_noalloc_host_validation(L):
    INV, UNS, WS = lms.LMS_ERR_INVALID_ARG, lms.LMS_ERR_UNSUPPORTED, lms.LMS_ERR_WORKSPACE

    def topk(k=4, D=64, H=FAKE, ws_bytes=1 << 24, p=None):
        p = _params() if p is None else p
        return L.lms_lmhead_sample_topk(H, 64, FAKE, 64, 4, D, 1000, k, ctypes.byref(p), FAKE, None,
                                        FAKE, ws_bytes, None)
    assert topk(k=0) == INV and topk(k=17) == INV
    assert topk(D=60) == UNS and topk(H=ctypes.c_void_p(0x100008)) == UNS
    assert topk(p=_params(path=lms.PATH_GEMV)) == UNS
    assert topk(ws_bytes=L.lms_workspace_bytes_topk(4, 1000, 4) - 1) == WS

    def fp8(w_scale=FAKE, D=64, ldw8=64, ws_bytes=1 << 24):
        p = _params()
        return L.lms_lmhead_sample_fp8(FAKE, 64, FAKE, ldw8, w_scale, 4, D, 1000, ctypes.byref(p), FAKE,
                                       FAKE, ws_bytes, None)
    assert fp8(w_scale=None) == INV
    assert fp8(D=24, ldw8=24) == UNS                    # D must be a multiple of 16
    assert fp8(ldw8=72) == UNS                          # ldw8 must be a multiple of 16
    assert fp8(ws_bytes=16) == WS

    def filtered(filters=True, k_max=1024, p=None, ld=0):
        p = _params() if p is None else p
        f = lms.FilterParams()
        f.k_max = k_max
        return L.lms_sample_from_logits_filtered(FAKE, 1, ld, 4, 1000, ctypes.byref(p),
                                                 ctypes.byref(f) if filters else None, FAKE, None)
    assert filtered(filters=False) == INV
    assert filtered(k_max=1025) == INV and filtered(k_max=-1) == INV
    assert filtered(p=_params(tile_v=256)) == INV
    assert filtered(ld=999) == INV

    # the allocation-free entry: B * ceil(V / 128) candidates beyond its static scratch are rejected
    p = _params()
    st = L.lms_lmhead_sample_noalloc(FAKE, 4096, FAKE, 4096, 65536, 4096, 151936, ctypes.byref(p), FAKE, None)
    assert st == WS and b"static scratch" in L.lms_last_error()


def test_mxfp4_host_validation(L):
    INV, UNS, WS = lms.LMS_ERR_INVALID_ARG, lms.LMS_ERR_UNSUPPORTED, lms.LMS_ERR_WORKSPACE
    # one 4352-byte block per (128-row tile, 64-element K chunk)
    assert L.lms_mxfp4_tiled_bytes(1000, 96) == 8 * 2 * 4352
    assert L.lms_mxfp4_tiled_bytes(151936, 4096) == 1187 * 64 * 4352
    assert L.lms_mxfp4_tiled_bytes(1000, 48) == 0 and L.lms_mxfp4_tiled_bytes(0, 64) == 0
    need = L.lms_mxfp4_tiled_bytes(1000, 64)

    def pack(ldw4=32, lds=1000, Wt=FAKE, n=need, D=64):
        return L.lms_mxfp4_pack(FAKE, ldw4, FAKE, lds, 1000, D, Wt, n, None)
    assert pack(Wt=None) == INV and pack(D=48) == INV
    assert pack(ldw4=31) == INV and pack(lds=999) == INV
    assert pack(Wt=ctypes.c_void_p(0x100008)) == UNS and pack(n=need - 1) == WS

    def mx(D=64, Wt=FAKE, n=need, ws_bytes=1 << 24, p=None):
        p = _params() if p is None else p
        return L.lms_lmhead_sample_mxfp4(FAKE, 64, Wt, n, 4, D, 1000, ctypes.byref(p), FAKE, FAKE,
                                         ws_bytes, None)
    assert mx(Wt=None) == INV and mx(n=need - 1) == INV
    assert mx(D=48) == UNS                              # D must be a multiple of 32
    assert mx(Wt=ctypes.c_void_p(0x100008)) == UNS
    assert mx(p=_params(path=lms.PATH_GEMV)) == UNS
    assert mx(ws_bytes=lms.workspace_bytes(lms.OP_LMHEAD, 4, 64, 1000) - 1) == WS


def test_read_status_rejects_a_missing_workspace(L):
    bits = ctypes.c_uint32(7)
    assert L.lms_read_status(None, None, ctypes.byref(bits)) == lms.LMS_ERR_INVALID_ARG
    assert bits.value == 7
    assert b"workspace" in L.lms_last_error()
