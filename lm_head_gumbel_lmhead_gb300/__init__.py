"""Exact Gumbel-max token sampling fused into the LM-head projection, for GB300 (sm_103a).

A thin ctypes binding over the C ABI in ``include/lms.h`` (library ``_lib/liblms.so``).  Every
step of the computation runs in the library's CUDA kernels; this module only checks tensor
metadata, allocates the workspace with PyTorch and passes raw device pointers and the current
CUDA stream.  There is no CPU fallback: if the library is missing or no GPU is present, calls
raise.

    tokens = lmhead_sample(H, W, temperature=T, seeds=seeds, positions=pos)
    tokens = sample_from_logits(logits, temperature=T, seeds=seeds, positions=pos)
    noise  = philox_fill_noise(B, V, kind="gumbel", seeds=seeds, positions=pos)
"""
from __future__ import annotations

import ctypes
import os
import threading
from typing import Optional

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "_lib", "liblms.so")

LMS_OK, LMS_ERR_INVALID_ARG, LMS_ERR_UNSUPPORTED, LMS_ERR_WORKSPACE, LMS_ERR_CUDA, LMS_ERR_TIMEOUT = range(6)
NOISE_FP32, NOISE_WIDE53 = 0, 1
DTYPE_F32, DTYPE_BF16 = 0, 1
OP_LMHEAD, OP_LOGITS, OP_LMHEAD_FP8 = 0, 1, 2
PATH_AUTO, PATH_GEMV, PATH_TCGEN05, PATH_TCGEN05_PAIR = 0, 1, 2, 3
NOISE_KINDS = {"words": 0, "uniform": 1, "exponential": 2, "gumbel": 3}
ROW_OK, ROW_NO_CANDIDATE, ROW_BAD_TEMPERATURE, ROW_DEVICE_TIMEOUT = range(4)
DEBUG_WITHHOLD_FIRST_LOAD = 1
FUSED_TILE_V = 128
GEMV_MAX_B = 8


class LmsError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"lms status {status}: {message}")
        self.status = status


class SampleParams(ctypes.Structure):
    """Mirror of ``lms_sample_params``."""
    _fields_ = [
        ("temperature", ctypes.c_void_p),
        ("seeds", ctypes.c_void_p),
        ("positions", ctypes.c_void_p),
        ("bias", ctypes.c_void_p),
        ("ld_bias", ctypes.c_int64),
        ("allow_mask", ctypes.c_void_p),
        ("ld_mask", ctypes.c_int64),
        ("base_seed", ctypes.c_uint64),
        ("offset", ctypes.c_uint64),
        ("noise_mode", ctypes.c_int32),
        ("tile_v", ctypes.c_int32),
        ("path", ctypes.c_int32),
        ("timeout_ms", ctypes.c_uint32),
        ("row_status", ctypes.c_void_p),
        ("debug_flags", ctypes.c_uint32),
        ("reserved", ctypes.c_uint32),
    ]


class FilterParams(ctypes.Structure):
    """Mirror of ``lms_filter_params``."""
    _fields_ = [("top_k", ctypes.c_void_p), ("top_p", ctypes.c_void_p), ("min_p", ctypes.c_void_p),
                ("k_max", ctypes.c_int32), ("reserved", ctypes.c_int32)]


_lock = threading.Lock()
_lib = None


def lib() -> ctypes.CDLL:
    """The loaded C library (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(f"{LIB_PATH} is missing: build it with "
                                   "`python -m lm_head_gumbel_lmhead_gb300.build` (needs nvcc)")
            L = ctypes.CDLL(LIB_PATH)
            P, i32, i64, u64, sz = (ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64,
                                    ctypes.c_uint64, ctypes.c_size_t)
            L.lms_version.restype = ctypes.c_char_p
            L.lms_last_error.restype = ctypes.c_char_p
            L.lms_tile_info.argtypes = [i32, i64, i64, i64, i32, P, P, P, P]
            L.lms_tile_info.restype = i32
            L.lms_workspace_bytes.argtypes = [i32, i64, i64, i64, i32]
            L.lms_workspace_bytes.restype = sz
            L.lms_lmhead_sample.argtypes = [P, i64, P, i64, i64, i64, i64,
                                            ctypes.POINTER(SampleParams), P, P, sz, P]
            L.lms_lmhead_sample.restype = i32
            L.lms_sample_from_logits.argtypes = [P, i32, i64, i64, i64, ctypes.POINTER(SampleParams),
                                                 P, P, sz, P]
            L.lms_sample_from_logits.restype = i32
            L.lms_lmhead_sample_noalloc.argtypes = [P, i64, P, i64, i64, i64, i64,
                                                    ctypes.POINTER(SampleParams), P, P]
            L.lms_lmhead_sample_noalloc.restype = i32
            L.lms_lmhead_sample_fp8.argtypes = [P, i64, P, i64, P, i64, i64, i64,
                                                ctypes.POINTER(SampleParams), P, P, sz, P]
            L.lms_lmhead_sample_fp8.restype = i32
            L.lms_mxfp4_tiled_bytes.argtypes = [i64, i64]
            L.lms_mxfp4_tiled_bytes.restype = sz
            L.lms_mxfp4_pack.argtypes = [P, i64, P, i64, i64, i64, P, sz, P]
            L.lms_mxfp4_pack.restype = i32
            L.lms_lmhead_sample_mxfp4.argtypes = [P, i64, P, sz, i64, i64, i64,
                                                  ctypes.POINTER(SampleParams), P, P, sz, P]
            L.lms_lmhead_sample_mxfp4.restype = i32
            L.lms_sample_from_logits_filtered.argtypes = [P, i32, i64, i64, i64,
                                                          ctypes.POINTER(SampleParams),
                                                          ctypes.POINTER(FilterParams), P, P]
            L.lms_sample_from_logits_filtered.restype = i32
            L.lms_workspace_bytes_topk.argtypes = [i64, i64, i32]
            L.lms_workspace_bytes_topk.restype = sz
            L.lms_lmhead_sample_topk.argtypes = [P, i64, P, i64, i64, i64, i64, i32,
                                                 ctypes.POINTER(SampleParams), P, P, P, sz, P]
            L.lms_lmhead_sample_topk.restype = i32
            L.lms_workspace_bytes_verify.argtypes = [i64, i32, i64]
            L.lms_workspace_bytes_verify.restype = sz
            L.lms_verify_from_logits.argtypes = [P, P, i32, i64, i64, i32, i64, P,
                                                 ctypes.POINTER(SampleParams), P, P, P, sz, P]
            L.lms_verify_from_logits.restype = i32
            L.lms_philox_fill_noise.argtypes = [P, i32, i32, i64, i64, P, P, u64, u64, P]
            L.lms_philox_fill_noise.restype = i32
            L.lms_read_status.argtypes = [P, P, P]
            L.lms_read_status.restype = i32
            _lib = L
    return _lib


def _check(status: int):
    if status != LMS_OK:
        raise LmsError(status, lib().lms_last_error().decode())


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _dev(t: Optional[torch.Tensor], dtype, name, device):
    if t is None:
        return None
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if t.device != device:
        raise ValueError(f"{name} must be on {device}, got {t.device}")
    if not t.is_contiguous() and t.dim() == 1:
        raise ValueError(f"{name} must be contiguous")
    return t


def _row_ld(t: Optional[torch.Tensor], name) -> int:
    if t is None or t.dim() == 1:
        if t is not None and t.stride(0) != 1:
            raise ValueError(f"{name} must have unit stride")
        return 0
    if t.stride(1) != 1:
        raise ValueError(f"{name} must be row-major with unit inner stride")
    return t.stride(0)


def _stream(stream) -> ctypes.c_void_p:
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def tile_info(op: int, B: int, D: int, V: int, tile_v: int = 0):
    """(tile_v, n_tiles, workspace_bytes, auto_path) for a call of these sizes."""
    tv, nt, ws, path = ctypes.c_int32(), ctypes.c_int64(), ctypes.c_size_t(), ctypes.c_int32()
    _check(lib().lms_tile_info(op, B, D, V, tile_v, ctypes.byref(tv), ctypes.byref(nt),
                               ctypes.byref(ws), ctypes.byref(path)))
    return tv.value, nt.value, ws.value, path.value


def workspace_bytes(op: int, B: int, D: int, V: int, tile_v: int = 0) -> int:
    return int(lib().lms_workspace_bytes(op, B, D, V, tile_v))


STATUS_BLOCK_BYTES = 256   # every workspace starts with the call's status word


def split_workspace(ws: torch.Tensor, B: int, n_tiles: int):
    """Views of the Stage-1 candidates in a workspace: (score f32 [B, nt], index i32 [B, nt])."""
    n = B * n_tiles
    off = STATUS_BLOCK_BYTES + (4 * n + 255) // 256 * 256
    raw = ws.view(torch.uint8)
    score = raw[STATUS_BLOCK_BYTES: STATUS_BLOCK_BYTES + 4 * n].view(torch.float32).view(B, n_tiles)
    index = raw[off: off + 4 * n].view(torch.int32).view(B, n_tiles)
    return score, index


def read_status(workspace: torch.Tensor, stream=None):
    """(lms_status, status_bits) of the last call that used `workspace`: synchronises the stream
    and reads the status word (bit s set when some row ended with row status s).  Returns
    LMS_ERR_TIMEOUT as the status when a device-side wait ran out; raises on other errors."""
    bits = ctypes.c_uint32(0)
    st = lib().lms_read_status(_ptr(workspace), _stream(stream), ctypes.byref(bits))
    if st not in (LMS_OK, LMS_ERR_TIMEOUT):
        _check(st)
    return st, bits.value


def _params(B, device, temperature, seeds, positions, bias, mask, base_seed, offset, wide, tile_v,
            path, row_status, timeout_ms, debug_flags):
    temperature = _dev(temperature, torch.float32, "temperature", device)
    seeds = _dev(seeds, torch.int64, "seeds", device)
    positions = _dev(positions, torch.int64, "positions", device)
    bias = _dev(bias, torch.float32, "bias", device)
    mask = _dev(mask, torch.int32, "mask", device)
    row_status = _dev(row_status, torch.int32, "row_status", device)
    for t, n in ((temperature, "temperature"), (seeds, "seeds"), (positions, "positions"),
                 (row_status, "row_status")):
        if t is not None and (t.dim() != 1 or t.shape[0] < B or t.stride(0) != 1):
            raise ValueError(f"{n} must be a contiguous vector of length >= {B}")
    p = SampleParams()
    p.temperature = temperature.data_ptr() if temperature is not None else None
    p.seeds = seeds.data_ptr() if seeds is not None else None
    p.positions = positions.data_ptr() if positions is not None else None
    p.bias = bias.data_ptr() if bias is not None else None
    p.ld_bias = _row_ld(bias, "bias")
    p.allow_mask = mask.data_ptr() if mask is not None else None
    p.ld_mask = _row_ld(mask, "mask")
    p.base_seed = int(base_seed) & (2**64 - 1)
    p.offset = int(offset) & (2**64 - 1)
    p.noise_mode = NOISE_WIDE53 if wide else NOISE_FP32
    p.tile_v = int(tile_v)
    p.path = int(path)
    p.timeout_ms = int(timeout_ms)
    p.row_status = row_status.data_ptr() if row_status is not None else None
    p.debug_flags = int(debug_flags)
    p.reserved = 0
    return p


class Prepared:
    """One C-ABI call with its arguments marshalled once, for a loop that repeats the call on the
    same buffers and stream: the buffers' contents may change between calls, their addresses and
    sizes may not, and the stream is the one given (or current) when the call was prepared.
    Calling it makes the C call (the same one the plain wrapper makes) and returns its outputs."""

    def __init__(self, fn, args, keep, result):
        self._fn, self._args, self._keep, self._result = fn, args, keep, result

    def __call__(self):
        _check(self._fn(*self._args))
        return self._result


def lmhead_sample(H: torch.Tensor, W: torch.Tensor, *, temperature=None, seeds=None,
                  positions=None, bias=None, mask=None, base_seed: int = 0, offset: int = 0,
                  wide: bool = False, path: int = PATH_AUTO, out=None, workspace=None,
                  row_status=None, timeout_ms: int = 0, debug_flags: int = 0,
                  stream=None) -> torch.Tensor:
    """Sample one token per row of H [B, D] from softmax((H W^T + bias) / T) with W [V, D].

    bf16 H and W on the GPU; per-row temperature (fp32, 0 = greedy), seeds / positions (int64,
    seed < 0 = unseeded), bias fp32 [B, V] or [V], mask int32 allow-bit words [B, ceil(V/32)].
    Returns int64 [B] (-1 on rows whose status is not 0)."""
    return prepare_lmhead_sample(H, W, temperature=temperature, seeds=seeds, positions=positions,
                                 bias=bias, mask=mask, base_seed=base_seed, offset=offset, wide=wide,
                                 path=path, out=out, workspace=workspace, row_status=row_status,
                                 timeout_ms=timeout_ms, debug_flags=debug_flags, stream=stream)()


def prepare_lmhead_sample(H: torch.Tensor, W: torch.Tensor, *, temperature=None, seeds=None,
                          positions=None, bias=None, mask=None, base_seed: int = 0, offset: int = 0,
                          wide: bool = False, path: int = PATH_AUTO, out=None, workspace=None,
                          row_status=None, timeout_ms: int = 0, debug_flags: int = 0,
                          stream=None) -> Prepared:
    """lmhead_sample's call, checked and marshalled once (see Prepared)."""
    if H.dtype != torch.bfloat16 or W.dtype != torch.bfloat16:
        raise TypeError("H and W must be bfloat16")
    if not H.is_cuda or W.device != H.device:
        raise ValueError("H and W must be on the same CUDA device")
    if H.dim() != 2 or W.dim() != 2 or H.shape[1] != W.shape[1]:
        raise ValueError("H must be [B, D] and W [V, D]")
    if H.stride(1) != 1 or W.stride(1) != 1:
        raise ValueError("H and W must be row-major with unit inner stride")
    B, D = H.shape
    V = W.shape[0]
    dev = H.device
    p = _params(B, dev, temperature, seeds, positions, bias, mask, base_seed, offset, wide, 0, path,
                row_status, timeout_ms, debug_flags)
    if out is None:
        out = torch.empty(B, dtype=torch.int64, device=dev)
    if workspace is None:
        workspace = torch.empty(workspace_bytes(OP_LMHEAD, B, D, V), dtype=torch.uint8, device=dev)
    args = (_ptr(H), H.stride(0), _ptr(W), W.stride(0), B, D, V, ctypes.byref(p), _ptr(out),
            _ptr(workspace), workspace.numel() * workspace.element_size(), _stream(stream))
    return Prepared(lib().lms_lmhead_sample, args,
                    (H, W, temperature, seeds, positions, bias, mask, row_status, workspace, p), out)


TOPK_MAX = 16


def lmhead_sample_topk(H: torch.Tensor, W: torch.Tensor, k: int, *, temperature=None, seeds=None,
                       positions=None, bias=None, mask=None, base_seed: int = 0, offset: int = 0,
                       wide: bool = False, out=None, scores=None, want_scores: bool = True,
                       workspace=None, row_status=None, timeout_ms: int = 0, debug_flags: int = 0,
                       stream=None):
    """Gumbel-top-k of the fused path: per row of H [B, D], the k largest perturbed scores of
    lmhead_sample's race (k draws without replacement), larger first, then the smaller index.
    Returns (indices int64 [B, k], -1 past a row's finite scores; scores fp32 [B, k] or None)."""
    return prepare_lmhead_sample_topk(
        H, W, k, temperature=temperature, seeds=seeds, positions=positions, bias=bias, mask=mask,
        base_seed=base_seed, offset=offset, wide=wide, out=out, scores=scores,
        want_scores=want_scores, workspace=workspace, row_status=row_status,
        timeout_ms=timeout_ms, debug_flags=debug_flags, stream=stream)()


def prepare_lmhead_sample_topk(H: torch.Tensor, W: torch.Tensor, k: int, *, temperature=None,
                               seeds=None, positions=None, bias=None, mask=None, base_seed: int = 0,
                               offset: int = 0, wide: bool = False, out=None, scores=None,
                               want_scores: bool = True, workspace=None, row_status=None,
                               timeout_ms: int = 0, debug_flags: int = 0, stream=None) -> Prepared:
    """lmhead_sample_topk's call, checked and marshalled once (see Prepared)."""
    if H.dtype != torch.bfloat16 or W.dtype != torch.bfloat16:
        raise TypeError("H and W must be bfloat16")
    if not H.is_cuda or W.device != H.device:
        raise ValueError("H and W must be on the same CUDA device")
    if H.dim() != 2 or W.dim() != 2 or H.shape[1] != W.shape[1]:
        raise ValueError("H must be [B, D] and W [V, D]")
    if H.stride(1) != 1 or W.stride(1) != 1:
        raise ValueError("H and W must be row-major with unit inner stride")
    B, D = H.shape
    V = W.shape[0]
    dev = H.device
    p = _params(B, dev, temperature, seeds, positions, bias, mask, base_seed, offset, wide, 0,
                PATH_AUTO, row_status, timeout_ms, debug_flags)
    if out is None:
        out = torch.empty(B, k, dtype=torch.int64, device=dev)
    if scores is None and want_scores:
        scores = torch.empty(B, k, dtype=torch.float32, device=dev)
    if workspace is None:
        need = lib().lms_workspace_bytes_topk(B, V, k)
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=dev)
    args = (_ptr(H), H.stride(0), _ptr(W), W.stride(0), B, D, V, k, ctypes.byref(p), _ptr(out),
            _ptr(scores) if scores is not None else None, _ptr(workspace),
            workspace.numel() * workspace.element_size(), _stream(stream))
    return Prepared(lib().lms_lmhead_sample_topk, args,
                    (H, W, temperature, seeds, positions, bias, mask, row_status, workspace, p),
                    (out, scores))


def lmhead_sample_fp8(H: torch.Tensor, W8: torch.Tensor, w_scale: torch.Tensor, *, temperature=None,
                      seeds=None, positions=None, bias=None, mask=None, base_seed: int = 0,
                      offset: int = 0, wide: bool = False, out=None, workspace=None,
                      row_status=None, timeout_ms: int = 0, debug_flags: int = 0,
                      stream=None) -> torch.Tensor:
    """lmhead_sample with FP8 inputs: W8 E4M3 codes (uint8 or float8_e4m3fn [V, D]) with per-row
    fp32 w_scale [V]; H bf16 [B, D] is quantised per row (power-of-two scale) by the call."""
    return prepare_lmhead_sample_fp8(
        H, W8, w_scale, temperature=temperature, seeds=seeds, positions=positions, bias=bias,
        mask=mask, base_seed=base_seed, offset=offset, wide=wide, out=out, workspace=workspace,
        row_status=row_status, timeout_ms=timeout_ms, debug_flags=debug_flags, stream=stream)()


def prepare_lmhead_sample_fp8(H: torch.Tensor, W8: torch.Tensor, w_scale: torch.Tensor, *,
                              temperature=None, seeds=None, positions=None, bias=None, mask=None,
                              base_seed: int = 0, offset: int = 0, wide: bool = False, out=None,
                              workspace=None, row_status=None, timeout_ms: int = 0,
                              debug_flags: int = 0, stream=None) -> Prepared:
    """lmhead_sample_fp8's call, checked and marshalled once (see Prepared)."""
    if H.dtype != torch.bfloat16:
        raise TypeError("H must be bfloat16")
    if W8.dtype not in (torch.uint8, torch.float8_e4m3fn):
        raise TypeError("W8 must be uint8 or float8_e4m3fn")
    if w_scale.dtype != torch.float32 or w_scale.dim() != 1 or w_scale.shape[0] != W8.shape[0]:
        raise ValueError("w_scale must be float32 [V]")
    if H.dim() != 2 or W8.dim() != 2 or H.shape[1] != W8.shape[1]:
        raise ValueError("H must be [B, D] and W8 [V, D]")
    if H.stride(1) != 1 or W8.stride(1) != 1:
        raise ValueError("H and W8 must be row-major with unit inner stride")
    B, D = H.shape
    V = W8.shape[0]
    dev = H.device
    p = _params(B, dev, temperature, seeds, positions, bias, mask, base_seed, offset, wide, 0,
                PATH_AUTO, row_status, timeout_ms, debug_flags)
    if out is None:
        out = torch.empty(B, dtype=torch.int64, device=dev)
    if workspace is None:
        workspace = torch.empty(workspace_bytes(OP_LMHEAD_FP8, B, D, V), dtype=torch.uint8, device=dev)
    args = (_ptr(H), H.stride(0), _ptr(W8), W8.stride(0), _ptr(w_scale), B, D, V, ctypes.byref(p),
            _ptr(out), _ptr(workspace), workspace.numel() * workspace.element_size(), _stream(stream))
    return Prepared(lib().lms_lmhead_sample_fp8, args,
                    (H, W8, w_scale, temperature, seeds, positions, bias, mask, row_status,
                     workspace, p), out)


def mxfp4_pack(W4: torch.Tensor, S: torch.Tensor, stream=None) -> torch.Tensor:
    """The library's tiled MXFP4 weights from the logical layout: W4 uint8 [V, D/2] packed E2M1
    codes (element d in the low nibble of byte d/2 when d is even), S uint8 [D/32, V] UE8M0 block
    scales (any row stride >= V), both on the GPU.  Returns uint8 [lms_mxfp4_tiled_bytes(V, D)]."""
    if W4.dtype != torch.uint8 or S.dtype != torch.uint8 or W4.dim() != 2 or S.dim() != 2:
        raise TypeError("W4 and S must be 2-D uint8 tensors")
    V, D = W4.shape[0], W4.shape[1] * 2
    if S.shape[0] * 32 != D or S.shape[1] != V:
        raise ValueError(f"S must be [{D // 32}, {V}] for W4 [{V}, {D // 2}]")
    if W4.stride(1) != 1 or S.stride(1) != 1 or not W4.is_cuda or S.device != W4.device:
        raise ValueError("W4 and S must be row-major CUDA tensors on one device")
    n = int(lib().lms_mxfp4_tiled_bytes(V, D))
    Wt = torch.empty(max(n, 1), dtype=torch.uint8, device=W4.device)
    _check(lib().lms_mxfp4_pack(_ptr(W4), W4.stride(0), _ptr(S), S.stride(0), V, D, _ptr(Wt), n,
                                _stream(stream)))
    return Wt


def lmhead_sample_mxfp4(H: torch.Tensor, Wt: torch.Tensor, V: int, *, temperature=None, seeds=None,
                        positions=None, bias=None, mask=None, base_seed: int = 0, offset: int = 0,
                        wide: bool = False, out=None, workspace=None, row_status=None,
                        timeout_ms: int = 0, debug_flags: int = 0, stream=None) -> torch.Tensor:
    """lmhead_sample with MXFP4 weights (W4A16): Wt the tiled weights of a V x D matrix
    (mxfp4_pack), H bf16 [B, D].  The workspace is lmhead_sample's (workspace_bytes(OP_LMHEAD, ...))."""
    return prepare_lmhead_sample_mxfp4(
        H, Wt, V, temperature=temperature, seeds=seeds, positions=positions, bias=bias, mask=mask,
        base_seed=base_seed, offset=offset, wide=wide, out=out, workspace=workspace,
        row_status=row_status, timeout_ms=timeout_ms, debug_flags=debug_flags, stream=stream)()


def prepare_lmhead_sample_mxfp4(H: torch.Tensor, Wt: torch.Tensor, V: int, *, temperature=None,
                                seeds=None, positions=None, bias=None, mask=None, base_seed: int = 0,
                                offset: int = 0, wide: bool = False, out=None, workspace=None,
                                row_status=None, timeout_ms: int = 0, debug_flags: int = 0,
                                stream=None) -> Prepared:
    """lmhead_sample_mxfp4's call, checked and marshalled once (see Prepared)."""
    if H.dtype != torch.bfloat16 or H.dim() != 2 or H.stride(1) != 1:
        raise TypeError("H must be a row-major bfloat16 [B, D] tensor")
    if Wt.dtype != torch.uint8 or not H.is_cuda or Wt.device != H.device:
        raise ValueError("Wt must be the uint8 tiled weights on H's device")
    B, D = H.shape
    dev = H.device
    p = _params(B, dev, temperature, seeds, positions, bias, mask, base_seed, offset, wide, 0,
                PATH_AUTO, row_status, timeout_ms, debug_flags)
    if out is None:
        out = torch.empty(B, dtype=torch.int64, device=dev)
    if workspace is None:
        workspace = torch.empty(workspace_bytes(OP_LMHEAD, B, D, V), dtype=torch.uint8, device=dev)
    args = (_ptr(H), H.stride(0), _ptr(Wt), Wt.numel(), B, D, V, ctypes.byref(p), _ptr(out),
            _ptr(workspace), workspace.numel() * workspace.element_size(), _stream(stream))
    return Prepared(lib().lms_lmhead_sample_mxfp4, args,
                    (H, Wt, temperature, seeds, positions, bias, mask, row_status, workspace, p), out)


def split_workspace_fp8(ws: torch.Tensor, B: int, D: int, n_tiles: int):
    """(score, index, quantised activations uint8 [B, round_up(D,16)], exponents int32 [B]) views
    of an FP8-path workspace."""
    score, index = split_workspace(ws, B, n_tiles)
    n = B * n_tiles
    off = STATUS_BLOCK_BYTES + 2 * ((4 * n + 255) // 256 * 256)
    ldq = (D + 15) // 16 * 16
    raw = ws.view(torch.uint8)
    q = raw[off: off + B * ldq].view(B, ldq)
    off2 = off + (B * ldq + 255) // 256 * 256
    e = raw[off2: off2 + 4 * B].view(torch.int32)
    return score, index, q, e


def lmhead_sample_noalloc(H: torch.Tensor, W: torch.Tensor, *, temperature=None, seeds=None,
                          positions=None, bias=None, mask=None, base_seed: int = 0,
                          offset: int = 0, wide: bool = False, path: int = PATH_AUTO, out=None,
                          row_status=None, stream=None) -> torch.Tensor:
    """lmhead_sample without a workspace, for callers that cannot allocate device memory: the
    Stage-1 candidates go to the library's fixed 4 MiB device array (B * ceil(V/128) <= 524288).
    Calls that overlap on the GPU share that array and race; serialise them.  `out` (and
    `row_status`) are still the caller's: pass preallocated tensors to allocate nothing."""
    if H.dtype != torch.bfloat16 or W.dtype != torch.bfloat16:
        raise TypeError("H and W must be bfloat16")
    if H.dim() != 2 or W.dim() != 2 or H.shape[1] != W.shape[1] or W.device != H.device:
        raise ValueError("H must be [B, D] and W [V, D] on one device")
    B, D = H.shape
    V = W.shape[0]
    p = _params(B, H.device, temperature, seeds, positions, bias, mask, base_seed, offset, wide, 0,
                path, row_status, 0, 0)
    if out is None:
        out = torch.empty(B, dtype=torch.int64, device=H.device)
    _check(lib().lms_lmhead_sample_noalloc(_ptr(H), H.stride(0), _ptr(W), W.stride(0), B, D, V,
                                           ctypes.byref(p), _ptr(out), _stream(stream)))
    return out


def sample_from_logits(logits: torch.Tensor, *, B: Optional[int] = None, temperature=None,
                       seeds=None, positions=None, bias=None, mask=None, base_seed: int = 0,
                       offset: int = 0, wide: bool = False, tile_v: int = 0, out=None,
                       workspace=None, row_status=None, stream=None) -> torch.Tensor:
    """The same race over materialised logits: fp32 or bf16 [B, V] (row-major), or one row [V]
    broadcast to B draws (pass B)."""
    if logits.dtype not in (torch.float32, torch.bfloat16):
        raise TypeError("logits must be float32 or bfloat16")
    if not logits.is_cuda:
        raise ValueError("logits must be on a CUDA device")
    if logits.dim() == 1:
        if B is None:
            raise ValueError("pass B for a broadcast row")
        ld, V = 0, logits.shape[0]
        if logits.stride(0) != 1:
            raise ValueError("logits must be contiguous")
    else:
        if logits.stride(1) != 1:
            raise ValueError("logits must be row-major with unit inner stride")
        B = logits.shape[0] if B is None else B
        ld, V = logits.stride(0), logits.shape[1]
    dev = logits.device
    p = _params(B, dev, temperature, seeds, positions, bias, mask, base_seed, offset, wide, tile_v,
                PATH_AUTO, row_status, 0, 0)
    if out is None:
        out = torch.empty(B, dtype=torch.int64, device=dev)
    if workspace is None:
        workspace = torch.empty(workspace_bytes(OP_LOGITS, B, 0, V, tile_v), dtype=torch.uint8,
                                device=dev)
    dt = DTYPE_F32 if logits.dtype == torch.float32 else DTYPE_BF16
    _check(lib().lms_sample_from_logits(_ptr(logits), dt, ld, B, V, ctypes.byref(p), _ptr(out),
                                        _ptr(workspace), workspace.numel() * workspace.element_size(),
                                        _stream(stream)))
    return out


def sample_from_logits_filtered(logits: torch.Tensor, *, B: Optional[int] = None, top_k=None,
                                top_p=None, min_p=None, k_max: int = 1024, temperature=None,
                                seeds=None, positions=None, bias=None, mask=None,
                                base_seed: int = 0, offset: int = 0, wide: bool = False, out=None,
                                row_status=None, stream=None) -> torch.Tensor:
    """The race over materialised logits after top-k -> top-p -> min-p filters (per-row [B]
    tensors: top_k int32, top_p / min_p float32; None = off)."""
    if logits.dtype not in (torch.float32, torch.bfloat16):
        raise TypeError("logits must be float32 or bfloat16")
    if logits.dim() == 1:
        if B is None:
            raise ValueError("pass B for a broadcast row")
        ld, V = 0, logits.shape[0]
    else:
        if logits.stride(1) != 1:
            raise ValueError("logits must be row-major with unit inner stride")
        B = logits.shape[0] if B is None else B
        ld, V = logits.stride(0), logits.shape[1]
    dev = logits.device
    p = _params(B, dev, temperature, seeds, positions, bias, mask, base_seed, offset, wide, 0,
                PATH_AUTO, row_status, 0, 0)
    fp = FilterParams()
    tk = _dev(top_k, torch.int32, "top_k", dev)
    tp = _dev(top_p, torch.float32, "top_p", dev)
    mp = _dev(min_p, torch.float32, "min_p", dev)
    fp.top_k = tk.data_ptr() if tk is not None else None
    fp.top_p = tp.data_ptr() if tp is not None else None
    fp.min_p = mp.data_ptr() if mp is not None else None
    fp.k_max = int(k_max)
    fp.reserved = 0
    if out is None:
        out = torch.empty(B, dtype=torch.int64, device=dev)
    dt = DTYPE_F32 if logits.dtype == torch.float32 else DTYPE_BF16
    _check(lib().lms_sample_from_logits_filtered(_ptr(logits), dt, ld, B, V, ctypes.byref(p),
                                                 ctypes.byref(fp), _ptr(out), _stream(stream)))
    return out


VERIFY_MAX_K = 32


def verify_from_logits(target: torch.Tensor, draft: torch.Tensor, draft_tokens: torch.Tensor, *,
                       temperature=None, seeds=None, positions=None, base_seed: int = 0,
                       offset: int = 0, wide: bool = False, accept_len=None, out=None,
                       workspace=None, row_status=None, stream=None):
    """Speculative-decoding verification: target logits [B, k+1, V], draft logits [B, k, V]
    (fp32 or bf16, same dtype, unit inner stride, rows ld apart within each tensor's [B, k(+1)]
    block as laid out contiguously), draft_tokens int64 [B, k].  Draft token x_i is accepted with
    probability min(1, p_t / p_d) in order; the first rejection is replaced by a draw from
    max(p_t - p_d, 0), and a fully accepted row draws a bonus token from the target at position k.
    Returns (accept_len int64 [B], out int64 [B, k+1] with -1 after the emitted tokens)."""
    if target.dtype not in (torch.float32, torch.bfloat16) or draft.dtype != target.dtype:
        raise TypeError("target and draft must both be float32 or both bfloat16")
    if not target.is_cuda or draft.device != target.device:
        raise ValueError("target and draft must be on the same CUDA device")
    if target.dim() != 3 or draft.dim() != 3:
        raise ValueError("target must be [B, k+1, V] and draft [B, k, V]")
    B, K1, V = target.shape
    k = K1 - 1
    if tuple(draft.shape) != (B, k, V) or k < 1:
        raise ValueError("draft must be [B, k, V] with k >= 1 and target [B, k+1, V]")
    ld = target.stride(1)
    for t, n, rows in ((target, "target", K1), (draft, "draft", k)):
        if t.stride(2) != 1 or t.stride(1) != ld or t.stride(0) != rows * ld:
            raise ValueError(f"{n} rows must be ld elements apart with unit inner stride")
    dev = target.device
    draft_tokens = _dev(draft_tokens, torch.int64, "draft_tokens", dev)
    if tuple(draft_tokens.shape) != (B, k) or not draft_tokens.is_contiguous():
        raise ValueError("draft_tokens must be a contiguous int64 [B, k]")
    p = _params(B, dev, temperature, seeds, positions, None, None, base_seed, offset, wide, 0,
                PATH_AUTO, row_status, 0, 0)
    if accept_len is None:
        accept_len = torch.empty(B, dtype=torch.int64, device=dev)
    if out is None:
        out = torch.empty(B, K1, dtype=torch.int64, device=dev)
    if workspace is None:
        need = lib().lms_workspace_bytes_verify(B, k, V)
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=dev)
    dt = DTYPE_F32 if target.dtype == torch.float32 else DTYPE_BF16
    _check(lib().lms_verify_from_logits(_ptr(target), _ptr(draft), dt, ld, B, k, V,
                                        _ptr(draft_tokens), ctypes.byref(p), _ptr(accept_len),
                                        _ptr(out), _ptr(workspace),
                                        workspace.numel() * workspace.element_size(),
                                        _stream(stream)))
    return accept_len, out


def philox_fill_noise(B: int, V: int, *, kind: str = "gumbel", wide: bool = False, seeds=None,
                      positions=None, base_seed: int = 0, offset: int = 0, device=None,
                      out=None, stream=None) -> torch.Tensor:
    """Noise grid [B, V] as the samplers compute it: kind 'words' (int32 [B, V, 4] holding the
    uint32 Philox words), 'uniform' (float64, exact), 'exponential' or 'gumbel' (float32)."""
    k = NOISE_KINDS[kind]
    device = torch.device(device or "cuda")
    if out is None:
        if k == 0:
            out = torch.empty(B, V, 4, dtype=torch.int32, device=device)
        elif k == 1:
            out = torch.empty(B, V, dtype=torch.float64, device=device)
        else:
            out = torch.empty(B, V, dtype=torch.float32, device=device)
    seeds = _dev(seeds, torch.int64, "seeds", out.device)
    positions = _dev(positions, torch.int64, "positions", out.device)
    _check(lib().lms_philox_fill_noise(_ptr(out), k, NOISE_WIDE53 if wide else NOISE_FP32, B, V,
                                       _ptr(seeds), _ptr(positions), int(base_seed) & (2**64 - 1),
                                       int(offset) & (2**64 - 1), _stream(stream)))
    return out


def version() -> str:
    return lib().lms_version().decode()
