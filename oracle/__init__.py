"""CPU oracle for exact Gumbel-max token sampling fused with the LM-head projection.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s
CPU-baseline / reference leg may import this package.  It shares no code with the CUDA library
in ``lm_head_gumbel_lmhead_gb300`` and never imports it.

The arithmetic lives in ``lms_oracle.c`` (plain C, fp64, compiled with gcc on first use); this
module only marshals numpy arrays.  Each function cites the page passage it follows; the
readings taken where the pages are silent are listed in ``lms_oracle.c``'s header.

Every function here has a pin in ``tests/test_oracle_*.py`` (Philox against Triton's own
Philox run in its CPU interpreter, the noise ranges the Megatron-LM PR prints, the tail-rate
closed form, chi-square against softmax, brute force over tile widths, fp64 GEMM against
numpy's matmul, greedy against numpy's argmax, the filters' hand-worked kept sets, the E4M3
codec against torch's cast, the Plackett-Luce law of Gumbel-top-k).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "lms_oracle.c")
_LIB_DIR = os.path.join(_HERE, "_build")
_LIB = os.path.join(_LIB_DIR, "liblms_oracle.so")
_lock = threading.Lock()
_lib = None

FP32_NOISE = 0
WIDE53_NOISE = 1


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (no CUDA).  Returns the shared-library path."""
    os.makedirs(_LIB_DIR, exist_ok=True)
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fPIC", "-shared", "-pthread",
               _SRC, "-o", tmp, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            P = ctypes.c_void_p
            i64, u64, i32 = ctypes.c_int64, ctypes.c_uint64, ctypes.c_int
            lib.orc_philox4x32_many.argtypes = [i64, P, P, i32, P]
            lib.orc_noise_fill.argtypes = [i64, i64, P, P, u64, u64, i32, P, P, P, P]
            lib.orc_sample_from_logits.argtypes = [P, i64, i64, i64, P, P, P, P, i64, P, i64, u64,
                                                   u64, i32, i64, P, P, P, P, P, P, P, i32]
            lib.orc_lmhead_logits.argtypes = [P, i64, P, i64, i64, i64, i64, P, i32]
            lib.orc_lmhead_sample.argtypes = [P, i64, P, i64, i64, i64, i64, P, P, P, P, i64, P,
                                              i64, u64, u64, i32, i64, P, P, P, P, P, P, P, i32]
            lib.orc_lmhead_sample.restype = ctypes.c_int
            lib.orc_lmhead_scores_at.argtypes = [P, i64, P, i64, i64, i64, i64, P, P, P, P, i64,
                                                 P, i64, u64, u64, i32, i64, P, P, P]
            lib.orc_lmhead_sample_rows.argtypes = [P, i64, P, i64, i64, i64, i64, P, i64, P, P,
                                                   P, P, i64, P, i64, u64, u64, i32, i64, P, P,
                                                   P, P, P, P, P, i32]
            lib.orc_lmhead_sample_rows.restype = ctypes.c_int
            lib.orc_sample_filtered.argtypes = [P, i64, i64, i64, P, P, P, P, i64, P, i64, u64, u64,
                                                i32, P, P, P, i32, ctypes.c_double,
                                                ctypes.c_double, P, P, P, P, P, i32]
            lib.orc_e4m3_decode.argtypes = [ctypes.c_uint8]
            lib.orc_e4m3_decode.restype = ctypes.c_double
            lib.orc_e4m3_encode.argtypes = [ctypes.c_double]
            lib.orc_e4m3_encode.restype = ctypes.c_uint8
            lib.orc_quantize_rows_e4m3.argtypes = [P, i64, i64, i64, P, i64, P]
            lib.orc_lmhead_logits_fp8.argtypes = [P, i64, P, P, i64, P, i64, i64, i64, P, i64, P, i32]
            lib.orc_lmhead_sample_fp8.argtypes = [P, i64, P, i64, P, i64, i64, i64, P, i64, P, P, P,
                                                  P, i64, P, i64, u64, u64, i32, i64, P, P, P, P,
                                                  P, P, i32]
            lib.orc_lmhead_sample_fp8.restype = ctypes.c_int
            lib.orc_e2m1_decode.argtypes = [ctypes.c_uint8]
            lib.orc_e2m1_decode.restype = ctypes.c_double
            lib.orc_e2m1_encode.argtypes = [ctypes.c_double]
            lib.orc_e2m1_encode.restype = ctypes.c_uint8
            lib.orc_ue8m0_decode.argtypes = [ctypes.c_uint8]
            lib.orc_ue8m0_decode.restype = ctypes.c_double
            lib.orc_mxfp4_weight.argtypes = [P, i64, P, i64, i64, i64]
            lib.orc_mxfp4_weight.restype = ctypes.c_double
            lib.orc_lmhead_logits_mxfp4.argtypes = [P, i64, P, i64, P, i64, i64, i64, i64, P, i64, P, i32]
            lib.orc_lmhead_sample_mxfp4.argtypes = [P, i64, P, i64, P, i64, i64, i64, i64, P, i64, P,
                                                    P, P, P, i64, P, i64, u64, u64, i32, i64, P, P, P,
                                                    P, P, P, i32]
            lib.orc_lmhead_sample_mxfp4.restype = ctypes.c_int
            lib.orc_noise_row.argtypes = [i32, i64, i64, u64, u64, i64, i64, i32, P]
            lib.orc_accept_uniform.argtypes = [i32, i64, i64, u64, u64, i64, i32]
            lib.orc_accept_uniform.restype = ctypes.c_double
            lib.orc_uniform.argtypes = [ctypes.c_uint32, ctypes.c_uint32, i32]
            lib.orc_uniform.restype = ctypes.c_double
            _lib = lib
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return None if a is None else np.ascontiguousarray(a, dtype=dtype)


def default_threads() -> int:
    return max(1, min(64, os.cpu_count() or 1))


def philox4x32(ctr, key, rounds: int = 10) -> np.ndarray:
    """Philox4x32-R (Salmon et al., SC'11) on arrays ctr [n,4] and key [n,2] (uint32)."""
    ctr = _c(np.asarray(ctr).reshape(-1, 4), np.uint32)
    key = _c(np.asarray(key).reshape(-1, 2), np.uint32)
    assert ctr.shape[0] == key.shape[0]
    out = np.empty_like(ctr)
    _load().orc_philox4x32_many(ctr.shape[0], _ptr(ctr), _ptr(key), rounds, _ptr(out))
    return out


def uniform(lo: int, hi: int, wide: bool) -> float:
    """The midpoint uniform (k + 1/2) / 2^m from an entry's word (fp32 noise: k = lo >> 8) or
    two words (wide noise: k = ((hi << 32) | lo) >> 12)."""
    return _load().orc_uniform(int(lo) & 0xFFFFFFFF, int(hi) & 0xFFFFFFFF, int(bool(wide)))


def entry_words(call_words, v, wide: bool):
    """The (lo, hi) words vocabulary entry v takes from its call's four words: fp32 noise uses
    word v & 3 of call v >> 2; wide noise words 2(v & 1), 2(v & 1) + 1 of call v >> 1."""
    w = np.asarray(call_words)
    v = np.asarray(v)
    if wide:
        j = 2 * (v & 1)
        return np.take_along_axis(w, j[..., None], -1)[..., 0], np.take_along_axis(w, (j + 1)[..., None], -1)[..., 0]
    return np.take_along_axis(w, (v & 3)[..., None], -1)[..., 0], np.zeros_like(w[..., 0])


def noise(B, V, seeds, positions, base_seed, offset, wide):
    """Noise grid [B, V]: the four words of the Philox call each entry draws from [B,V,4], u,
    E = -log u, g = -log E (fp64).

    Keyed by (request seed, absolute position, vocabulary index) for seeded rows, as in the
    Megatron-LM PR ("The change"); unseeded rows by (base_seed, offset, row).  A call serves
    four consecutive entries (fp32 noise) or two (wide noise)."""
    seeds = _c(seeds, np.int64)
    positions = _c(positions, np.int64)
    words = np.empty((B, V, 4), np.uint32)
    u = np.empty((B, V)); E = np.empty((B, V)); g = np.empty((B, V))
    _load().orc_noise_fill(B, V, _ptr(seeds), _ptr(positions), base_seed, offset, int(bool(wide)),
                           _ptr(words), _ptr(u), _ptr(E), _ptr(g))
    return words, u, E, g


class RowResult:
    """Per-row outcome of the race: index (-1 if none), status, top-two scores, tile maxima."""

    def __init__(self, out, status, top1, top2, tile_max, tile_idx, scores):
        self.out, self.status, self.top1, self.top2 = out, status, top1, top2
        self.tile_max, self.tile_idx, self.scores = tile_max, tile_idx, scores


def _row_outputs(B, V, tile_v, want_scores):
    nt = (V + tile_v - 1) // tile_v if tile_v else 0
    return (np.empty(B, np.int64), np.empty(B, np.int32), np.empty(B), np.empty(B),
            np.empty((B, nt)), np.empty((B, nt), np.int64),
            np.empty((B, V)) if want_scores else None)


def sample_from_logits(logits, *, B=None, temperature=None, seeds=None, positions=None, bias=None,
                       mask=None, base_seed=0, offset=0, wide=False, tile_v=0,
                       want_scores=False, threads=None) -> RowResult:
    """Gumbel-max race over materialised logits [B, V] (or one broadcast row [V] with B given).

    FlashSampling "method step details" steps 2-6 and Stage 2, with the transform order of the
    sampling-kernel guide (bias before temperature; T == 0 greedy)."""
    y = np.asarray(logits, dtype=np.float64)
    if y.ndim == 1:
        assert B is not None
        ld_y, V = 0, y.shape[0]
    else:
        B = y.shape[0] if B is None else B
        ld_y, V = y.shape[1], y.shape[1]
    y = np.ascontiguousarray(y)
    T = _c(temperature, np.float64)
    bias_a = _c(bias, np.float64)
    ld_bias = 0 if bias_a is None or bias_a.ndim == 1 else bias_a.shape[1]
    mask_a = _c(mask, np.uint32)
    ld_mask = 0 if mask_a is None or mask_a.ndim == 1 else mask_a.shape[1]
    seeds_a, pos_a = _c(seeds, np.int64), _c(positions, np.int64)
    outs = _row_outputs(B, V, tile_v, want_scores)
    _load().orc_sample_from_logits(
        _ptr(y), ld_y, B, V, _ptr(T), _ptr(seeds_a), _ptr(pos_a), _ptr(bias_a), ld_bias,
        _ptr(mask_a), ld_mask, base_seed, offset, int(bool(wide)), tile_v,
        *[_ptr(o) for o in outs], threads or default_threads())
    return RowResult(*outs)


def _bits16(t):
    """bf16 bit patterns as uint16 from a torch bf16 tensor or a uint16/int16 array."""
    if hasattr(t, "view") and hasattr(t, "dtype") and str(t.dtype) == "torch.bfloat16":
        import torch
        t = t.detach().cpu().contiguous().view(torch.int16).numpy()
    a = np.asarray(t)
    if a.dtype != np.uint16:
        a = a.view(np.uint16)
    return np.ascontiguousarray(a)


def lmhead_logits(H_bits, W_bits, threads=None) -> np.ndarray:
    """Y = H W^T in fp64 from bf16 bit patterns H [B, D], W [V, D] (FlashSampling step 1)."""
    H, W = _bits16(H_bits), _bits16(W_bits)
    B, D = H.shape
    V = W.shape[0]
    y = np.empty((B, V))
    _load().orc_lmhead_logits(_ptr(H), D, _ptr(W), D, B, D, V, _ptr(y), threads or default_threads())
    return y


def lmhead_sample(H_bits, W_bits, *, temperature=None, seeds=None, positions=None, bias=None,
                  mask=None, base_seed=0, offset=0, wide=False, tile_v=128, want_scores=False,
                  threads=None) -> RowResult:
    """The fused path's result: fp64 logits from bf16 H, W, then the per-row race."""
    H, W = _bits16(H_bits), _bits16(W_bits)
    B, D = H.shape
    V = W.shape[0]
    T = _c(temperature, np.float64)
    bias_a = _c(bias, np.float64)
    ld_bias = 0 if bias_a is None or bias_a.ndim == 1 else bias_a.shape[1]
    mask_a = _c(mask, np.uint32)
    ld_mask = 0 if mask_a is None or mask_a.ndim == 1 else mask_a.shape[1]
    seeds_a, pos_a = _c(seeds, np.int64), _c(positions, np.int64)
    outs = _row_outputs(B, V, tile_v, want_scores)
    rc = _load().orc_lmhead_sample(
        _ptr(H), D, _ptr(W), D, B, D, V, _ptr(T), _ptr(seeds_a), _ptr(pos_a), _ptr(bias_a),
        ld_bias, _ptr(mask_a), ld_mask, base_seed, offset, int(bool(wide)), tile_v,
        *[_ptr(o) for o in outs], threads or default_threads())
    if rc != 0:
        raise MemoryError("oracle could not allocate the fp64 logits")
    return RowResult(*outs)


def lmhead_sample_rows(H_bits, W_bits, rows, *, temperature=None, seeds=None, positions=None,
                       bias=None, mask=None, base_seed=0, offset=0, wide=False, tile_v=128,
                       want_scores=False, threads=None) -> RowResult:
    """The fused path's result for chosen batch rows of a B-row problem (each row keeps its own
    parameters and its batch index), for sampled checks at full size; with want_scores, also
    every perturbed score of those rows."""
    H, W = _bits16(H_bits), _bits16(W_bits)
    B, D = H.shape
    V = W.shape[0]
    rows = _c(rows, np.int64)
    n = rows.shape[0]
    T = _c(temperature, np.float64)
    bias_a = _c(bias, np.float64)
    ld_bias = 0 if bias_a is None or bias_a.ndim == 1 else bias_a.shape[1]
    mask_a = _c(mask, np.uint32)
    ld_mask = 0 if mask_a is None or mask_a.ndim == 1 else mask_a.shape[1]
    seeds_a, pos_a = _c(seeds, np.int64), _c(positions, np.int64)
    outs = _row_outputs(n, V, tile_v, want_scores)
    rc = _load().orc_lmhead_sample_rows(
        _ptr(H), D, _ptr(W), D, B, D, V, _ptr(rows), n, _ptr(T), _ptr(seeds_a), _ptr(pos_a),
        _ptr(bias_a), ld_bias, _ptr(mask_a), ld_mask, base_seed, offset, int(bool(wide)), tile_v,
        *[_ptr(o) for o in outs], threads or default_threads())
    if rc != 0:
        raise MemoryError("oracle could not allocate the fp64 logits")
    return RowResult(*outs)


def lmhead_scores_at(H_bits, W_bits, rows, cols, *, temperature=None, seeds=None, positions=None,
                     bias=None, mask=None, base_seed=0, offset=0, wide=False) -> np.ndarray:
    """Perturbed scores s[b, v] of the fused path at chosen (b, v) pairs, one by one."""
    H, W = _bits16(H_bits), _bits16(W_bits)
    B, D = H.shape
    V = W.shape[0]
    rows = _c(rows, np.int64); cols = _c(cols, np.int64)
    T = _c(temperature, np.float64)
    bias_a = _c(bias, np.float64)
    ld_bias = 0 if bias_a is None or bias_a.ndim == 1 else bias_a.shape[1]
    mask_a = _c(mask, np.uint32)
    ld_mask = 0 if mask_a is None or mask_a.ndim == 1 else mask_a.shape[1]
    seeds_a, pos_a = _c(seeds, np.int64), _c(positions, np.int64)
    s = np.empty(rows.shape[0])
    _load().orc_lmhead_scores_at(
        _ptr(H), D, _ptr(W), D, B, D, V, _ptr(T), _ptr(seeds_a), _ptr(pos_a), _ptr(bias_a),
        ld_bias, _ptr(mask_a), ld_mask, base_seed, offset, int(bool(wide)), rows.shape[0],
        _ptr(rows), _ptr(cols), _ptr(s))
    return s


def sample_filtered(logits, *, B=None, temperature=None, seeds=None, positions=None, bias=None,
                    mask=None, base_seed=0, offset=0, wide=False, top_k=None, top_p=None,
                    min_p=None, k_max=1024, p_shift=0.0, minp_scale=1.0, threads=None,
                    want_top2=False):
    """Filtered race over materialised logits: top-k -> top-p -> min-p on t = (y + bias) / T,
    then the Gumbel race over the kept tokens (spec-decode-ops "Semantics"; sampling-kernel
    guide steps 6-8).  Returns (out, status, kept-set size[, top1, top2]): top1 / top2 are the
    two best perturbed scores of the kept set.  p_shift / minp_scale move the top-p / min-p
    thresholds, to find out which decisions sit on a floating-point boundary."""
    y = np.asarray(logits, dtype=np.float64)
    if y.ndim == 1:
        ld_y, V = 0, y.shape[0]
    else:
        B = y.shape[0] if B is None else B
        ld_y, V = y.shape[1], y.shape[1]
    y = np.ascontiguousarray(y)
    T = _c(temperature, np.float64)
    bias_a = _c(bias, np.float64)
    ld_bias = 0 if bias_a is None or bias_a.ndim == 1 else bias_a.shape[1]
    mask_a = _c(mask, np.uint32)
    ld_mask = 0 if mask_a is None or mask_a.ndim == 1 else mask_a.shape[1]
    seeds_a, pos_a = _c(seeds, np.int64), _c(positions, np.int64)
    tk, tp, mp = _c(top_k, np.int32), _c(top_p, np.float64), _c(min_p, np.float64)
    out = np.empty(B, np.int64); status = np.empty(B, np.int32); kept = np.empty(B, np.int32)
    top1 = np.empty(B); top2 = np.empty(B)
    _load().orc_sample_filtered(_ptr(y), ld_y, B, V, _ptr(T), _ptr(seeds_a), _ptr(pos_a),
                                _ptr(bias_a), ld_bias, _ptr(mask_a), ld_mask, base_seed, offset,
                                int(bool(wide)), _ptr(tk), _ptr(tp), _ptr(mp), int(k_max),
                                float(p_shift), float(minp_scale), _ptr(out), _ptr(status),
                                _ptr(kept), _ptr(top1), _ptr(top2), threads or default_threads())
    if want_top2:
        return out, status, kept, top1, top2
    return out, status, kept


# ---- Gumbel-top-k: k draws without replacement ----

def topk_from_scores(scores, k: int):
    """Gumbel-top-k (FlashSampling "Limitations" and "Future directions": sampling without
    replacement through Gumbel-top-k): per row, the k largest perturbed scores, in order (larger
    score first, then the smaller index); -inf is never taken.  Returns (indices [B, k] int64,
    with -1 where fewer than k scores are finite; scores [B, k], -inf there)."""
    s = np.asarray(scores, dtype=np.float64)
    B = s.shape[0]
    idx = np.full((B, k), -1, np.int64)
    val = np.full((B, k), -np.inf)
    for b in range(B):
        fin = np.nonzero(s[b] > -np.inf)[0]
        order = fin[np.lexsort((fin, -s[b][fin]))]     # score descending, then index ascending
        m = min(k, order.shape[0])
        idx[b, :m] = order[:m]
        val[b, :m] = s[b][order[:m]]
    return idx, val


def tile_topk_from_scores(scores, k: int, tile_v: int):
    """The same selection within each vocabulary tile of tile_v entries: ([B, nt, k], [B, nt, k])."""
    s = np.asarray(scores, dtype=np.float64)
    B, V = s.shape
    nt = (V + tile_v - 1) // tile_v
    idx = np.full((B, nt, k), -1, np.int64)
    val = np.full((B, nt, k), -np.inf)
    for t in range(nt):
        i, x = topk_from_scores(s[:, t * tile_v:(t + 1) * tile_v], k)
        idx[:, t] = np.where(i >= 0, i + t * tile_v, -1)
        val[:, t] = x
    return idx, val


def gumbel_topk(logits, k: int, **race_kw):
    """Gumbel-top-k over materialised logits: the race's perturbed scores (``sample_from_logits``,
    same transform and noise), then ``topk_from_scores``.  Returns (indices [B, k], scores [B, k],
    status [B]) with the race's statuses (1: no finite score, 2: invalid temperature)."""
    r = sample_from_logits(logits, want_scores=True, **race_kw)
    idx, val = topk_from_scores(r.scores, k)
    return idx, val, r.status


def lmhead_gumbel_topk(H_bits, W_bits, k: int, rows=None, **race_kw):
    """Gumbel-top-k of the fused path (fp64 logits H W^T, then ``gumbel_topk``'s selection), for
    all rows or for chosen batch rows of a larger batch (each keeps its parameters and index)."""
    H = _bits16(H_bits)
    if rows is None:
        rows = np.arange(H.shape[0])
    race_kw.setdefault("tile_v", 128)
    r = lmhead_sample_rows(H_bits, W_bits, rows, want_scores=True, **race_kw)
    idx, val = topk_from_scores(r.scores, k)
    return idx, val, r.status, r.scores


# ---- Speculative-decoding verification ----

def noise_row(seeded, seed, pos, base_seed, offset, row, V, wide):
    """Gumbel noise [V] of one row with an explicit row index and absolute position."""
    g = np.empty(V)
    _load().orc_noise_row(int(bool(seeded)), int(seed), int(pos), int(base_seed), int(offset),
                          int(row), int(V), int(bool(wide)), _ptr(g))
    return g


def accept_uniform(seeded, seed, pos, base_seed, offset, row, wide) -> float:
    """The acceptance uniform of one verification step (Philox call index 0xffffffff)."""
    return _load().orc_accept_uniform(int(bool(seeded)), int(seed), int(pos), int(base_seed),
                                      int(offset), int(row), int(bool(wide)))


def _softmax(z):
    m = np.max(z)
    if not np.isfinite(m):
        return np.zeros_like(z)
    e = np.exp(z - m)
    return e / e.sum()


def verify_from_logits(target, draft, draft_tokens, *, temperature=None, seeds=None,
                       positions=None, base_seed=0, offset=0, wide=False, want_detail=False):
    """Speculative-decoding verification (spec-decode-ops "verify": the canonical rejection
    sampling of Leviathan et al. and Chen et al.).  target [B, k+1, V] and draft [B, k, V]
    logits, draft_tokens [B, k]; p = softmax(logits / T) per position, T per row.

    Draft token x_i is accepted when u_i * p_d(x_i) < p_t(x_i) (probability min(1, p_t / p_d)),
    in order; the first rejection j is replaced by a draw from the residual max(p_t - p_d, 0) at
    position j (Gumbel race over log r + g; p_t itself if no entry of r is positive); with every
    draft accepted a bonus token is drawn from p_t at position k (the plain race).  T == 0 rows:
    accept while x_i is the target's argmax (smallest index on ties), then emit the argmax.  A
    draft token outside [0, V) is rejected.  NaN logits count as -inf (never drawn), as in the
    race; a row with nothing finite at the drawn position emits no token at all.

    Noise: row b's draw at step position i uses the race's Philox noise at absolute position
    positions[b] + i (seeded rows) or row index b (k + 1) + i with (base_seed, offset)
    (unseeded rows); u_i is ``accept_uniform`` with the same keying.

    Returns (accept_len [B] int64, out [B, k+1] int64 with -1 after the emitted tokens,
    status [B] int32: 0 ok, 1 no finite target entry at the drawn position, 2 invalid T).
    With want_detail, also the margins u_i p_d(x_i) - p_t(x_i) [B, k] (nan where not reached),
    the top-two scores of the final draw [B, 2] and its scores [B, V] (-inf on rows that made
    no draw)."""
    t = np.asarray(target, np.float64)
    d = np.asarray(draft, np.float64)
    t = np.where(np.isnan(t), -np.inf, t)
    d = np.where(np.isnan(d), -np.inf, d)
    x = np.asarray(draft_tokens, np.int64)
    B, K1, V = t.shape
    k = K1 - 1
    T = np.ones(B) if temperature is None else np.asarray(temperature, np.float64)
    acc = np.zeros(B, np.int64)
    out = np.full((B, K1), -1, np.int64)
    status = np.zeros(B, np.int32)
    margin = np.full((B, k), np.nan)
    top2 = np.full((B, 2), -np.inf)
    scores = np.full((B, V), -np.inf) if want_detail else None
    for b in range(B):
        Tb = T[b]
        if not (Tb >= 0.0):
            status[b] = 2
            continue
        seeded = seeds is not None and seeds[b] >= 0
        seed = int(seeds[b]) if seeded else 0
        pos0 = int(positions[b]) if seeded else 0

        def keying(i):
            return dict(seeded=seeded, seed=seed, pos=pos0 + i if seeded else 0, base_seed=base_seed,
                        offset=offset, row=b * K1 + i, wide=wide)

        j = k
        if Tb == 0.0:
            for i in range(k):
                a = int(np.argmax(t[b, i]))
                if x[b, i] == a and np.isfinite(t[b, i, a]):
                    out[b, i] = x[b, i]
                else:
                    j = i
                    break
            s = t[b, j].copy()
        else:
            for i in range(k):
                pt = _softmax(t[b, i] / Tb)
                pd = _softmax(d[b, i] / Tb)
                u = accept_uniform(**keying(i))
                xi = x[b, i]
                if not 0 <= xi < V:                     # not a vocabulary entry: rejected
                    j = i
                    break
                margin[b, i] = u * pd[xi] - pt[xi]
                if u * pd[xi] < pt[xi]:
                    out[b, i] = xi
                else:
                    j = i
                    break
            g = noise_row(V=V, **keying(j))
            if j < k:
                r = np.maximum(_softmax(t[b, j] / Tb) - _softmax(d[b, j] / Tb), 0.0)
                if (r > 0).any():
                    with np.errstate(divide="ignore"):
                        s = np.where(r > 0, np.log(r), -np.inf) + g
                else:
                    s = t[b, j] / Tb + g
            else:
                s = t[b, k] / Tb + g
        s = np.where(np.isnan(s), -np.inf, s)
        if not np.isfinite(s).any() and not (s == np.inf).any():
            status[b] = 1
            out[b] = -1
            continue
        a = int(np.argmax(s))                      # the first maximum: smallest index on ties
        srt = np.sort(s)[::-1]
        top2[b] = srt[:2] if V > 1 else (srt[0], -np.inf)
        if want_detail:
            scores[b] = s
        out[b, j] = a
        acc[b] = j
    if want_detail:
        return acc, out, status, margin, top2, scores
    return acc, out, status


# ---- FP8 (E4M3) inputs: W8A8 with per-row scales ----

def e4m3_decode(codes) -> np.ndarray:
    """E4M3 ("fn") codes -> fp64 values."""
    lib = _load()
    c = np.asarray(codes, dtype=np.uint8)
    return np.array([lib.orc_e4m3_decode(int(x)) for x in c.ravel()]).reshape(c.shape)


def e4m3_encode(x) -> np.ndarray:
    """Nearest finite E4M3 code (ties to even, saturating at +-448) of fp64 values."""
    lib = _load()
    a = np.asarray(x, dtype=np.float64)
    return np.array([lib.orc_e4m3_encode(float(v)) for v in a.ravel()], np.uint8).reshape(a.shape)


def quantize_rows_e4m3(H_bits):
    """Per-row power-of-two quantisation of bf16 H [B, D]: (E4M3 codes uint8 [B, D], e int32 [B])
    with e the smallest integer such that max |h| * 2^-e <= 448."""
    H = _bits16(H_bits)
    B, D = H.shape
    q = np.empty((B, D), np.uint8)
    e = np.empty(B, np.int32)
    _load().orc_quantize_rows_e4m3(_ptr(H), D, B, D, _ptr(q), D, _ptr(e))
    return q, e


def lmhead_logits_fp8(H8, e_h, W8, w_scale, rows=None, threads=None) -> np.ndarray:
    """y = 2^e_h[b] * w_scale[v] * sum_d E4M3(H8) E4M3(W8) in fp64 (rows: subset of H's rows)."""
    H8 = _c(H8, np.uint8); W8 = _c(W8, np.uint8)
    e_h = _c(e_h, np.int32); ws = _c(w_scale, np.float64)
    B, D = H8.shape
    V = W8.shape[0]
    r = _c(rows, np.int64)
    nb = B if r is None else r.shape[0]
    y = np.empty((nb, V))
    _load().orc_lmhead_logits_fp8(_ptr(H8), D, _ptr(e_h), _ptr(W8), D, _ptr(ws), B, D, V, _ptr(r),
                                  0 if r is None else nb, _ptr(y), threads or default_threads())
    return y


def lmhead_sample_fp8(H_bits, W8, w_scale, *, rows=None, temperature=None, seeds=None,
                      positions=None, bias=None, mask=None, base_seed=0, offset=0, wide=False,
                      tile_v=128, threads=None) -> RowResult:
    """The fused FP8 path's result: quantise H per row (power-of-two scale), fp64 logits from the
    E4M3 operands and scales, then the per-row race; rows = a subset of the batch (or all)."""
    H = _bits16(H_bits)
    B, D = H.shape
    W8 = _c(W8, np.uint8)
    V = W8.shape[0]
    ws = _c(w_scale, np.float64)
    r = _c(rows, np.int64)
    nb = B if r is None else r.shape[0]
    T = _c(temperature, np.float64)
    bias_a = _c(bias, np.float64)
    ld_bias = 0 if bias_a is None or bias_a.ndim == 1 else bias_a.shape[1]
    mask_a = _c(mask, np.uint32)
    ld_mask = 0 if mask_a is None or mask_a.ndim == 1 else mask_a.shape[1]
    seeds_a, pos_a = _c(seeds, np.int64), _c(positions, np.int64)
    outs = _row_outputs(nb, V, tile_v, False)
    rc = _load().orc_lmhead_sample_fp8(
        _ptr(H), D, _ptr(W8), D, _ptr(ws), B, D, V, _ptr(r), 0 if r is None else nb, _ptr(T),
        _ptr(seeds_a), _ptr(pos_a), _ptr(bias_a), ld_bias, _ptr(mask_a), ld_mask, base_seed,
        offset, int(bool(wide)), tile_v, *[_ptr(o) for o in outs[:6]], threads or default_threads())
    if rc != 0:
        raise MemoryError("oracle could not allocate")
    return RowResult(*outs)


# ---- MXFP4 weights (W4A16): E2M1 elements with one UE8M0 scale per block of 32 ----

def e2m1_decode(codes) -> np.ndarray:
    """E2M1 codes (4-bit, 0..15) -> fp64 values (OCP Microscaling element format)."""
    lib = _load()
    c = np.asarray(codes, dtype=np.uint8)
    return np.array([lib.orc_e2m1_decode(int(x)) for x in c.ravel()]).reshape(c.shape)


def e2m1_encode(x) -> np.ndarray:
    """Nearest E2M1 code of fp64 values (ties to the even mantissa, saturating at +-6)."""
    lib = _load()
    a = np.asarray(x, dtype=np.float64)
    return np.array([lib.orc_e2m1_encode(float(v)) for v in a.ravel()], np.uint8).reshape(a.shape)


def ue8m0_decode(codes) -> np.ndarray:
    """UE8M0 scale codes -> 2^(s - 127) (NaN for 255)."""
    lib = _load()
    c = np.asarray(codes, dtype=np.uint8)
    return np.array([lib.orc_ue8m0_decode(int(x)) for x in c.ravel()]).reshape(c.shape)


def mxfp4_weight(W4, S, v, d) -> float:
    """The decoded weight W[v][d] of an MXFP4 matrix: packed codes W4 [V, D/2] (element d in the
    low nibble of byte d/2 when d is even, the high nibble when odd), scales S [D/32, V]."""
    W4 = _c(W4, np.uint8); S = _c(S, np.uint8)
    return _load().orc_mxfp4_weight(_ptr(W4), W4.shape[1], _ptr(S), S.shape[1], int(v), int(d))


def lmhead_logits_mxfp4(H_bits, W4, S, rows=None, threads=None) -> np.ndarray:
    """y = H W^T in fp64 from bf16 H [B, D] and MXFP4 W (W4 [V, D/2], S [D/32, V])."""
    H = _bits16(H_bits)
    W4 = _c(W4, np.uint8); S = _c(S, np.uint8)
    B, D = H.shape
    V = W4.shape[0]
    r = _c(rows, np.int64)
    nb = B if r is None else r.shape[0]
    y = np.empty((nb, V))
    _load().orc_lmhead_logits_mxfp4(_ptr(H), D, _ptr(W4), W4.shape[1], _ptr(S), S.shape[1], B, D, V,
                                    _ptr(r), 0 if r is None else nb, _ptr(y),
                                    threads or default_threads())
    return y


def lmhead_sample_mxfp4(H_bits, W4, S, *, rows=None, temperature=None, seeds=None, positions=None,
                        bias=None, mask=None, base_seed=0, offset=0, wide=False, tile_v=128,
                        threads=None) -> RowResult:
    """The fused MXFP4 path's result: fp64 logits from bf16 H and the decoded MXFP4 weights, then
    the per-row race (FlashSampling Stage 1 and 2); rows = a subset of the batch (or all)."""
    H = _bits16(H_bits)
    B, D = H.shape
    W4 = _c(W4, np.uint8); S = _c(S, np.uint8)
    V = W4.shape[0]
    r = _c(rows, np.int64)
    nb = B if r is None else r.shape[0]
    T = _c(temperature, np.float64)
    bias_a = _c(bias, np.float64)
    ld_bias = 0 if bias_a is None or bias_a.ndim == 1 else bias_a.shape[1]
    mask_a = _c(mask, np.uint32)
    ld_mask = 0 if mask_a is None or mask_a.ndim == 1 else mask_a.shape[1]
    seeds_a, pos_a = _c(seeds, np.int64), _c(positions, np.int64)
    outs = _row_outputs(nb, V, tile_v, False)
    rc = _load().orc_lmhead_sample_mxfp4(
        _ptr(H), D, _ptr(W4), W4.shape[1], _ptr(S), S.shape[1], B, D, V, _ptr(r),
        0 if r is None else nb, _ptr(T), _ptr(seeds_a), _ptr(pos_a), _ptr(bias_a), ld_bias,
        _ptr(mask_a), ld_mask, base_seed, offset, int(bool(wide)), tile_v,
        *[_ptr(o) for o in outs[:6]], threads or default_threads())
    if rc != 0:
        raise MemoryError("oracle could not allocate")
    return RowResult(*outs)
