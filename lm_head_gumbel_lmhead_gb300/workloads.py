"""Seeded synthetic inputs for the fused LM-head + Gumbel-max sampler.

This module only draws inputs: it holds none of the sampling method's arithmetic, so both the
CUDA path and the CPU oracle can be fed from it.  Shapes and distributions follow the
workloads the FlashSampling page measures ("reproduction" section: D = 4096, V = 151936,
BF16 inputs, B from 1 to 256; D = 8192 with a larger vocabulary) and the Megatron-LM PR's tail
rows ("Problem": float32 rows [0, -D, ..., -D] with V = 131072).  Nothing here is a dataset:
the pages' vLLM / AIME / GSM8K runs are replaced by these seeded tensors.

All tensors are made on the host by ``torch.Generator().manual_seed(seed)``; callers copy
them to the device.  Masks are packed allow-bits (bit v % 32 of word v // 32 set = allowed)
stored in int32 tensors (torch has no general uint32 arithmetic); padding bits are zero.
"""
from __future__ import annotations

import math
from dataclasses import dataclass
from typing import Optional

import torch

NOISE_FP32 = 0
NOISE_WIDE53 = 1


@dataclass
class Workload:
    name: str
    B: int
    D: int
    V: int
    H: torch.Tensor                 # bf16 [B, D]
    W: torch.Tensor                 # bf16 [V, D]
    temperature: torch.Tensor       # fp32 [B]
    seeds: torch.Tensor             # int64 [B]; -1 = unseeded row
    positions: torch.Tensor         # int64 [B]
    bias: Optional[torch.Tensor]    # fp32 [B, V] or None
    mask: Optional[torch.Tensor]    # int32 [B, ceil(V/32)] allow-bit words or None
    noise_mode: int
    base_seed: int = 0
    offset: int = 0


def _gen(seed: int) -> torch.Generator:
    return torch.Generator().manual_seed(int(seed))


def normal_bf16(rows: int, cols: int, std: float, seed: int, chunk_rows: int = 8192) -> torch.Tensor:
    """N(0, std^2) entries rounded to bf16, drawn in row chunks to bound host memory."""
    g = _gen(seed)
    out = torch.empty(rows, cols, dtype=torch.bfloat16)
    for r0 in range(0, rows, chunk_rows):
        r1 = min(rows, r0 + chunk_rows)
        out[r0:r1] = (torch.randn(r1 - r0, cols, generator=g) * std).to(torch.bfloat16)
    return out


def rms_normalised_bf16(rows: int, cols: int, seed: int) -> torch.Tensor:
    """Hidden states: N(0,1) rows divided by their RMS, rounded to bf16 (round-to-nearest-even)."""
    x = torch.randn(rows, cols, generator=_gen(seed), dtype=torch.float64)
    x = x / torch.sqrt((x * x).mean(dim=1, keepdim=True))
    return x.to(torch.float32).to(torch.bfloat16)


def pack_allow_bits(allowed: torch.Tensor) -> torch.Tensor:
    """bool [B, V] -> int32 words [B, ceil(V/32)], bit v % 32 of word v // 32 = allowed."""
    B, V = allowed.shape
    nw = (V + 31) // 32
    padded = torch.zeros(B, nw * 32, dtype=torch.int64)
    padded[:, :V] = allowed.to(torch.int64)
    weights = (torch.ones(32, dtype=torch.int64) << torch.arange(32, dtype=torch.int64))
    words = (padded.view(B, nw, 32) * weights).sum(dim=2)          # values in [0, 2^32)
    words = torch.where(words >= 2**31, words - 2**32, words)        # same bits as int32
    return words.to(torch.int32)


def tiny(seed: int = 0) -> Workload:
    """B=4, D=512, V=8192: H ~ N(0,1), W ~ N(0, 1/sqrt(D)), zero bias, T = 1, seed 1234,
    positions 0..3, fp32 noise (small enough for the oracle to finish in seconds)."""
    B, D, V = 4, 512, 8192
    H = torch.randn(B, D, generator=_gen(seed + 1)).to(torch.bfloat16)
    W = normal_bf16(V, D, 1.0 / math.sqrt(D), seed + 2)
    return Workload("tiny fused decode B=4 D=512 V=8192", B, D, V, H, W,
                    torch.ones(B), torch.full((B,), 1234, dtype=torch.int64),
                    torch.arange(B, dtype=torch.int64), None, None, NOISE_FP32)


def qwen3_8b(B: int, step: int = 0, seed: int = 0, V: int = 151936, D: int = 4096) -> Workload:
    """Qwen3-8B-shaped decode: D=4096, V=151936, W ~ N(0, 0.02) bf16, H RMS-normalised N(0,1)
    bf16, uniform T = 0.7, per-row seeds 1000 + b, positions = step."""
    H = rms_normalised_bf16(B, D, seed + 11)
    W = normal_bf16(V, D, 0.02, seed + 12)
    return Workload(f"qwen3-8b-shaped fused decode B={B} D={D} V={V}", B, D, V, H, W,
                    torch.full((B,), 0.7), 1000 + torch.arange(B, dtype=torch.int64),
                    torch.full((B,), step, dtype=torch.int64), None, None, NOISE_FP32)


def llama3_hetero(B: int = 64, seed: int = 0, V: int = 128256, D: int = 4096) -> Workload:
    """Llama-3-shaped heterogeneous batch: D=4096, V=128256, B=64; T ~ U[0.3, 1.2] with rows
    0, 8, ..., 56 greedy (T = 0); bias ~ N(0, 0.5) fp32 [B, V]; a random 90% -inf mask
    (10% of tokens allowed) on rows b < B/2; rows with b % 4 == 3 unseeded, the others seeded
    with 1000 + b at position 7 + b."""
    g = _gen(seed + 21)
    H = rms_normalised_bf16(B, D, seed + 22)
    W = normal_bf16(V, D, 0.02, seed + 23)
    T = 0.3 + 0.9 * torch.rand(B, generator=g)
    T[0::8] = 0.0
    bias = torch.randn(B, V, generator=g) * 0.5
    allowed = torch.ones(B, V, dtype=torch.bool)
    allowed[: B // 2] = torch.rand(B // 2, V, generator=g) < 0.1
    seeds = 1000 + torch.arange(B, dtype=torch.int64)
    seeds[3::4] = -1
    positions = 7 + torch.arange(B, dtype=torch.int64)
    return Workload(f"llama-3-shaped heterogeneous fused decode B={B} D={D} V={V}", B, D, V, H, W,
                    T, seeds, positions, bias, pack_allow_bits(allowed), NOISE_FP32,
                    base_seed=4321, offset=17)


def large_vocab(B: int, seed: int = 0, V: int = 262144, D: int = 8192) -> Workload:
    """Large-vocabulary sweep: D=8192, V=262144, W ~ N(0, 0.015) bf16, T = 1, wide noise."""
    H = rms_normalised_bf16(B, D, seed + 31)
    W = normal_bf16(V, D, 0.015, seed + 32)
    return Workload(f"large-vocab fused decode B={B} D={D} V={V}", B, D, V, H, W,
                    torch.ones(B), 1000 + torch.arange(B, dtype=torch.int64),
                    torch.zeros(B, dtype=torch.int64), None, None, NOISE_WIDE53)


def tail_row(V: int, r: float) -> torch.Tensor:
    """The Megatron-LM PR's tail row in fp32: [0, -D, ..., -D] with D = -ln r."""
    row = torch.full((V,), -math.log(r), dtype=torch.float32).neg_()
    row[0] = 0.0
    return row


def logits_normal(B: int, V: int, std: float = 2.0, seed: int = 0,
                  dtype: torch.dtype = torch.float32) -> torch.Tensor:
    """Materialised logits ~ N(0, std^2) in fp32 or bf16."""
    return (torch.randn(B, V, generator=_gen(seed + 41)) * std).to(dtype)


def spec_logits(B: int, k: int, V: int, seed: int = 0, dtype: torch.dtype = torch.bfloat16,
                std: float = 2.0, draft_corr: float = 0.8):
    """Target logits [B, k+1, V] ~ N(0, std^2) and draft logits [B, k, V] correlated with the
    target's first k positions (draft = c * target + sqrt(1 - c^2) * independent N(0, std^2)),
    a draft that agrees with the target often but not always."""
    g = _gen(seed + 57)
    tgt = torch.randn(B, k + 1, V, generator=g) * std
    noise = torch.randn(B, k, V, generator=g) * std
    dft = draft_corr * tgt[:, :k] + (1.0 - draft_corr ** 2) ** 0.5 * noise
    return tgt.to(dtype), dft.to(dtype)


def quantize_weight_e4m3(W: torch.Tensor, chunk_rows: int = 8192):
    """Offline per-row FP8 (E4M3) weight quantisation, as a model would ship its LM head:
    w_scale[v] = max_d |W[v][d]| / 448 (fp32, 1 for an all-zero row), W8 = E4M3(W / w_scale)
    (torch's float8_e4m3fn cast), returned as (uint8 codes [V, D], fp32 scales [V])."""
    V, D = W.shape
    W8 = torch.empty(V, D, dtype=torch.uint8)
    scale = torch.empty(V, dtype=torch.float32)
    for r0 in range(0, V, chunk_rows):
        r1 = min(V, r0 + chunk_rows)
        w = W[r0:r1].float()
        s = w.abs().amax(dim=1) / 448.0
        s = torch.where(s > 0, s, torch.ones_like(s))
        scale[r0:r1] = s
        W8[r0:r1] = (w / s[:, None]).to(torch.float8_e4m3fn).view(torch.uint8)
    return W8, scale


def quantize_weight_mxfp4(W: torch.Tensor, chunk_rows: int = 8192):
    """Offline MXFP4 weight quantisation (Open Compute Project Microscaling: E2M1 elements, one
    UE8M0 scale per block of 32 along D), as a model would ship its LM head.  Per block the scale
    is 2^e with e the smallest integer such that max |w| <= 6 * 2^e (e = -127 for an all-zero
    block), and each element is w / 2^e rounded to the nearest E2M1 magnitude (0, 0.5, 1, 1.5, 2,
    3, 4, 6; ties to the even mantissa) with its sign.  Returns (W4 uint8 [V, D/2]: element d in
    the low nibble of byte d/2 when d is even, the high nibble when odd; S uint8 [D/32, V]: the
    scale code e + 127 of block d/32 of row v)."""
    V, D = W.shape
    assert D % 32 == 0, "MXFP4 blocks are 32 elements along D"
    W4 = torch.empty(V, D // 2, dtype=torch.uint8)
    S = torch.empty(D // 32, V, dtype=torch.uint8)
    mags = torch.tensor([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])
    mids = (mags[1:] + mags[:-1]) / 2
    for r0 in range(0, V, chunk_rows):
        r1 = min(V, r0 + chunk_rows)
        w = W[r0:r1].double().reshape(r1 - r0, D // 32, 32)
        amax = w.abs().amax(dim=2)
        m, ex = torch.frexp(amax / 6.0)                 # amax / 6 = m 2^ex, m in [0.5, 1)
        e = torch.where(m == 0.5, ex - 1, ex)           # ceil(log2(amax / 6))
        e = torch.where(amax > 0, e, torch.full_like(e, -127)).clamp(-127, 127)
        x = (w / torch.pow(2.0, e.double())[:, :, None]).float()
        a = x.abs().clamp(max=6.0)
        code = torch.searchsorted(mids, a, right=False)  # the lower magnitude at a midpoint
        tie = (code < 7) & (a == mids[code.clamp(max=6)]) & (code % 2 == 1)
        code = code + tie.to(code.dtype)                 # ties go to the even mantissa
        code = code | ((x < 0) | ((x == 0) & torch.signbit(x))).to(code.dtype) * 8
        code = code.reshape(r1 - r0, D).to(torch.uint8)
        W4[r0:r1] = code[:, 0::2] | (code[:, 1::2] << 4)
        S[:, r0:r1] = (e + 127).to(torch.uint8).T
    return W4, S
