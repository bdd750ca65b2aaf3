// Fused LM-head + Gumbel-max Stage 1 with MXFP4 weights (W4A16) on the tcgen05 tensor cores.
//
// FlashSampling ("Limitations", "Future directions"): low-precision inputs cut the bytes of the
// memory-bound regime.  The weights here are MXFP4 (Open Compute Project Microscaling): E2M1
// elements, two per byte, with one UE8M0 scale per block of 32 elements along K, streamed at
// 0.53 bytes per weight.  The activations stay bf16.  Stage 1 is the same method as the bf16
// kernel (logits on chip, transform, Philox noise, per-tile argmax); only the weight operand
// differs: it is rebuilt in shared memory as the exact bf16 values E2M1 x 2^(s - 127), in the
// 128-byte-swizzled K-major layout tcgen05.mma kind::f16 reads, so the tensor cores run the same
// bf16 x bf16 -> fp32 contraction.
//
// Warp roles (one persistent CTA per SM):
//   warp 0           bulk-copy producer of the packed weights: the library's tiled MXFP4 format
//                    (lms_mxfp4_pack) stores each (128-row vocabulary tile, 64-element K chunk)
//                    as one contiguous 4352-byte block, 4 KB of codes then 256 bytes of scales, so
//                    one cp.async.bulk of contiguous bytes fills a ring-A stage.
//   warp 1           allocates TMEM; one lane issues tcgen05.mma (M = 128 vocabulary rows,
//                    N = n_pad batch rows, K = 16 per instruction) into two TMEM accumulators.
//   warp 2           TMA producer of H [n_pad x 64] bf16 chunks into ring H.
//   warps 3..10      converters: converter w owns the K chunks j = w, w + 8, ... of the CTA's
//                    sequence and turns each whole chunk (ring-A stage: 128 rows x 64 codes and
//                    their scales) into the bf16 weight tile of ring C (byte permutes and one
//                    bf16x2 multiply per pair of weights), then a proxy fence so that the tensor
//                    cores see it.  Eight chunks are converted at once, each by one warp.
//   warps 11..18     epilogue: as in the bf16 kernel (transform, noise, argmax per tile).
// Ring A (packed codes and scales, 4.25 KB a stage) is deep so that enough weight bytes are in
// flight to keep HBM busy; ring C holds converted tiles (16 KB) and ring H the activations
// (n_pad * 128 bytes).  Every wait is bounded in time; a CTA whose wait runs out flags the
// error, drains its copies and MMAs, poisons its remaining candidates (row status 3), frees
// TMEM and exits.
#include <cuda.h>
#include <cuda_bf16.h>

#include "lms.h"
#include "lms_device.cuh"
#include "lms_kernels.h"
#include "tcgen05_common.cuh"

namespace lms {
namespace {

using namespace tc;

constexpr int kMxConvWarps = 8;
constexpr int kMxEpiWarps = 8;
constexpr int kMxFirstConv = 3;
constexpr int kMxFirstEpi = kMxFirstConv + kMxConvWarps;
constexpr int kMxThreads = 32 * (kMxFirstEpi + kMxEpiWarps);
// Ring A and ring C have a multiple of kMxConvWarps stages: then chunks j and j + S, which share a
// slot, are converted by the same warp, in order, so no warp can wait on a slot's next phase while
// its current one is incomplete.
constexpr int kMaxStagesA = 16;
constexpr int kStagesC = kMxConvWarps;
constexpr int kMaxStagesH = 8;
constexpr uint32_t kW4StageBytes = kTileV * kBK / 2;   // 128 rows x 64 codes = 4 KB
constexpr uint32_t kS4StageBytes = 2 * kTileV;         // 2 scale blocks x 128 rows
constexpr uint32_t kAStageBytes = kW4StageBytes + kS4StageBytes;   // one tiled block
constexpr int kUnitsPerLane = 2 * kTileV / 32;        // (row, scale block) units of a chunk per lane

struct MxParams {
    SampleArgs a;
    int nk;              // K chunks of 64, ceil(D / 64)
    int n_pad;
    int stages_a, stages_c, stages_h;
    uint32_t h_stage_bytes;   // n_pad * 128
    uint32_t tmem_cols;
    uint64_t timeout_ns;
    uint32_t debug_flags;
};

// Shared memory (offsets from a 1024-byte aligned base): ring C (converted 16 KB tiles) and ring H
// (activation chunks), both 1024-aligned for the 128-byte swizzle; ring A's packed codes and
// scales; barriers; then the epilogue's buffers.
struct MxLayout {
    uint32_t c_off, h_off, a_off, bars_off, misc_off, rows_off, red_off, tr_off, total;
    __host__ __device__ MxLayout(int sa, int sc, int sh, uint32_t h_stage_bytes, int n_pad) {
        c_off = 0;
        h_off = c_off + sc * kWStageBytes;
        a_off = h_off + sh * h_stage_bytes;
        bars_off = a_off + sa * kAStageBytes;
        // fullA, emptyA [SA]; fullC, emptyC [SC]; fullH, emptyH [SH]; acc_full[2], acc_empty[2],
        // drain
        misc_off = bars_off + (2 * sa + 2 * sc + 2 * sh + 5) * 8;
        rows_off = (misc_off + 16 + 15) & ~15u;   // misc: tmem slot, error flag
        red_off = rows_off + n_pad * static_cast<uint32_t>(sizeof(RowParams));
        tr_off = red_off + n_pad * 8;
        total = tr_off + kMxEpiWarps * kTrWarpBytes;
    }
};

// E2M1 magnitudes 0, 0.5, 1, 1.5, 2, 3, 4, 6 as bf16 bit patterns, split into high and low bytes:
// byte m of the 8-byte tables {a, b} is the high (low) byte of magnitude m.
constexpr uint32_t kHiA = 0x3F3F3F00u, kHiB = 0x40404040u;
constexpr uint32_t kLoA = 0xC0800000u, kLoB = 0xC0804000u;

// Eight E2M1 codes (code j in bits 4j..4j+3) -> eight bf16 values (pairs in out[0..3], code 2i in
// the low half of out[i]), times the block scale sc2 (2^(s - 127) in both halves).
__device__ __forceinline__ void e2m1x8_to_bf16(uint32_t x, __nv_bfloat162 sc2, uint32_t (&out)[4]) {
    const uint32_t mag = x & 0x77777777u;
    uint32_t hb0 = __byte_perm(kHiA, kHiB, mag);
    const uint32_t lb0 = __byte_perm(kLoA, kLoB, mag);
    const uint32_t m1 = mag >> 16;
    uint32_t hb1 = __byte_perm(kHiA, kHiB, m1);
    const uint32_t lb1 = __byte_perm(kLoA, kLoB, m1);
    // sign of code 2k at bit 7 of byte k of se, of code 2k + 1 at bit 7 of byte k of so
    const uint32_t se = (x << 4) & 0x80808080u, so = x & 0x80808080u;
    hb0 |= __byte_perm(se, so, 0x5140);
    hb1 |= __byte_perm(se, so, 0x7362);
    const uint32_t p[4] = {__byte_perm(lb0, hb0, 0x5140), __byte_perm(lb0, hb0, 0x7362),
                           __byte_perm(lb1, hb1, 0x5140), __byte_perm(lb1, hb1, 0x7362)};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        __nv_bfloat162 v = *reinterpret_cast<const __nv_bfloat162*>(&p[i]);
        v = __hmul2(v, sc2);                       // a power of two: exact in the normal range
        out[i] = *reinterpret_cast<const uint32_t*>(&v);
    }
}

// UE8M0 scale code -> 2^(s - 127) as bf16 in both halves (s = 0: the subnormal 2^-127; s = 255:
// NaN).
__device__ __forceinline__ __nv_bfloat162 ue8m0_to_bf16x2(uint32_t s) {
    const uint32_t h = s == 0 ? 0x0040u : (s == 255 ? 0x7FC0u : (s << 7));
    const uint32_t w = h | (h << 16);
    return *reinterpret_cast<const __nv_bfloat162*>(&w);
}

// Contiguous global -> shared bulk copy completing on an mbarrier (addresses and size 16-byte
// multiples).
__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar,
                                          uint64_t policy) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1], %2, [%3], %4;" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(bar), "l"(policy)
        : "memory");
}

// The tiled MXFP4 format: block (t, c) at byte (t * nk + c) * kAStageBytes holds the codes of
// rows 128 t .. 128 t + 127 and elements 64 c .. 64 c + 63 (row r at r * 32, element 64 c + 2 i
// in the low nibble of byte i, 64 c + 2 i + 1 in the high nibble), then the scale codes of their
// two blocks of 32 (block k of row r at 4096 + 128 k + r); rows past V and elements past D are
// zero.  One CTA of 256 threads writes one block.
__global__ void __launch_bounds__(256) mxfp4_pack_kernel(const uint8_t* __restrict__ W4, int64_t ldw4,
                                                          const uint8_t* __restrict__ S, int64_t lds,
                                                          int64_t V, int64_t D, int nk,
                                                          uint8_t* __restrict__ out) {
    const int64_t t = blockIdx.x / nk;
    const int c = static_cast<int>(blockIdx.x - t * nk);
    uint8_t* blk = out + static_cast<int64_t>(blockIdx.x) * kAStageBytes;
    const int i = threadIdx.x;
    {
        const int r = i >> 1, half = i & 1;
        const int64_t v = t * kTileV + r;
        const int64_t byte0 = static_cast<int64_t>(c) * (kBK / 2) + half * 16;   // within the row
        uint8_t piece[16];
#pragma unroll
        for (int e = 0; e < 16; ++e)
            piece[e] = (v < V && byte0 + e < D / 2) ? W4[v * ldw4 + byte0 + e] : 0;
        uint4 w;
        w.x = piece[0] | (piece[1] << 8) | (piece[2] << 16) | (static_cast<uint32_t>(piece[3]) << 24);
        w.y = piece[4] | (piece[5] << 8) | (piece[6] << 16) | (static_cast<uint32_t>(piece[7]) << 24);
        w.z = piece[8] | (piece[9] << 8) | (piece[10] << 16) | (static_cast<uint32_t>(piece[11]) << 24);
        w.w = piece[12] | (piece[13] << 8) | (piece[14] << 16) | (static_cast<uint32_t>(piece[15]) << 24);
        *reinterpret_cast<uint4*>(blk + i * 16) = w;
    }
    {
        const int k = i >> 7, r = i & 127;
        const int64_t v = t * kTileV + r;
        const int64_t kb = 2 * static_cast<int64_t>(c) + k;
        blk[kW4StageBytes + i] = (v < V && kb < D / 32) ? S[kb * lds + v] : 0;
    }
}

template <bool kWide, bool kPlain>
__global__ void __launch_bounds__(kMxThreads, 1)
    lmhead_mx_kernel(const uint8_t* __restrict__ Wt, const __grid_constant__ CUtensorMap tmH,
                     const MxParams prm) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_addr = smem_addr(smem_raw);
    const uint32_t base_addr = (raw_addr + 1023u) & ~1023u;
    uint8_t* base = smem_raw + (base_addr - raw_addr);
    const MxLayout L(prm.stages_a, prm.stages_c, prm.stages_h, prm.h_stage_bytes, prm.n_pad);

    const SampleArgs& a = prm.a;
    const int SA = prm.stages_a, SC = prm.stages_c, SH = prm.stages_h;
    const int n_pad = prm.n_pad;
    const int B = static_cast<int>(a.B);
    const int64_t nt = a.n_tiles;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    const uint32_t bar0 = base_addr + L.bars_off;
    auto fullA = [&](int s) { return bar0 + 8u * s; };
    auto emptyA = [&](int s) { return bar0 + 8u * (SA + s); };
    auto fullC = [&](int s) { return bar0 + 8u * (2 * SA + s); };
    auto emptyC = [&](int s) { return bar0 + 8u * (2 * SA + SC + s); };
    auto fullH = [&](int s) { return bar0 + 8u * (2 * SA + 2 * SC + s); };
    auto emptyH = [&](int s) { return bar0 + 8u * (2 * SA + 2 * SC + SH + s); };
    const uint32_t acc0 = bar0 + 8u * (2 * SA + 2 * SC + 2 * SH);
    auto accf_bar = [&](int ab) { return acc0 + 8u * ab; };
    auto acce_bar = [&](int ab) { return acc0 + 8u * (2 + ab); };
    const uint32_t drain_bar = acc0 + 32u;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(base + L.misc_off);
    volatile int* err = reinterpret_cast<volatile int*>(base + L.misc_off + 4);
    RowParams* rows = reinterpret_cast<RowParams*>(base + L.rows_off);
    unsigned long long* red = reinterpret_cast<unsigned long long*>(base + L.red_off);

    if (threadIdx.x == 0) {
        for (int s = 0; s < SA; ++s) {
            mbar_init(fullA(s), 1);
            mbar_init(emptyA(s), 1);
        }
        for (int s = 0; s < SC; ++s) {
            mbar_init(fullC(s), 1);
            mbar_init(emptyC(s), 1);
        }
        for (int s = 0; s < SH; ++s) {
            mbar_init(fullH(s), 1);
            mbar_init(emptyH(s), 1);
        }
        for (int ab = 0; ab < 2; ++ab) {
            mbar_init(accf_bar(ab), 1);
            mbar_init(acce_bar(ab), kMxEpiWarps);
        }
        mbar_init(drain_bar, 1);
        *err = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    }
    clear_status_bits(a.status_bits, a.row0);
    if (warp == 0 && lane == 0) {
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmH)) : "memory");
    }
    for (int b = threadIdx.x; b < B; b += blockDim.x) {
        rows[b] = make_row_params(a.temperature, a.seeds, a.positions, a.base_seed, a.offset,
                                  a.row0 + b);
        red[b] = 0ull;
    }
    if (warp == 1) tmem_alloc(base_addr + L.misc_off, prm.tmem_cols);
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem_base = *tmem_slot;
    // this CTA's K chunks, in order: chunk j is K chunk j % nk of its (j / nk)-th tile
    const int64_t my_tiles = nt > blockIdx.x ? (nt - 1 - blockIdx.x) / gridDim.x + 1 : 0;
    const int64_t n_chunks = my_tiles * prm.nk;
    auto chunk_tile = [&](int64_t j) { return blockIdx.x + (j / prm.nk) * static_cast<int64_t>(gridDim.x); };

    if (warp == 0) {
        // ---------------- TMA producer: packed weights and scales (ring A) ----------------
        if (lane == 0) {
            const uint64_t pol_w = l2_policy_evict_first();
            uint32_t issued = 0, issued_parity = 0;
            for (int64_t j = 0; j < n_chunks && *err == 0; ++j) {
                const int stage = static_cast<int>(j % SA);
                const uint32_t phase = static_cast<uint32_t>((j / SA) & 1);
                if (!mbar_wait(emptyA(stage), phase ^ 1u, prm.timeout_ns, err)) {
                    *err = 1;
                    break;
                }
                const bool withhold = j == 0 && blockIdx.x == 0 &&
                                      (prm.debug_flags & LMS_DEBUG_WITHHOLD_FIRST_LOAD);
                if (!withhold) {
                    const int64_t block = chunk_tile(j) * prm.nk + j % prm.nk;
                    mbar_arrive_expect_tx(fullA(stage), kAStageBytes);
                    bulk_load(base_addr + L.a_off + stage * kAStageBytes, Wt + block * kAStageBytes,
                              kAStageBytes, fullA(stage), pol_w);
                    issued |= 1u << stage;
                    issued_parity = (issued_parity & ~(1u << stage)) | (phase << stage);
                }
            }
            for (int s = 0; s < SA; ++s)
                if (issued & (1u << s))
                    mbar_wait(fullA(s), (issued_parity >> s) & 1u, prm.timeout_ns, nullptr);
        }
    } else if (warp == 2) {
        // ---------------- TMA producer: activations (ring H) ----------------
        if (lane == 0) {
            const uint64_t pol_h = l2_policy_evict_last();
            uint32_t issued = 0, issued_parity = 0;
            for (int64_t j = 0; j < n_chunks && *err == 0; ++j) {
                const int stage = static_cast<int>(j % SH);
                const uint32_t phase = static_cast<uint32_t>((j / SH) & 1);
                if (!mbar_wait(emptyH(stage), phase ^ 1u, prm.timeout_ns, err)) {
                    *err = 1;
                    break;
                }
                mbar_arrive_expect_tx(fullH(stage), prm.h_stage_bytes);
                tma_load_2d(base_addr + L.h_off + stage * prm.h_stage_bytes, &tmH,
                            static_cast<int>(j % prm.nk) * kBK, static_cast<int>(a.row0), fullH(stage), pol_h);
                issued |= 1u << stage;
                issued_parity = (issued_parity & ~(1u << stage)) | (phase << stage);
            }
            for (int s = 0; s < SH; ++s)
                if (issued & (1u << s))
                    mbar_wait(fullH(s), (issued_parity >> s) & 1u, prm.timeout_ns, nullptr);
        }
    } else if (warp == 1) {
        // ---------------- MMA issuer ----------------
        if (lane == 0) {
            const uint32_t idesc = mma_idesc_bf16(n_pad, kTileV);
            bool ok = true;
            for (int64_t i = 0; i < my_tiles && ok; ++i) {
                const int ab = static_cast<int>(i & 1);
                const uint32_t use_parity = static_cast<uint32_t>((i >> 1) & 1);
                if (!mbar_wait(acce_bar(ab), use_parity ^ 1u, prm.timeout_ns, err)) { ok = false; break; }
                tc_fence_after_sync();
                const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(ab * n_pad);
                for (int kc = 0; kc < prm.nk; ++kc) {
                    const int64_t j = i * prm.nk + kc;
                    const int sc = static_cast<int>(j % SC), sh = static_cast<int>(j % SH);
                    if (!mbar_wait(fullH(sh), static_cast<uint32_t>((j / SH) & 1), prm.timeout_ns, err) ||
                        !mbar_wait(fullC(sc), static_cast<uint32_t>((j / SC) & 1), prm.timeout_ns, err)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after_sync();
                    const uint64_t adesc = kmajor_sw128_desc(base_addr + L.c_off + sc * kWStageBytes);
                    const uint64_t bdesc = kmajor_sw128_desc(base_addr + L.h_off + sh * prm.h_stage_bytes);
#pragma unroll
                    for (int k = 0; k < 4; ++k)
                        mma_bf16(d_tmem, adesc + 2u * k, bdesc + 2u * k, idesc, (kc | k) != 0 ? 1u : 0u);
                    mma_commit(emptyC(sc));
                    mma_commit(emptyH(sh));
                }
                if (!ok) break;
                mma_commit(accf_bar(ab));
            }
            if (!ok) *err = 1;
            mma_commit(drain_bar);
            mbar_wait(drain_bar, 0, prm.timeout_ns, nullptr);
        }
    } else if (warp < kMxFirstEpi) {
        // ---------------- converters: one whole chunk per warp at a time ----------------
        // Converter w takes chunks j = w, w + 8, ...  Lane l converts the (row, scale block)
        // units u = l + 32 m (m < 8) of the chunk: row r = u / 2, block k = u % 2: 16 bytes of
        // codes (32 weights) and one scale byte, written as four 16-byte pieces of the row's
        // 128-byte line at the 128-byte-swizzled positions (piece p of row r goes to p ^ (r % 8)),
        // the layout a TMA load with the 128-byte swizzle would give.
        const int cw = warp - kMxFirstConv;
        bool ok = true;
        for (int64_t j = cw; j < n_chunks && ok; j += kMxConvWarps) {
            const int sa = static_cast<int>(j % SA), sc = static_cast<int>(j % SC);
            if (!mbar_wait(fullA(sa), static_cast<uint32_t>((j / SA) & 1), prm.timeout_ns, err) ||
                !mbar_wait(emptyC(sc), static_cast<uint32_t>(((j / SC) & 1) ^ 1), prm.timeout_ns, err)) {
                ok = false;
                break;
            }
            const uint8_t* w4 = base + L.a_off + sa * kAStageBytes;
            const uint8_t* sf = w4 + kW4StageBytes;
            uint4 codes[kUnitsPerLane];
            uint32_t scale[kUnitsPerLane];
#pragma unroll
            for (int m = 0; m < kUnitsPerLane; ++m) {
                const int u = lane + 32 * m;
                codes[m] = *reinterpret_cast<const uint4*>(w4 + u * 16);   // row u/2, block u%2
                scale[m] = sf[(u & 1) * kTileV + (u >> 1)];
            }
            // the codes and scales are in registers: the ring-A stage is free for the producer
            __syncwarp();
            if (lane == 0) mbar_arrive(emptyA(sa));
            uint8_t* tile = base + L.c_off + sc * kWStageBytes;
#pragma unroll
            for (int m = 0; m < kUnitsPerLane; ++m) {
                const int u = lane + 32 * m;
                const int r = u >> 1, blk = u & 1;
                const __nv_bfloat162 sc2 = ue8m0_to_bf16x2(scale[m]);
                const uint32_t cw4[4] = {codes[m].x, codes[m].y, codes[m].z, codes[m].w};
#pragma unroll
                for (int w = 0; w < 4; ++w) {
                    uint32_t o[4];
                    e2m1x8_to_bf16(cw4[w], sc2, o);
                    const int piece = (4 * blk + w) ^ (r & 7);
                    *reinterpret_cast<uint4*>(tile + r * 128 + piece * 16) = make_uint4(o[0], o[1], o[2], o[3]);
                }
            }
            // generic-proxy writes made visible to the tensor cores' (async proxy) reads
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            __syncwarp();
            if (lane == 0) mbar_arrive(fullC(sc));
        }
        if (!ok) *err = 1;
    } else {
        // ---------------- epilogue ----------------
        const int epi_tid = threadIdx.x - 32 * kMxFirstEpi;
        const int epi_threads = 32 * kMxEpiWarps;
        const int quad = warp & 3;                       // TMEM lanes 32*quad .. 32*quad+31
        const int col_group = (warp - kMxFirstEpi) >> 2;
        float* tr = reinterpret_cast<float*>(base + L.tr_off + (warp - kMxFirstEpi) * kTrWarpBytes);
        int i = 0;
        bool ok = true;
        for (int64_t tile = blockIdx.x; tile < nt; tile += gridDim.x, ++i) {
            const int ab = i & 1;
            const uint32_t use_parity = (i >> 1) & 1;
            if (ok) ok = mbar_wait(accf_bar(ab), use_parity, prm.timeout_ns, err);
            ok = epi_barrier_and(epi_threads, ok);
            if (!ok) {
                if (epi_tid == 0) *err = 1;
                for (int b = epi_tid; b < B; b += epi_threads) {
                    a.cand_score[b * nt + tile] = -CUDART_INF_F;
                    a.cand_index[b * nt + tile] = kPoisonIndex;
                }
                continue;
            }
            tc_fence_after_sync();
            const uint32_t t_row = tmem_base + (static_cast<uint32_t>(32 * quad) << 16) +
                                   static_cast<uint32_t>(ab * n_pad);
            epilogue_tile_columns<kMxEpiWarps, kWide, kPlain>(a, rows, red, tr, t_row, tile, quad,
                                                              col_group, lane, B);
            tc_fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(acce_bar(ab));
            epi_barrier(epi_threads);
            for (int b = epi_tid; b < B; b += epi_threads) {
                const unsigned long long key = red[b];
                red[b] = 0ull;
                const float s = unpack_score(key);
                a.cand_score[b * nt + tile] = s;
                a.cand_index[b * nt + tile] = candidate_index(s, unpack_index(key));
            }
            epi_barrier(epi_threads);
        }
    }

    pdl_launch_dependents();
    tc_fence_before_sync();
    __syncthreads();
    if (warp == 1) {
        __syncwarp();
        tc_fence_after_sync();
        tmem_dealloc(tmem_base, prm.tmem_cols);
    }
}

template <bool kWide, bool kPlain>
cudaError_t launch_mx_variant(const uint8_t* Wt, const CUtensorMap& tmH, const MxParams& prm,
                              size_t smem, int grid, cudaStream_t stream) {
    auto kern = lmhead_mx_kernel<kWide, kPlain>;
    const cudaError_t e = ensure_dynamic_smem(reinterpret_cast<const void*>(kern), smem);
    if (e != cudaSuccess) return e;
    kern<<<grid, kMxThreads, smem, stream>>>(Wt, tmH, prm);
    return cudaGetLastError();
}

}  // namespace

size_t mxfp4_tiled_bytes(int64_t V, int64_t D) {
    return static_cast<size_t>((V + kTileV - 1) / kTileV) * static_cast<size_t>((D + kBK - 1) / kBK) *
           kAStageBytes;
}

cudaError_t launch_mxfp4_pack(const uint8_t* W4, int64_t ldw4, const uint8_t* S, int64_t lds, int64_t V,
                              int64_t D, uint8_t* out, cudaStream_t stream) {
    const int nk = static_cast<int>((D + kBK - 1) / kBK);
    const int64_t blocks = (V + kTileV - 1) / kTileV * nk;
    if (blocks > 0x7fffffff) return cudaErrorInvalidValue;
    mxfp4_pack_kernel<<<static_cast<unsigned>(blocks), 256, 0, stream>>>(W4, ldw4, S, lds, V, D, nk, out);
    return cudaGetLastError();
}

cudaError_t launch_lmhead_mx(const uint8_t* Wt, const CUtensorMap& tmH, int64_t D, int n_pad, bool wide,
                             uint32_t timeout_ms, uint32_t debug_flags, const SampleArgs& a,
                             cudaStream_t stream) {
    MxParams prm;
    prm.a = a;
    prm.nk = static_cast<int>((D + kBK - 1) / kBK);
    prm.n_pad = n_pad;
    prm.h_stage_bytes = static_cast<uint32_t>(n_pad * kBK * 2);
    const uint32_t budget = 227u * 1024u - 1024u;        // opt-in maximum minus alignment slack
    const uint32_t per_a = kAStageBytes;
    const uint32_t bar_bytes = (2 * kMaxStagesA + 2 * kStagesC + 2 * kMaxStagesH + 5) * 8;
    const uint32_t fixed = MxLayout(0, 0, 0, prm.h_stage_bytes, n_pad).total + bar_bytes;
    // ring C: one slot per converter warp; ring H as deep as fits, from 8 down to 4; then ring A
    // 16 deep when there is room, else 8
    const int sc = kStagesC;
    int sh = kMaxStagesH, sa = kMaxStagesA;
    auto used = [&]() { return fixed + sa * per_a + sh * prm.h_stage_bytes + sc * kWStageBytes; };
    while (used() > budget && sa > kMxConvWarps) sa -= kMxConvWarps;
    while (used() > budget && sh > 2) --sh;
    if (used() > budget) return cudaErrorInvalidValue;
    prm.stages_a = sa;
    prm.stages_c = sc;
    prm.stages_h = sh;
    uint32_t cols = 32;
    while (cols < static_cast<uint32_t>(2 * n_pad)) cols <<= 1;
    prm.tmem_cols = cols;
    prm.timeout_ns = static_cast<uint64_t>(timeout_ms) * 1000000ull;
    prm.debug_flags = debug_flags;
    const MxLayout L(sa, sc, sh, prm.h_stage_bytes, n_pad);
    const size_t smem = L.total + 1024;
    const int sms = device_sm_count();
    const int grid = static_cast<int>(a.n_tiles < sms ? a.n_tiles : sms);
    const bool plain = a.bias == nullptr && a.mask == nullptr;
    if (plain)
        return wide ? launch_mx_variant<true, true>(Wt, tmH, prm, smem, grid, stream)
                    : launch_mx_variant<false, true>(Wt, tmH, prm, smem, grid, stream);
    return wide ? launch_mx_variant<true, false>(Wt, tmH, prm, smem, grid, stream)
                : launch_mx_variant<false, false>(Wt, tmH, prm, smem, grid, stream);
}

}  // namespace lms
