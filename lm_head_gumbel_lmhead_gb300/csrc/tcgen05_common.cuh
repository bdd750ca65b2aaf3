// Building blocks shared by the tcgen05 kernels: PTX wrappers for mbarriers, TMA, TMEM and
// tcgen05.mma, the operand descriptors, the ordered 64-bit candidate key, and the epilogue's
// per-tile column loop (transform, Philox noise and argmax over one TMEM accumulator).
#pragma once
#include <cuda.h>

#include "lms_device.cuh"
#include "lms_kernels.h"

namespace lms {
namespace tc {

constexpr int kTileV = 128;                       // rows of W per accumulator (TMEM lanes)
constexpr int kBK = 64;                           // K elements per stage (one 128-byte row)
constexpr int kWStageBytes = kTileV * kBK * 2;    // 16 KB
constexpr uint32_t kEpiBarrierId = 1;

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(bar), "r"(parity)
        : "memory");
    return done != 0;
}

__device__ __forceinline__ uint64_t global_timer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Waits until the barrier phase of the given parity has completed.  Gives up (returns false)
// when `timeout_ns` passes or, if `err` is non-null, when another role has flagged an error.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, uint64_t timeout_ns,
                                          const volatile int* err) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t deadline = global_timer_ns() + timeout_ns;
    for (uint32_t spin = 1;; ++spin) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((spin & 31u) == 0u) {
            if (err != nullptr && *err != 0) return false;
            if (global_timer_ns() > deadline) return false;
        }
    }
}

// As mbar_wait, but each try suspends the thread for up to `suspend_ns` while the phase is
// incomplete (the thread resumes when the phase completes), so a long wait issues almost no
// instructions and leaves the issue slots to the warps doing work.  The error flag and the
// deadline are checked after every try.
__device__ __forceinline__ bool mbar_wait_suspend(uint32_t bar, uint32_t parity, uint64_t timeout_ns,
                                                  const volatile int* err, uint32_t suspend_ns) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t deadline = global_timer_ns() + timeout_ns;
    for (;;) {
        uint32_t done;
        asm volatile(
            "{\n\t.reg .pred p;\n\t"
            "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
            "selp.u32 %0, 1, 0, p;\n\t}"
            : "=r"(done)
            : "r"(bar), "r"(parity), "r"(suspend_ns)
            : "memory");
        if (done) return true;
        if (err != nullptr && *err != 0) return false;
        if (global_timer_ns() > deadline) return false;
    }
}

__device__ __forceinline__ uint64_t l2_policy_evict_first() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

__device__ __forceinline__ uint64_t l2_policy_evict_last() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

// 2-D tiled TMA load (box given by the descriptor) completing on an mbarrier.
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* tm, int x, int y,
                                            uint32_t bar, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(tm)), "r"(x), "r"(y), "r"(bar), "l"(policy)
        : "memory");
}

__device__ __forceinline__ void tmem_alloc(uint32_t slot, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(slot),
                 "r"(ncols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
                 : "memory");
}

__device__ __forceinline__ void tc_fence_before_sync() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tc_fence_after_sync() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// D[tmem] (+)= A[smem] * B[smem]^T, bf16 inputs, fp32 accumulate; issued by one thread.
__device__ __forceinline__ void mma_bf16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                         uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// D[tmem] (+)= A[smem] * B[smem]^T, E4M3 inputs (K = 32 per instruction), fp32 accumulate.
__device__ __forceinline__ void mma_e4m3(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                         uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Arrive once on `bar` when all tcgen05 operations issued so far by this thread have completed.
__device__ __forceinline__ void mma_commit(uint32_t bar) {
    asm volatile(
        "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
        : "memory");
}

// 32 TMEM lanes x 8 consecutive 32-bit columns -> 8 registers per thread (lane = thread).
__device__ __forceinline__ void tmem_load_8(uint32_t taddr, uint32_t (&r)[8]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void epi_barrier(int threads) {
    asm volatile("bar.sync %0, %1;" ::"r"(kEpiBarrierId), "r"(threads) : "memory");
}

// Barrier over the epilogue warps that also ANDs a flag across them, so that every epilogue
// thread takes the same branch after a bounded wait (no thread can be left at a barrier).
__device__ __forceinline__ bool epi_barrier_and(int threads, bool flag) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.u32 p, %1, 0;\n\t"
        "bar.red.and.pred p, %2, %3, p;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(r)
        : "r"(flag ? 1u : 0u), "r"(kEpiBarrierId), "r"(threads)
        : "memory");
    return r != 0;
}

// (score, index) as one 64-bit key whose unsigned order is the lexicographic order "larger
// score, then smaller index": the score's bits mapped to a monotone unsigned integer in the high
// half (-0 folded onto +0 first; scores are never NaN here), the complemented index in the low
// half.  Key 0 is below every real candidate.
__device__ __forceinline__ unsigned long long pack_candidate(float s, int idx) {
    const uint32_t f = __float_as_uint(s + 0.0f);
    const uint32_t ord = (f & 0x80000000u) ? ~f : (f | 0x80000000u);
    return (static_cast<unsigned long long>(ord) << 32) | static_cast<uint32_t>(~static_cast<uint32_t>(idx));
}

__device__ __forceinline__ float unpack_score(unsigned long long key) {
    const uint32_t ord = static_cast<uint32_t>(key >> 32);
    return __uint_as_float((ord & 0x80000000u) ? (ord & 0x7fffffffu) : ~ord);
}

__device__ __forceinline__ int unpack_index(unsigned long long key) {
    return static_cast<int>(~static_cast<uint32_t>(key));
}

// Shared-memory matrix descriptor for a K-major operand tile written by TMA with the 128-byte
// swizzle: rows of 128 bytes, 8-row groups 1024 bytes apart (stride byte offset), the leading
// byte offset unused for this layout, descriptor version 1, layout code 2 = 128-byte swizzle.
__device__ __forceinline__ uint64_t kmajor_sw128_desc(uint32_t saddr) {
    uint64_t d = 0;
    d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
    d |= static_cast<uint64_t>(1u) << 16;
    d |= static_cast<uint64_t>(1024u >> 4) << 32;
    d |= static_cast<uint64_t>(1u) << 46;
    d |= static_cast<uint64_t>(2u) << 61;
    return d;
}

// Instruction descriptor, kind::f8f6f4: fp32 accumulator, E4M3 A and B (format code 0), both
// K-major, N and M.
__host__ __device__ constexpr uint32_t mma_idesc_e4m3(int n, int m) {
    return (1u << 4) | (static_cast<uint32_t>(n >> 3) << 17) | (static_cast<uint32_t>(m >> 4) << 24);
}

// Instruction descriptor, kind::f16: fp32 accumulator, bf16 A and B, both K-major, N and M.
__host__ __device__ constexpr uint32_t mma_idesc_bf16(int n, int m) {
    return (1u << 4) | (1u << 7) | (1u << 10) | (static_cast<uint32_t>(n >> 3) << 17) |
           (static_cast<uint32_t>(m >> 4) << 24);
}

// Per epilogue warp: an 8-column x 32-row transpose tile, rows padded to 36 floats so that both
// the row-wise stores and the 16-byte column-wise loads are free of bank conflicts.
constexpr int kTrStride = 36;
constexpr uint32_t kTrWarpBytes = 8 * kTrStride * 4;


// One tile's epilogue over this warp's share of the batch columns: for each 8-column chunk,
// load the warp's 32 TMEM lanes (rows), transpose through the warp's shared-memory tile so that
// each thread owns 8 consecutive rows of one column, add bias / mask / temperature and the
// Philox Gumbel noise (2 calls fp32, 4 wide), take the argmax, combine the 4 threads sharing
// the column, and fold the result into red[b] (the tile's best key per column) with atomicMax.
template <int kEpiWarps, bool kWide, bool kPlain = false>
__device__ __forceinline__ void epilogue_tile_columns(const SampleArgs& a, const RowParams* rows,
                                                      unsigned long long* red, float* tr,
                                                      uint32_t t_row, int64_t tile, int quad,
                                                      int col_group, int lane, int B) {
    constexpr int kColGroups = kEpiWarps / 4;
    const int n_chunks = (B + 7) / 8;
    const int my_col = lane & 7;
    const int my_r0 = (lane >> 3) * 8;
    const int64_t v0 = tile * kTileV + 32 * quad + my_r0;   // a multiple of 8
    for (int cc = col_group; cc < n_chunks; cc += kColGroups) {
        uint32_t acc[8];
        tmem_load_8(t_row + 8u * cc, acc);
#pragma unroll
        for (int j = 0; j < 8; ++j) tr[j * kTrStride + lane] = __uint_as_float(acc[j]);
        __syncwarp();
        float y[8];
        const float4 y0 = *reinterpret_cast<const float4*>(tr + my_col * kTrStride + my_r0);
        const float4 y1 = *reinterpret_cast<const float4*>(tr + my_col * kTrStride + my_r0 + 4);
        __syncwarp();
        y[0] = y0.x; y[1] = y0.y; y[2] = y0.z; y[3] = y0.w;
        y[4] = y1.x; y[5] = y1.y; y[6] = y1.z; y[7] = y1.w;
        const int b = cc * 8 + my_col;
        float best_s = -CUDART_INF_F;
        int best_i = kNoIndex;
        if (b < B && v0 < a.V) {
            const RowParams p = rows[b];
            if (!(p.flags & kRowInvalid)) {
                float g[8];
                if (p.flags & kRowGreedy) {
#pragma unroll
                    for (int e = 0; e < 8; ++e) g[e] = 0.0f;
                } else {
                    gumbel_run<kWide, 8>(p.key, static_cast<uint32_t>(v0), g);
                }
                const int64_t row = a.row0 + b;
                if (a.w_scale) {                 // FP8 inputs: logits = acc * 2^e_h * w_scale
                    // w_scale * 2^e_h is exact while 2^e_h is a normal float, so the product
                    // equals ldexpf(w_scale, e_h); below that range ldexpf per entry keeps it
                    const int eh = a.h_exp[row];
                    const float* ws = a.w_scale + v0;
                    if (eh >= -126 && eh <= 127 && v0 + 8 <= a.V &&
                        (reinterpret_cast<uintptr_t>(ws) & 15u) == 0) {
                        const float hs = __int_as_float((eh + 127) << 23);
                        const float4 w0 = __ldg(reinterpret_cast<const float4*>(ws));
                        const float4 w1 = __ldg(reinterpret_cast<const float4*>(ws) + 1);
                        y[0] *= w0.x * hs; y[1] *= w0.y * hs; y[2] *= w0.z * hs; y[3] *= w0.w * hs;
                        y[4] *= w1.x * hs; y[5] *= w1.y * hs; y[6] *= w1.z * hs; y[7] *= w1.w * hs;
                    } else {
#pragma unroll
                        for (int e = 0; e < 8; ++e)
                            if (v0 + e < a.V) y[e] *= ldexpf(__ldg(ws + e), eh);
                    }
                }
                if constexpr (kPlain) {
                    // no bias and no mask in this launch: s = y / T + g (greedy: y), no per-entry
                    // tests on a whole chunk; a NaN score never compares above the running best,
                    // so it loses as -inf does
                    const float scale = (p.flags & kRowGreedy) ? 1.0f : p.inv_t;
                    const int v0i = static_cast<int>(v0);
                    if (v0 + 8 <= a.V) {
#pragma unroll
                        for (int e = 0; e < 8; ++e) {
                            const float sc = fmaf(y[e], scale, g[e]);
                            if (sc > best_s) { best_s = sc; best_i = v0i + e; }
                        }
                    } else {
#pragma unroll
                        for (int e = 0; e < 8; ++e) {
                            const float sc = fmaf(y[e], scale, g[e]);
                            if (v0 + e < a.V && sc > best_s) { best_s = sc; best_i = v0i + e; }
                        }
                    }
                } else {
                    const float* brow = a.bias ? a.bias + row * a.ld_bias : nullptr;
                    // the eight entries share one mask word (v0 is a multiple of 8)
                    const uint32_t mword =
                        a.mask ? (__ldg(a.mask + row * a.ld_mask + (v0 >> 5)) >> (v0 & 31)) : 0xffu;
                    const float scale = (p.flags & kRowGreedy) ? 1.0f : p.inv_t;
                    if (v0 + 8 <= a.V) {
                        // a whole chunk: the bias as two 16-byte loads when the row allows it;
                        // s = (y + bias) / T + g, masked entries -inf; a NaN score never
                        // compares above the running best, so it loses as -inf does
                        float bias[8];
                        if (brow != nullptr && (reinterpret_cast<uintptr_t>(brow + v0) & 15u) == 0) {
                            const float4 b0 = __ldg(reinterpret_cast<const float4*>(brow + v0));
                            const float4 b1 = __ldg(reinterpret_cast<const float4*>(brow + v0) + 1);
                            bias[0] = b0.x; bias[1] = b0.y; bias[2] = b0.z; bias[3] = b0.w;
                            bias[4] = b1.x; bias[5] = b1.y; bias[6] = b1.z; bias[7] = b1.w;
                        } else {
#pragma unroll
                            for (int e = 0; e < 8; ++e) bias[e] = brow ? __ldg(brow + v0 + e) : 0.0f;
                        }
                        const int v0i = static_cast<int>(v0);
#pragma unroll
                        for (int e = 0; e < 8; ++e) {
                            const float t = fmaf(y[e] + bias[e], scale, g[e]);
                            const float sc = ((mword >> e) & 1u) ? t : -CUDART_INF_F;
                            if (sc > best_s) { best_s = sc; best_i = v0i + e; }
                        }
                    } else {
#pragma unroll
                        for (int e = 0; e < 8; ++e) {
                            const int64_t v = v0 + e;
                            if (v < a.V) {
                                const float bias = brow ? __ldg(brow + v) : 0.0f;
                                const float sc = perturb(p, y[e], bias, (mword >> e) & 1u, g[e]);
                                if (sc > best_s) { best_s = sc; best_i = static_cast<int>(v); }
                            }
                        }
                    }
                }
            }
        }
        // the four threads holding this column (lanes c, c + 8, c + 16, c + 24)
#pragma unroll
        for (int off = 8; off <= 16; off <<= 1) {
            const float so = __shfl_xor_sync(0xffffffffu, best_s, off);
            const int io = __shfl_xor_sync(0xffffffffu, best_i, off);
            if (better(so, io, best_s, best_i)) { best_s = so; best_i = io; }
        }
        if (lane < 8 && b < B) atomicMax(red + b, pack_candidate(best_s, best_i));
    }
}

// ---------------------------------------------------------------------------------------------
// Gumbel-top-k epilogue (k draws without replacement: the k largest perturbed scores)
// ---------------------------------------------------------------------------------------------
constexpr int kMaxTopK = 16;
// Written in place of a tile's keys when a bounded wait ran out; above every real key (a real
// key's high half is at most the order key of +inf, 0xff800000).
constexpr unsigned long long kPoisonKey = ~0ull;

// One tile's Gumbel-top-k epilogue.  Scores as in epilogue_tile_columns, then as ordered 64-bit
// keys (0 for -inf).  Per column, the 4 threads holding its 32 rows (this warp's TMEM quadrant)
// extract their best keys by rounds of shuffle-max with removal, at most k, and the warp writes
// that ordered list to a.cand_keys[((b * n_tiles + tile) * 4 + quad) * k + r], ended by a key 0
// when shorter than k (the slots after it are not written).
// thr[quad * n_pad + b] holds the k-th key of this warp's last full list for column b: k keys of
// the row lie above it, so entries not above it cannot be among the row's k best and are dropped
// before the rounds, which stop once no column of the warp has a key left.  Every key among the
// row's k best therefore reaches some list; Stage 2 merges them.  No step crosses warps.
template <int kEpiWarps, bool kWide, bool kPlain = false>
__device__ __forceinline__ void epilogue_tile_topk(const SampleArgs& a, const RowParams* rows,
                                                   float* tr, unsigned long long* thr, int n_pad,
                                                   uint32_t t_row, int64_t tile, int quad,
                                                   int col_group, int lane, int B) {
    constexpr int kColGroups = kEpiWarps / 4;
    const int k = a.topk;
    const int n_chunks = (B + 7) / 8;
    const int my_col = lane & 7;
    const int my_r0 = (lane >> 3) * 8;
    const int64_t v0 = tile * kTileV + 32 * quad + my_r0;   // a multiple of 8
    for (int cc = col_group; cc < n_chunks; cc += kColGroups) {
        uint32_t acc[8];
        tmem_load_8(t_row + 8u * cc, acc);
#pragma unroll
        for (int j = 0; j < 8; ++j) tr[j * kTrStride + lane] = __uint_as_float(acc[j]);
        __syncwarp();
        float y[8];
        const float4 y0 = *reinterpret_cast<const float4*>(tr + my_col * kTrStride + my_r0);
        const float4 y1 = *reinterpret_cast<const float4*>(tr + my_col * kTrStride + my_r0 + 4);
        __syncwarp();
        y[0] = y0.x; y[1] = y0.y; y[2] = y0.z; y[3] = y0.w;
        y[4] = y1.x; y[5] = y1.y; y[6] = y1.z; y[7] = y1.w;
        const int b = cc * 8 + my_col;
        unsigned long long* th = thr + quad * n_pad + (b < B ? b : 0);
        const unsigned long long theta = b < B ? *th : 0ull;
        unsigned long long ky[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) ky[e] = 0ull;
        if (b < B && v0 < a.V) {
            const RowParams p = rows[b];
            if (!(p.flags & kRowInvalid)) {
                float g[8];
                if (p.flags & kRowGreedy) {
#pragma unroll
                    for (int e = 0; e < 8; ++e) g[e] = 0.0f;
                } else {
                    gumbel_run<kWide, 8>(p.key, static_cast<uint32_t>(v0), g);
                }
                const int64_t row = a.row0 + b;
                if constexpr (kPlain) {
                    // no bias and no mask in this launch: s = y / T + g (greedy: y); a NaN score
                    // fails the -inf test below and gets no key, as a masked entry
                    const float scale = (p.flags & kRowGreedy) ? 1.0f : p.inv_t;
                    const int v0i = static_cast<int>(v0);
                    const int n_in = (a.V - v0 < 8) ? static_cast<int>(a.V - v0) : 8;
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        const float sc = fmaf(y[e], scale, g[e]);
                        const unsigned long long key = pack_candidate(sc, v0i + e);
                        ky[e] = (e < n_in && sc > -CUDART_INF_F && key > theta) ? key : 0ull;
                    }
                } else {
                    const float* brow = a.bias ? a.bias + row * a.ld_bias : nullptr;
                    const uint32_t mword =
                        a.mask ? (__ldg(a.mask + row * a.ld_mask + (v0 >> 5)) >> (v0 & 31)) : 0xffu;
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        const int64_t v = v0 + e;
                        if (v < a.V) {
                            const float bias = brow ? __ldg(brow + v) : 0.0f;
                            const float sc = perturb(p, y[e], bias, (mword >> e) & 1u, g[e]);
                            const unsigned long long key = pack_candidate(sc, static_cast<int>(v));
                            ky[e] = (sc > -CUDART_INF_F && key > theta) ? key : 0ull;
                        }
                    }
                }
            }
        }
        unsigned long long* out =
            a.cand_keys + ((static_cast<int64_t>(b < B ? b : 0) * a.n_tiles + tile) * 4 + quad) * k;
        // rounds: the column's best remaining key; its owner drops it
        int r = 0;
        unsigned long long last = 0ull;
        for (; r < k; ++r) {
            unsigned long long bk = 0ull;
#pragma unroll
            for (int e = 0; e < 8; ++e) bk = ky[e] > bk ? ky[e] : bk;
            unsigned long long wk = bk;
#pragma unroll
            for (int off = 8; off <= 16; off <<= 1) {
                const unsigned long long o = __shfl_xor_sync(0xffffffffu, wk, off);
                wk = o > wk ? o : wk;
            }
            if (!__any_sync(0xffffffffu, wk != 0ull)) break;   // no column of the warp has one left
            if (wk != 0ull && wk == bk) {
#pragma unroll
                for (int e = 0; e < 8; ++e) ky[e] = ky[e] == bk ? 0ull : ky[e];
            }
            if (lane < 8 && b < B) out[r] = wk;
            last = wk;
        }
        if (lane < 8 && b < B) {
            if (r < k) out[r] = 0ull;                    // a shorter list ends with key 0
            if (r == k && last != 0ull) *th = last;     // a full list: its k-th key
        }
    }
}

// Gumbel-top-k with running lists (used when they fit in shared memory): per TMEM quadrant and
// batch column, the ordered k largest keys of the quadrant's rows over the CTA's tiles so far,
// run[(quad * n_pad + b) * k + r], larger first, key 0 for an empty slot.  The list of (b, quad)
// belongs to one epilogue lane (lane b % 8 of the quadrant's warp that takes b's column chunk),
// which alone writes it while the tiles run.  Scores and extraction rounds as in
// epilogue_tile_topk.  The threshold is the largest k-th key among row b's four quadrant lists:
// that quadrant alone holds k keys above it, so no key at or below it is among the row's k best,
// and since the lists' k-th keys only grow, reading another quadrant's while its owner updates it
// gives a threshold that is still valid, if lower.  After a CTA's first tiles almost every chunk
// ends before its first round.  Nothing is written to global memory per tile:
// topk_running_lists_publish writes each list once, after the CTA's last tile.
template <int kEpiWarps, bool kWide, bool kPlain = false>
__device__ __forceinline__ void epilogue_tile_topk_running(const SampleArgs& a, const RowParams* rows,
                                                           float* tr, unsigned long long* run, int n_pad,
                                                           uint32_t t_row, int64_t tile, int quad,
                                                           int col_group, int lane, int B) {
    constexpr int kColGroups = kEpiWarps / 4;
    const int k = a.topk;
    const int n_chunks = (B + 7) / 8;
    const int my_col = lane & 7;
    const int my_r0 = (lane >> 3) * 8;
    const int64_t v0 = tile * kTileV + 32 * quad + my_r0;   // a multiple of 8
    for (int cc = col_group; cc < n_chunks; cc += kColGroups) {
        uint32_t acc[8];
        tmem_load_8(t_row + 8u * cc, acc);
#pragma unroll
        for (int j = 0; j < 8; ++j) tr[j * kTrStride + lane] = __uint_as_float(acc[j]);
        __syncwarp();
        float y[8];
        const float4 y0 = *reinterpret_cast<const float4*>(tr + my_col * kTrStride + my_r0);
        const float4 y1 = *reinterpret_cast<const float4*>(tr + my_col * kTrStride + my_r0 + 4);
        __syncwarp();
        y[0] = y0.x; y[1] = y0.y; y[2] = y0.z; y[3] = y0.w;
        y[4] = y1.x; y[5] = y1.y; y[6] = y1.z; y[7] = y1.w;
        const int b = cc * 8 + my_col;
        const int bb = b < B ? b : 0;
        unsigned long long* lst = run + (static_cast<int64_t>(quad) * n_pad + bb) * k;
        unsigned long long theta = 0ull;
        if (b < B) {
#pragma unroll
            for (int q4 = 0; q4 < 4; ++q4) {
                const unsigned long long t = *reinterpret_cast<volatile const unsigned long long*>(
                    run + (static_cast<int64_t>(q4) * n_pad + bb) * k + (k - 1));
                theta = t > theta ? t : theta;
            }
        }
        unsigned long long ky[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) ky[e] = 0ull;
        if (b < B && v0 < a.V) {
            const RowParams p = rows[b];
            if (!(p.flags & kRowInvalid)) {
                float g[8];
                if (p.flags & kRowGreedy) {
#pragma unroll
                    for (int e = 0; e < 8; ++e) g[e] = 0.0f;
                } else {
                    gumbel_run<kWide, 8>(p.key, static_cast<uint32_t>(v0), g);
                }
                const int64_t row = a.row0 + b;
                if constexpr (kPlain) {
                    // no bias and no mask in this launch: s = y / T + g (greedy: y); a NaN score
                    // fails the -inf test below and gets no key, as a masked entry
                    const float scale = (p.flags & kRowGreedy) ? 1.0f : p.inv_t;
                    const int v0i = static_cast<int>(v0);
                    const int n_in = (a.V - v0 < 8) ? static_cast<int>(a.V - v0) : 8;
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        const float sc = fmaf(y[e], scale, g[e]);
                        const unsigned long long key = pack_candidate(sc, v0i + e);
                        ky[e] = (e < n_in && sc > -CUDART_INF_F && key > theta) ? key : 0ull;
                    }
                } else {
                    const float* brow = a.bias ? a.bias + row * a.ld_bias : nullptr;
                    const uint32_t mword =
                        a.mask ? (__ldg(a.mask + row * a.ld_mask + (v0 >> 5)) >> (v0 & 31)) : 0xffu;
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        const int64_t v = v0 + e;
                        if (v < a.V) {
                            const float bias = brow ? __ldg(brow + v) : 0.0f;
                            const float sc = perturb(p, y[e], bias, (mword >> e) & 1u, g[e]);
                            const unsigned long long key = pack_candidate(sc, static_cast<int>(v));
                            ky[e] = (sc > -CUDART_INF_F && key > theta) ? key : 0ull;
                        }
                    }
                }
            }
        }
        // rounds: the column's best remaining key; its owner drops it and, while it beats the
        // threshold (the row-wide one, raised by the owner's own list as it fills), inserts it;
        // after each round the 4 lanes of a column take the owner's threshold.  A chunk with no
        // key left above its thresholds (most chunks after a CTA's first tiles) skips the rounds.
        unsigned long long kth = theta;
        bool mine = false;
#pragma unroll
        for (int e = 0; e < 8; ++e) mine = mine || ky[e] != 0ull;
        const int rounds = __any_sync(0xffffffffu, mine) ? k : 0;
        for (int r = 0; r < rounds; ++r) {
            unsigned long long bk = 0ull;
#pragma unroll
            for (int e = 0; e < 8; ++e) bk = ky[e] > bk ? ky[e] : bk;
            unsigned long long wk = bk;
#pragma unroll
            for (int off = 8; off <= 16; off <<= 1) {
                const unsigned long long o = __shfl_xor_sync(0xffffffffu, wk, off);
                wk = o > wk ? o : wk;
            }
            // no column of the warp has a key left that would enter its list
            if (!__any_sync(0xffffffffu, wk > kth)) break;
            if (wk != 0ull && wk == bk) {
#pragma unroll
                for (int e = 0; e < 8; ++e) ky[e] = ky[e] == bk ? 0ull : ky[e];
            }
            if (lane < 8 && b < B && wk > kth) {
                // insertion into the ordered list: carry the displaced key down.  The list's new
                // k-th key is the smaller of wk and its old (k-1)-th (for k = 1: wk), kept in a
                // register rather than read back.
                unsigned long long cur = wk, before_last = wk;
#pragma unroll
                for (int i = 0; i < kMaxTopK; ++i) {
                    if (i < k) {
                        const unsigned long long li = lst[i];
                        if (i == k - 2) before_last = li;
                        lst[i] = cur > li ? cur : li;
                        cur = cur > li ? li : cur;
                    }
                }
                const unsigned long long own = (k >= 2 && before_last < wk) ? before_last : wk;
                kth = own > kth ? own : kth;
            }
            kth = __shfl_sync(0xffffffffu, kth, lane & 7);
        }
    }
}

// After the CTA's last tile: each owner lane writes its running lists to the workspace,
// uint64 [B][4 G][k] (G = gridDim.x): list (b, blockIdx.x, quad) at ((b * 4 G) + 4 blockIdx.x +
// quad) * k.  A CTA whose bounded wait ran out (ok false, the same in every epilogue thread)
// heads each list with the poison key instead.
template <int kEpiWarps>
__device__ __forceinline__ void topk_running_lists_publish(const SampleArgs& a, const unsigned long long* run,
                                                           int n_pad, int quad, int col_group, int lane,
                                                           int B, bool ok) {
    constexpr int kColGroups = kEpiWarps / 4;
    const int k = a.topk;
    const int n_chunks = (B + 7) / 8;
    for (int cc = col_group; cc < n_chunks; cc += kColGroups) {
        const int b = cc * 8 + (lane & 7);
        if (lane < 8 && b < B) {
            const unsigned long long* lst = run + (static_cast<int64_t>(quad) * n_pad + b) * k;
            unsigned long long* out =
                a.cand_keys + ((static_cast<int64_t>(b) * 4 * gridDim.x + 4 * blockIdx.x + quad) * k);
            out[0] = ok ? lst[0] : kPoisonKey;
            for (int i = 1; i < k; ++i) out[i] = lst[i];
        }
    }
}

}  // namespace tc
}  // namespace lms
