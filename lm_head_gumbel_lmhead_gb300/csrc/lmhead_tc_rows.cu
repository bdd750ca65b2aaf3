// Fused LM-head + Gumbel-max Stage 1 for batches above 256 rows: row groups that stream W once.
//
// FlashSampling ("method step details", Stage 1; "Limitations": the portable kernel trails a
// library GEMM at large batch).  One CTA holds at most 256 batch rows: two 128 x 256 fp32
// accumulators fill the 512 TMEM columns.  Above 256 rows this kernel serves up to four groups of
// 256 rows in one launch: CTA c takes group c mod G and walks the vocabulary tiles c / G,
// c / G + grid / G, ..., so the G CTAs that share a tile read it within a short window and every
// read of W but the first hits L2.  Run as separate launches of 256 rows, each launch would stream
// all of W from HBM.
//
// The roles, ring, barriers, bounded waits and epilogue are those of the single-group kernel
// (lmhead_tc.cu, bf16 race only), which this translation unit leaves untouched: warp 0 is the
// TMA producer (W[128 x 64] and this group's H[256 x 64] per stage), warp 1 allocates TMEM and
// issues tcgen05.mma (M = 128 vocabulary rows, N = 256 batch rows, K = 16), the epilogue warps
// transform, add the Philox Gumbel noise and write one candidate per row and tile.  A CTA whose
// wait runs out poisons its group's remaining candidates (row status 3).
#include <cuda.h>

#include "lms.h"
#include "lms_device.cuh"
#include "lms_kernels.h"
#include "tcgen05_common.cuh"

namespace lms {
namespace {

using namespace tc;

constexpr int kRgMaxStages = 8;
constexpr int kRgEpiWarps = 16;
constexpr int kRgRows = 256;                 // batch rows per group (MMA N)

struct RgParams {
    SampleArgs a;         // the whole launch: rows a.row0 .. a.row0 + a.B - 1
    int groups;           // G = ceil(a.B / 256), at most kMaxRowGroups
    int nk;               // K chunks of 64
    int stages;
    uint32_t stage_bytes;
    uint64_t timeout_ns;
    uint32_t debug_flags;
};

// Shared memory (offsets from a 1024-byte aligned base): the ring, barriers, then the epilogue's
// buffers (row parameters, per-column best keys, transposition tiles).
struct RgLayout {
    uint32_t stages_off, bars_off, misc_off, rows_off, red_off, tr_off, total;
    __host__ __device__ RgLayout(int stages, uint32_t stage_bytes) {
        stages_off = 0;
        bars_off = stages * stage_bytes;
        // full[S], empty[S], acc_full[2], acc_empty[2], drain
        misc_off = bars_off + (2 * stages + 5) * 8;
        rows_off = (misc_off + 16 + 15) & ~15u;   // misc: tmem slot, error flag
        red_off = rows_off + kRgRows * static_cast<uint32_t>(sizeof(RowParams));
        tr_off = red_off + kRgRows * 8;
        total = tr_off + kRgEpiWarps * kTrWarpBytes;
    }
};

// W is read by every group's CTAs within a short window, so its lines keep the normal L2 priority
// (the single-group kernel marks them evict-first).
__device__ __forceinline__ uint64_t l2_policy_evict_normal() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_normal.b64 %0, 1.0;" : "=l"(p));
    return p;
}

template <bool kWide, bool kPlain>
__global__ void __launch_bounds__(32 * (2 + kRgEpiWarps), 1)
    lmhead_tc_rows_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmH,
                          const RgParams prm) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_addr = smem_addr(smem_raw);
    const uint32_t base_addr = (raw_addr + 1023u) & ~1023u;
    uint8_t* base = smem_raw + (base_addr - raw_addr);
    const RgLayout L(prm.stages, prm.stage_bytes);

    // This CTA's group: rows row_off .. row_off + B - 1 of the launch, tiles t0, t0 + tstride, ...
    const int G = prm.groups;
    const int grp = static_cast<int>(blockIdx.x) % G;
    const int64_t row_off = static_cast<int64_t>(grp) * kRgRows;
    const int64_t t0 = blockIdx.x / G, tstride = gridDim.x / G;
    const int64_t nt = prm.a.n_tiles;
    SampleArgs a = prm.a;
    a.row0 += row_off;
    a.B = (prm.a.B - row_off < kRgRows) ? prm.a.B - row_off : kRgRows;
    a.cand_score += row_off * nt;
    a.cand_index += row_off * nt;
    const int S = prm.stages;
    const int n_pad = kRgRows;
    const int B = static_cast<int>(a.B);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    const uint32_t bar0 = base_addr + L.bars_off;
    auto full_bar = [&](int s) { return bar0 + 8u * s; };
    auto empty_bar = [&](int s) { return bar0 + 8u * (S + s); };
    auto accf_bar = [&](int ab) { return bar0 + 8u * (2 * S + ab); };
    auto acce_bar = [&](int ab) { return bar0 + 8u * (2 * S + 2 + ab); };
    const uint32_t drain_bar = bar0 + 8u * (2 * S + 4);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(base + L.misc_off);
    volatile int* err = reinterpret_cast<volatile int*>(base + L.misc_off + 4);
    RowParams* rows = reinterpret_cast<RowParams*>(base + L.rows_off);
    unsigned long long* red = reinterpret_cast<unsigned long long*>(base + L.red_off);

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(full_bar(s), 1);
            mbar_init(empty_bar(s), 1);
        }
        for (int ab = 0; ab < 2; ++ab) {
            mbar_init(accf_bar(ab), 1);
            mbar_init(acce_bar(ab), kRgEpiWarps);
        }
        mbar_init(drain_bar, 1);
        *err = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    }
    clear_status_bits(prm.a.status_bits, prm.a.row0);
    if (warp == 0 && lane == 0) {
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmW)) : "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmH)) : "memory");
    }
    for (int b = threadIdx.x; b < B; b += blockDim.x) {
        rows[b] = make_row_params(a.temperature, a.seeds, a.positions, a.base_seed, a.offset,
                                  a.row0 + b);
        red[b] = 0ull;
    }
    if (warp == 1) tmem_alloc(base_addr + L.misc_off, 2 * kRgRows);
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem_base = *tmem_slot;

    if (warp == 0) {
        // ---------------- TMA producer ----------------
        if (lane == 0) {
            const uint64_t pol_w = l2_policy_evict_normal();
            const uint64_t pol_h = l2_policy_evict_last();
            uint32_t issued = 0, issued_parity = 0;   // per-stage: load in flight, its phase
            int stage = 0;
            uint32_t phase = 0;
            bool first = true;
            for (int64_t tile = t0; tile < nt && *err == 0; tile += tstride) {
                for (int kc = 0; kc < prm.nk; ++kc) {
                    if (!mbar_wait(empty_bar(stage), phase ^ 1u, prm.timeout_ns, err)) {
                        *err = 1;
                        break;
                    }
                    const bool withhold = first && blockIdx.x == 0 &&
                                          (prm.debug_flags & LMS_DEBUG_WITHHOLD_FIRST_LOAD);
                    first = false;
                    if (!withhold) {
                        const uint32_t dst = base_addr + L.stages_off + stage * prm.stage_bytes;
                        mbar_arrive_expect_tx(full_bar(stage), prm.stage_bytes);
                        const int kx = kc * kBK;
                        tma_load_2d(dst, &tmW, kx, static_cast<int>(tile * kTileV), full_bar(stage), pol_w);
                        tma_load_2d(dst + kWStageBytes, &tmH, kx, static_cast<int>(a.row0), full_bar(stage),
                                    pol_h);
                        issued |= 1u << stage;
                        issued_parity = (issued_parity & ~(1u << stage)) | (phase << stage);
                    }
                    if (++stage == S) { stage = 0; phase ^= 1u; }
                }
            }
            // Drain: every copy this thread started must land before the CTA may exit.
            for (int s = 0; s < S; ++s)
                if (issued & (1u << s))
                    mbar_wait(full_bar(s), (issued_parity >> s) & 1u, prm.timeout_ns, nullptr);
        }
    } else if (warp == 1) {
        // ---------------- MMA issuer ----------------
        if (lane == 0) {
            const uint32_t idesc = mma_idesc_bf16(n_pad, kTileV);
            int stage = 0;
            uint32_t phase = 0;
            int i = 0;
            bool ok = true;
            for (int64_t tile = t0; tile < nt && ok; tile += tstride, ++i) {
                const int ab = i & 1;
                const uint32_t use_parity = (i >> 1) & 1;
                if (!mbar_wait(acce_bar(ab), use_parity ^ 1u, prm.timeout_ns, err)) { ok = false; break; }
                tc_fence_after_sync();
                const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(ab * n_pad);
                for (int kc = 0; kc < prm.nk; ++kc) {
                    if (!mbar_wait(full_bar(stage), phase, prm.timeout_ns, err)) { ok = false; break; }
                    tc_fence_after_sync();
                    const uint32_t sa = base_addr + L.stages_off + stage * prm.stage_bytes;
                    const uint64_t adesc = kmajor_sw128_desc(sa);
                    const uint64_t bdesc = kmajor_sw128_desc(sa + kWStageBytes);
#pragma unroll
                    for (int k = 0; k < 4; ++k)
                        mma_bf16(d_tmem, adesc + 2u * k, bdesc + 2u * k, idesc, (kc | k) != 0 ? 1u : 0u);
                    mma_commit(empty_bar(stage));
                    if (++stage == S) { stage = 0; phase ^= 1u; }
                }
                if (!ok) break;
                mma_commit(accf_bar(ab));
            }
            if (!ok) *err = 1;
            // Drain: all MMAs issued by this thread complete before TMEM is freed.
            mma_commit(drain_bar);
            mbar_wait(drain_bar, 0, prm.timeout_ns, nullptr);
        }
    } else {
        // ---------------- epilogue ----------------
        const int epi_tid = threadIdx.x - 64;
        const int epi_threads = 32 * kRgEpiWarps;
        const int quad = warp & 3;                       // TMEM lanes 32*quad .. 32*quad+31
        const int col_group = (warp - 2) >> 2;           // which column chunks this warp takes
        float* tr = reinterpret_cast<float*>(base + L.tr_off + (warp - 2) * kTrWarpBytes);
        int i = 0;
        bool ok = true;
        for (int64_t tile = t0; tile < nt; tile += tstride, ++i) {
            const int ab = i & 1;
            const uint32_t use_parity = (i >> 1) & 1;
            if (ok) ok = mbar_wait(accf_bar(ab), use_parity, prm.timeout_ns, err);
            ok = epi_barrier_and(epi_threads, ok);
            if (!ok) {
                // Poison this tile's candidates (and, through the loop, every later one).
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
            epilogue_tile_columns<kRgEpiWarps, kWide, kPlain>(a, rows, red, tr, t_row, tile, quad,
                                                              col_group, lane, B);
            // The accumulator buffer is free for the MMA of tile i+2.
            tc_fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(acce_bar(ab));
            epi_barrier(epi_threads);
            for (int b = epi_tid; b < B; b += epi_threads) {
                const unsigned long long key = red[b];
                red[b] = 0ull;                           // ready for the next tile
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
        tmem_dealloc(tmem_base, 2 * kRgRows);
    }
}

template <bool kWide, bool kPlain>
cudaError_t launch_rows_variant(const CUtensorMap& tmW, const CUtensorMap& tmH, const RgParams& prm,
                                size_t smem, int grid, cudaStream_t stream) {
    auto kern = lmhead_tc_rows_kernel<kWide, kPlain>;
    const cudaError_t e = ensure_dynamic_smem(reinterpret_cast<const void*>(kern), smem);
    if (e != cudaSuccess) return e;
    kern<<<grid, 32 * (2 + kRgEpiWarps), smem, stream>>>(tmW, tmH, prm);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_lmhead_tc_rows(const CUtensorMap& tmW, const CUtensorMap& tmH, int64_t D, bool wide,
                                  uint32_t timeout_ms, uint32_t debug_flags, const SampleArgs& a,
                                  cudaStream_t stream) {
    if (a.B <= kRgRows || a.B > static_cast<int64_t>(kMaxRowGroups) * kRgRows) return cudaErrorInvalidValue;
    RgParams prm;
    prm.a = a;
    prm.groups = static_cast<int>((a.B + kRgRows - 1) / kRgRows);
    prm.nk = static_cast<int>((D + kBK - 1) / kBK);
    prm.stage_bytes = static_cast<uint32_t>(kWStageBytes + kRgRows * kBK * 2);
    const uint32_t budget = 227u * 1024u - 1024u;   // opt-in maximum minus alignment slack
    const RgLayout fixed(0, prm.stage_bytes);
    int stages = static_cast<int>((budget - fixed.total - (2 * kRgMaxStages + 5) * 8) / prm.stage_bytes);
    if (stages > kRgMaxStages) stages = kRgMaxStages;
    if (stages < 2) return cudaErrorInvalidValue;
    prm.stages = stages;
    prm.timeout_ns = static_cast<uint64_t>(timeout_ms) * 1000000ull;
    prm.debug_flags = debug_flags;
    const RgLayout L(stages, prm.stage_bytes);
    const size_t smem = L.total + 1024;
    // a whole number of CTAs per group, at most one per SM
    const int sms = device_sm_count();
    const int64_t per_group = a.n_tiles < sms / prm.groups ? a.n_tiles : sms / prm.groups;
    const int grid = static_cast<int>(per_group) * prm.groups;
    if (grid < prm.groups) return cudaErrorInvalidValue;
    const bool plain = a.bias == nullptr && a.mask == nullptr;
    if (plain)
        return wide ? launch_rows_variant<true, true>(tmW, tmH, prm, smem, grid, stream)
                    : launch_rows_variant<false, true>(tmW, tmH, prm, smem, grid, stream);
    return wide ? launch_rows_variant<true, false>(tmW, tmH, prm, smem, grid, stream)
                : launch_rows_variant<false, false>(tmW, tmH, prm, smem, grid, stream);
}

}  // namespace lms
