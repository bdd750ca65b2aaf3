// Fused LM-head + Gumbel-max Stage 1 on the 5th-generation tensor cores (sm_103a).
//
// FlashSampling ("method step details", Stage 1): for each vocabulary tile, compute
// Y = H W^T on chip (step 1), transform it (step 2), add Gumbel noise (steps 3-4), keep the
// per-row (max, index) (step 5) and write that candidate (step 6).  The logits never reach
// memory.
//
// Design for GB300 (one persistent CTA per SM, warp-specialised):
//   warp 0      TMA producer: W[128 x 64] and H[n_pad x 64] bf16 chunks, 128-byte swizzle, into an
//               S-stage shared-memory ring guarded by mbarriers (no multicast).
//   warp 1      allocates TMEM; one lane issues tcgen05.mma (kind::f16, bf16 x bf16 -> fp32) with
//               "swap-AB": M = 128 vocabulary rows of W, N = n_pad batch rows of H, K = 16 per
//               instruction, into one of two TMEM accumulators [128 lanes x n_pad columns].
//   warps 2..   epilogue (kEpilogueWarps, a multiple of 4): tcgen05.ld the accumulator (thread = one vocabulary row,
//               registers = batch columns), apply bias / mask / temperature, run Philox and the
//               noise per element, reduce the argmax over the 128 rows (16 columns at a time
//               across the 32 lanes, then across the 4 lane quadrants in shared memory), write
//               one candidate per batch row.
// The double-buffered accumulator lets the epilogue of tile i overlap the loads and MMAs of
// tile i+1.  Every mbarrier wait is bounded in time; a CTA whose wait runs out flags the error,
// drains its in-flight copies and MMAs, poisons its remaining candidates (index -2, reported
// as row status 3 by Stage 2), frees TMEM and exits.
#include <cuda.h>

#include "lms.h"
#include "lms_device.cuh"
#include "lms_kernels.h"
#include "tcgen05_common.cuh"

namespace lms {
namespace {

using namespace tc;
// At most 8 stages in flight per SM: more lets each SM keep more W loads outstanding, which
// measured slower on GB300 (Qwen3-8B shape, B = 1: 194.9 us with 11 stages, 188.8 with 10, 186.4
// with 8, 189.4 with 6; B = 64 takes 8 either way).
constexpr int kMaxStages = 8;
#ifndef LMS_TC_EPILOGUE_WARPS
#define LMS_TC_EPILOGUE_WARPS 16
#endif
// Epilogue warps: a multiple of 4 (each TMEM lane quadrant gets the same number of warps, which
// split the batch columns between them).
constexpr int kEpilogueWarps = LMS_TC_EPILOGUE_WARPS;
static_assert(kEpilogueWarps % 4 == 0, "epilogue warps come in groups of four");

struct TcParams {
    SampleArgs a;
    int nk;              // number of K chunks, ceil(D / 64)
    int n_pad;           // MMA N: batch rows padded to a multiple of 16 (16..256)
    int stages;
    uint32_t stage_bytes;
    uint32_t tmem_cols;
    uint64_t timeout_ns;
    uint32_t debug_flags;
};

// ------------------------------------------------------------------------------------------
// Shared-memory layout (offsets from a 1024-byte aligned base)
// ------------------------------------------------------------------------------------------
struct SmemLayout {
    uint32_t stages_off, bars_off, misc_off, rows_off, red_off, tr_off, run_off, total;
    // Gumbel-top-k only: run_keys 64-bit keys (per TMEM quadrant and batch column, the threshold
    // key of the per-tile lists, or the whole running list)
    __host__ __device__ SmemLayout(int stages, uint32_t stage_bytes, int n_pad, int epi_warps,
                                   uint32_t run_keys = 0) {
        stages_off = 0;
        bars_off = stages * stage_bytes;
        // full[S], empty[S], acc_full[2], acc_empty[2], drain
        misc_off = bars_off + (2 * stages + 5) * 8;
        rows_off = (misc_off + 16 + 15) & ~15u;   // misc: tmem slot, error flag
        red_off = rows_off + n_pad * static_cast<uint32_t>(sizeof(RowParams));
        tr_off = red_off + n_pad * 8;
        run_off = tr_off + epi_warps * kTrWarpBytes;
        total = run_off + run_keys * 8u;
    }
};

// Gumbel-top-k keys in shared memory: the per-tile lists' thresholds (4 n_pad keys) or the running
// lists (4 n_pad k keys).
__host__ __device__ inline uint32_t topk_run_keys(int mode, int n_pad, int k) {
    return mode == 0 ? 0u : static_cast<uint32_t>(4 * n_pad) * (mode == kTopKRunning ? static_cast<uint32_t>(k) : 1u);
}

// kTopK: 0 = the race; kTopKTileLists = Gumbel-top-k with per-tile lists; kTopKRunning = with
// running lists in shared memory.
template <int kEpiWarps, bool kWide, bool kFp8, int kTopK, bool kPlain>
__global__ void __launch_bounds__(32 * (2 + kEpiWarps), 1)
    lmhead_tc_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmH,
                     const TcParams prm) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_addr = smem_addr(smem_raw);
    const uint32_t base_addr = (raw_addr + 1023u) & ~1023u;
    uint8_t* base = smem_raw + (base_addr - raw_addr);
    const SmemLayout L(prm.stages, prm.stage_bytes, prm.n_pad, kEpiWarps,
                       topk_run_keys(kTopK, prm.n_pad, prm.a.topk));

    const SampleArgs& a = prm.a;
    const int S = prm.stages;
    const int n_pad = prm.n_pad;
    const int B = static_cast<int>(a.B);
    const int64_t nt = a.n_tiles;
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
    // per batch column: the best (score, index) of the tile so far, as one ordered 64-bit key
    unsigned long long* red = reinterpret_cast<unsigned long long*>(base + L.red_off);

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(full_bar(s), 1);
            mbar_init(empty_bar(s), 1);
        }
        for (int ab = 0; ab < 2; ++ab) {
            mbar_init(accf_bar(ab), 1);
            mbar_init(acce_bar(ab), kEpiWarps);
        }
        mbar_init(drain_bar, 1);
        *err = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    }
    clear_status_bits(a.status_bits, a.row0);
    if (warp == 0 && lane == 0) {
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmW)) : "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmH)) : "memory");
    }
    for (int b = threadIdx.x; b < B; b += blockDim.x) {
        rows[b] = make_row_params(a.temperature, a.seeds, a.positions, a.base_seed, a.offset,
                                  a.row0 + b);
        red[b] = 0ull;
    }
    if constexpr (kTopK != 0) {
        unsigned long long* run = reinterpret_cast<unsigned long long*>(base + L.run_off);
        const int run_keys = static_cast<int>(topk_run_keys(kTopK, n_pad, a.topk));
        for (int i = threadIdx.x; i < run_keys; i += blockDim.x) run[i] = 0ull;
    }
    if (warp == 1) tmem_alloc(base_addr + L.misc_off, prm.tmem_cols);
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem_base = *tmem_slot;

    if (warp == 0) {
        // ---------------- TMA producer ----------------
        if (lane == 0) {
            const uint64_t pol_w = l2_policy_evict_first();
            const uint64_t pol_h = l2_policy_evict_last();
            uint32_t issued = 0, issued_parity = 0;   // per-stage: load in flight, its phase
            int stage = 0;
            uint32_t phase = 0;
            bool first = true;
            // FP8 inputs: H8 is written by the quantisation kernel this launch overlaps.  The W
            // loads do not depend on it, so the first stages of the ring are filled with W before
            // the wait, and their H loads (each stage's barrier expects both) follow it.
            bool h_ready = !kFp8;
            uint32_t h_pending = 0;                   // stages whose H load waits for the quantiser
            int h_kx[kMaxStages];
            auto release_h = [&]() {
                pdl_wait_primary();
                for (int s = 0; s < S; ++s)
                    if (h_pending & (1u << s))
                        tma_load_2d(base_addr + L.stages_off + s * prm.stage_bytes + kWStageBytes, &tmH,
                                    h_kx[s], static_cast<int>(a.row0), full_bar(s), pol_h);
                h_pending = 0;
                h_ready = true;
            };
            for (int64_t tile = blockIdx.x; tile < nt && *err == 0; tile += gridDim.x) {
                for (int kc = 0; kc < prm.nk; ++kc) {
                    if (!h_ready && (h_pending & (1u << stage))) release_h();   // the ring is full
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
                        // one stage is 128 bytes of K: 64 bf16 or 128 E4M3 elements
                        const int kx = kc * (kFp8 ? 2 * kBK : kBK);
                        tma_load_2d(dst, &tmW, kx, static_cast<int>(tile * kTileV),
                                    full_bar(stage), pol_w);
                        if (h_ready) {
                            tma_load_2d(dst + kWStageBytes, &tmH, kx, static_cast<int>(a.row0),
                                        full_bar(stage), pol_h);
                        } else {
                            h_kx[stage] = kx;
                            h_pending |= 1u << stage;
                        }
                        issued |= 1u << stage;
                        issued_parity = (issued_parity & ~(1u << stage)) | (phase << stage);
                    }
                    if (++stage == S) { stage = 0; phase ^= 1u; }
                }
            }
            if (!h_ready) release_h();               // fewer loads than stages, or an error
            // Drain: every copy this thread started must land before the CTA may exit.
            for (int s = 0; s < S; ++s)
                if (issued & (1u << s))
                    mbar_wait(full_bar(s), (issued_parity >> s) & 1u, prm.timeout_ns, nullptr);
        }
    } else if (warp == 1) {
        // ---------------- MMA issuer ----------------
        if (lane == 0) {
            const uint32_t idesc = kFp8 ? mma_idesc_e4m3(n_pad, kTileV) : mma_idesc_bf16(n_pad, kTileV);
            int stage = 0;
            uint32_t phase = 0;
            int i = 0;
            bool ok = true;
            for (int64_t tile = blockIdx.x; tile < nt && ok; tile += gridDim.x, ++i) {
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
                    for (int k = 0; k < 4; ++k) {
                        // advance 32 bytes along K inside the swizzle atom (16 bf16 / 32 E4M3)
                        if (kFp8)
                            mma_e4m3(d_tmem, adesc + 2u * k, bdesc + 2u * k, idesc, (kc | k) != 0 ? 1u : 0u);
                        else
                            mma_bf16(d_tmem, adesc + 2u * k, bdesc + 2u * k, idesc, (kc | k) != 0 ? 1u : 0u);
                    }
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
        if (kFp8) pdl_wait_primary();   // the activation exponents come from the quantisation kernel
        const int epi_threads = 32 * kEpiWarps;
        const int quad = warp & 3;                       // TMEM lanes 32*quad .. 32*quad+31
        const int col_group = (warp - 2) >> 2;           // which column chunks this warp takes
        float* tr = reinterpret_cast<float*>(base + L.tr_off + (warp - 2) * kTrWarpBytes);
        int i = 0;
        bool ok = true;
        for (int64_t tile = blockIdx.x; tile < nt; tile += gridDim.x, ++i) {
            const int ab = i & 1;
            const uint32_t use_parity = (i >> 1) & 1;
            if (ok) ok = mbar_wait(accf_bar(ab), use_parity, prm.timeout_ns, err);
            ok = epi_barrier_and(epi_threads, ok);
            if (!ok) {
                // Poison this tile's candidates (and, through the loop, every later one); running
                // lists are poisoned by their owners when they publish them after the loop
                if (epi_tid == 0) *err = 1;
                for (int b = epi_tid; b < B && kTopK != kTopKRunning; b += epi_threads) {
                    if constexpr (kTopK == kTopKTileLists) {
                        for (int r = 0; r < 4 * a.topk; ++r)
                            a.cand_keys[(b * nt + tile) * 4 * a.topk + r] = kPoisonKey;
                    } else {
                        a.cand_score[b * nt + tile] = -CUDART_INF_F;
                        a.cand_index[b * nt + tile] = kPoisonIndex;
                    }
                }
                continue;
            }
            tc_fence_after_sync();
            const uint32_t t_row = tmem_base + (static_cast<uint32_t>(32 * quad) << 16) +
                                   static_cast<uint32_t>(ab * n_pad);
            if constexpr (kTopK == kTopKRunning) {
                unsigned long long* run = reinterpret_cast<unsigned long long*>(base + L.run_off);
                epilogue_tile_topk_running<kEpiWarps, kWide, kPlain>(a, rows, tr, run, n_pad, t_row,
                                                                     tile, quad, col_group, lane, B);
            } else if constexpr (kTopK == kTopKTileLists) {
                unsigned long long* thr = reinterpret_cast<unsigned long long*>(base + L.run_off);
                epilogue_tile_topk<kEpiWarps, kWide, kPlain>(a, rows, tr, thr, n_pad, t_row, tile,
                                                             quad, col_group, lane, B);
            } else {
                epilogue_tile_columns<kEpiWarps, kWide, kPlain>(a, rows, red, tr, t_row, tile, quad,
                                                                col_group, lane, B);
            }
            // The accumulator buffer is free for the MMA of tile i+2.
            tc_fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(acce_bar(ab));
            if constexpr (kTopK == 0) {
                epi_barrier(epi_threads);
                for (int b = epi_tid; b < B; b += epi_threads) {
                    const unsigned long long key = red[b];
                    red[b] = 0ull;                       // ready for the next tile
                    const float s = unpack_score(key);
                    a.cand_score[b * nt + tile] = s;
                    a.cand_index[b * nt + tile] = candidate_index(s, unpack_index(key));
                }
                epi_barrier(epi_threads);
            }
        }
        if constexpr (kTopK == kTopKRunning) {
            const unsigned long long* run = reinterpret_cast<const unsigned long long*>(base + L.run_off);
            topk_running_lists_publish<kEpiWarps>(a, run, n_pad, quad, col_group, lane, B, ok);
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

template <int kEpiWarps, bool kWide, bool kFp8, int kTopK = 0, bool kPlain = false>
cudaError_t launch_variant(const CUtensorMap& tmW, const CUtensorMap& tmH, const TcParams& prm,
                           size_t smem, int grid, cudaStream_t stream) {
    auto kern = lmhead_tc_kernel<kEpiWarps, kWide, kFp8, kTopK, kPlain>;
    cudaError_t e = ensure_dynamic_smem(reinterpret_cast<const void*>(kern), smem);
    if (e != cudaSuccess) return e;
    if (!kFp8) {
        kern<<<grid, 32 * (2 + kEpiWarps), smem, stream>>>(tmW, tmH, prm);
        return cudaGetLastError();
    }
    // FP8: a programmatic dependent of the activation quantisation, so the prologue (barriers,
    // TMEM, descriptor prefetch) overlaps it; the roles that read its output wait for it.
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(32 * (2 + kEpiWarps));
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, tmW, tmH, prm);
}

}  // namespace

cudaError_t launch_lmhead_tc(const CUtensorMap& tmW, const CUtensorMap& tmH, int64_t D, int n_pad,
                             bool wide, uint32_t timeout_ms, uint32_t debug_flags,
                             const SampleArgs& a, cudaStream_t stream, bool fp8) {
    TcParams prm;
    prm.a = a;
    const int64_t k_per_stage = fp8 ? 2 * kBK : kBK;
    prm.nk = static_cast<int>((D + k_per_stage - 1) / k_per_stage);
    prm.n_pad = n_pad;
    prm.stage_bytes = static_cast<uint32_t>(kWStageBytes + n_pad * kBK * 2);
    const uint32_t budget = 227u * 1024u - 1024u;   // opt-in maximum minus alignment slack
    const int topk_mode = a.topk > 0 ? a.topk_mode : 0;
    const uint32_t run_keys = topk_run_keys(topk_mode, n_pad, a.topk);
    const SmemLayout fixed(0, prm.stage_bytes, n_pad, kEpilogueWarps, run_keys);
    int stages = static_cast<int>((budget - fixed.total - (2 * kMaxStages + 5) * 8) / prm.stage_bytes);
    if (stages > kMaxStages) stages = kMaxStages;
    if (stages < 2) return cudaErrorInvalidValue;
    prm.stages = stages;
    uint32_t cols = 32;
    while (cols < static_cast<uint32_t>(2 * n_pad)) cols <<= 1;
    prm.tmem_cols = cols;
    prm.timeout_ns = static_cast<uint64_t>(timeout_ms) * 1000000ull;
    prm.debug_flags = debug_flags;
    const SmemLayout L(stages, prm.stage_bytes, n_pad, kEpilogueWarps, run_keys);
    const size_t smem = L.total + 1024;
    int sms = device_sm_count();
    int grid = static_cast<int>(a.n_tiles < sms ? a.n_tiles : sms);
    // no bias and no mask: the epilogues without per-entry bias, mask and bounds tests
    const bool plain = a.bias == nullptr && a.mask == nullptr;
    if (a.topk > 0) {
        if (fp8 || a.topk > kMaxTopK || a.cand_keys == nullptr) return cudaErrorInvalidValue;
        if (topk_mode == kTopKRunning) {
            if (plain)
                return wide ? launch_variant<kEpilogueWarps, true, false, kTopKRunning, true>(tmW, tmH, prm, smem, grid, stream)
                            : launch_variant<kEpilogueWarps, false, false, kTopKRunning, true>(tmW, tmH, prm, smem, grid, stream);
            return wide ? launch_variant<kEpilogueWarps, true, false, kTopKRunning>(tmW, tmH, prm, smem, grid, stream)
                        : launch_variant<kEpilogueWarps, false, false, kTopKRunning>(tmW, tmH, prm, smem, grid, stream);
        }
        if (topk_mode != kTopKTileLists) return cudaErrorInvalidValue;
        if (plain)
            return wide ? launch_variant<kEpilogueWarps, true, false, kTopKTileLists, true>(tmW, tmH, prm, smem, grid, stream)
                        : launch_variant<kEpilogueWarps, false, false, kTopKTileLists, true>(tmW, tmH, prm, smem, grid, stream);
        return wide ? launch_variant<kEpilogueWarps, true, false, kTopKTileLists>(tmW, tmH, prm, smem, grid, stream)
                    : launch_variant<kEpilogueWarps, false, false, kTopKTileLists>(tmW, tmH, prm, smem, grid, stream);
    }
    if (fp8) {
        if (plain)
            return wide ? launch_variant<kEpilogueWarps, true, true, false, true>(tmW, tmH, prm, smem, grid, stream)
                        : launch_variant<kEpilogueWarps, false, true, false, true>(tmW, tmH, prm, smem, grid, stream);
        return wide ? launch_variant<kEpilogueWarps, true, true>(tmW, tmH, prm, smem, grid, stream)
                    : launch_variant<kEpilogueWarps, false, true>(tmW, tmH, prm, smem, grid, stream);
    }
    if (plain)
        return wide ? launch_variant<kEpilogueWarps, true, false, false, true>(tmW, tmH, prm, smem, grid, stream)
                    : launch_variant<kEpilogueWarps, false, false, false, true>(tmW, tmH, prm, smem, grid, stream);
    return wide ? launch_variant<kEpilogueWarps, true, false>(tmW, tmH, prm, smem, grid, stream)
                : launch_variant<kEpilogueWarps, false, false>(tmW, tmH, prm, smem, grid, stream);
}

}  // namespace lms
