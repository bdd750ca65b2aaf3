// Fused LM-head + Gumbel-max Stage 1 on a CTA pair: tcgen05.mma.cta_group::2, M = 256.
//
// The same method as lmhead_tc.cu (FlashSampling "method step details", Stage 1 steps 1-6), with
// two CTAs of a cluster sharing each MMA.  Each CTA streams its own 128 rows of a 256-row
// vocabulary tile of W and HALF of the batch rows of H; the leader CTA (rank 0) issues
// tcgen05.mma.cta_group::2 with M = 256 and N = n_pad, whose D lands in both CTAs' TMEM (128 rows
// x n_pad columns each).  Per SM this halves the L2 traffic of H, which for large batches is
// re-read for every vocabulary tile, and frees shared memory for a deeper load pipeline.
// Measured on GB300 it is nonetheless slower than the single-CTA kernel at every batch size tried
// (the pair's coupling costs more than the saved H traffic), so it is an explicit path only.
//
// Synchronisation, every wait bounded in time:
//   full[s]       local; the CTA's own TMA completes on it (so each producer can drain its own
//                 copies on every exit path).
//   peer_full[s]  leader only; the peer's forwarder (its warp 1) arrives on it remotely once the
//                 peer's full[s] completes.  The leader's MMA waits on full[s] and peer_full[s].
//   empty[s]      local in both; the leader's tcgen05.commit multicasts to both CTAs.
//   acc_full[ab]  local in both; multicast commit after a tile's last MMA.
//   acc_empty[ab] leader only; both CTAs' epilogue warps arrive (the peer's remotely).
// A cluster barrier follows barrier initialisation and precedes TMEM deallocation; every path to
// it is bounded, so both CTAs always reach it.
#include <cuda.h>

#include "lms.h"
#include "lms_device.cuh"
#include "lms_kernels.h"
#include "tcgen05_common.cuh"

namespace lms {
namespace {

using namespace tc;

constexpr int kPairEpiWarps = 16;
constexpr int kPairMaxStages = 12;

struct PairParams {
    SampleArgs a;
    int nk;               // K chunks, ceil(D / 64)
    int n_pad;            // MMA N over both CTAs: batch rows padded to a multiple of 16 (16..256)
    int stages;
    uint32_t stage_bytes; // W 16 KB + (n_pad / 2) * 128 bytes of H
    uint32_t tmem_cols;
    uint64_t timeout_ns;
    uint32_t debug_flags;
};

__device__ __forceinline__ uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

__device__ __forceinline__ uint32_t cluster_index() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%clusterid.x;" : "=r"(r));
    return r;
}

__device__ __forceinline__ uint32_t cluster_count() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%nclusterid.x;" : "=r"(r));
    return r;
}

// The shared::cluster address of `addr` (a shared::cta address) in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t map_shared(uint32_t addr, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
    return r;
}

// Relaxed remote arrive for the forwarder: the data it announces was written by the TMA and its
// completion already observed on the peer's own barrier, so the arrive orders nothing of this
// thread's; a release at cluster scope here measured ~1 us per arrive and serialised the ring.
__device__ __forceinline__ void mbar_arrive_cluster_relaxed(uint32_t cluster_addr) {
    asm volatile("mbarrier.arrive.relaxed.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive_cluster(uint32_t cluster_addr) {
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait_acq_cluster(uint32_t bar, uint32_t parity) {
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(bar), "r"(parity)
        : "memory");
    return done != 0;
}

// mbar_wait with cluster-scope acquire (the barrier receives arrivals from the other CTA).
__device__ __forceinline__ bool mbar_wait_cl(uint32_t bar, uint32_t parity, uint64_t timeout_ns,
                                             const volatile int* err) {
    if (mbar_try_wait_acq_cluster(bar, parity)) return true;
    const uint64_t deadline = global_timer_ns() + timeout_ns;
    for (uint32_t spin = 1;; ++spin) {
        if (mbar_try_wait_acq_cluster(bar, parity)) return true;
        if ((spin & 31u) == 0u) {
            if (err != nullptr && *err != 0) return false;
            if (global_timer_ns() > deadline) return false;
        }
    }
}

__device__ __forceinline__ void cluster_sync_all() {
    asm volatile("barrier.cluster.arrive.release;" ::: "memory");
    asm volatile("barrier.cluster.wait.acquire;" ::: "memory");
}

__device__ __forceinline__ void tmem_alloc_pair(uint32_t slot, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(slot),
                 "r"(ncols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
                 : "memory");
}

// D[tmem of both CTAs] (+)= A[smem, 128 rows per CTA] * B[smem, n/2 rows per CTA]^T.
__device__ __forceinline__ void mma_pair_bf16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                              uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Arrive once, on the barrier at this offset in every CTA of `mask`, when the pair's MMAs issued
// so far by this thread have completed.
__device__ __forceinline__ void mma_pair_commit_multicast(uint32_t bar, uint16_t mask) {
    asm volatile(
        "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64"
        " [%0], %1;" ::"r"(bar),
        "h"(mask)
        : "memory");
}

struct PairLayout {
    uint32_t stages_off, bars_off, misc_off, rows_off, red_off, tr_off, total;
    __host__ __device__ PairLayout(int stages, uint32_t stage_bytes, int n_pad) {
        stages_off = 0;
        bars_off = stages * stage_bytes;
        // full[S], empty[S], peer_full[S], acc_full[2], acc_empty[2], drain
        misc_off = bars_off + (3 * stages + 5) * 8;
        rows_off = (misc_off + 16 + 15) & ~15u;
        red_off = rows_off + n_pad * static_cast<uint32_t>(sizeof(RowParams));
        tr_off = red_off + n_pad * 8;
        total = tr_off + kPairEpiWarps * kTrWarpBytes;
    }
};

template <bool kWide>
__global__ void __launch_bounds__(32 * (2 + kPairEpiWarps), 1)
    lmhead_tc_pair_kernel(const __grid_constant__ CUtensorMap tmW,
                          const __grid_constant__ CUtensorMap tmH, const PairParams prm) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_addr = smem_addr(smem_raw);
    const uint32_t base_addr = (raw_addr + 1023u) & ~1023u;
    uint8_t* base = smem_raw + (base_addr - raw_addr);
    const PairLayout L(prm.stages, prm.stage_bytes, prm.n_pad);

    const SampleArgs& a = prm.a;
    const int S = prm.stages;
    const int n_pad = prm.n_pad;
    const int B = static_cast<int>(a.B);
    const int64_t nt = a.n_tiles;
    const int64_t n_super = (nt + 1) / 2;          // 256-row tiles
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t rank = cluster_rank();          // 0: leader (issues the MMAs), 1: peer
    const int64_t cid = cluster_index();
    const int64_t ncl = cluster_count();

    const uint32_t bar0 = base_addr + L.bars_off;
    auto full_bar = [&](int s) { return bar0 + 8u * s; };
    auto empty_bar = [&](int s) { return bar0 + 8u * (S + s); };
    auto peer_full_bar = [&](int s) { return bar0 + 8u * (2 * S + s); };
    auto accf_bar = [&](int ab) { return bar0 + 8u * (3 * S + ab); };
    auto acce_bar = [&](int ab) { return bar0 + 8u * (3 * S + 2 + ab); };
    const uint32_t drain_bar = bar0 + 8u * (3 * S + 4);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(base + L.misc_off);
    volatile int* err = reinterpret_cast<volatile int*>(base + L.misc_off + 4);
    RowParams* rows = reinterpret_cast<RowParams*>(base + L.rows_off);
    unsigned long long* red = reinterpret_cast<unsigned long long*>(base + L.red_off);

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(full_bar(s), 1);
            mbar_init(empty_bar(s), 1);
            mbar_init(peer_full_bar(s), 1);
        }
        for (int ab = 0; ab < 2; ++ab) {
            mbar_init(accf_bar(ab), 1);
            mbar_init(acce_bar(ab), 2 * kPairEpiWarps);
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
    if (warp == 1) tmem_alloc_pair(base_addr + L.misc_off, prm.tmem_cols);
    tc_fence_before_sync();
    __syncthreads();
    cluster_sync_all();        // both CTAs' barriers exist before any remote arrive
    tc_fence_after_sync();
    const uint32_t tmem_base = *tmem_slot;

    if (warp == 0) {
        // ---------------- TMA producer (both CTAs) ----------------
        if (lane == 0) {
            const uint64_t pol_w = l2_policy_evict_first();
            const uint64_t pol_h = l2_policy_evict_last();
            uint32_t issued = 0, issued_parity = 0;
            int stage = 0;
            uint32_t phase = 0;
            bool first = true;
            const int h_row0 = static_cast<int>(a.row0) + static_cast<int>(rank) * (n_pad / 2);
            for (int64_t st = cid; st < n_super && *err == 0; st += ncl) {
                const int64_t tile = 2 * st + rank;
                for (int kc = 0; kc < prm.nk; ++kc) {
                    if (!mbar_wait_cl(empty_bar(stage), phase ^ 1u, prm.timeout_ns, err)) {
                        *err = 1;
                        break;
                    }
                    const bool withhold = first && cid == 0 && rank == 0 &&
                                          (prm.debug_flags & LMS_DEBUG_WITHHOLD_FIRST_LOAD);
                    first = false;
                    if (!withhold) {
                        const uint32_t dst = base_addr + L.stages_off + stage * prm.stage_bytes;
                        mbar_arrive_expect_tx(full_bar(stage), prm.stage_bytes);
                        tma_load_2d(dst, &tmW, kc * kBK, static_cast<int>(tile * kTileV),
                                    full_bar(stage), pol_w);
                        tma_load_2d(dst + kWStageBytes, &tmH, kc * kBK, h_row0, full_bar(stage), pol_h);
                        issued |= 1u << stage;
                        issued_parity = (issued_parity & ~(1u << stage)) | (phase << stage);
                    }
                    if (++stage == S) { stage = 0; phase ^= 1u; }
                }
            }
            for (int s = 0; s < S; ++s)
                if (issued & (1u << s))
                    mbar_wait(full_bar(s), (issued_parity >> s) & 1u, prm.timeout_ns, nullptr);
        }
    } else if (warp == 1) {
        if (lane == 0 && rank == 1) {
            // ---------------- forwarder (peer): "my half of stage s has landed" ----------------
            int stage = 0;
            uint32_t phase = 0;
            bool ok = true;
            for (int64_t st = cid; st < n_super && ok; st += ncl) {
                for (int kc = 0; kc < prm.nk; ++kc) {
                    if (!mbar_wait(full_bar(stage), phase, prm.timeout_ns, err)) { ok = false; break; }
                    mbar_arrive_cluster_relaxed(map_shared(peer_full_bar(stage), 0));
                    if (++stage == S) { stage = 0; phase ^= 1u; }
                }
            }
            if (!ok) *err = 1;
        } else if (lane == 0) {
            // ---------------- MMA issuer (leader) ----------------
            const uint32_t idesc = mma_idesc_bf16(n_pad, 2 * kTileV);
            int stage = 0;
            uint32_t phase = 0;
            int i = 0;
            bool ok = true;
            for (int64_t st = cid; st < n_super && ok; st += ncl, ++i) {
                const int ab = i & 1;
                const uint32_t use_parity = (i >> 1) & 1;
                if (!mbar_wait_cl(acce_bar(ab), use_parity ^ 1u, prm.timeout_ns, err)) { ok = false; break; }
                tc_fence_after_sync();
                const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(ab * n_pad);
                for (int kc = 0; kc < prm.nk; ++kc) {
                    if (!mbar_wait(full_bar(stage), phase, prm.timeout_ns, err) ||
                        !mbar_wait_cl(peer_full_bar(stage), phase, prm.timeout_ns, err)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after_sync();
                    const uint32_t sa = base_addr + L.stages_off + stage * prm.stage_bytes;
                    const uint64_t adesc = kmajor_sw128_desc(sa);
                    const uint64_t bdesc = kmajor_sw128_desc(sa + kWStageBytes);
#pragma unroll
                    for (int k = 0; k < kBK / 16; ++k)
                        mma_pair_bf16(d_tmem, adesc + 2u * k, bdesc + 2u * k, idesc, (kc | k) != 0 ? 1u : 0u);
                    mma_pair_commit_multicast(empty_bar(stage), 0x3);
                    if (++stage == S) { stage = 0; phase ^= 1u; }
                }
                if (!ok) break;
                mma_pair_commit_multicast(accf_bar(ab), 0x3);
            }
            if (!ok) *err = 1;
            // every MMA of the pair completes before either CTA frees its TMEM
            mma_pair_commit_multicast(drain_bar, 0x1);
            mbar_wait(drain_bar, 0, prm.timeout_ns, nullptr);
        }
    } else {
        // ---------------- epilogue (both CTAs, own TMEM rows) ----------------
        const int epi_tid = threadIdx.x - 64;
        const int epi_threads = 32 * kPairEpiWarps;
        const int quad = warp & 3;
        const int col_group = (warp - 2) >> 2;
        float* tr = reinterpret_cast<float*>(base + L.tr_off + (warp - 2) * kTrWarpBytes);
        const uint32_t acce_leader0 = map_shared(acce_bar(0), 0);
        const uint32_t acce_leader1 = map_shared(acce_bar(1), 0);
        int i = 0;
        bool ok = true;
        for (int64_t st = cid; st < n_super; st += ncl, ++i) {
            const int64_t tile = 2 * st + rank;
            const int ab = i & 1;
            const uint32_t use_parity = (i >> 1) & 1;
            if (ok) ok = mbar_wait_cl(accf_bar(ab), use_parity, prm.timeout_ns, err);
            ok = epi_barrier_and(epi_threads, ok);
            if (!ok) {
                if (epi_tid == 0) *err = 1;
                if (tile < nt)
                    for (int b = epi_tid; b < B; b += epi_threads) {
                        a.cand_score[b * nt + tile] = -CUDART_INF_F;
                        a.cand_index[b * nt + tile] = kPoisonIndex;
                    }
                continue;
            }
            tc_fence_after_sync();
            const uint32_t t_row = tmem_base + (static_cast<uint32_t>(32 * quad) << 16) +
                                   static_cast<uint32_t>(ab * n_pad);
            epilogue_tile_columns<kPairEpiWarps, kWide>(a, rows, red, tr, t_row, tile, quad,
                                                        col_group, lane, B);
            tc_fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive_cluster(ab ? acce_leader1 : acce_leader0);
            epi_barrier(epi_threads);
            for (int b = epi_tid; b < B; b += epi_threads) {
                const unsigned long long key = red[b];
                red[b] = 0ull;
                if (tile < nt) {
                    const float s = unpack_score(key);
                    a.cand_score[b * nt + tile] = s;
                    a.cand_index[b * nt + tile] = candidate_index(s, unpack_index(key));
                }
            }
            epi_barrier(epi_threads);
        }
    }

    pdl_launch_dependents();
    tc_fence_before_sync();
    __syncthreads();
    cluster_sync_all();        // no CTA frees TMEM or exits while its pair may still touch it
    tc_fence_after_sync();
    if (warp == 1) {
        __syncwarp();
        tmem_dealloc_pair(tmem_base, prm.tmem_cols);
    }
}

template <bool kWide>
cudaError_t launch_pair_variant(const CUtensorMap& tmW, const CUtensorMap& tmH, const PairParams& prm,
                                size_t smem, int64_t n_super, cudaStream_t stream) {
    auto kern = lmhead_tc_pair_kernel<kWide>;
    cudaError_t e = ensure_dynamic_smem(reinterpret_cast<const void*>(kern), smem);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.blockDim = dim3(32 * (2 + kPairEpiWarps));
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    // as many pairs as can be resident at once (the kernel is persistent), at most one per tile
    cfg.gridDim = dim3(2 * static_cast<unsigned>(device_sm_count() / 2));
    int max_clusters = 0;
    e = cudaOccupancyMaxActiveClusters(&max_clusters, kern, &cfg);
    if (e != cudaSuccess) return e;
    if (max_clusters < 1) return cudaErrorInvalidConfiguration;
    const int64_t clusters = n_super < max_clusters ? n_super : max_clusters;
    cfg.gridDim = dim3(2 * static_cast<unsigned>(clusters));
    return cudaLaunchKernelEx(&cfg, kern, tmW, tmH, prm);
}

}  // namespace

cudaError_t launch_lmhead_tc_pair(const CUtensorMap& tmW, const CUtensorMap& tmH, int64_t D,
                                  int n_pad, bool wide, uint32_t timeout_ms, uint32_t debug_flags,
                                  const SampleArgs& a, cudaStream_t stream) {
    PairParams prm;
    prm.a = a;
    prm.nk = static_cast<int>((D + kBK - 1) / kBK);
    prm.n_pad = n_pad;
    prm.stage_bytes = static_cast<uint32_t>(kWStageBytes + (n_pad / 2) * kBK * 2);
    const uint32_t budget = 227u * 1024u - 1024u;
    const PairLayout fixed(0, prm.stage_bytes, n_pad);
    int stages = static_cast<int>((budget - fixed.total - 3 * kPairMaxStages * 8) / prm.stage_bytes);
    if (stages > kPairMaxStages) stages = kPairMaxStages;
    if (stages < 2) return cudaErrorInvalidValue;
    prm.stages = stages;
    uint32_t cols = 32;
    while (cols < static_cast<uint32_t>(2 * n_pad)) cols <<= 1;
    prm.tmem_cols = cols;
    prm.timeout_ns = static_cast<uint64_t>(timeout_ms) * 1000000ull;
    prm.debug_flags = debug_flags;
    const PairLayout L(stages, prm.stage_bytes, n_pad);
    const size_t smem = L.total + 1024;
    const int64_t n_super = (a.n_tiles + 1) / 2;
    return wide ? launch_pair_variant<true>(tmW, tmH, prm, smem, n_super, stream)
                : launch_pair_variant<false>(tmW, tmH, prm, smem, n_super, stream);
}

}  // namespace lms
