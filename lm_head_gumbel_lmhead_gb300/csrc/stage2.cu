// Stage 2 (FlashSampling "method step details", Stage 2): per row, the candidate of the best
// vocabulary tile, t* = argmax_t m_b^(t), output idx_b^(t*).  Ties between tiles go to the
// smaller index, which is the earlier tile.  Also writes the per-row status.
#include "lms_device.cuh"
#include "lms_kernels.h"
#include "tcgen05_common.cuh"

namespace lms {
namespace {

constexpr int kStage2Threads = 128;

__global__ void __launch_bounds__(kStage2Threads) stage2_kernel(
    const float* __restrict__ cand_score, const int* __restrict__ cand_index, int64_t n_tiles,
    const float* __restrict__ temperature, int64_t* __restrict__ out, int32_t* __restrict__ row_status) {
    // Wait for Stage 1 when launched as its programmatic dependent.
    pdl_wait_primary();
    const int64_t b = blockIdx.x;
    const float* s_row = cand_score + b * n_tiles;
    const int* i_row = cand_index + b * n_tiles;
    float best_s = -CUDART_INF_F;
    int best_i = kNoIndex;
    int poisoned = 0;
    for (int64_t t = threadIdx.x; t < n_tiles; t += kStage2Threads) {
        const int idx = i_row[t];
        if (idx == kPoisonIndex) {
            poisoned = 1;
        } else if (idx >= 0) {
            const float s = s_row[t];
            if (better(s, idx, best_s, best_i)) { best_s = s; best_i = idx; }
        }
    }
    warp_argmax(best_s, best_i);
    poisoned = __any_sync(0xffffffffu, poisoned);
    __shared__ float sh_s[kStage2Threads / 32];
    __shared__ int sh_i[kStage2Threads / 32];
    __shared__ int sh_p[kStage2Threads / 32];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (lane == 0) { sh_s[warp] = best_s; sh_i[warp] = best_i; sh_p[warp] = poisoned; }
    __syncthreads();
    if (threadIdx.x == 0) {
        for (int w = 1; w < kStage2Threads / 32; ++w) {
            if (better(sh_s[w], sh_i[w], best_s, best_i)) { best_s = sh_s[w]; best_i = sh_i[w]; }
            poisoned |= sh_p[w];
        }
        const float T = temperature ? temperature[b] : 1.0f;
        int32_t status;
        int64_t token;
        if (poisoned) {
            status = 3; token = -1;
        } else if (!(T >= 0.0f)) {
            status = 2; token = -1;
        } else if (candidate_index(best_s, best_i) < 0) {
            status = 1; token = -1;
        } else {
            status = 0; token = best_i;
        }
        out[b] = token;
        if (row_status) row_status[b] = status;
    }
}

// Stage 2 of Gumbel-top-k: row b's candidates are n_lists ordered lists of k keys (larger score,
// then smaller index first; key 0 and the keys of -inf scores are below every finite one).  Each
// thread folds lists tid, tid + 512, ... into its own ordered k best, inserting a list's keys in
// order until one is not above the thread's current k-th (a list shorter than k ends with key 0).
// The 512 lists are then merged pairwise in 9 rounds.  The merged list's first k keys are the
// row's k best, since the lists hold every one of them (Stage 1's selection guarantees it).  Launched in stream order,
// not as a programmatic dependent: its resident, waiting CTAs slowed the top-k Stage 1 (measured).
constexpr int kTopKThreads = 512;

template <int kM>
__global__ void __launch_bounds__(kTopKThreads) stage2_topk_kernel(
    const unsigned long long* __restrict__ cand_keys, int64_t n_lists, int k,
    const float* __restrict__ temperature, int64_t* __restrict__ out, float* __restrict__ scores,
    int32_t* __restrict__ row_status) {
    // lst[r * kTopKThreads + t]: rank r of thread t's list (thread-minor, so that the threads of
    // a warp touch distinct banks)
    extern __shared__ unsigned long long lst[];
    const int tid = threadIdx.x;
    const int64_t b = blockIdx.x;
    const unsigned long long* keys = cand_keys + b * n_lists * k;
    unsigned long long* mine = lst + tid;
    auto at = [&](unsigned long long* l, int r) -> unsigned long long& { return l[r * kTopKThreads]; };
    // This thread's best kM >= k keys, ordered, in registers (the first k are used); insertion
    // is a branch-free pass over the kM slots, so no slot is indexed at run time.
    unsigned long long best[kM];
#pragma unroll
    for (int i = 0; i < kM; ++i) best[i] = 0ull;
    // First keys of 4 lists at a time are loaded together; a list is read further only when its
    // first key beats this thread's current k-th (most lists of a warmed-up Stage 1 are empty).
    unsigned long long kth = 0ull;
    constexpr int kBatch = 4;
    for (int64_t base = tid; base < n_lists; base += static_cast<int64_t>(kBatch) * kTopKThreads) {
        unsigned long long first[kBatch];
#pragma unroll
        for (int j = 0; j < kBatch; ++j) {
            const int64_t t = base + static_cast<int64_t>(j) * kTopKThreads;
            first[j] = t < n_lists ? __ldg(keys + t * k) : 0ull;
        }
#pragma unroll
        for (int j = 0; j < kBatch; ++j) {
            if (first[j] <= kth) continue;
            // the list's k slots are loaded together (one latency); a shorter list ends with a key
            // 0, and the stale slots after it (left by an earlier call) are zeroed before use
            const unsigned long long* tl = keys + (base + static_cast<int64_t>(j) * kTopKThreads) * k;
            // keys in groups of 4 loaded together; the list is ordered and ends with a key 0, so
            // the first key not above kth ends it
            for (int r0 = 0; r0 < k; r0 += 4) {
                unsigned long long q[4];
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const int r = r0 + u;
                    q[u] = r == 0 ? first[j] : (r < k ? __ldg(tl + r) : 0ull);
                }
                bool stop = false;
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    stop = stop || !(q[u] > kth);
                    const unsigned long long x = stop ? 0ull : q[u];     // 0 changes nothing
#pragma unroll
                    for (int i = kM - 1; i > 0; --i)                     // past the kM-th: dropped
                        best[i] = x > best[i - 1] ? best[i - 1] : (x > best[i] ? x : best[i]);
                    best[0] = x > best[0] ? x : best[0];
                }
                if (stop) break;
            }
            // the k-th key, as the least of the first k (the list is ordered); written as a min so
            // that it is not folded into a run-time index of best[]
            unsigned long long t = ~0ull;
#pragma unroll
            for (int i = 0; i < kM; ++i) t = (i < k && best[i] < t) ? best[i] : t;
            kth = t;
        }
    }
#pragma unroll
    for (int r = 0; r < kM; ++r)
        if (r < k) lst[r * kTopKThreads + tid] = best[r];
    __syncthreads();
    for (int stride = 1; stride < kTopKThreads; stride <<= 1) {
        const bool merging = (tid & (2 * stride - 1)) == 0;
        unsigned long long m[kM];
        if (merging) {
            unsigned long long* x = lst + tid;
            unsigned long long* y = lst + tid + stride;
            int i = 0, j = 0;
#pragma unroll
            for (int r = 0; r < kM; ++r) {
                if (r < k) {
                    const unsigned long long xv = i < k ? at(x, i) : 0ull, yv = j < k ? at(y, j) : 0ull;
                    if (xv >= yv) { m[r] = xv; ++i; } else { m[r] = yv; ++j; }
                }
            }
        }
        __syncthreads();
        if (merging) {
#pragma unroll
            for (int r = 0; r < kM; ++r)
                if (r < k) at(mine, r) = m[r];
        }
        __syncthreads();
    }
    if (tid == 0) {
        const float T = temperature ? temperature[b] : 1.0f;
        const bool poisoned = at(lst, 0) == tc::kPoisonKey;
        const bool invalid = !(T >= 0.0f);
        int found = 0;
        for (int r = 0; r < k; ++r) {
            const unsigned long long key = at(lst, r);
            float s = -CUDART_INF_F;
            int64_t idx = -1;
            if (!poisoned && !invalid && key != 0ull) {
                s = tc::unpack_score(key);
                idx = candidate_index(s, tc::unpack_index(key));
                if (idx < 0) s = -CUDART_INF_F;
            }
            found += idx >= 0;
            out[b * k + r] = idx;
            if (scores) scores[b * k + r] = s;
        }
        if (row_status) row_status[b] = poisoned ? 3 : invalid ? 2 : (found > 0 ? 0 : 1);
    }
}

}  // namespace

cudaError_t launch_stage2_topk(const unsigned long long* cand_keys, int64_t n_lists, int k, int64_t B,
                               const float* temperature, int64_t* out, float* scores,
                               int32_t* row_status, cudaStream_t stream) {
    if (k < 1 || k > tc::kMaxTopK) return cudaErrorInvalidValue;
    const size_t smem = static_cast<size_t>(kTopKThreads) * k * sizeof(unsigned long long);
    for (const void* f : {reinterpret_cast<const void*>(stage2_topk_kernel<1>),
                          reinterpret_cast<const void*>(stage2_topk_kernel<2>),
                          reinterpret_cast<const void*>(stage2_topk_kernel<4>),
                          reinterpret_cast<const void*>(stage2_topk_kernel<8>),
                          reinterpret_cast<const void*>(stage2_topk_kernel<16>)}) {
        const cudaError_t e = ensure_dynamic_smem(f, smem);
        if (e != cudaSuccess) return e;
    }
    auto kern = k <= 1 ? stage2_topk_kernel<1> : k <= 2 ? stage2_topk_kernel<2>
              : k <= 4 ? stage2_topk_kernel<4> : k <= 8 ? stage2_topk_kernel<8> : stage2_topk_kernel<16>;
    kern<<<static_cast<unsigned>(B), kTopKThreads, smem, stream>>>(cand_keys, n_lists, k, temperature,
                                                                    out, scores, row_status);
    return cudaGetLastError();
}

cudaError_t launch_stage2(const float* cand_score, const int* cand_index, int64_t n_tiles,
                          int64_t B, const float* temperature, int64_t* out, int32_t* row_status,
                          cudaStream_t stream) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(B));
    cfg.blockDim = dim3(kStage2Threads);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, stage2_kernel, cand_score, cand_index, n_tiles, temperature,
                              out, row_status);
}

}  // namespace lms
