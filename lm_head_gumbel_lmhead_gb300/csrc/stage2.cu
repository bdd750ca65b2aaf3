// Stage 2 (FlashSampling "method step details", Stage 2): per row, the candidate of the best
// vocabulary tile, t* = argmax_t m_b^(t), output idx_b^(t*).  Ties between tiles go to the
// smaller index, which is the earlier tile.  Also writes the per-row status.
#include "lms_device.cuh"
#include "lms_kernels.h"
#include "tcgen05_common.cuh"

namespace lms {
namespace {

constexpr int kStage2Threads = 256;
constexpr int kStage2PerThread = 8;   // candidates a thread loads before it compares any

__global__ void __launch_bounds__(kStage2Threads) stage2_kernel(
    const float* __restrict__ cand_score, const int* __restrict__ cand_index, int64_t n_tiles,
    const float* __restrict__ temperature, int64_t* __restrict__ out, int32_t* __restrict__ row_status,
    uint32_t* __restrict__ status_bits) {
    const int64_t b = blockIdx.x;
    // T is an input of the step, not a Stage-1 result: read it before the wait.
    const float T = temperature ? temperature[b] : 1.0f;
    // Wait for Stage 1 when launched as its programmatic dependent.
    pdl_wait_primary();
    const float* s_row = cand_score + b * n_tiles;
    const int* i_row = cand_index + b * n_tiles;
    float best_s = -CUDART_INF_F;
    int best_i = kNoIndex;
    int poisoned = 0;
    // All of a thread's loads of a round are issued before its comparisons, so a round costs one
    // trip to L2 (1187 candidates per row at the Qwen3-8B shape: one round).
    for (int64_t base = threadIdx.x; base < n_tiles; base += kStage2Threads * kStage2PerThread) {
        int idx[kStage2PerThread];
        float sc[kStage2PerThread];
#pragma unroll
        for (int j = 0; j < kStage2PerThread; ++j) {
            const int64_t t = base + j * kStage2Threads;
            idx[j] = t < n_tiles ? i_row[t] : -1;
            sc[j] = t < n_tiles ? s_row[t] : -CUDART_INF_F;
        }
#pragma unroll
        for (int j = 0; j < kStage2PerThread; ++j) {
            if (idx[j] == kPoisonIndex) {
                poisoned = 1;
            } else if (idx[j] >= 0 && better(sc[j], idx[j], best_s, best_i)) {
                best_s = sc[j];
                best_i = idx[j];
            }
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
        note_row_status(status_bits, status);
    }
}

// Stage 2 of Gumbel-top-k, part 1: row b's candidates are n_lists ordered lists of k keys (larger
// score, then smaller index first; key 0 and the keys of -inf scores are below every finite one).
// The lists of a row are split over S CTAs.  Each thread folds lists lo + tid, lo + tid + 256, ...
// (read whole, two at a time) into its own ordered kM best by a bitonic merge per list; the CTA's
// 256 lists are then merged pairwise in 8 rounds and its first k keys written out.  The union of the parts holds
// every one of the row's k best, since the lists do (Stage 1's selection guarantees it).
// Launched in stream order, not as a programmatic dependent: resident, waiting Stage-2 CTAs slowed
// the top-k Stage 1 (measured).
constexpr int kTopKThreads = 256;
constexpr int kTopKMaxSplit = 32;
// rows with at most this many lists are merged by one CTA of kTopKThreads threads (a few lists a
// thread), which also writes the outputs
constexpr int64_t kTopKOneCtaLists = 4 * kTopKThreads;

// best <- the kM largest keys of best and q, both ordered largest first (kM a power of two).
// The elementwise maximum of best and q reversed is a bitonic sequence holding the kM largest
// (Batcher's merge); half-cleaners at distances kM/2, ..., 1 order it.
template <int kM>
__device__ __forceinline__ void merge_top(unsigned long long (&best)[kM], const unsigned long long (&q)[kM]) {
#pragma unroll
    for (int i = 0; i < kM; ++i) {
        const unsigned long long x = q[kM - 1 - i];
        best[i] = best[i] > x ? best[i] : x;
    }
#pragma unroll
    for (int d = kM / 2; d > 0; d /= 2) {
#pragma unroll
        for (int i = 0; i < kM; ++i) {
            if ((i & d) == 0) {
                const unsigned long long a = best[i], b = best[i + d];
                best[i] = a > b ? a : b;
                best[i + d] = a > b ? b : a;
            }
        }
    }
}

// The row's k best keys, ordered, in the lanes r < k of one warp (0 past the finite ones) -> the
// indices, scores and status of row b.
__device__ __forceinline__ void write_topk_row(int64_t b, unsigned long long mine, int k, int lane,
                                               const float* __restrict__ temperature,
                                               int64_t* __restrict__ out, float* __restrict__ scores,
                                               int32_t* __restrict__ row_status,
                                               uint32_t* __restrict__ status_bits) {
    const unsigned long long top = __shfl_sync(0xffffffffu, mine, 0);
    const float T = temperature ? temperature[b] : 1.0f;
    const bool poisoned = top == tc::kPoisonKey;
    const bool invalid = !(T >= 0.0f);
    float sc = -CUDART_INF_F;
    int64_t idx = -1;
    if (lane < k && !poisoned && !invalid && mine != 0ull) {
        sc = tc::unpack_score(mine);
        idx = candidate_index(sc, tc::unpack_index(mine));
        if (idx < 0) sc = -CUDART_INF_F;
    }
    if (lane < k) {
        out[b * k + lane] = idx;
        if (scores) scores[b * k + lane] = sc;
    }
    const int found = __popc(__ballot_sync(0xffffffffu, lane < k && idx >= 0));
    if (lane == 0) {
        const int status = poisoned ? 3 : invalid ? 2 : (found > 0 ? 0 : 1);
        if (row_status) row_status[b] = status;
        note_row_status(status_bits, status);
    }
}

// kFinal: one CTA takes all of a row's lists (gridDim.x == 1) and its first warp writes the row's
// indices, scores and status directly (no part lists, no second kernel).
template <int kM, bool kFinal>
__global__ void __launch_bounds__(kTopKThreads) stage2_topk_part(
    const unsigned long long* __restrict__ cand_keys, int64_t n_lists, int k,
    unsigned long long* __restrict__ part_keys, const float* __restrict__ temperature,
    int64_t* __restrict__ out, float* __restrict__ scores, int32_t* __restrict__ row_status,
    uint32_t* __restrict__ status_bits) {
    // lst[r * kTopKThreads + t]: rank r of thread t's list (thread-minor, so that the threads of
    // a warp touch distinct banks)
    extern __shared__ unsigned long long lst[];
    const int tid = threadIdx.x;
    const int S = gridDim.x, s = blockIdx.x;
    const int64_t b = blockIdx.y;
    const int64_t lo = n_lists * s / S, hi = n_lists * (s + 1) / S;
    const unsigned long long* keys = cand_keys + b * n_lists * k;
    unsigned long long* mine = lst + tid;
    auto at = [&](unsigned long long* l, int r) -> unsigned long long& { return l[r * kTopKThreads]; };
    // This thread's best kM >= k keys, ordered, in registers (the first k are used); merges are
    // branch-free networks over the kM slots, so no slot is indexed at run time.
    unsigned long long best[kM];
#pragma unroll
    for (int i = 0; i < kM; ++i) best[i] = 0ull;
    // Two whole lists at a time are loaded together (the candidate lists have usually left L2 by
    // now, so one round trip per batch matters more than the bytes).  A list shorter than k ends
    // with a key 0; the stale slots after it (left by an earlier call) are cleared.  A list whose
    // first key beats this thread's kM-th is merged in.
    constexpr int kBatch = 2;
    for (int64_t base = lo + tid; base < hi; base += static_cast<int64_t>(kBatch) * kTopKThreads) {
        unsigned long long q[kBatch][kM];
#pragma unroll
        for (int j = 0; j < kBatch; ++j) {
            const int64_t t = base + static_cast<int64_t>(j) * kTopKThreads;
#pragma unroll
            for (int r = 0; r < kM; ++r) q[j][r] = (t < hi && r < k) ? __ldg(keys + t * k + r) : 0ull;
        }
#pragma unroll
        for (int j = 0; j < kBatch; ++j) {
            bool alive = true;
#pragma unroll
            for (int r = 0; r < kM; ++r) {
                alive = alive && q[j][r] != 0ull;
                q[j][r] = alive ? q[j][r] : 0ull;
            }
            if (q[j][0] > best[kM - 1]) merge_top<kM>(best, q[j]);
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
    if constexpr (kFinal) {
        if (tid < 32) {
            const unsigned long long mine = tid < k ? at(lst, tid) : 0ull;
            write_topk_row(b, mine, k, tid, temperature, out, scores, row_status, status_bits);
        }
    } else {
        if (tid < k) part_keys[(b * S + s) * k + tid] = at(lst, tid);
    }
}

// Part 2: one warp per row takes the k best of the row's S ordered part lists by k rounds of a
// warp-wide maximum (each lane holds up to kM keys of its lists, ordered), and writes the indices,
// scores and status.  A programmatic dependent of part 1.
template <int kM>
__global__ void __launch_bounds__(256) stage2_topk_final(
    const unsigned long long* __restrict__ part_keys, int S, int k, int64_t B,
    const float* __restrict__ temperature, int64_t* __restrict__ out, float* __restrict__ scores,
    int32_t* __restrict__ row_status, uint32_t* __restrict__ status_bits) {
    pdl_wait_primary();
    const int64_t b = static_cast<int64_t>(blockIdx.x) * 8 + (threadIdx.x >> 5);
    if (b >= B) return;                            // warp-uniform
    const int lane = threadIdx.x & 31;
    // lane l holds the keys l, l + 32, ... of the row's S * k part keys, ordered (kM slots)
    unsigned long long best[kM];
#pragma unroll
    for (int i = 0; i < kM; ++i) best[i] = 0ull;
    const unsigned long long* pk = part_keys + b * S * k;
    for (int x = lane; x < S * k; x += 32) {
        const unsigned long long v = pk[x];
#pragma unroll
        for (int i = kM - 1; i > 0; --i)
            best[i] = v > best[i - 1] ? best[i - 1] : (v > best[i] ? v : best[i]);
        best[0] = v > best[0] ? v : best[0];
    }
    unsigned long long mine = 0ull;                 // lane r keeps the row's r-th key
    for (int r = 0; r < k; ++r) {
        unsigned long long m = best[0];
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
            const unsigned long long o = __shfl_xor_sync(0xffffffffu, m, off);
            m = o > m ? o : m;
        }
        if (lane == r) mine = m;
        // the lane that held the maximum drops it (keys are distinct unless 0)
        if (best[0] == m && m != 0ull) {
#pragma unroll
            for (int i = 0; i < kM - 1; ++i) best[i] = best[i + 1];
            best[kM - 1] = 0ull;
        }
    }
    write_topk_row(b, mine, k, lane, temperature, out, scores, row_status, status_bits);
}

}  // namespace

int64_t stage2_topk_split(int64_t B) {
    // about two CTAs' worth of rows per SM
    const int64_t want = (2 * static_cast<int64_t>(device_sm_count()) + B - 1) / B;
    return want < 1 ? 1 : (want > kTopKMaxSplit ? kTopKMaxSplit : want);
}

size_t stage2_topk_part_bytes(int64_t B, int k) {
    return static_cast<size_t>(B) * kTopKMaxSplit * static_cast<size_t>(k) * sizeof(unsigned long long);
}

cudaError_t launch_stage2_topk(const unsigned long long* cand_keys, int64_t n_lists, int k, int64_t B,
                               const float* temperature, int64_t* out, float* scores,
                               int32_t* row_status, uint32_t* status_bits,
                               unsigned long long* part_keys, cudaStream_t stream) {
    if (k < 1 || k > tc::kMaxTopK) return cudaErrorInvalidValue;
    const size_t smem = static_cast<size_t>(kTopKThreads) * k * sizeof(unsigned long long);
    // A row of at most kTopKOneCtaLists lists (the running lists: 4 per Stage-1 CTA) is merged by
    // one CTA, which writes the outputs; more lists (one per tile and quadrant) are split over S
    // CTAs per row and merged by the final kernel.
    const bool one_cta = n_lists <= kTopKOneCtaLists;
    auto part = one_cta ? (k <= 1 ? stage2_topk_part<1, true> : k <= 2 ? stage2_topk_part<2, true>
                           : k <= 4 ? stage2_topk_part<4, true> : k <= 8 ? stage2_topk_part<8, true>
                                                                        : stage2_topk_part<16, true>)
                        : (k <= 1 ? stage2_topk_part<1, false> : k <= 2 ? stage2_topk_part<2, false>
                           : k <= 4 ? stage2_topk_part<4, false> : k <= 8 ? stage2_topk_part<8, false>
                                                                        : stage2_topk_part<16, false>);
    cudaError_t e = ensure_dynamic_smem(reinterpret_cast<const void*>(part), smem);
    if (e != cudaSuccess) return e;
    const int S = one_cta ? 1 : static_cast<int>(stage2_topk_split(B));
    part<<<dim3(static_cast<unsigned>(S), static_cast<unsigned>(B)), kTopKThreads, smem, stream>>>(
        cand_keys, n_lists, k, part_keys, temperature, out, scores, row_status, status_bits);
    e = cudaGetLastError();
    if (e != cudaSuccess || one_cta) return e;
    auto fin = k <= 1 ? stage2_topk_final<1> : k <= 2 ? stage2_topk_final<2>
             : k <= 4 ? stage2_topk_final<4> : k <= 8 ? stage2_topk_final<8> : stage2_topk_final<16>;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>((B + 7) / 8));
    cfg.blockDim = dim3(256);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, fin, static_cast<const unsigned long long*>(part_keys), S, k, B,
                              temperature, out, scores, row_status, status_bits);
}

cudaError_t launch_stage2(const float* cand_score, const int* cand_index, int64_t n_tiles,
                          int64_t B, const float* temperature, int64_t* out, int32_t* row_status,
                          uint32_t* status_bits, cudaStream_t stream) {
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
                              out, row_status, status_bits);
}

}  // namespace lms
