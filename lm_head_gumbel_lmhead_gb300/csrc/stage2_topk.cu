// Stage 2 of Gumbel-top-k (FlashSampling "Future directions": the k largest perturbed scores are
// k draws without replacement).  Row b's candidates are n_lists ordered lists of k keys,
// cand_keys[b][l][r]: larger score, then smaller index first; key 0 and the keys of -inf scores
// are below every finite one; a list shorter than k ends with a key 0, and the slots after it may
// hold stale keys of an earlier call.  Every vocabulary entry belongs to one list, so the nonzero
// keys of a row are distinct, except the poison key that heads the lists of a Stage-1 CTA whose
// bounded wait ran out.  The union of a row's lists holds every one of its k best keys (Stage 1's
// selection guarantees it), so the row's k best keys are the k best of the union.
#include "lms_device.cuh"
#include "lms_kernels.h"
#include "tcgen05_common.cuh"

namespace lms {
namespace {

constexpr int kTopKThreads = 256;
constexpr int kTopKWarps = kTopKThreads / 32;
constexpr int kTopKMaxSplit = 32;
// Rows of at most kRowLists lists (always, with running lists: 4 per Stage-1 CTA) are taken by one
// CTA, kRowListsPerThread whole lists a thread; longer rows are split over several CTAs.
constexpr int kRowListsPerThread = 4;
constexpr int64_t kRowLists = kRowListsPerThread * kTopKThreads;

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

// A list as loaded: the slots after its first key 0 are stale and are cleared.
template <int kM>
__device__ __forceinline__ void clear_after_end(unsigned long long (&q)[kM]) {
    bool alive = true;
#pragma unroll
    for (int r = 0; r < kM; ++r) {
        alive = alive && q[r] != 0ull;
        q[r] = alive ? q[r] : 0ull;
    }
}

// v into the ordered (largest first) slots c.
template <int kM>
__device__ __forceinline__ void insert_ordered(unsigned long long (&c)[kM], unsigned long long v) {
#pragma unroll
    for (int i = kM - 1; i > 0; --i) c[i] = v > c[i - 1] ? c[i - 1] : (v > c[i] ? v : c[i]);
    c[0] = v > c[0] ? v : c[0];
}

// The warp's k best keys by k rounds of a warp-wide maximum over the lanes' ordered slots best:
// lane r < k ends with the warp's r-th key (0 past its last nonzero key).  Every lane whose first
// slot holds the round's nonzero maximum drops it: nonzero keys are distinct, except the poison
// key, which ends the row as poisoned whatever follows it.
template <int kM>
__device__ __forceinline__ unsigned long long warp_top_k(unsigned long long (&best)[kM], int k, int lane) {
    unsigned long long mine = 0ull;
    for (int r = 0; r < k; ++r) {
        unsigned long long m = best[0];
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
            const unsigned long long o = __shfl_xor_sync(0xffffffffu, m, off);
            m = o > m ? o : m;
        }
        if (lane == r) mine = m;
        if (best[0] == m && m != 0ull) {
#pragma unroll
            for (int i = 0; i < kM - 1; ++i) best[i] = best[i + 1];
            best[kM - 1] = 0ull;
        }
    }
    return mine;
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

// Rows of at most kRowLists lists: one CTA per row, a programmatic dependent of Stage 1.  Each
// thread loads its lists t, t + 256, ... whole and all at once (one trip to memory), folds them
// into its own ordered kM best by Batcher's merge, each warp takes its k best by k rounds of a
// warp-wide maximum, and the first warp takes the row's k best from the eight warps' lists the
// same way and writes the indices, scores and status.
template <int kM>
__global__ void __launch_bounds__(kTopKThreads, 1) stage2_topk_row(
    const unsigned long long* __restrict__ cand_keys, int64_t n_lists, int k,
    const float* __restrict__ temperature, int64_t* __restrict__ out, float* __restrict__ scores,
    int32_t* __restrict__ row_status, uint32_t* __restrict__ status_bits) {
    __shared__ unsigned long long warp_keys[kTopKWarps * kM];   // warp w's r-th key at w * k + r
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int64_t b = blockIdx.x;
    pdl_wait_primary();                             // the lists are Stage 1's output
    const unsigned long long* keys = cand_keys + b * n_lists * k;
    unsigned long long q[kRowListsPerThread][kM];
#pragma unroll
    for (int j = 0; j < kRowListsPerThread; ++j) {
        const int64_t l = tid + static_cast<int64_t>(j) * kTopKThreads;
#pragma unroll
        for (int r = 0; r < kM; ++r) q[j][r] = (l < n_lists && r < k) ? __ldg(keys + l * k + r) : 0ull;
    }
    unsigned long long best[kM];
#pragma unroll
    for (int i = 0; i < kM; ++i) best[i] = 0ull;
#pragma unroll
    for (int j = 0; j < kRowListsPerThread; ++j) {
        clear_after_end<kM>(q[j]);
        if (q[j][0] > best[kM - 1]) merge_top<kM>(best, q[j]);
    }
    const unsigned long long wk = warp_top_k<kM>(best, k, lane);
    if (lane < k) warp_keys[warp * k + lane] = wk;
    __syncthreads();
    if (warp == 0) {
        // lane l takes the warp keys l, l + 32, ... (at most kTopKWarps * kM / 32), ordered
        constexpr int kPer = (kTopKWarps * kM + 31) / 32;
        unsigned long long c[kPer];
#pragma unroll
        for (int i = 0; i < kPer; ++i) c[i] = 0ull;
        for (int x = lane; x < kTopKWarps * k; x += 32) insert_ordered<kPer>(c, warp_keys[x]);
        const unsigned long long mine = warp_top_k<kPer>(c, k, lane);
        write_topk_row(b, mine, k, lane, temperature, out, scores, row_status, status_bits);
    }
}

// Longer rows (one list per tile and quadrant), part 1: the row's lists are split over S CTAs.
// Each thread folds lists lo + tid, lo + tid + 256, ... (read whole, two at a time) into its own
// ordered kM best by Batcher's merge; the CTA's 256 lists are then merged pairwise in 8 rounds and
// its first k keys written out.  The union of the parts holds every one of the row's k best.
// Launched in stream order, not as a programmatic dependent: resident, waiting CTAs of this
// many-CTA grid slowed the top-k Stage 1 (measured).
template <int kM>
__global__ void __launch_bounds__(kTopKThreads) stage2_topk_part(
    const unsigned long long* __restrict__ cand_keys, int64_t n_lists, int k,
    unsigned long long* __restrict__ part_keys) {
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
    // now, so one round trip per batch matters more than the bytes).  A list whose first key beats
    // this thread's kM-th is merged in.
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
            clear_after_end<kM>(q[j]);
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
    if (tid < k) part_keys[(b * S + s) * k + tid] = at(lst, tid);
}

// Part 2: one warp per row takes the k best of the row's S ordered part lists (lane l holds the
// keys l, l + 32, ... of them, ordered, in kM slots) by k rounds of a warp-wide maximum, and writes
// the indices, scores and status.  A programmatic dependent of part 1.
template <int kM>
__global__ void __launch_bounds__(256) stage2_topk_final(
    const unsigned long long* __restrict__ part_keys, int S, int k, int64_t B,
    const float* __restrict__ temperature, int64_t* __restrict__ out, float* __restrict__ scores,
    int32_t* __restrict__ row_status, uint32_t* __restrict__ status_bits) {
    pdl_wait_primary();
    const int64_t b = static_cast<int64_t>(blockIdx.x) * 8 + (threadIdx.x >> 5);
    if (b >= B) return;                            // warp-uniform
    const int lane = threadIdx.x & 31;
    unsigned long long best[kM];
#pragma unroll
    for (int i = 0; i < kM; ++i) best[i] = 0ull;
    const unsigned long long* pk = part_keys + b * S * k;
    for (int x = lane; x < S * k; x += 32) insert_ordered<kM>(best, pk[x]);
    const unsigned long long mine = warp_top_k<kM>(best, k, lane);
    write_topk_row(b, mine, k, lane, temperature, out, scores, row_status, status_bits);
}

// A programmatic dependent launch of kern on the stream.
template <typename... Params, typename... Args>
cudaError_t launch_dependent(void (*kern)(Params...), dim3 grid, cudaStream_t stream, Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(kTopKThreads);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, args...);
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
    if (n_lists <= kRowLists) {
        auto row = k <= 1 ? stage2_topk_row<1> : k <= 2 ? stage2_topk_row<2>
                 : k <= 4 ? stage2_topk_row<4> : k <= 8 ? stage2_topk_row<8> : stage2_topk_row<16>;
        return launch_dependent(row, dim3(static_cast<unsigned>(B)), stream, cand_keys, n_lists, k,
                                temperature, out, scores, row_status, status_bits);
    }
    auto part = k <= 1 ? stage2_topk_part<1> : k <= 2 ? stage2_topk_part<2>
              : k <= 4 ? stage2_topk_part<4> : k <= 8 ? stage2_topk_part<8> : stage2_topk_part<16>;
    const size_t smem = static_cast<size_t>(kTopKThreads) * k * sizeof(unsigned long long);
    cudaError_t e = ensure_dynamic_smem(reinterpret_cast<const void*>(part), smem);
    if (e != cudaSuccess) return e;
    const int S = static_cast<int>(stage2_topk_split(B));
    part<<<dim3(static_cast<unsigned>(S), static_cast<unsigned>(B)), kTopKThreads, smem, stream>>>(
        cand_keys, n_lists, k, part_keys);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    auto fin = k <= 1 ? stage2_topk_final<1> : k <= 2 ? stage2_topk_final<2>
             : k <= 4 ? stage2_topk_final<4> : k <= 8 ? stage2_topk_final<8> : stage2_topk_final<16>;
    return launch_dependent(fin, dim3(static_cast<unsigned>((B + 7) / 8)), stream,
                            static_cast<const unsigned long long*>(part_keys), S, k, B, temperature,
                            out, scores, row_status, status_bits);
}

}  // namespace lms
