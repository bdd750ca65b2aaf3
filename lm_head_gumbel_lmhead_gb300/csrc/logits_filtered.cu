// Filtered Gumbel race over materialised logits: top-k -> top-p -> min-p on t = (y + bias) / T,
// then the race over the kept tokens (spec-decode-ops "Semantics": top-p keeps the shortest
// sorted prefix whose mass, normalised over the top-k prefix, reaches top_p, crossing token
// included; min-p keeps p >= min_p * p_max; every filter keeps at least one token.  The
// sampling-kernel guide, reasoning steps 6-8: top-k before top-p, a compile-time bound K_MAX on
// the candidate set).  The race over a subset samples the renormalised softmax, so nothing is
// normalised except the top-p prefix mass.
//
// One CTA of 1024 threads per row:
//   1. radix select (4 passes of 8 bits over order-preserving 32-bit keys of t) finds the key of
//      the k-th largest entry, k = min(top_k, k_max) (k_max when only top-p is on);
//   2. one pass gathers exactly k candidates: every key above it and, in index order, the first
//      entries equal to it (ties keep the smallest indices);
//   3. a bitonic sort in shared memory orders them by (t descending, v ascending);
//   4. fp32 prefix sums of exp(t_i - t_0) give the top-p cut, a threshold t_0 + log(min_p) the
//      min-p cut;
//   5. the race over the kept prefix with the same Philox noise as the unfiltered race.
// Rows with only min-p (or no filter) skip 1-4: one pass for t_max, one threshold race.
#include <cuda_bf16.h>

#include "lms_device.cuh"
#include "lms_kernels.h"

namespace lms {
namespace {

constexpr int kThreads = 1024;
constexpr int kWarps = kThreads / 32;
constexpr int kMaxK = 1024;

template <typename T>
__device__ __forceinline__ float to_f(T x);
template <>
__device__ __forceinline__ float to_f<float>(float x) { return x; }
template <>
__device__ __forceinline__ float to_f<__nv_bfloat16>(__nv_bfloat16 x) { return __bfloat162float(x); }

// Order-preserving 32-bit key of a (non-NaN) float; -0 folded onto +0.
__device__ __forceinline__ uint32_t order_key(float t) {
    const uint32_t f = __float_as_uint(t + 0.0f);
    return (f & 0x80000000u) ? ~f : (f | 0x80000000u);
}

__device__ __forceinline__ float key_value(uint32_t k) {
    return __uint_as_float((k & 0x80000000u) ? (k & 0x7fffffffu) : ~k);
}

struct RowView {
    const void* y;
    const float* bias;
    const uint32_t* mask;
    RowParams p;
    int64_t V;
};

// Transformed logit t (no noise): -inf when masked or NaN.
template <typename T>
__device__ __forceinline__ float t_of(const RowView& r, int64_t v) {
    if (r.mask && !((__ldg(r.mask + (v >> 5)) >> (v & 31)) & 1u)) return -CUDART_INF_F;
    const float y = to_f<T>(static_cast<const T*>(r.y)[v]) + (r.bias ? __ldg(r.bias + v) : 0.0f);
    const float t = (r.p.flags & kRowGreedy) ? y : y * r.p.inv_t;
    return t == t ? t : -CUDART_INF_F;
}

template <typename X>
__device__ __forceinline__ X block_sum(X x, X* sh) {
    for (int off = 16; off > 0; off >>= 1) x += __shfl_xor_sync(0xffffffffu, x, off);
    const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
    __syncthreads();
    if (l == 0) sh[w] = x;
    __syncthreads();
    x = (threadIdx.x < kWarps) ? sh[threadIdx.x] : X(0);
    if (w == 0)
        for (int off = 16; off > 0; off >>= 1) x += __shfl_xor_sync(0xffffffffu, x, off);
    if (threadIdx.x == 0) sh[0] = x;
    __syncthreads();
    return sh[0];
}

__device__ __forceinline__ float block_max(float x, float* sh) {
    for (int off = 16; off > 0; off >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, off));
    const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
    __syncthreads();
    if (l == 0) sh[w] = x;
    __syncthreads();
    x = (threadIdx.x < kWarps) ? sh[threadIdx.x] : -CUDART_INF_F;
    if (w == 0)
        for (int off = 16; off > 0; off >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, off));
    if (threadIdx.x == 0) sh[0] = x;
    __syncthreads();
    return sh[0];
}

// Inclusive prefix sum over the block (thread order), returns this thread's inclusive value.
template <typename X>
__device__ __forceinline__ X block_scan_incl(X x, X* sh) {
    const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
    for (int off = 1; off < 32; off <<= 1) {
        const X y = __shfl_up_sync(0xffffffffu, x, off);
        if (l >= off) x += y;
    }
    __syncthreads();
    if (l == 31) sh[w] = x;
    __syncthreads();
    if (w == 0) {
        X s = sh[l];
        for (int off = 1; off < 32; off <<= 1) {
            const X y = __shfl_up_sync(0xffffffffu, s, off);
            if (l >= off) s += y;
        }
        sh[l] = s;
    }
    __syncthreads();
    return w > 0 ? x + sh[w - 1] : x;
}

// Block argmax of (score, index), larger score then smaller index; result in every thread.
__device__ __forceinline__ void block_argmax(float& s, int& i, float* shs, int* shi) {
    warp_argmax(s, i);
    const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
    __syncthreads();
    if (l == 0) { shs[w] = s; shi[w] = i; }
    __syncthreads();
    if (w == 0) {
        s = shs[l];
        i = shi[l];
        warp_argmax(s, i);
        if (l == 0) { shs[0] = s; shi[0] = i; }
    }
    __syncthreads();
    s = shs[0];
    i = shi[0];
}

template <typename T, bool kWide>
__global__ void __launch_bounds__(kThreads, 1) filtered_race_kernel(const T* __restrict__ logits,
                                                                    int64_t ld, FilterArgs f) {
    __shared__ unsigned long long cand[kMaxK];       // (key << 32) | ~v, sorted descending
    __shared__ float shf[kWarps];
    __shared__ int shi[kWarps];
    __shared__ int hist[256];
    __shared__ int sh_int[4];

    const SampleArgs& a = f.a;
    const int64_t b = blockIdx.x;
    const int64_t row = a.row0 + b;
    const int tid = threadIdx.x;
    RowView r;
    r.p = make_row_params(a.temperature, a.seeds, a.positions, a.base_seed, a.offset, row);
    r.y = logits + row * ld;
    r.bias = a.bias ? a.bias + row * a.ld_bias : nullptr;
    r.mask = a.mask ? a.mask + row * a.ld_mask : nullptr;
    r.V = a.V;
    const int64_t V = a.V;

    if (r.p.flags & kRowInvalid) {
        if (tid == 0) { f.out[b] = -1; if (f.row_status) f.row_status[b] = 2; }
        return;
    }
    const int tk = f.top_k ? f.top_k[row] : 0;
    const float tp = f.top_p ? f.top_p[row] : 1.0f;
    const float mp = f.min_p ? f.min_p[row] : 0.0f;
    const bool topk_on = tk >= 1 && tk < V;
    const bool topp_on = tp > 0.0f && tp < 1.0f;
    const bool minp_on = mp > 0.0f && mp <= 1.0f;
    const bool greedy = r.p.flags & kRowGreedy;

    // t_max over the row (also tells whether any entry is above -inf)
    float tmax = -CUDART_INF_F;
    for (int64_t v = tid; v < V; v += kThreads) tmax = fmaxf(tmax, t_of<T>(r, v));
    tmax = block_max(tmax, shf);
    if (!(tmax > -CUDART_INF_F)) {
        if (tid == 0) { f.out[b] = -1; if (f.row_status) f.row_status[b] = 1; }
        return;
    }

    float best_s = -CUDART_INF_F;
    int best_i = kNoIndex;
    if (greedy || !(topk_on || topp_on)) {
        // greedy rows, min-p only, or no filter: one threshold race over the row.  Greedy rows
        // need no filter (every filter keeps the top token).
        const float thr = (minp_on && !greedy) ? tmax + logf(mp) : -CUDART_INF_F;
        for (int64_t v0 = static_cast<int64_t>(tid) * 4; v0 < V; v0 += kThreads * 4) {
            float g[4] = {0.0f, 0.0f, 0.0f, 0.0f};
            if (!greedy) gumbel_run<kWide, 4>(r.p.key, static_cast<uint32_t>(v0), g);
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int64_t v = v0 + e;
                if (v < V) {
                    const float t = t_of<T>(r, v);
                    if (t > -CUDART_INF_F && t >= thr) {
                        const float s = greedy ? t : t + g[e];
                        if (s > best_s) { best_s = s; best_i = static_cast<int>(v); }
                    }
                }
            }
        }
        block_argmax(best_s, best_i, shf, shi);
    } else {
        const int k_cap = f.k_max;
        const int k = topk_on ? (tk < k_cap ? tk : k_cap) : k_cap;
        // ---- 1. radix select: key of the k-th largest entry (or the smallest, if V < k) ----
        uint32_t prefix = 0, pmask = 0;
        int remaining = k < V ? k : static_cast<int>(V);
        for (int shift = 24; shift >= 0; shift -= 8) {
            if (tid < 256) hist[tid] = 0;
            __syncthreads();
            for (int64_t v = tid; v < V; v += kThreads) {
                const uint32_t key = order_key(t_of<T>(r, v));
                if ((key & pmask) == prefix) atomicAdd(&hist[(key >> shift) & 255u], 1);
            }
            __syncthreads();
            if (tid == 0) {
                int cum = 0, d = 255;
                for (; d > 0; --d) {
                    if (cum + hist[d] >= remaining) break;
                    cum += hist[d];
                }
                sh_int[0] = d;
                sh_int[1] = remaining - cum;
            }
            __syncthreads();
            prefix |= static_cast<uint32_t>(sh_int[0]) << shift;
            pmask |= 255u << shift;
            remaining = sh_int[1];
            __syncthreads();
        }
        const uint32_t kstar = prefix;   // the k-th largest key
        const int need_eq = remaining;   // entries equal to it that are kept (smallest indices)
        // ---- 2. gather exactly min(k, V) candidates ----
        if (tid == 0) { sh_int[2] = 0; sh_int[3] = 0; }
        cand[tid] = 0ull;                // below every real candidate (kMaxK == kThreads)
        __syncthreads();
        for (int64_t base = 0; base < V; base += kThreads) {
            const int64_t v = base + tid;
            const uint32_t key = v < V ? order_key(t_of<T>(r, v)) : 0u;
            const int eq = (v < V && key == kstar) ? 1 : 0;
            const int taken_before = sh_int[3];
            int eq_rank = 0;
            if (__syncthreads_or(eq)) eq_rank = block_scan_incl<int>(eq, hist) - eq;
            const bool take = (v < V && key > kstar) || (eq && taken_before + eq_rank < need_eq);
            if (take) {
                const int pos = atomicAdd(&sh_int[2], 1);
                if (pos < kMaxK)
                    cand[pos] = (static_cast<unsigned long long>(key) << 32) |
                                static_cast<uint32_t>(~static_cast<uint32_t>(v));
            }
            const int eq_total = __syncthreads_count(eq);
            if (tid == 0) sh_int[3] = taken_before + eq_total;
            __syncthreads();
        }
        const int n_cand = sh_int[2] < kMaxK ? sh_int[2] : kMaxK;
        // ---- 3. bitonic sort, descending ----
        for (int size = 2; size <= kMaxK; size <<= 1) {
            for (int stride = size >> 1; stride > 0; stride >>= 1) {
                const int j = tid ^ stride;
                if (j > tid) {
                    const unsigned long long x = cand[tid], y = cand[j];
                    const bool desc = (tid & size) == 0;
                    if (desc ? (x < y) : (x > y)) { cand[tid] = y; cand[j] = x; }
                }
                __syncthreads();
            }
        }
        // ---- 4. top-p and min-p cuts on the sorted prefix ----
        const float t0 = key_value(static_cast<uint32_t>(cand[0] >> 32));
        const float ti = key_value(static_cast<uint32_t>(cand[tid] >> 32));
        int n_keep = n_cand;
        if (topp_on) {
            const float e = tid < n_cand ? __expf(ti - t0) : 0.0f;
            const float z = block_sum<float>(e, shf);
            const float c = block_scan_incl<float>(e, shf);
            if (tid == 0) sh_int[0] = n_cand;
            __syncthreads();
            if (tid < n_cand && c >= tp * z) atomicMin(&sh_int[0], tid + 1);
            __syncthreads();
            n_keep = sh_int[0];
        }
        if (minp_on) {
            const float thr = t0 + logf(mp);
            if (tid == 0) sh_int[1] = n_keep;
            __syncthreads();
            if (tid < n_keep && tid > 0 && ti < thr) atomicMin(&sh_int[1], tid);
            __syncthreads();
            n_keep = sh_int[1];
        }
        if (n_keep < 1) n_keep = 1;
        // ---- 5. the race over the kept prefix ----
        if (tid < n_keep) {
            const int v = static_cast<int>(~static_cast<uint32_t>(cand[tid]));
            if (ti > -CUDART_INF_F) {
                best_s = ti + gumbel_one<kWide>(r.p.key, static_cast<uint32_t>(v));
                best_i = v;
            }
        }
        block_argmax(best_s, best_i, shf, shi);
    }
    if (tid == 0) {
        const bool found = best_s > -CUDART_INF_F && best_i != kNoIndex;
        f.out[b] = found ? best_i : -1;
        if (f.row_status) f.row_status[b] = found ? 0 : 1;
    }
}

template <typename T>
cudaError_t launch_typed(const void* logits, int64_t ld, bool wide, const FilterArgs& f,
                         cudaStream_t stream) {
    const unsigned grid = static_cast<unsigned>(f.a.B);
    const T* y = static_cast<const T*>(logits);
    if (wide) {
        filtered_race_kernel<T, true><<<grid, kThreads, 0, stream>>>(y, ld, f);
    } else {
        filtered_race_kernel<T, false><<<grid, kThreads, 0, stream>>>(y, ld, f);
    }
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_filtered_race(const void* logits, bool bf16, int64_t ld, bool wide,
                                 const FilterArgs& f, cudaStream_t stream) {
    return bf16 ? launch_typed<__nv_bfloat16>(logits, ld, wide, f, stream)
                : launch_typed<float>(logits, ld, wide, f, stream);
}

}  // namespace lms
