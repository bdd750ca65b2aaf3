// Filtered Gumbel race over materialised logits: top-k -> top-p -> min-p on t = (y + bias) / T,
// then the race over the kept tokens (spec-decode-ops "Semantics": top-p keeps the shortest
// sorted prefix whose mass, normalised over the top-k prefix, reaches top_p, crossing token
// included; min-p keeps p >= min_p * p_max; every filter keeps at least one token.  The
// sampling-kernel guide, reasoning steps 6-8: top-k before top-p, a compile-time bound K_MAX on
// the candidate set).  The race over a subset samples the renormalised softmax, so nothing is
// normalised except the top-p prefix mass.
//
// One CTA of 1024 threads per row:
//   1. radix select (4 passes of 8 bits over order-preserving 32-bit keys of t, histograms built
//      with warp-aggregated shared-memory atomics) finds the key K of the k-th largest entry,
//      k = min(top_k, k_max) (k_max when only top-p is on); if fewer entries equal to K are kept
//      than exist, a second radix select over their indices finds the largest kept index, so ties
//      keep the smallest indices;
//   2. one pass gathers exactly k candidates (key > K, or key == K and index <= that bound);
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

// hist[bin] += 1 for every thread with `in`, one shared-memory atomic per distinct bin per warp.
// Every lane of the warp must call it (full-mask ballot).
__device__ __forceinline__ void hist_add(int* hist, uint32_t bin, bool in) {
    const unsigned active = __ballot_sync(0xffffffffu, in);
    if (in) {
        const unsigned peers = __match_any_sync(active, bin);
        if ((threadIdx.x & 31) == __ffs(peers) - 1) atomicAdd(&hist[bin], __popc(peers));
    }
}

// Warp 0 (called by its 32 lanes): the bin where the count from the top (bin 255 down) reaches
// `need`; writes the bin and the rank left inside it.  Lane l owns bins 255-8l .. 248-8l.
__device__ __forceinline__ void find_bin_desc(const int* hist, int need, int* bin_out, int* rem_out) {
    const int l = threadIdx.x & 31;
    int local = 0;
#pragma unroll
    for (int j = 0; j < 8; ++j) local += hist[255 - 8 * l - j];
    int incl = local;
    for (int off = 1; off < 32; off <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, off);
        if (l >= off) incl += y;
    }
    const int excl = incl - local;
    if (excl < need && need <= incl) {
        int cum = excl, j = 0;
        for (; j < 7; ++j) {
            const int h = hist[255 - 8 * l - j];
            if (cum + h >= need) break;
            cum += h;
        }
        *bin_out = 255 - 8 * l - j;
        *rem_out = need - cum;
    }
}

// The same from the bottom (bin 0 up), for the ascending index select.
__device__ __forceinline__ void find_bin_asc(const int* hist, int need, int* bin_out, int* rem_out) {
    const int l = threadIdx.x & 31;
    int local = 0;
#pragma unroll
    for (int j = 0; j < 8; ++j) local += hist[8 * l + j];
    int incl = local;
    for (int off = 1; off < 32; off <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, off);
        if (l >= off) incl += y;
    }
    const int excl = incl - local;
    if (excl < need && need <= incl) {
        int cum = excl, j = 0;
        for (; j < 7; ++j) {
            const int h = hist[8 * l + j];
            if (cum + h >= need) break;
            cum += h;
        }
        *bin_out = 8 * l + j;
        *rem_out = need - cum;
    }
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

    float best_s = -CUDART_INF_F;
    int best_i = kNoIndex;
    if (greedy || !(topk_on || topp_on)) {
        // t_max over the row (for the min-p threshold)
        float tmax = -CUDART_INF_F;
        for (int64_t v = tid; v < V; v += kThreads) tmax = fmaxf(tmax, t_of<T>(r, v));
        tmax = block_max(tmax, shf);
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
            // whole 1024-wide chunks, so that every lane of every warp reaches hist_add
            for (int64_t base = 0; base < V; base += kThreads) {
                const int64_t v = base + tid;
                const bool valid = v < V;
                const uint32_t key = valid ? order_key(t_of<T>(r, v)) : 0u;
                hist_add(hist, (key >> shift) & 255u, valid && (key & pmask) == prefix);
            }
            __syncthreads();
            if (tid < 32) find_bin_desc(hist, remaining, &sh_int[0], &sh_int[1]);
            __syncthreads();
            prefix |= static_cast<uint32_t>(sh_int[0]) << shift;
            pmask |= 255u << shift;
            remaining = sh_int[1];
            __syncthreads();
        }
        const uint32_t kstar = prefix;   // the k-th largest key
        const int need_eq = remaining;   // entries equal to it that are kept (smallest indices)
        // ties at K: the need_eq-th smallest index among entries with key == K, by a radix select
        // over the index bits (ascending); skipped when every such entry is kept
        int eq_count = 0;
        for (int64_t v = tid; v < V; v += kThreads) eq_count += order_key(t_of<T>(r, v)) == kstar;
        eq_count = block_sum<int>(eq_count, shi);
        uint32_t vmax = 0xffffffffu;
        if (need_eq < eq_count) {
            int bits = 1;
            while ((int64_t{1} << bits) < V) ++bits;
            uint32_t vprefix = 0, vmask = 0;
            int rem = need_eq;
            for (int shift = ((bits + 7) / 8 - 1) * 8; shift >= 0; shift -= 8) {
                if (tid < 256) hist[tid] = 0;
                __syncthreads();
                for (int64_t base = 0; base < V; base += kThreads) {
                    const int64_t v = base + tid;
                    const bool in = v < V && order_key(t_of<T>(r, v)) == kstar &&
                                    (static_cast<uint32_t>(v) & vmask) == vprefix;
                    hist_add(hist, (static_cast<uint32_t>(v) >> shift) & 255u, in);
                }
                __syncthreads();
                if (tid < 32) find_bin_asc(hist, rem, &sh_int[0], &sh_int[1]);
                __syncthreads();
                vprefix |= static_cast<uint32_t>(sh_int[0]) << shift;
                vmask |= 255u << shift;
                rem = sh_int[1];
                __syncthreads();
            }
            vmax = vprefix;
        }
        // ---- 2. gather exactly min(k, V) candidates (unordered; sorted next) ----
        if (tid == 0) sh_int[2] = 0;
        cand[tid] = 0ull;                // below every real candidate (kMaxK == kThreads)
        __syncthreads();
        for (int64_t v = tid; v < V; v += kThreads) {
            const uint32_t key = order_key(t_of<T>(r, v));
            if (key > kstar || (key == kstar && static_cast<uint32_t>(v) <= vmax)) {
                const int pos = atomicAdd(&sh_int[2], 1);
                if (pos < kMaxK)
                    cand[pos] = (static_cast<unsigned long long>(key) << 32) |
                                static_cast<uint32_t>(~static_cast<uint32_t>(v));
            }
        }
        __syncthreads();
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
