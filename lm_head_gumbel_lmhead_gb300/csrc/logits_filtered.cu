// Filtered Gumbel race over materialised logits: top-k -> top-p -> min-p on t = (y + bias) / T,
// then the race over the kept tokens (spec-decode-ops "Semantics": top-p keeps the shortest
// sorted prefix whose mass, normalised over the top-k prefix, reaches top_p, crossing token
// included; min-p keeps p >= min_p * p_max; every filter keeps at least one token.  The
// sampling-kernel guide, reasoning steps 6-8: top-k before top-p, a compile-time bound K_MAX on
// the candidate set).  The race over a subset samples the renormalised softmax, so nothing is
// normalised except the top-p prefix mass.
//
// One thread-block cluster per row; CTA c of the cluster owns the slice [c S, (c + 1) S) of the
// vocabulary (S a multiple of 8).
//   0. Each CTA reads its slice once (16-byte loads, several in flight per thread), turns every
//      entry into an order-preserving 32-bit key of t (kept in shared memory when the slice fits,
//      else recomputed from global memory on every pass) and finds the slice's largest key; the
//      CTAs exchange these through distributed shared memory, so each knows the row's largest key.
//   1. Radix select, over the cluster, of the kk-th smallest rank row_max - key, kk = min(top_k,
//      k_max) (k_max when only top-p is on).  A first pass histograms only the entries within 2^24
//      keys of the row max (about two octaves of t) on rank bits 23..16; the others, usually most
//      of the row, cost no atomic.  When at least kk entries are that close the top level is
//      settled, else the select starts from the top byte.  Per 8-bit level each CTA sums the
//      cluster's histograms (per-warp copies folded per CTA, then read remotely) and finds the
//      same bin.  It stops as soon as the bin holding the kk-th entry is kept whole, or the entries
//      ahead of it plus the bin number at most 2048 with at most 256 in the bin; otherwise it runs
//      down to the full key K, and of the entries equal to K the smallest indices are kept: slices
//      are in index order, so each CTA works out how many of its own to keep and finds its cut
//      with a block scan.
//   2. Every CTA appends its entries to the leader CTA's candidate list with
//      distributed-shared-memory atomics and stores; the other CTAs then exit.
//   3. The leader, with the candidates in no particular order: keeps the kk best (ranking the
//      boundary bin's entries among themselves when it holds more), cuts top-p with a radix
//      select over per-bin masses exp(t - t0) in 2^-40 fixed point (exact, order-independent
//      sums; ties at the crossing key kept by index), applies the min-p threshold
//      t0 + log(min_p), and runs the race over what is left with the unfiltered race's Philox
//      noise.  Nothing is sorted.
// Rows with only min-p (or no filter, or greedy rows) skip 1-3: every CTA races over its slice
// above the threshold and the leader takes the best of the cluster's candidates.
//
// Every decision that selects a cluster barrier is made from row parameters or from values every
// CTA of the cluster computes identically (merged histograms, the exchanged maxima), so all CTAs
// pass the same sequence of barriers; a CTA exits only after the last barrier behind which a peer
// reads its shared memory.  There are no spin-waits.
#include <cuda_bf16.h>

#include <mutex>

#include "lms_device.cuh"
#include "lms_kernels.h"

namespace lms {
namespace {

constexpr int kThreads = 512;
constexpr int kWarps = kThreads / 32;
// The leader's candidate list: the kk <= 1024 entries of the top-k cut, or a superset of at most
// kCap entries made of the entries above the bin holding the kk-th one plus that whole bin, when
// the bin holds at most kTie entries (the leader then ranks the bin's entries among themselves).
constexpr int kCap = 2048;
constexpr int kTie = 256;
static_assert(kCap == 4 * kThreads, "the leader gives each thread four candidates");
// Largest slice whose keys stay in shared memory (176 KiB of keys; with the static shared memory
// below, within the 227 KiB a block may opt into).
constexpr int64_t kMaxSmemSlice = 44 * 1024;
// Key of t = -inf; every entry of a row has a key >= this one.
constexpr uint32_t kKeyNegInf = 0x007fffffu;

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
};

// Transformed logit t (no noise): -inf when masked or NaN.
template <typename T>
__device__ __forceinline__ float t_of(const RowView& r, int64_t v) {
    if (r.mask && !((__ldg(r.mask + (v >> 5)) >> (v & 31)) & 1u)) return -CUDART_INF_F;
    const float y = to_f<T>(static_cast<const T*>(r.y)[v]) + (r.bias ? __ldg(r.bias + v) : 0.0f);
    const float t = (r.p.flags & kRowGreedy) ? y : y * r.p.inv_t;
    return t == t ? t : -CUDART_INF_F;
}

// Load pass over a slice: t of each entry as an order key (stored in `keys` when kSmemKeys),
// returns the largest key this thread saw.  Units of 8 entries (v a multiple of 8); each thread
// issues the loads of kUnits units before it uses any of them (fewer when a bias row is read too).
template <int kUnits, bool kBias, bool kSmemKeys, typename T>
__device__ __forceinline__ uint32_t load_slice(const RowView& r, const T* yrow, const float* brow,
                                               int64_t v_begin, int n_loc, uint32_t* keys) {
    const int tid = threadIdx.x;
    const bool vec_y = (reinterpret_cast<uintptr_t>(yrow) & 15u) == 0;
    const bool vec_b = kBias && (reinterpret_cast<uintptr_t>(brow) & 15u) == 0;
    const int n_units = (n_loc + 7) >> 3;
    uint32_t kmax = 0u;
    for (int base = 0; base < n_units; base += kUnits * kThreads) {
        const int u0 = base + tid;
        float y[kUnits][8];
        float bs[kBias ? kUnits : 1][8];
        uint32_t bits[kUnits];
#pragma unroll
        for (int q = 0; q < kUnits; ++q) {
            const int j0 = 8 * (u0 + q * kThreads);
            const int n = n_loc - j0;             // entries of this unit (<= 0: none)
            load8(yrow + j0, n, vec_y, y[q]);
            if constexpr (kBias) load8(brow + j0, n, vec_b, bs[q]);
            const int64_t v0 = v_begin + j0;
            bits[q] = (r.mask == nullptr || n <= 0) ? 0xffu
                                                    : (__ldg(r.mask + (v0 >> 5)) >> (v0 & 31)) & 0xffu;
        }
#pragma unroll
        for (int q = 0; q < kUnits; ++q) {
            const int j0 = 8 * (u0 + q * kThreads);
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                if (j0 + e < n_loc) {
                    const float yb = kBias ? y[q][e] + bs[kBias ? q : 0][e] : y[q][e];
                    float t = (r.p.flags & kRowGreedy) ? yb : yb * r.p.inv_t;
                    t = (((bits[q] >> e) & 1u) && t == t) ? t : -CUDART_INF_F;
                    const uint32_t key = order_key(t);
                    if constexpr (kSmemKeys) keys[j0 + e] = key;
                    kmax = max(kmax, key);
                }
            }
        }
    }
    return kmax;
}

// ---- cluster plumbing ----
__device__ __forceinline__ uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

__device__ __forceinline__ uint32_t cluster_size() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(r));
    return r;
}

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// The shared::cluster address of shared::cta address `addr` in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t map_rank(uint32_t addr, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
    return r;
}

__device__ __forceinline__ uint32_t ld_cluster_u32(uint32_t caddr) {
    uint32_t v;
    asm volatile("ld.shared::cluster.u32 %0, [%1];" : "=r"(v) : "r"(caddr));
    return v;
}

// Sum (or max) of the u32 at shared::cta address `addr` over CTAs 0 .. n-1 of the cluster
// (n <= 16): the remote loads are issued together, then combined.
template <bool kMax>
__device__ __forceinline__ uint32_t cluster_reduce_u32(uint32_t addr, uint32_t n) {
    uint32_t v[16];
#pragma unroll
    for (uint32_t c = 0; c < 16; ++c) v[c] = c < n ? ld_cluster_u32(map_rank(addr, c)) : 0u;
    uint32_t acc = 0u;
#pragma unroll
    for (int c = 0; c < 16; ++c) acc = kMax ? max(acc, v[c]) : acc + v[c];
    return acc;
}

__device__ __forceinline__ void st_cluster_u32(uint32_t caddr, uint32_t v) {
    asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(caddr), "r"(v) : "memory");
}

__device__ __forceinline__ void st_cluster_u64(uint32_t caddr, unsigned long long v) {
    asm volatile("st.shared::cluster.u64 [%0], %1;" ::"r"(caddr), "l"(v) : "memory");
}

__device__ __forceinline__ uint32_t atom_add_cluster(uint32_t caddr, uint32_t v) {
    uint32_t old;
    asm volatile("atom.shared::cluster.add.u32 %0, [%1], %2;" : "=r"(old) : "r"(caddr), "r"(v) : "memory");
    return old;
}

// Every thread of every CTA of the cluster; orders shared-memory accesses across the cluster.
__device__ __forceinline__ void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
    asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// ---- block helpers (all threads of the CTA call them) ----
__device__ __forceinline__ uint32_t block_max_u32(uint32_t x, uint32_t* sh) {
    for (int off = 16; off > 0; off >>= 1) x = max(x, __shfl_xor_sync(0xffffffffu, x, off));
    const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
    __syncthreads();
    if (l == 0) sh[w] = x;
    __syncthreads();
    x = (threadIdx.x < kWarps) ? sh[threadIdx.x] : 0u;
    if (w == 0)
        for (int off = 16; off > 0; off >>= 1) x = max(x, __shfl_xor_sync(0xffffffffu, x, off));
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
        X s = l < kWarps ? sh[l] : X(0);
        for (int off = 1; off < 32; off <<= 1) {
            const X y = __shfl_up_sync(0xffffffffu, s, off);
            if (l >= off) s += y;
        }
        if (l < kWarps) sh[l] = s;
    }
    __syncthreads();
    const X r = w > 0 ? x + sh[w - 1] : x;
    __syncthreads();
    return r;
}

// Block argmax of (score, index), larger score then smaller index; result in every thread.
__device__ __forceinline__ void block_argmax(float& s, int& i, float* shs, int* shi) {
    warp_argmax(s, i);
    const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
    __syncthreads();
    if (l == 0) { shs[w] = s; shi[w] = i; }
    __syncthreads();
    if (w == 0) {
        s = l < kWarps ? shs[l] : -CUDART_INF_F;
        i = l < kWarps ? shi[l] : kNoIndex;
        warp_argmax(s, i);
        if (l == 0) { shs[0] = s; shi[0] = i; }
    }
    __syncthreads();
    s = shs[0];
    i = shi[0];
}

// Histogram add with run-length aggregation: a thread's consecutive entries that fall in the same
// bin cost one shared-memory atomic.  No warp-synchronous step.
struct RunCount {
    uint32_t bin = 0xffffffffu;
    int n = 0;
    __device__ __forceinline__ void add(int* hist, uint32_t b) {
        if (b == bin) { ++n; return; }
        if (n) atomicAdd(&hist[bin], n);
        bin = b;
        n = 1;
    }
    __device__ __forceinline__ void flush(int* hist) {
        if (n) atomicAdd(&hist[bin], n);
        n = 0;
    }
};

// hist[t] = sum of the warps' histograms at bin t, which are cleared for the next pass (threads
// t < 256; the caller separates the warps' adds from this with a block barrier).
__device__ __forceinline__ void fold_warp_hists(int (*whist)[256], int* hist) {
    const int t = threadIdx.x;
    if (t < 256) {
        int sum = 0;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) {
            sum += whist[w][t];
            whist[w][t] = 0;
        }
        hist[t] = sum;
    }
}

// Warp 0 (called by its 32 lanes): the bin where the count from the bottom (bin 0 up) reaches
// `need`; writes the bin, the rank left inside it and the bin's count.  Lane l owns bins
// 8l .. 8l + 7.  0 < need <= the histogram's total.
__device__ __forceinline__ void find_bin_asc(const int* hist, int need, int* out3) {
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
        out3[0] = 8 * l + j;
        out3[1] = need - cum;
        out3[2] = hist[8 * l + j];
    }
}

__device__ __forceinline__ int block_sum_int(int x, int* sh) {
    for (int off = 16; off > 0; off >>= 1) x += __shfl_xor_sync(0xffffffffu, x, off);
    const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
    __syncthreads();
    if (l == 0) sh[w] = x;
    __syncthreads();
    x = l < kWarps ? sh[l] : 0;
    for (int off = 16; off > 0; off >>= 1) x += __shfl_xor_sync(0xffffffffu, x, off);
    __syncthreads();
    return x;
}

// exp(d) for d <= 0 in 2^-40 fixed point (1.0 -> 2^40).
__device__ __forceinline__ unsigned long long fixed_mass(float d) {
    return static_cast<unsigned long long>(__expf(d) * 0x1p40f + 0.5f);
}

__device__ __forceinline__ unsigned long long block_sum_u64(unsigned long long x, unsigned long long* sh) {
    for (int off = 16; off > 0; off >>= 1) x += __shfl_xor_sync(0xffffffffu, x, off);
    const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
    __syncthreads();
    if (l == 0) sh[w] = x;
    __syncthreads();
    x = l < kWarps ? sh[l] : 0ull;
    for (int off = 16; off > 0; off >>= 1) x += __shfl_xor_sync(0xffffffffu, x, off);
    __syncthreads();
    return x;
}

// ceil(p * Z) for 0 < p < 1 (fp32) and Z < 2^63, exactly: p = m 2^-s with m < 2^24, so
// p Z = m Z / 2^s with the 128-bit product m Z.
__device__ __forceinline__ unsigned long long ceil_frac_times(float p, unsigned long long Z) {
    const uint32_t bits = __float_as_uint(p);
    const uint32_t e = (bits >> 23) & 255u;
    const unsigned long long m = e ? ((bits & 0x7fffffu) | 0x800000u) : (bits & 0x7fffffu);
    const int s = e ? 150 - static_cast<int>(e) : 149;   // p = m / 2^s, s >= 24 for p < 1
    const unsigned long long lo = m * Z, hi = __umul64hi(m, Z);
    if (s >= 128) return (lo | hi) ? 1ull : 0ull;
    unsigned long long q, rem;
    if (s >= 64) {
        q = hi >> (s - 64);
        rem = lo | (s > 64 ? (hi & ((1ull << (s - 64)) - 1ull)) : 0ull);
    } else {
        q = (lo >> s) | (hi << (64 - s));
        rem = lo & ((1ull << s) - 1ull);
    }
    return q + (rem ? 1ull : 0ull);
}

// Warp 0 (called by its 32 lanes): scanning the bins from 0 up, the first bin where the
// cumulative mass (bin b holds mhi[b] 2^20 + mlo[b]) reaches `need` (> 0); writes the bin to out[0] and the mass of the bins before
// it to mass_out[0].  If the total is below `need`, the last non-empty bin.
__device__ __forceinline__ void find_mass_bin_asc(const uint32_t* mlo, const uint32_t* mhi,
                                                  unsigned long long need, int* out,
                                                  unsigned long long* mass_out) {
    auto mh = [&](int bin) -> unsigned long long {
        return (static_cast<unsigned long long>(mhi[bin]) << 20) + mlo[bin];
    };
    const int l = threadIdx.x & 31;
    unsigned long long local = 0ull;
#pragma unroll
    for (int j = 0; j < 8; ++j) local += mh(8 * l + j);
    unsigned long long incl = local;
    for (int off = 1; off < 32; off <<= 1) {
        const unsigned long long y = __shfl_up_sync(0xffffffffu, incl, off);
        if (l >= off) incl += y;
    }
    const unsigned long long excl = incl - local;
    const unsigned long long total = __shfl_sync(0xffffffffu, incl, 31);
    const unsigned long long goal = total < need ? total : need;
    if (excl < goal && goal <= incl) {
        unsigned long long cum = excl;
        int j = 0;
        for (; j < 7; ++j) {
            const unsigned long long h = mh(8 * l + j);
            if (cum + h >= goal) break;
            cum += h;
        }
        out[0] = 8 * l + j;
        mass_out[0] = cum;
    }
}

template <typename T, bool kWide, bool kSmemKeys>
__global__ void __launch_bounds__(kThreads, 2) filtered_race_cluster_kernel(
    const T* __restrict__ logits, int64_t ld, FilterArgs f, int64_t S) {
    extern __shared__ __align__(16) uint32_t keys[];     // [S] when kSmemKeys
    __shared__ unsigned long long cand[kCap];            // leader: (key << 32) | ~v
    __shared__ unsigned long long tiebuf[kTie];          // leader: entries of one key bin or tie
    __shared__ uint32_t mlo[256], mhi[256];              // leader: per-bin masses, low 20 bits / rest
    __shared__ unsigned long long shl[kWarps];
    __shared__ uint32_t tie_count;
    __shared__ int whist[kWarps][256];                   // per-warp histograms of the current pass
    __shared__ int hist[2][256];                         // this CTA's histograms, read by peers
    __shared__ int ghist[256];                           // the cluster's merged histogram
    __shared__ uint32_t xch_max;                         // this CTA's largest key, read by peers
    __shared__ uint32_t cand_count;                      // leader: candidates appended
    __shared__ float slot_s[16];                         // leader: per-CTA race winners
    __shared__ int slot_i[16];
    __shared__ float shf[kWarps];
    __shared__ int shi[kWarps];
    __shared__ uint32_t shu[kWarps];
    __shared__ int sh_int[8];
    __shared__ uint32_t xch_near;                        // this CTA's entries near the row max

    const SampleArgs& a = f.a;
    const uint32_t rank = cluster_rank();
    const uint32_t csize = cluster_size();
    const int64_t b = blockIdx.x / csize;
    const int64_t row = a.row0 + b;
    const int tid = threadIdx.x;
    const int64_t V = a.V;
    RowView r;
    r.p = make_row_params(a.temperature, a.seeds, a.positions, a.base_seed, a.offset, row);
    r.y = logits + row * ld;
    r.bias = a.bias ? a.bias + row * a.ld_bias : nullptr;
    r.mask = a.mask ? a.mask + row * a.ld_mask : nullptr;
    const int64_t v_begin = static_cast<int64_t>(rank) * S;
    const int n_loc = static_cast<int>(v_begin < V ? (V - v_begin < S ? V - v_begin : S) : 0);

    if (r.p.flags & kRowInvalid) {     // uniform over the cluster; no shared memory touched
        if (rank == 0 && tid == 0) { f.out[b] = -1; if (f.row_status) f.row_status[b] = 2; }
        return;
    }
    const int tk = f.top_k ? f.top_k[row] : 0;
    const float tp = f.top_p ? f.top_p[row] : 1.0f;
    const float mp = f.min_p ? f.min_p[row] : 0.0f;
    const bool topk_on = tk >= 1 && tk < V;
    const bool topp_on = tp > 0.0f && tp < 1.0f;
    const bool minp_on = mp > 0.0f && mp <= 1.0f;
    const bool greedy = r.p.flags & kRowGreedy;
    const bool select = !greedy && (topk_on || topp_on);

    auto key_at = [&](int j) -> uint32_t {
        if constexpr (kSmemKeys) return keys[j];
        else return order_key(t_of<T>(r, v_begin + j));
    };

    if (tid < 256) {
#pragma unroll
        for (int w = 0; w < kWarps; ++w) whist[w][tid] = 0;
    }
    if (tid == 0) cand_count = 0u;
    __syncthreads();

    // ---- 0. load: keys and the slice's largest key ----
    uint32_t kmax;
    {
        const T* yrow = static_cast<const T*>(r.y) + v_begin;
        const float* brow = r.bias ? r.bias + v_begin : nullptr;
        kmax = brow ? load_slice<2, true, kSmemKeys>(r, yrow, brow, v_begin, n_loc, keys)
                    : load_slice<4, false, kSmemKeys>(r, yrow, brow, v_begin, n_loc, keys);
    }
    kmax = block_max_u32(kmax, shu);     // ends with a block barrier: the keys are complete
    if (tid == 0) xch_max = kmax;
    cluster_sync();                      // (A) the slices' maxima are visible
    uint32_t row_max = 0u;
    {
        if (tid == 0) sh_int[3] = static_cast<int>(cluster_reduce_u32<true>(smem_u32(&xch_max), csize));
    }
    // (read below, after the next block barrier)

    float best_s = -CUDART_INF_F;
    int best_i = kNoIndex;
    if (!select) {
        __syncthreads();
        row_max = static_cast<uint32_t>(sh_int[3]);
        // Greedy rows, min-p only, or no filter: one threshold race over the slice.  Greedy rows
        // need no filter (every filter keeps the top token).
        const float tmax = key_value(row_max);
        const float thr = (minp_on && !greedy) ? tmax + logf(mp) : -CUDART_INF_F;
        for (int j0 = 4 * tid; j0 < n_loc; j0 += 4 * kThreads) {
            float g[4] = {0.0f, 0.0f, 0.0f, 0.0f};
            if (!greedy) gumbel_run<kWide, 4>(r.p.key, static_cast<uint32_t>(v_begin + j0), g);
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int j = j0 + e;
                if (j < n_loc) {
                    const float t = key_value(key_at(j));
                    if (t > -CUDART_INF_F && t >= thr) {
                        const float s = greedy ? t : t + g[e];
                        const int v = static_cast<int>(v_begin + j);
                        if (better(s, v, best_s, best_i)) { best_s = s; best_i = v; }
                    }
                }
            }
        }
        block_argmax(best_s, best_i, shf, shi);
        if (tid == 0) {
            st_cluster_u32(map_rank(smem_u32(&slot_s[rank]), 0), __float_as_uint(best_s));
            st_cluster_u32(map_rank(smem_u32(&slot_i[rank]), 0), static_cast<uint32_t>(best_i));
        }
        cluster_sync();                  // (B) winners in the leader; peers' maxima read
        if (rank != 0) return;
        if (tid == 0) {
            for (uint32_t c = 0; c < csize; ++c)
                if (better(slot_s[c], slot_i[c], best_s, best_i)) { best_s = slot_s[c]; best_i = slot_i[c]; }
        }
    } else {
        const int k_cap = f.k_max;
        const int k = topk_on ? (tk < k_cap ? tk : k_cap) : k_cap;
        const int kk = static_cast<int>(k < V ? k : V);   // entries kept by the top-k cut
        __syncthreads();
        row_max = static_cast<uint32_t>(sh_int[3]);
        const bool nothing = row_max <= kKeyNegInf;   // no finite entry in the row
        // Ranks rk = row_max - key (0 for the largest entry; larger for smaller t).  The select
        // finds the kk-th smallest rank, 8 bits per level from the top.
        auto rank_at = [&](int j) -> uint32_t { return row_max - key_at(j); };
        int remaining = kk;
        uint32_t prefix = 0u, pmask = 0u;      // on ranks
        bool gather_all = kk == V;             // every entry kept (V <= k_max): no select
        int last_buf = 0, last_bin = 0;
        int level = 0;
        bool level1_built = false;
        if (!gather_all && !nothing) {
            // Near pass: the entries within 2^24 keys (about two octaves) of the row max are
            // counted and histogrammed on rank bits 23..16; the others, usually most of the row,
            // cost no atomic.  If at least kk entries are near, the top level is settled (its bin
            // is 0) and the next one is built already.
            int near = 0;
            {
                int* wh = whist[tid >> 5];
                RunCount rc;
#pragma unroll 4
                for (int j = tid; j < n_loc; j += kThreads) {
                    const uint32_t rk = rank_at(j);
                    if (rk < (1u << 24)) {
                        ++near;
                        rc.add(wh, rk >> 16);
                    }
                }
                rc.flush(wh);
            }
            near = block_sum_int(near, shi);     // its block barriers also order the warps' adds
            fold_warp_hists(whist, hist[1]);
            if (tid == 0) xch_near = static_cast<uint32_t>(near);
            cluster_sync();                  // (N) near counts and hist[1] visible
            if (tid == 0) sh_int[4] = static_cast<int>(cluster_reduce_u32<false>(smem_u32(&xch_near), csize));
            __syncthreads();
            if (sh_int[4] >= kk) {
                pmask = 0xff000000u;
                level = 1;
                level1_built = true;
            }
        }
        // ---- 1. radix select over the cluster, 8 bits per level ----
        for (; level < 4 && !gather_all && !nothing; ++level) {
            const int shift = 24 - 8 * level;
            const int buf = level & 1;
            if (!(level == 1 && level1_built)) {
                // hist[buf] (rewritten by the fold) was last read by peers two barriers ago (at
                // barrier (N) or a previous level's), and every peer has passed the barrier after
                // that read
                {
                    int* wh = whist[tid >> 5];
                    RunCount rc;
#pragma unroll 4
                    for (int j = tid; j < n_loc; j += kThreads) {
                        const uint32_t rk = rank_at(j);
                        if ((rk & pmask) == prefix) rc.add(wh, (rk >> shift) & 255u);
                    }
                    rc.flush(wh);
                }
                __syncthreads();
                fold_warp_hists(whist, hist[buf]);
                cluster_sync();
            }
            if (tid < 256) {
                ghist[tid] = static_cast<int>(cluster_reduce_u32<false>(smem_u32(&hist[buf][tid]), csize));
            }
            __syncthreads();
            if (tid < 32) find_bin_asc(ghist, remaining, sh_int);
            __syncthreads();
            const int bin = sh_int[0];
            prefix |= static_cast<uint32_t>(bin) << shift;
            pmask |= 255u << shift;
            last_buf = buf;
            last_bin = bin;
            remaining = sh_int[1];
            // gather now if the bin is kept whole (exactly kk entries), or if the entries ahead of
            // the bin (kk - remaining) plus the bin fit the leader's list and the bin is small
            // enough for the leader to rank its entries among themselves
            gather_all = sh_int[2] == remaining || (kk - remaining + sh_int[2] <= kCap && sh_int[2] <= kTie);
            __syncthreads();
        }
        // gather_all: every entry with (rank & pmask) <= prefix goes to the leader (kk of them, or
        // at most kCap with at most kTie in the boundary bin).
        // Otherwise all 32 bits are resolved to the rank R of key K = row_max - R: entries with a
        // smaller rank are kept and, of those equal to it, `remaining`, smallest index first.
        int j_cut = 0x7fffffff;                // keep entries of rank R with local offset <= j_cut
        if (!nothing && !gather_all) {
            // counts of R in the lower-ranked slices (their last histograms, read remotely)
            if (tid == 0) {
                sh_int[0] = static_cast<int>(cluster_reduce_u32<false>(smem_u32(&hist[last_buf][last_bin]), rank));
            }
            __syncthreads();
            const int eq_here = hist[last_buf][last_bin];
            int keep = remaining - sh_int[0];
            keep = keep < 0 ? 0 : (keep > eq_here ? eq_here : keep);
            __syncthreads();
            if (keep == 0) {
                j_cut = -1;
            } else if (keep < eq_here) {
                // contiguous runs of C offsets per thread, so the block scan follows index order
                // (C odd: the lanes of a warp start in distinct shared-memory banks)
                const int C = ((n_loc + kThreads - 1) / kThreads) | 1;
                const int j0 = tid * C;
                const int j1 = j0 + C < n_loc ? j0 + C : n_loc;
                int cnt = 0;
                for (int j = j0; j < j1; ++j) cnt += rank_at(j) == prefix;
                const int incl = block_scan_incl<int>(cnt, shi);
                const int excl = incl - cnt;
                if (excl < keep && keep <= incl) {
                    int c = excl;
                    for (int j = j0; j < j1; ++j) {
                        if (rank_at(j) == prefix && ++c == keep) { sh_int[1] = j; break; }
                    }
                }
                __syncthreads();
                j_cut = sh_int[1];
            }
        }
        // ---- 2. append the kept entries to the leader's candidate list ----
        if (!nothing) {
            const uint32_t count_addr = map_rank(smem_u32(&cand_count), 0);
            const uint32_t cand_addr = map_rank(smem_u32(&cand[0]), 0);
            const int lane = tid & 31;
#pragma unroll 4
            for (int base = 0; base < n_loc; base += kThreads) {      // uniform trip count
                const int j = base + tid;
                bool in = false;
                uint32_t key = 0u;
                if (j < n_loc) {
                    key = key_at(j);
                    const uint32_t m = (row_max - key) & pmask;
                    in = gather_all ? m <= prefix : (m < prefix || (m == prefix && j <= j_cut));
                }
                const unsigned bal = __ballot_sync(0xffffffffu, in);
                if (bal) {
                    uint32_t pos0 = 0u;
                    if (lane == 0) pos0 = atom_add_cluster(count_addr, __popc(bal));
                    pos0 = __shfl_sync(0xffffffffu, pos0, 0);
                    if (in) {
                        const uint32_t pos = pos0 + __popc(bal & ((1u << lane) - 1u));
                        const uint32_t v = static_cast<uint32_t>(v_begin + j);
                        if (pos < static_cast<uint32_t>(kCap))
                            st_cluster_u64(cand_addr + 8u * pos,
                                           (static_cast<unsigned long long>(key) << 32) | (~v));
                    }
                }
            }
        }
        cluster_sync();                  // (C) candidates in the leader; peers' histograms read
        if (rank != 0) return;
        // ---- 3. leader: top-k membership, top-p cut, min-p threshold, race ----
        // Thread t holds candidates t + h kThreads (h < 4); the list's order is arbitrary and
        // nothing below needs it sorted.
        const int n = nothing ? 0 : (cand_count < static_cast<uint32_t>(kCap) ? static_cast<int>(cand_count) : kCap);
        const float t0 = key_value(row_max);
        unsigned long long c[4];
        bool kept[4];
#pragma unroll
        for (int h = 0; h < 4; ++h) {
            const int i = tid + h * kThreads;
            c[h] = i < n ? cand[i] : 0ull;
            kept[h] = i < n;
        }
        if (n > kk) {
            // The entries ahead of the boundary bin plus the whole bin: keep the `remaining` best
            // entries of the bin (larger key, then smaller index), ranked among themselves.
            if (tid == 0) tie_count = 0u;
            __syncthreads();
#pragma unroll
            for (int h = 0; h < 4; ++h) {
                if (kept[h] && ((row_max - static_cast<uint32_t>(c[h] >> 32)) & pmask) == prefix) {
                    const uint32_t pos = atomicAdd(&tie_count, 1u);
                    if (pos < static_cast<uint32_t>(kTie)) tiebuf[pos] = c[h];
                }
            }
            __syncthreads();
            const int nb = tie_count < static_cast<uint32_t>(kTie) ? static_cast<int>(tie_count) : kTie;
#pragma unroll
            for (int h = 0; h < 4; ++h) {
                if (kept[h] && ((row_max - static_cast<uint32_t>(c[h] >> 32)) & pmask) == prefix) {
                    int ahead = 0;
                    for (int j = 0; j < nb; ++j) ahead += tiebuf[j] > c[h];
                    kept[h] = ahead < remaining;
                }
            }
            __syncthreads();
#pragma unroll
            for (int h = 0; h < 4; ++h)
                if (tid + h * kThreads < n && !kept[h]) cand[tid + h * kThreads] = 0ull;   // dropped
            __syncthreads();
        }
        if (topp_on && kk > 1) {
            // Top-p: keep the entries whose mass strictly before them in (t desc, v asc) order
            // is below top_p * Z.  Masses exp(t - t0) in 2^-40 fixed point, so every sum is exact
            // and independent of the order of the atomics; the cut is found by a radix select
            // on the ranks with per-bin masses.
            // (each mass is recomputed where it is needed rather than held in registers)
            auto mass = [&](int h) -> unsigned long long {
                return fixed_mass(key_value(static_cast<uint32_t>(c[h] >> 32)) - t0);
            };
            unsigned long long msum = 0ull;
#pragma unroll
            for (int h = 0; h < 4; ++h)
                if (kept[h]) msum += mass(h);
            const unsigned long long Z = block_sum_u64(msum, shl);
            const unsigned long long target = ceil_frac_times(tp, Z);   // keep iff mass before < target
            // radix select on ranks row_max - key (ascending = t descending); every candidate of
            // the near select has rank < 2^24, so its top byte is settled
            uint32_t pfx = 0u, pm = level1_built ? 0xff000000u : 0u;
            unsigned long long before = 0ull;    // mass of the entries ahead of the current bin
            int ties = 0;
            for (int level = level1_built ? 1 : 0; level < 4; ++level) {
                const int shift = 24 - 8 * level;
                if (tid < 256) { mlo[tid] = 0u; mhi[tid] = 0u; hist[0][tid] = 0; }
                __syncthreads();
#pragma unroll
                for (int h = 0; h < 4; ++h) {
                    const uint32_t rk = row_max - static_cast<uint32_t>(c[h] >> 32);
                    if (kept[h] && (rk & pm) == pfx) {
                        const uint32_t bin = (rk >> shift) & 255u;
                        const unsigned long long mh = mass(h);
                        atomicAdd(&mlo[bin], static_cast<uint32_t>(mh & 0xfffffull));
                        atomicAdd(&mhi[bin], static_cast<uint32_t>(mh >> 20));
                        atomicAdd(&hist[0][bin], 1);
                    }
                }
                __syncthreads();
                if (tid < 32) find_mass_bin_asc(mlo, mhi, target - before, sh_int, shl);
                __syncthreads();
                const int bin = sh_int[0];
                before += shl[0];
                ties = hist[0][bin];
                pfx |= static_cast<uint32_t>(bin) << shift;
                pm |= 255u << shift;
                __syncthreads();
            }
            // pfx is the rank of the crossing key; the entries equal to it have one mass each, and
            // the first m_keep of them (smallest index first) are kept
            const uint32_t kcross = row_max - pfx;
            const unsigned long long mk = fixed_mass(key_value(kcross) - t0);
            int m_keep = ties;
            if (mk > 0ull && target > before) {
                const unsigned long long q = (target - before + mk - 1ull) / mk;
                m_keep = q < static_cast<unsigned long long>(ties) ? static_cast<int>(q) : ties;
            }
            m_keep = m_keep < 1 ? 1 : m_keep;
            if (m_keep < ties) {
                // rank the kept entries equal to kcross by index: in a compact list when few
                if (tid == 0) tie_count = 0u;
                __syncthreads();
#pragma unroll
                for (int h = 0; h < 4; ++h) {
                    if (kept[h] && static_cast<uint32_t>(c[h] >> 32) == kcross) {
                        const uint32_t pos = atomicAdd(&tie_count, 1u);
                        if (pos < static_cast<uint32_t>(kTie)) tiebuf[pos] = c[h];
                    }
                }
                __syncthreads();
                const bool listed = ties <= kTie;
                const unsigned long long tie_hi = (static_cast<unsigned long long>(kcross) + 1ull) << 32;
#pragma unroll
                for (int h = 0; h < 4; ++h) {
                    if (kept[h] && static_cast<uint32_t>(c[h] >> 32) == kcross) {
                        int ahead = 0;             // kept ties with a smaller index
                        if (listed) {
                            for (int j = 0; j < ties; ++j) ahead += tiebuf[j] > c[h];
                        } else {
                            for (int j = 0; j < n; ++j) ahead += cand[j] > c[h] && cand[j] < tie_hi;
                        }
                        kept[h] = ahead < m_keep;
                    }
                }
            }
#pragma unroll
            for (int h = 0; h < 4; ++h)
                if (kept[h] && static_cast<uint32_t>(c[h] >> 32) < kcross) kept[h] = false;
        }
        const float thr = minp_on ? t0 + logf(mp) : -CUDART_INF_F;
#pragma unroll
        for (int h = 0; h < 4; ++h) {
            if (!kept[h]) continue;
            const float t = key_value(static_cast<uint32_t>(c[h] >> 32));
            const int v = static_cast<int>(~static_cast<uint32_t>(c[h]));
            if (t > -CUDART_INF_F && t >= thr) {
                const float sc = t + gumbel_one<kWide>(r.p.key, static_cast<uint32_t>(v));
                if (better(sc, v, best_s, best_i)) { best_s = sc; best_i = v; }
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

// Cluster size per row: about 8K entries per CTA for small batches (many SMs on one row), 16K
// for larger ones, at most 16; S rounded up to a multiple of 8 (aligned Philox groups).
struct Plan {
    int csize;
    int64_t S;
};

Plan make_plan(int64_t B, int64_t V, int max_cluster) {
    const int64_t per_cta = B * 8 < 152 ? 8192 : 16384;
    int64_t c = (V + per_cta - 1) / per_cta;
    if (c < 1) c = 1;
    if (c > max_cluster) c = max_cluster;
    int64_t S = (V + c - 1) / c;
    S = (S + 7) / 8 * 8;
    return {static_cast<int>(c), S};
}

// Per device and variant, once: the kernel's attributes (largest dynamic shared memory, cluster
// sizes above 8) and the largest cluster size the device can co-schedule (16 if allowed, else 8).
template <typename T, bool kWide, bool kSmemKeys>
cudaError_t prepare_variant(int* max_cluster) {
    constexpr int kMaxDevices = 64;
    static std::mutex mu;
    static bool ready[kMaxDevices] = {};
    static int best[kMaxDevices] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(mu);
    if (!ready[dev]) {
        auto kern = filtered_race_cluster_kernel<T, kWide, kSmemKeys>;
        const size_t smem = kSmemKeys ? static_cast<size_t>(kMaxSmemSlice) * 4 : 0;
        e = ensure_dynamic_smem(reinterpret_cast<const void*>(kern), smem);
        if (e != cudaSuccess) return e;
        int b = 8;
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) == cudaSuccess) {
            cudaLaunchConfig_t cfg = {};
            cudaLaunchAttribute attr[1];
            attr[0].id = cudaLaunchAttributeClusterDimension;
            attr[0].val.clusterDim.x = 16;
            attr[0].val.clusterDim.y = 1;
            attr[0].val.clusterDim.z = 1;
            cfg.gridDim = dim3(16);
            cfg.blockDim = dim3(kThreads);
            cfg.dynamicSmemBytes = smem;
            cfg.attrs = attr;
            cfg.numAttrs = 1;
            int nclusters = 0;
            if (cudaOccupancyMaxActiveClusters(&nclusters, kern, &cfg) == cudaSuccess && nclusters > 0) b = 16;
        }
        cudaGetLastError();   // a refused query is not an error of the caller's launch
        best[dev] = b;
        ready[dev] = true;
    }
    *max_cluster = best[dev];
    return cudaSuccess;
}

template <typename T, bool kWide, bool kSmemKeys>
cudaError_t launch_variant(const T* y, int64_t ld, const FilterArgs& f, const Plan& pl,
                           cudaStream_t stream) {
    if (f.a.B * pl.csize > 0x7fffffffll) return cudaErrorInvalidConfiguration;   // grid.x limit
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = static_cast<unsigned>(pl.csize);
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.gridDim = dim3(static_cast<unsigned>(f.a.B * pl.csize));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = kSmemKeys ? static_cast<size_t>(pl.S) * 4 : 0;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, filtered_race_cluster_kernel<T, kWide, kSmemKeys>, y, ld, f, pl.S);
}

template <typename T, bool kWide>
cudaError_t launch_typed(const void* logits, int64_t ld, const FilterArgs& f, cudaStream_t stream) {
    const T* y = static_cast<const T*>(logits);
    int max_cluster = 8;
    cudaError_t e = prepare_variant<T, kWide, true>(&max_cluster);
    if (e != cudaSuccess) return e;
    Plan pl = make_plan(f.a.B, f.a.V, max_cluster);
    if (pl.S <= kMaxSmemSlice) return launch_variant<T, kWide, true>(y, ld, f, pl, stream);
    e = prepare_variant<T, kWide, false>(&max_cluster);
    if (e != cudaSuccess) return e;
    pl = make_plan(f.a.B, f.a.V, max_cluster);
    return launch_variant<T, kWide, false>(y, ld, f, pl, stream);
}

}  // namespace

cudaError_t launch_filtered_race(const void* logits, bool bf16, int64_t ld, bool wide,
                                 const FilterArgs& f, cudaStream_t stream) {
    if (bf16) {
        return wide ? launch_typed<__nv_bfloat16, true>(logits, ld, f, stream)
                    : launch_typed<__nv_bfloat16, false>(logits, ld, f, stream);
    }
    return wide ? launch_typed<float, true>(logits, ld, f, stream)
                : launch_typed<float, false>(logits, ld, f, stream);
}

}  // namespace lms
