// Speculative-decoding verification over materialised target and draft logits (spec-decode-ops
// "verify": the canonical rejection sampling of speculative decoding).  Draft token x_i is
// accepted when u_i p_d(x_i) < p_t(x_i), i.e. with probability min(1, p_t / p_d), in order; the
// first rejection j is replaced by a draw from the residual max(p_t - p_d, 0) at position j (the
// target's own race when no entry of the residual is positive); with every draft accepted, a
// bonus token is drawn from the target at position k.  p = softmax(logits / T), one T per row;
// T == 0 rows accept while x_i is the target's argmax and then emit the argmax.
//
// Noise: row b's draws at step position i use the race's Philox noise at absolute position
// positions[b] + i (seeded rows) or row index b (k + 1) + i with (base_seed, offset) (unseeded
// rows).  The acceptance uniform u_i is the same key's Philox call with counter word 0 =
// 0xffffffff, which no vocabulary entry uses.
//
// Four kernels, chained by programmatic dependent launch:
//   1. verify_partials: per (row, chunk of 8192 entries) of the 2k + 1 target and draft rows of
//      each batch row, the softmax partials in base 2 (max m of y log2(e) / T, sum of
//      2^(z - m)) and, on greedy rows, the first index of the max.  Every logit is read here once.
//   2. verify_decide: per batch row (one warp), the normalisers, the k acceptance tests side by
//      side (u in double), the first rejection j; greedy and invalid rows are finished here.
//   3. verify_race: per (batch row, chunk of 4096 entries), the best of log(p_t - p_d) + g
//      (residual) and of y / T + g (the target's race, rounded exactly as the plain race) at j.
//      The two rows at j are read a second time.
//   4. verify_finalize: per batch row, the chunk candidates reduced to the emitted token.
// Logits of +inf are outside the domain (the normalisers are not finite).
#include <cuda_bf16.h>

#include "lms_device.cuh"
#include "lms_kernels.h"

namespace lms {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kPartUnits = 4;                           // units of 8 entries per thread
constexpr int kPartChunk = kThreads * kPartUnits * 8;   // 8192 entries per partials block
constexpr int kRaceUnits = 2;
constexpr int kRaceChunk = kThreads * kRaceUnits * 8;   // 4096 entries per race block
constexpr int kModeDone = 0, kModeRace = 1;
constexpr int kMaxRowsPerBatch = 2 * 32 + 1;            // 2k + 1 for the largest k
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

// 2^x and log2(x) of the special function unit (ex2 / lg2 approx, flush-to-zero): relative
// error about 2^-22, 2^-inf = 0.
__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
__device__ __forceinline__ float lg2(float x) {
    float y;
    asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

template <typename T>
__device__ __forceinline__ float ld_f(const T* p);
template <>
__device__ __forceinline__ float ld_f<float>(const float* p) { return __ldg(p); }
template <>
__device__ __forceinline__ float ld_f<__nv_bfloat16>(const __nv_bfloat16* p) {
    return __bfloat162float(p[0]);
}

__device__ __forceinline__ bool aligned16(const void* p) {
    return (reinterpret_cast<uintptr_t>(p) & 15u) == 0;
}

// Base-2 softmax partial: the max m, the sum s of 2^(z - m), the first index of the max (greedy
// rows only; 0x7fffffff otherwise).
struct Part {
    float m, s;
    int a;
};

__device__ __forceinline__ Part combine(Part x, Part y) {
    Part r;
    r.m = fmaxf(x.m, y.m);
    if (r.m == -CUDART_INF_F) return {-CUDART_INF_F, 0.0f, x.a < y.a ? x.a : y.a};
    r.s = x.s * ex2(x.m - r.m) + y.s * ex2(y.m - r.m);   // 2^-inf = 0 for an empty side
    r.a = x.m > y.m ? x.a : (y.m > x.m ? y.a : (x.a < y.a ? x.a : y.a));
    return r;
}

__device__ __forceinline__ Part warp_combine(Part p) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        Part o;
        o.m = __shfl_xor_sync(0xffffffffu, p.m, off);
        o.s = __shfl_xor_sync(0xffffffffu, p.s, off);
        o.a = __shfl_xor_sync(0xffffffffu, p.a, off);
        p = combine(p, o);
    }
    return p;
}

// log2 of the normaliser sum_v 2^(z_v) of a row's combined partial.
__device__ __forceinline__ float log2_norm(const Part& p) { return p.m + lg2(p.s); }

// The generator of row b's draws at step position i.
__device__ __forceinline__ RowKey step_key(const VerifyArgs& a, int64_t b, int i) {
    RowKey r;
    if (a.seeds != nullptr && a.seeds[b] >= 0) {
        const uint64_t s = static_cast<uint64_t>(a.seeds[b]);
        const uint64_t p = static_cast<uint64_t>(a.positions[b] + i);
        r.ka = static_cast<uint32_t>(s);
        r.kb = static_cast<uint32_t>(s >> 32);
        r.c1 = static_cast<uint32_t>(p);
        r.c2 = static_cast<uint32_t>(p >> 32);
        r.c3 = 0u;
    } else {
        r.ka = static_cast<uint32_t>(a.base_seed);
        r.kb = static_cast<uint32_t>(a.base_seed >> 32);
        r.c1 = static_cast<uint32_t>(a.offset);
        r.c2 = static_cast<uint32_t>(a.offset >> 32);
        r.c3 = 0x80000000u | static_cast<uint32_t>(b * (a.k + 1) + i);
    }
    return r;
}

// The acceptance uniform (k + 1/2) / 2^m from the call with counter word 0 = 0xffffffff, in
// double (exact for both widths).
__device__ __forceinline__ double accept_uniform(const RowKey& key, bool wide) {
    const Words w = row_call(key, 0xffffffffu);
    if (wide) {
        const uint64_t k52 = ((static_cast<uint64_t>(w.w1) << 32) | w.w0) >> 12;
        return (static_cast<double>(k52) + 0.5) * 0x1p-52;
    }
    return (static_cast<double>(w.w0 >> 8) + 0.5) * 0x1p-24;
}

// 1 / T of a sampled row (1 on greedy and invalid rows).
__device__ __forceinline__ float row_scale(const float* temperature, int64_t b, bool* greedy,
                                           bool* invalid) {
    const float T = temperature ? temperature[b] : 1.0f;
    *invalid = !(T >= 0.0f);
    *greedy = T == 0.0f;
    return (*invalid || *greedy) ? 1.0f : 1.0f / T;
}

// The factor from logits to base-2 exponents: log2(e) / T (1 on greedy rows, whose partials hold
// the raw max and its index).
__device__ __forceinline__ float base2_scale(float scale, bool greedy) {
    return greedy ? 1.0f : scale * kLog2e;
}

template <typename T>
__global__ void __launch_bounds__(kThreads) verify_partials(VerifyArgs a) {
    pdl_launch_dependents();                       // the decision kernel may take its slots now
    const int K2 = 2 * a.k + 1;
    const int64_t idx = blockIdx.x;
    const int64_t row = idx / a.nc;
    const int64_t c = idx % a.nc;
    const int64_t b = row / K2;
    const int q = static_cast<int>(row % K2);
    const T* y = q <= a.k ? static_cast<const T*>(a.target) + (b * (a.k + 1) + q) * a.ld
                          : static_cast<const T*>(a.draft) + (b * a.k + (q - a.k - 1)) * a.ld;
    bool greedy, invalid;
    const float scale2 = base2_scale(row_scale(a.temperature, b, &greedy, &invalid), greedy);
    Part p = {-CUDART_INF_F, 0.0f, 0x7fffffff};
    if (!invalid) {                                // block-uniform
        // every load of the thread's units is issued before any of them is used
        const bool vec = aligned16(y);
        const int64_t v_chunk = c * kPartChunk;
        float z[kPartUnits][8];
#pragma unroll
        for (int u = 0; u < kPartUnits; ++u) {
            const int64_t v0 = v_chunk + (static_cast<int64_t>(u) * kThreads + threadIdx.x) * 8;
            const int64_t n = a.V - v0;
            if (n > 0) {
                load8(y + v0, n < 8 ? static_cast<int>(n) : 8, vec, z[u]);
            } else {
#pragma unroll
                for (int e = 0; e < 8; ++e) z[u][e] = 0.0f;
            }
        }
        float m = -CUDART_INF_F;
        if (v_chunk + kPartChunk <= a.V) {         // whole chunk (block-uniform)
#pragma unroll
            for (int u = 0; u < kPartUnits; ++u)
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    z[u][e] *= scale2;
                    m = fmaxf(m, z[u][e]);         // NaN is never the max
                }
        } else {
#pragma unroll
            for (int u = 0; u < kPartUnits; ++u) {
                const int64_t v0 = v_chunk + (static_cast<int64_t>(u) * kThreads + threadIdx.x) * 8;
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    z[u][e] = v0 + e < a.V ? z[u][e] * scale2 : -CUDART_INF_F;
                    m = fmaxf(m, z[u][e]);
                }
            }
        }
        float s = 0.0f;
        if (m > -CUDART_INF_F) {
#pragma unroll
            for (int u = 0; u < kPartUnits; ++u)
#pragma unroll
                for (int e = 0; e < 8; ++e) s += ex2(fmaxf(z[u][e] - m, -CUDART_INF_F));  // NaN -> 0
            if (greedy) {
                int arg = 0x7fffffff;
#pragma unroll
                for (int u = kPartUnits - 1; u >= 0; --u) {
                    const int v0 = static_cast<int>(v_chunk) + (u * kThreads + static_cast<int>(threadIdx.x)) * 8;
#pragma unroll
                    for (int e = 7; e >= 0; --e)
                        if (z[u][e] == m) arg = v0 + e;   // the smallest index of the max wins
                }
                p.a = arg;
            }
        }
        p.m = m;
        p.s = s;
    }
    p = warp_combine(p);
    __shared__ Part sh[kWarps];
    const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
    if (l == 0) sh[w] = p;
    __syncthreads();
    if (threadIdx.x == 0) {
        Part r = sh[0];
        for (int i = 1; i < kWarps; ++i) r = combine(r, sh[i]);
        a.pmax[row * a.nc + c] = r.m;
        a.psum[row * a.nc + c] = r.s;
        a.parg[row * a.nc + c] = r.a;
    }
}

// One row's partials combined serially by one thread (independent loads, issued ahead).
__device__ __forceinline__ Part row_total(const VerifyArgs& a, int64_t row) {
    Part p = {-CUDART_INF_F, 0.0f, 0x7fffffff};
    const int64_t base = row * a.nc;
#pragma unroll 4
    for (int64_t c = 0; c < a.nc; ++c)
        p = combine(p, {a.pmax[base + c], a.psum[base + c], a.parg[base + c]});
    return p;
}

// One warp per batch row.  The lanes first combine the 2k + 1 rows' partials (lane l takes rows
// l, l + 32, ...), then lane i < k takes acceptance test i; the tests do not depend on one
// another, and the first failing lane is the rejection position j.
template <typename T>
__global__ void __launch_bounds__(kThreads) verify_decide(VerifyArgs a, bool wide) {
    pdl_launch_dependents();
    __shared__ Part rows_sh[kWarps][kMaxRowsPerBatch];
    const int w = threadIdx.x >> 5;
    const int64_t b = static_cast<int64_t>(blockIdx.x) * kWarps + w;
    const int lane = threadIdx.x & 31;
    pdl_wait_primary();                            // the partials
    if (b >= a.B) return;                          // warp-uniform
    const int k = a.k, K1 = a.k + 1, K2 = 2 * a.k + 1;
    bool greedy, invalid;
    const float scale2 = base2_scale(row_scale(a.temperature, b, &greedy, &invalid), greedy);
    int64_t* out = a.out + b * K1;
    if (invalid) {
        for (int i = lane; i < K1; i += 32) out[i] = -1;
        if (lane == 0) {
            a.accept_len[b] = 0;
            if (a.row_status) a.row_status[b] = 2;
            a.dec_mode[b] = kModeDone;
        }
        return;
    }
    Part* rows = rows_sh[w];
    for (int q = lane; q < K2; q += 32) rows[q] = row_total(a, b * K2 + q);
    __syncwarp();
    bool reject = false;
    if (lane < k) {
        const int i = lane;
        const int64_t x = a.tokens[b * k + i];
        const Part pt = rows[i];
        if (x < 0 || x >= a.V) {
            reject = true;                         // not a vocabulary entry
        } else if (greedy) {
            reject = !(pt.m > -CUDART_INF_F && x == pt.a);
        } else {
            const Part pd = rows[k + 1 + i];
            const T* tgt = static_cast<const T*>(a.target) + (b * K1 + i) * a.ld;
            const T* dft = static_cast<const T*>(a.draft) + (b * k + i) * a.ld;
            // 2^(z - log2 Z); NaN and -inf entries and empty rows give 0
            const float zt = ld_f<T>(tgt + x) * scale2, zd = ld_f<T>(dft + x) * scale2;
            const float p_t = pt.m > -CUDART_INF_F ? ex2(fmaxf(zt - log2_norm(pt), -CUDART_INF_F)) : 0.0f;
            const float p_d = pd.m > -CUDART_INF_F ? ex2(fmaxf(zd - log2_norm(pd), -CUDART_INF_F)) : 0.0f;
            const double u = accept_uniform(step_key(a, b, i), wide);
            reject = !(u * static_cast<double>(p_d) < static_cast<double>(p_t));
        }
    }
    const unsigned rejected = __ballot_sync(0xffffffffu, reject);
    const int j = rejected ? __ffs(rejected) - 1 : k;
    const Part pj = rows[j];
    const bool none = pj.m == -CUDART_INF_F;       // nothing finite to draw: the row emits nothing
    for (int i = lane; i < K1; i += 32)
        if (i != j || none) out[i] = (i < j && !none) ? a.tokens[b * k + i] : -1;
    if (lane == 0) {
        a.accept_len[b] = none ? 0 : j;
        if (greedy || none) {
            if (!none) out[j] = pj.a;
            if (a.row_status) a.row_status[b] = none ? 1 : 0;
            a.dec_mode[b] = kModeDone;
        } else {
            a.dec_j[b] = j;
            a.dec_lt[b] = log2_norm(pj);
            if (j < k) {
                const Part pd = rows[k + 1 + j];
                a.dec_ld[b] = pd.m > -CUDART_INF_F ? log2_norm(pd) : CUDART_INF_F;
            }
            a.dec_mode[b] = kModeRace;
        }
    }
}

template <typename T, bool kWide>
__global__ void __launch_bounds__(kThreads) verify_race(VerifyArgs a) {
    pdl_launch_dependents();
    const int64_t idx = blockIdx.x;
    const int64_t b = idx / a.ncr;
    const int64_t c = idx % a.ncr;
    pdl_wait_primary();                            // the decisions
    if (a.dec_mode[b] != kModeRace) return;        // block-uniform
    const int k = a.k, K1 = a.k + 1;
    const int j = a.dec_j[b];
    const bool resid = j < k;
    bool greedy, invalid;
    const float scale = row_scale(a.temperature, b, &greedy, &invalid);
    const float scale2 = scale * kLog2e;
    const float lt = a.dec_lt[b];
    const float ldr = resid ? a.dec_ld[b] : 0.0f;
    const RowKey key = step_key(a, b, j);
    const T* trow = static_cast<const T*>(a.target) + (b * K1 + j) * a.ld;
    const T* drow = resid ? static_cast<const T*>(a.draft) + (b * k + j) * a.ld : trow;
    const bool vec_t = aligned16(trow), vec_d = aligned16(drow);
    const int64_t v_chunk = c * kRaceChunk;
    float yt[kRaceUnits][8], yd[kRaceUnits][8];
#pragma unroll
    for (int u = 0; u < kRaceUnits; ++u) {
        const int64_t v0 = v_chunk + (static_cast<int64_t>(u) * kThreads + threadIdx.x) * 8;
        const int64_t n = a.V - v0;
        const int nn = n < 8 ? static_cast<int>(n) : 8;
        if (n > 0) {
            load8(trow + v0, nn, vec_t, yt[u]);
            if (resid) load8(drow + v0, nn, vec_d, yd[u]);
        }
    }
    float bs_t = -CUDART_INF_F, bs_r = -CUDART_INF_F;
    int bi_t = kNoIndex, bi_r = kNoIndex;
#pragma unroll
    for (int u = 0; u < kRaceUnits; ++u) {
        const int64_t v0 = v_chunk + (static_cast<int64_t>(u) * kThreads + threadIdx.x) * 8;
        if (v0 >= a.V) break;
        float g[8];
        gumbel_run<kWide, 8>(key, static_cast<uint32_t>(v0), g);
        const int n = a.V - v0 < 8 ? static_cast<int>(a.V - v0) : 8;
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            if (e < n) {
                const int v = static_cast<int>(v0) + e;
                const float y = yt[u][e] == yt[u][e] ? yt[u][e] : -CUDART_INF_F;
                // the plain race's score, rounded as the race rounds it
                const float s_t = fmaf(y, scale, g[e]);
                if (s_t > bs_t) { bs_t = s_t; bi_t = v; }
                if (resid) {
                    const float p_t = ex2(y * scale2 - lt);
                    const float p_d = ex2(fmaxf(yd[u][e] * scale2 - ldr, -CUDART_INF_F));  // NaN -> 0
                    const float r = p_t - p_d;
                    const float s_r = r > 0.0f ? fmaf(lg2(r), kLn2, g[e]) : -CUDART_INF_F;
                    if (s_r > bs_r) { bs_r = s_r; bi_r = v; }
                }
            }
        }
    }
    warp_argmax(bs_t, bi_t);
    warp_argmax(bs_r, bi_r);
    __shared__ float ss[2][kWarps];
    __shared__ int si[2][kWarps];
    const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
    if (l == 0) { ss[0][w] = bs_r; si[0][w] = bi_r; ss[1][w] = bs_t; si[1][w] = bi_t; }
    __syncthreads();
    if (threadIdx.x == 0) {
        for (int q = 0; q < 2; ++q) {
            float s = ss[q][0];
            int i = si[q][0];
            for (int x = 1; x < kWarps; ++x)
                if (better(ss[q][x], si[q][x], s, i)) { s = ss[q][x]; i = si[q][x]; }
            a.c_s[(b * a.ncr + c) * 2 + q] = s;
            a.c_i[(b * a.ncr + c) * 2 + q] = i;
        }
    }
}

__global__ void __launch_bounds__(kThreads) verify_finalize(VerifyArgs a) {
    const int64_t b = static_cast<int64_t>(blockIdx.x) * kWarps + (threadIdx.x >> 5);
    pdl_wait_primary();                            // the race candidates
    if (b >= a.B || a.dec_mode[b] != kModeRace) return;   // warp-uniform
    const int lane = threadIdx.x & 31;
    float sr = -CUDART_INF_F, st = -CUDART_INF_F;
    int ir = kNoIndex, it = kNoIndex;
    for (int64_t c = lane; c < a.ncr; c += 32) {
        const float s0 = a.c_s[(b * a.ncr + c) * 2], s1 = a.c_s[(b * a.ncr + c) * 2 + 1];
        const int i0 = a.c_i[(b * a.ncr + c) * 2], i1 = a.c_i[(b * a.ncr + c) * 2 + 1];
        if (better(s0, i0, sr, ir)) { sr = s0; ir = i0; }
        if (better(s1, i1, st, it)) { st = s1; it = i1; }
    }
    warp_argmax(sr, ir);
    warp_argmax(st, it);
    if (lane == 0) {
        const int j = a.dec_j[b];
        const int ri = candidate_index(sr, ir), ti = candidate_index(st, it);
        // the residual's draw; the target's own race if no residual entry is positive or j = k
        const int64_t tok = (j < a.k && ri >= 0) ? ri : ti;
        a.out[b * (a.k + 1) + j] = tok;
        if (a.row_status) a.row_status[b] = tok >= 0 ? 0 : 1;
    }
}

// Launch with programmatic stream serialization: the kernel may start while its predecessor
// finishes and waits for it with griddepcontrol.wait.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kern)(KArgs...), unsigned grid, cudaStream_t s, Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, args...);
}

template <typename T>
cudaError_t launch_typed(const VerifyArgs& a, bool wide, cudaStream_t s) {
    const unsigned parts = static_cast<unsigned>(a.B * (2 * a.k + 1) * a.nc);
    const unsigned warps_grid = static_cast<unsigned>((a.B + kWarps - 1) / kWarps);
    const unsigned race = static_cast<unsigned>(a.B * a.ncr);
    verify_partials<T><<<parts, kThreads, 0, s>>>(a);
    cudaError_t e = cudaGetLastError();
    if (e == cudaSuccess) e = launch_pdl(verify_decide<T>, warps_grid, s, a, wide);
    if (e == cudaSuccess)
        e = wide ? launch_pdl(verify_race<T, true>, race, s, a) : launch_pdl(verify_race<T, false>, race, s, a);
    if (e == cudaSuccess) e = launch_pdl(verify_finalize, warps_grid, s, a);
    return e;
}

}  // namespace

void verify_chunks(int64_t V, int64_t* partial_chunks, int64_t* race_chunks) {
    *partial_chunks = (V + kPartChunk - 1) / kPartChunk;
    *race_chunks = (V + kRaceChunk - 1) / kRaceChunk;
}

cudaError_t launch_verify(const VerifyArgs& a, bool bf16, bool wide, cudaStream_t stream) {
    return bf16 ? launch_typed<__nv_bfloat16>(a, wide, stream) : launch_typed<float>(a, wide, stream);
}

}  // namespace lms
