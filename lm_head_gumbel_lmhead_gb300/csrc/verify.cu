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
// Three kernels, chained by programmatic dependent launch:
//   1. verify_partials: per (chunk, row) of the 2k + 1 target and draft rows of each batch row
//      (128 bytes per thread, loaded before use), one softmax partial per warp in base 2: the
//      max m of z = y log2(e) / T, the sum of 2^(z - m) and, on greedy rows, the first index of
//      the max.  Every logit is read here once; nothing else happens in this pass.
//   2. verify_decide: per batch row, the normalisers, the k acceptance tests side by side (u in
//      double), the first rejection j; greedy and invalid rows are finished here.  What does not
//      depend on the partials (the tokens, the logits at them, the uniforms) is read before the
//      wait on the partials pass.
//   3. verify_race: per (chunk, batch row) of the rows left to draw, the best of
//      log(p_t - p_d) + g (residual) and of y / T + g (the target's race, rounded exactly as the
//      plain race) at j; the two rows at j are read a second time.  The block that completes a
//      row's last chunk reduces the chunk candidates to the emitted token.
// The decision kernel zeroes each row's race counter, so a call needs no zeroed workspace.
// Logits of +inf are outside the domain (the normalisers are not finite).
#include <cuda_bf16.h>

#include "lms_device.cuh"
#include "lms_kernels.h"

namespace lms {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kMaxGridYZ = 65535;
constexpr int64_t kMaxGridX = 0x7fffffff;
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

// Units of 8 entries that a thread loads before it uses any of them: 128 bytes per thread in the
// partials pass, 64 bytes of each row (target and draft) in the race pass.
template <typename T>
__host__ __device__ constexpr int part_units() { return 128 / (8 * static_cast<int>(sizeof(T))); }   // bf16 8, fp32 4
template <typename T>
__host__ __device__ constexpr int race_units() { return 64 / (8 * static_cast<int>(sizeof(T))); }    // bf16 4, fp32 2
template <typename T>
__host__ __device__ constexpr int part_chunk() { return kThreads * part_units<T>() * 8; }             // 16384 / 8192
template <typename T>
__host__ __device__ constexpr int race_chunk() { return kThreads * race_units<T>() * 8; }             // 8192 / 4096

// A unit of 8 entries as loaded (bf16 pairs in four words, or eight floats); entries past the
// row's end read as -inf.
template <typename T>
struct Raw;
template <>
struct Raw<__nv_bfloat16> {
    uint32_t w[4];
    __device__ __forceinline__ void load(const __nv_bfloat16* p, int n, bool vec) {
        if (vec && n >= 8) {
            const uint4 x = __ldg(reinterpret_cast<const uint4*>(p));
            w[0] = x.x; w[1] = x.y; w[2] = x.z; w[3] = x.w;
        } else {
            const unsigned short* h = reinterpret_cast<const unsigned short*>(p);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const uint32_t lo = 2 * i < n ? __ldg(h + 2 * i) : 0xff80u;        // -inf
                const uint32_t hi = 2 * i + 1 < n ? __ldg(h + 2 * i + 1) : 0xff80u;
                w[i] = lo | (hi << 16);
            }
        }
    }
    __device__ __forceinline__ float at(int e) const {
        return __uint_as_float((e & 1) ? (w[e >> 1] & 0xffff0000u) : (w[e >> 1] << 16));
    }
    // the largest entry, by packed bf16 pairs (NaN is never the max)
    __device__ __forceinline__ float max8() const {
        __nv_bfloat162 m = __hmax2(as_pair(w[0]), as_pair(w[1]));
        m = __hmax2(m, __hmax2(as_pair(w[2]), as_pair(w[3])));
        return fmaxf(__low2float(m), __high2float(m));
    }
    static __device__ __forceinline__ __nv_bfloat162 as_pair(uint32_t x) {
        __nv_bfloat162 r;
        *reinterpret_cast<uint32_t*>(&r) = x;
        return r;
    }
};
template <>
struct Raw<float> {
    float f[8];
    __device__ __forceinline__ void load(const float* p, int n, bool vec) {
        if (vec && n >= 8) {
            const float4 x = __ldg(reinterpret_cast<const float4*>(p));
            const float4 y = __ldg(reinterpret_cast<const float4*>(p) + 1);
            f[0] = x.x; f[1] = x.y; f[2] = x.z; f[3] = x.w;
            f[4] = y.x; f[5] = y.y; f[6] = y.z; f[7] = y.w;
        } else {
#pragma unroll
            for (int e = 0; e < 8; ++e) f[e] = e < n ? __ldg(p + e) : -CUDART_INF_F;
        }
    }
    __device__ __forceinline__ float at(int e) const { return f[e]; }
    // the largest entry (NaN is never the max)
    __device__ __forceinline__ float max8() const {
        float m = fmaxf(f[0], f[1]);
#pragma unroll
        for (int e = 2; e < 8; ++e) m = fmaxf(m, f[e]);
        return m;
    }
};

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

// The thread's sum of 2^(z - m) with NaN entries counted as -inf, over its units read again.
template <typename T, int kUnits>
__device__ __noinline__ float rescan_sum(const T* y, int64_t v_chunk, int64_t V, bool vec,
                                         float scale2, float m) {
    float s = 0.0f;
#pragma unroll 1
    for (int u = 0; u < kUnits; ++u) {
        const int64_t v0 = v_chunk + (u * kThreads + static_cast<int>(threadIdx.x)) * 8;
        const int64_t n = V - v0;
        if (n <= 0) break;
        Raw<T> r;
        r.load(y + v0, n < 8 ? static_cast<int>(n) : 8, vec);
#pragma unroll
        for (int e = 0; e < 8; ++e) s += ex2(fmaxf(fmaf(r.at(e), scale2, -m), -CUDART_INF_F));
    }
    return s;
}

// The first index among the thread's units whose entry equals the max m_raw.
template <typename T, int kUnits>
__device__ __noinline__ int rescan_first_max(const T* y, int64_t v_chunk, int64_t V, bool vec,
                                             float m_raw) {
#pragma unroll 1
    for (int u = 0; u < kUnits; ++u) {
        const int64_t v0 = v_chunk + (u * kThreads + static_cast<int>(threadIdx.x)) * 8;
        const int64_t n = V - v0;
        if (n <= 0) break;
        Raw<T> r;
        r.load(y + v0, n < 8 ? static_cast<int>(n) : 8, vec);
#pragma unroll
        for (int e = 0; e < 8; ++e)
            if (r.at(e) == m_raw) return static_cast<int>(v0) + e;
    }
    return 0x7fffffff;
}

// Units of one partials item (chunk c of row q of batch row b), loaded before any is used.
template <typename T>
struct PartItem {
    static constexpr int kUnits = part_units<T>();
    Raw<T> raw[kUnits];
    const T* y;
    int64_t v_chunk;
    bool vec, skip;

    __device__ __forceinline__ void load(const VerifyArgs& a, int64_t b, int q, int64_t c, bool invalid) {
        y = q <= a.k ? static_cast<const T*>(a.target) + (b * (a.k + 1) + q) * a.ld
                     : static_cast<const T*>(a.draft) + (b * a.k + (q - a.k - 1)) * a.ld;
        v_chunk = c * part_chunk<T>();
        vec = aligned16(y);
        skip = invalid;
        if (skip) return;                          // block-uniform
#pragma unroll
        for (int u = 0; u < kUnits; ++u) {
            const int64_t v0 = v_chunk + (u * kThreads + static_cast<int>(threadIdx.x)) * 8;
            const int64_t n = a.V - v0;
            raw[u].load(y + (n > 0 ? v0 : 0), n <= 0 ? 0 : (n < 8 ? static_cast<int>(n) : 8), vec);
        }
    }

    // The warp's partial (every lane holds it).
    __device__ __forceinline__ Part partial(int64_t V, float scale2, bool greedy) const {
        Part p = {-CUDART_INF_F, 0.0f, 0x7fffffff};
        if (!skip) {
            float m_raw = -CUDART_INF_F;
#pragma unroll
            for (int u = 0; u < kUnits; ++u) m_raw = fmaxf(m_raw, raw[u].max8());
            if (m_raw > -CUDART_INF_F) {
                // scale2 > 0, so the max of the scaled entries is the scaled max, rounding included
                const float m = m_raw * scale2;
                float s0 = 0.0f, s1 = 0.0f;
#pragma unroll
                for (int u = 0; u < kUnits; ++u)
#pragma unroll
                    for (int e = 0; e < 8; e += 2) {
                        s0 += ex2(fmaf(raw[u].at(e), scale2, -m));
                        s1 += ex2(fmaf(raw[u].at(e + 1), scale2, -m));
                    }
                float s = s0 + s1;
                // the rare paths read the units again (from L2) rather than keep them live
                if (s != s) s = rescan_sum<T, kUnits>(y, v_chunk, V, vec, scale2, m);
                const int arg = greedy ? rescan_first_max<T, kUnits>(y, v_chunk, V, vec, m_raw) : 0x7fffffff;
                p = {m, s, arg};
            }
        }
        return warp_combine(p);
    }
};

// Grid (chunk, row q of the batch row: target 0..k then draft k+1..2k, batch row - b_base).
// Each warp writes its own partial: no block-wide step, no atomics.
template <typename T>
__global__ void __launch_bounds__(kThreads, 4) verify_partials(VerifyArgs a, int64_t b_base) {
    pdl_launch_dependents();                       // the decision kernel may take its slots now
    clear_status_bits(a.status_bits, b_base);
    const int c = blockIdx.x, q = blockIdx.y;
    const int64_t b = b_base + blockIdx.z;
    bool greedy, invalid;
    const float scale2 = base2_scale(row_scale(a.temperature, b, &greedy, &invalid), greedy);
    PartItem<T> item;
    item.load(a, b, q, c, invalid);
    const Part p = item.partial(a.V, scale2, greedy);
    if ((threadIdx.x & 31) == 0) {
        const int64_t at = ((b * (2 * a.k + 1) + q) * a.nc + c) * kWarps + (threadIdx.x >> 5);
        a.pmax[at] = p.m;
        a.psum[at] = p.s;
        a.parg[at] = p.a;
    }
}

// The decision of batch row b, one block per row: the warps combine the 2k + 1 rows' partials
// (warp w takes rows w, w + 8, ...; lanes take the row's warp partials), then lane i < k of warp
// 0 takes acceptance test i.  The tests do not depend on one another; the first failing lane is
// the rejection position j.  Warp 0 writes the accept length, the accepted prefix and -1 after
// it, the token and status of rows finished here, and the decision for the race pass.
template <typename T>
__global__ void __launch_bounds__(kThreads) verify_decide(VerifyArgs a, int64_t b_base, bool wide) {
    __shared__ Part rows[kMaxRowsPerBatch];
    pdl_launch_dependents();                       // the race kernel may take its slots now
    const int64_t b = b_base + blockIdx.x;
    const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int k = a.k, K1 = a.k + 1, K2 = 2 * a.k + 1;
    bool greedy, invalid;
    const float scale2 = base2_scale(row_scale(a.temperature, b, &greedy, &invalid), greedy);
    int64_t* out = a.out + b * K1;
    VerifyDecision d = {k, kModeDone, 0.0f, CUDART_INF_F};
    // what does not depend on the partials comes first: lane i < k of warp 0 reads x_i, the two
    // logits at x_i and draws u_i while the partials pass finishes
    int64_t x = -1;
    float zt = 0.0f, zd = 0.0f;
    double u = 0.0;
    if (w == 0 && lane < k && !invalid) {
        const int i = lane;
        x = a.tokens[b * k + i];
        if (x >= 0 && x < a.V && !greedy) {
            zt = ld_f<T>(static_cast<const T*>(a.target) + (b * K1 + i) * a.ld + x) * scale2;
            zd = ld_f<T>(static_cast<const T*>(a.draft) + (b * k + i) * a.ld + x) * scale2;
            u = accept_uniform(step_key(a, b, i), wide);
        }
    }
    pdl_wait_primary();                            // the partials
    if (invalid) {                                 // block-uniform
        if (w == 0) {
            for (int i = lane; i < K1; i += 32) out[i] = -1;
            if (lane == 0) {
                a.accept_len[b] = 0;
                if (a.row_status) a.row_status[b] = 2;
                note_row_status(a.status_bits, 2);
                a.dec[b] = d;
            }
        }
        return;
    }
    const int64_t per_row = a.nc * kWarps;
    for (int q = w; q < K2; q += kWarps) {
        Part p = {-CUDART_INF_F, 0.0f, 0x7fffffff};
        const int64_t base = (b * K2 + q) * per_row;
        for (int64_t e = lane; e < per_row; e += 32)
            p = combine(p, {a.pmax[base + e], a.psum[base + e], a.parg[base + e]});
        p = warp_combine(p);
        if (lane == 0) rows[q] = p;
    }
    __syncthreads();
    if (w != 0) return;
    bool reject = false;
    if (lane < k) {
        const Part pt = rows[lane];
        if (x < 0 || x >= a.V) {
            reject = true;                         // not a vocabulary entry
        } else if (greedy) {
            reject = !(pt.m > -CUDART_INF_F && x == pt.a);
        } else {
            const Part pd = rows[k + 1 + lane];
            // 2^(z - log2 Z); NaN and -inf entries and empty rows give 0
            const float p_t = pt.m > -CUDART_INF_F ? ex2(fmaxf(zt - log2_norm(pt), -CUDART_INF_F)) : 0.0f;
            const float p_d = pd.m > -CUDART_INF_F ? ex2(fmaxf(zd - log2_norm(pd), -CUDART_INF_F)) : 0.0f;
            reject = !(u * static_cast<double>(p_d) < static_cast<double>(p_t));
        }
    }
    const unsigned rejected = __ballot_sync(0xffffffffu, reject);
    const int j = rejected ? __ffs(rejected) - 1 : k;
    const Part pj = rows[j];
    const bool none = pj.m == -CUDART_INF_F;       // nothing finite to draw: the row emits nothing
    for (int i = lane; i < K1; i += 32)
        if (i != j || none || greedy) out[i] = (i < j && !none) ? a.tokens[b * k + i]
                                               : (i == j && !none) ? pj.a : -1;
    if (lane == 0) {
        a.accept_len[b] = none ? 0 : j;
        if ((greedy || none) && a.row_status) a.row_status[b] = none ? 1 : 0;
        if (none) note_row_status(a.status_bits, 1);
        d.j = j;
        if (!greedy && !none) {
            d.mode = kModeRace;
            d.lt = log2_norm(pj);
            if (j < k && rows[k + 1 + j].m > -CUDART_INF_F) d.ld = log2_norm(rows[k + 1 + j]);
        }
        a.dec[b] = d;
        a.cnt_r[b] = 0;                            // the race pass counts from zero
    }
}

// The emitted token of batch row b from its race candidates, by the block that completed the
// row's last race chunk (warp 0).
__device__ __forceinline__ void finalize_row(const VerifyArgs& a, int64_t b, int j) {
    const int lane = threadIdx.x & 31;
    float sr = -CUDART_INF_F, st = -CUDART_INF_F;
    int ir = kNoIndex, it = kNoIndex;
    for (int64_t c = lane; c < a.ncr; c += 32) {
        const int64_t at = (b * a.ncr + c) * 2;
        const float s0 = __ldcg(a.c_s + at), s1 = __ldcg(a.c_s + at + 1);
        const int i0 = __ldcg(a.c_i + at), i1 = __ldcg(a.c_i + at + 1);
        if (better(s0, i0, sr, ir)) { sr = s0; ir = i0; }
        if (better(s1, i1, st, it)) { st = s1; it = i1; }
    }
    warp_argmax(sr, ir);
    warp_argmax(st, it);
    if (lane == 0) {
        const int ri = candidate_index(sr, ir), ti = candidate_index(st, it);
        // the residual's draw; the target's own race if no residual entry is positive or j = k
        const int64_t tok = (j < a.k && ri >= 0) ? ri : ti;
        a.out[b * (a.k + 1) + j] = tok;
        if (a.row_status) a.row_status[b] = tok >= 0 ? 0 : 1;
        if (tok < 0) note_row_status(a.status_bits, 1);
    }
}

// Grid (chunk, batch row - b_base).  Rows finished by their decision leave at once.
template <typename T, bool kWide>
__global__ void __launch_bounds__(kThreads) verify_race(VerifyArgs a, int64_t b_base) {
    constexpr int kUnits = race_units<T>();
    constexpr int kChunk = race_chunk<T>();
    __shared__ float ss[2][kWarps];
    __shared__ int si[2][kWarps];
    __shared__ int last;
    const int c = blockIdx.x;
    const int64_t b = b_base + blockIdx.y;
    const int k = a.k, K1 = a.k + 1;
    bool greedy, invalid;
    const float scale = row_scale(a.temperature, b, &greedy, &invalid);
    pdl_wait_primary();                            // the partials and decisions
    const VerifyDecision dec = a.dec[b];
    if (dec.mode != kModeRace) return;             // block-uniform
    const int j = dec.j;
    const bool resid = j < k;
    const float scale2 = scale * kLog2e;
    const float lt = dec.lt, ldr = dec.ld;
    const RowKey key = step_key(a, b, j);
    const T* trow = static_cast<const T*>(a.target) + (b * K1 + j) * a.ld;
    const T* drow = resid ? static_cast<const T*>(a.draft) + (b * k + j) * a.ld : trow;
    const bool vec_t = aligned16(trow), vec_d = aligned16(drow);
    const int64_t v_chunk = static_cast<int64_t>(c) * kChunk;
    Raw<T> rt[kUnits], rd[kUnits];
#pragma unroll
    for (int u = 0; u < kUnits; ++u) {
        const int64_t v0 = v_chunk + (u * kThreads + static_cast<int>(threadIdx.x)) * 8;
        const int64_t n = a.V - v0;
        const int nn = n <= 0 ? 0 : (n < 8 ? static_cast<int>(n) : 8);
        rt[u].load(trow + (n > 0 ? v0 : 0), nn, vec_t);
        if (resid) rd[u].load(drow + (n > 0 ? v0 : 0), nn, vec_d);
    }
    float bs_t = -CUDART_INF_F, bs_r = -CUDART_INF_F;
    int bi_t = kNoIndex, bi_r = kNoIndex;
#pragma unroll
    for (int u = 0; u < kUnits; ++u) {
        const int64_t v0 = v_chunk + (u * kThreads + static_cast<int>(threadIdx.x)) * 8;
        if (v0 >= a.V) break;
        float g[8];
        gumbel_run<kWide, 8>(key, static_cast<uint32_t>(v0), g);
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            const int v = static_cast<int>(v0) + e;
            float y = rt[u].at(e);                 // -inf past the row's end
            y = y == y ? y : -CUDART_INF_F;
            // the plain race's score, rounded as the race rounds it
            const float s_t = fmaf(y, scale, g[e]);
            if (s_t > bs_t) { bs_t = s_t; bi_t = v; }
            if (resid) {
                const float p_t = ex2(fmaf(y, scale2, -lt));
                const float p_d = ex2(fmaxf(fmaf(rd[u].at(e), scale2, -ldr), -CUDART_INF_F));  // NaN -> 0
                const float r = p_t - p_d;
                const float s_r = r > 0.0f ? fmaf(lg2(r), kLn2, g[e]) : -CUDART_INF_F;
                if (s_r > bs_r) { bs_r = s_r; bi_r = v; }
            }
        }
    }
    warp_argmax(bs_t, bi_t);
    warp_argmax(bs_r, bi_r);
    const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
    if (l == 0) { ss[0][w] = bs_r; si[0][w] = bi_r; ss[1][w] = bs_t; si[1][w] = bi_t; }
    __syncthreads();
    if (threadIdx.x == 0) {
        for (int qd = 0; qd < 2; ++qd) {
            float s = ss[qd][0];
            int i = si[qd][0];
            for (int x = 1; x < kWarps; ++x)
                if (better(ss[qd][x], si[qd][x], s, i)) { s = ss[qd][x]; i = si[qd][x]; }
            a.c_s[(b * a.ncr + c) * 2 + qd] = s;
            a.c_i[(b * a.ncr + c) * 2 + qd] = i;
        }
        __threadfence();
        last = atomicAdd(a.cnt_r + b, 1) == static_cast<int>(a.ncr) - 1;
    }
    __syncthreads();
    if (!last) return;                             // block-uniform
    __threadfence();
    if (threadIdx.x < 32) finalize_row(a, b, j);
}

// Launch with programmatic stream serialization: the kernel may start while its predecessor
// finishes and waits for it with griddepcontrol.wait.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, cudaStream_t s, Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
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
    const unsigned K2 = static_cast<unsigned>(2 * a.k + 1);
    for (int64_t b0 = 0; b0 < a.B; b0 += kMaxGridYZ) {
        const unsigned nb = static_cast<unsigned>(a.B - b0 < kMaxGridYZ ? a.B - b0 : kMaxGridYZ);
        verify_partials<T><<<dim3(static_cast<unsigned>(a.nc), K2, nb), kThreads, 0, s>>>(a, b0);
        const cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    for (int64_t b0 = 0; b0 < a.B; b0 += kMaxGridX) {
        const unsigned nb = static_cast<unsigned>(a.B - b0 < kMaxGridX ? a.B - b0 : kMaxGridX);
        const cudaError_t e = launch_pdl(verify_decide<T>, dim3(nb), s, a, b0, wide);
        if (e != cudaSuccess) return e;
    }
    for (int64_t b0 = 0; b0 < a.B; b0 += kMaxGridYZ) {
        const unsigned nb = static_cast<unsigned>(a.B - b0 < kMaxGridYZ ? a.B - b0 : kMaxGridYZ);
        const dim3 rg(static_cast<unsigned>(a.ncr), nb);
        const cudaError_t e = wide ? launch_pdl(verify_race<T, true>, rg, s, a, b0)
                                   : launch_pdl(verify_race<T, false>, rg, s, a, b0);
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

}  // namespace

void verify_chunks(int64_t V, bool bf16, int64_t* partial_chunks, int64_t* race_chunks) {
    const int64_t pc = bf16 ? part_chunk<__nv_bfloat16>() : part_chunk<float>();
    const int64_t rc = bf16 ? race_chunk<__nv_bfloat16>() : race_chunk<float>();
    *partial_chunks = (V + pc - 1) / pc;
    *race_chunks = (V + rc - 1) / rc;
}

cudaError_t launch_verify(const VerifyArgs& a, bool bf16, bool wide, cudaStream_t stream) {
    return bf16 ? launch_typed<__nv_bfloat16>(a, wide, stream) : launch_typed<float>(a, wide, stream);
}

}  // namespace lms
