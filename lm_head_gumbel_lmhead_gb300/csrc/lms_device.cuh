// Device-side building blocks shared by the sampling kernels: the Philox4x32-10 generator, the
// uniform -> exponential -> Gumbel noise in fp32, the per-row transform, and the
// lexicographic (score, index) argmax.  Every kernel computes the noise through these
// functions, so the noise-fill kernel tests exactly what the samplers use.
#pragma once
#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <math_constants.h>

namespace lms {

// ---------------------------------------------------------------------------------------------
// Philox4x32-10 (Salmon, Moraes, Dror, Shaw, "Parallel Random Numbers: As Easy as 1, 2, 3",
// SC'11): ten rounds of two 32x32->64-bit products whose high halves are xored with the other
// two words and the round key; the key advances by the Weyl constants between rounds.
// ---------------------------------------------------------------------------------------------
constexpr uint32_t kPhiloxMulA = 0xD2511F53u;
constexpr uint32_t kPhiloxMulB = 0xCD9E8D57u;
constexpr uint32_t kWeylA = 0x9E3779B9u;
constexpr uint32_t kWeylB = 0xBB67AE85u;

struct Words { uint32_t w0, w1, w2, w3; };

__device__ __forceinline__ Words philox4x32_10(uint32_t x0, uint32_t x1, uint32_t x2, uint32_t x3,
                                               uint32_t ka, uint32_t kb) {
#pragma unroll
    for (int round = 0; round < 10; ++round) {
        // the two products as separate high and low halves (32-bit multiplies)
        const uint32_t hi_a = __umulhi(kPhiloxMulA, x0), lo_a = kPhiloxMulA * x0;
        const uint32_t hi_b = __umulhi(kPhiloxMulB, x2), lo_b = kPhiloxMulB * x2;
        const uint32_t n0 = hi_b ^ x1 ^ (ka + static_cast<uint32_t>(round) * kWeylA);
        const uint32_t n2 = hi_a ^ x3 ^ (kb + static_cast<uint32_t>(round) * kWeylB);
        x1 = lo_b;
        x3 = lo_a;
        x0 = n0;
        x2 = n2;
    }
    return {x0, x1, x2, x3};
}

// Per-row generator state: the key and the counter words that do not depend on v.
struct RowKey {
    uint32_t ka, kb;      // key
    uint32_t c1, c2, c3;  // counter words 1..3 (word 0 is the vocabulary index)
};

// (request seed, absolute position) for seeded rows; (base_seed, offset, row) otherwise.
__device__ __forceinline__ RowKey make_row_key(const int64_t* seeds, const int64_t* positions,
                                               uint64_t base_seed, uint64_t offset, int64_t row) {
    RowKey k;
    if (seeds != nullptr && seeds[row] >= 0) {
        const uint64_t s = static_cast<uint64_t>(seeds[row]);
        const uint64_t p = static_cast<uint64_t>(positions[row]);
        k.ka = static_cast<uint32_t>(s);
        k.kb = static_cast<uint32_t>(s >> 32);
        k.c1 = static_cast<uint32_t>(p);
        k.c2 = static_cast<uint32_t>(p >> 32);
        k.c3 = 0u;
    } else {
        k.ka = static_cast<uint32_t>(base_seed);
        k.kb = static_cast<uint32_t>(base_seed >> 32);
        k.c1 = static_cast<uint32_t>(offset);
        k.c2 = static_cast<uint32_t>(offset >> 32);
        k.c3 = 0x80000000u | static_cast<uint32_t>(row);
    }
    return k;
}

// One Philox call of a row: counter (n, c1, c2, c3) under the row's key.  With fp32 noise the
// call n serves the four vocabulary entries 4n..4n+3 (entry v takes word v & 3); with wide noise
// it serves 2n and 2n+1 (entry v takes words 2(v & 1) and 2(v & 1) + 1, low half first).  The
// variate of an entry is therefore a function of (seed, position, v) alone, and no word is
// dropped.
__device__ __forceinline__ Words row_call(const RowKey& k, uint32_t n) {
    return philox4x32_10(n, k.c1, k.c2, k.c3, k.ka, k.kb);
}

// ---------------------------------------------------------------------------------------------
// Uniform -> E = -log u -> g = -log E, in fp32.
//
// u = (k + 1/2) / 2^m is written as n / 2^(m+1) with n = 2k + 1 odd, and its complement
// c = 1 - u = j / 2^(m+1) with j = 2^(m+1) - n, both from integers.  Two evaluations of E, one
// kept:
//  * c >= 3/8 (u <= 5/8, E >= 0.47): E = -ln2 * log2(u) with the hardware base-2 logarithm,
//    whose absolute error near 1 is about 2^-22, i.e. at most 2^-21 relative to E here;
//  * c < 3/8: E = -log(1 - c) = 2 atanh(z) with z = c / (2 - c) = j / (2^(m+2) - j) < 3/13,
//    summed to z^9/9 (the first omitted term, z^11/11, is below 2^-24 z).
// The tail (u -> 1, E -> 0, the largest g) therefore keeps full relative precision: E reaches
// 2^-25 (fp32 noise) and 2^-53 (wide noise), the ranges the Megatron-LM PR gives.
// ---------------------------------------------------------------------------------------------

// Hardware base-2 logarithm and reciprocal (PTX lg2.approx / rcp.approx, flush-to-zero forms).
// Every argument passed to them here is a normal float (at least 2^-53), so the subnormal
// handling of the non-ftz forms is not needed.
__device__ __forceinline__ float lg2_approx(float x) {
    float r;
    asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
    return r;
}
__device__ __forceinline__ float rcp_approx(float x) {
    float r;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
    return r;
}
constexpr float kLn2f = 0.693147180559945309f;

// -log(1 - c) = 2 atanh(z) from z = c / (2 - c) <= 3/13: 2 z (1 + z^2/3 + z^4/5 + z^6/7 + z^8/9).
__device__ __forceinline__ float two_atanh_series(float z) {
    const float z2 = z * z;
    float p = 2.0f / 9.0f;
    p = fmaf(p, z2, 2.0f / 7.0f);
    p = fmaf(p, z2, 2.0f / 5.0f);
    p = fmaf(p, z2, 2.0f / 3.0f);
    p = fmaf(p, z2, 2.0f);
    return z * p;
}

// E from the entry's word, fp32 noise: n = 2 (w >> 8) + 1, u = n / 2^25.
__device__ __forceinline__ float exponential_fp32(uint32_t w) {
    const uint32_t n = (w >> 7) | 1u;
    const uint32_t j = (1u << 25) - n;
    const float from_u = -kLn2f * lg2_approx(static_cast<float>(n) * 0x1p-25f);
    const float jf = static_cast<float>(j);                       // exact when it is used
    const float from_c = two_atanh_series(jf * rcp_approx(0x1p26f - jf));
    return j < (3u << 22) ? from_c : from_u;
}

// A 53-bit integer to fp32 (one rounding of the low part, then one of the sum).
__device__ __forceinline__ float int53_to_float(uint64_t n) {
    return fmaf(static_cast<float>(static_cast<uint32_t>(n >> 32)), 0x1p32f,
                static_cast<float>(static_cast<uint32_t>(n)));
}

// E from the entry's two words, wide noise: n = 2 k + 1 with k = ((hi << 32) | lo) >> 12,
// u = n / 2^53.
__device__ __forceinline__ float exponential_wide(uint32_t lo, uint32_t hi) {
    const uint64_t n = (((static_cast<uint64_t>(hi) << 32) | lo) >> 11) | 1ull;
    const uint64_t j = (1ull << 53) - n;
    const float from_u = -kLn2f * lg2_approx(int53_to_float(n) * 0x1p-53f);
    const float jf = int53_to_float(j);
    const float from_c = two_atanh_series(jf * rcp_approx(0x1p54f - jf));
    return j < (3ull << 50) ? from_c : from_u;
}

__device__ __forceinline__ float gumbel_from_exponential(float E) { return -kLn2f * lg2_approx(E); }

// Gumbel noise of one entry (a whole call per entry: for kernels that visit entries one by one).
template <bool kWide>
__device__ __forceinline__ float gumbel_one(const RowKey& k, uint32_t v) {
    if (kWide) {
        const Words w = row_call(k, v >> 1);
        const bool second = v & 1u;
        return gumbel_from_exponential(exponential_wide(second ? w.w2 : w.w0, second ? w.w3 : w.w1));
    }
    const Words w = row_call(k, v >> 2);
    const uint32_t j = v & 3u;
    const uint32_t word = j == 0 ? w.w0 : j == 1 ? w.w1 : j == 2 ? w.w2 : w.w3;
    return gumbel_from_exponential(exponential_fp32(word));
}

// Gumbel noise of kN consecutive entries v0 .. v0 + kN - 1 from kN / 4 calls (fp32 noise) or
// kN / 2 calls (wide noise).  v0 must be a multiple of 4 (fp32) or 2 (wide), kN of the same.
template <bool kWide, int kN>
__device__ __forceinline__ void gumbel_run(const RowKey& k, uint32_t v0, float (&g)[kN]) {
    if constexpr (kWide) {
        static_assert(kN % 2 == 0, "wide noise: entries come in pairs");
#pragma unroll
        for (int c = 0; c < kN / 2; ++c) {
            const Words w = row_call(k, (v0 >> 1) + c);
            g[2 * c] = gumbel_from_exponential(exponential_wide(w.w0, w.w1));
            g[2 * c + 1] = gumbel_from_exponential(exponential_wide(w.w2, w.w3));
        }
    } else {
        static_assert(kN % 4 == 0, "fp32 noise: entries come in fours");
#pragma unroll
        for (int c = 0; c < kN / 4; ++c) {
            const Words w = row_call(k, (v0 >> 2) + c);
            g[4 * c] = gumbel_from_exponential(exponential_fp32(w.w0));
            g[4 * c + 1] = gumbel_from_exponential(exponential_fp32(w.w1));
            g[4 * c + 2] = gumbel_from_exponential(exponential_fp32(w.w2));
            g[4 * c + 3] = gumbel_from_exponential(exponential_fp32(w.w3));
        }
    }
}

// Entries p[0 .. 7] as floats (0 past n): one or two 16-byte loads when the unit is whole and
// p is 16-byte aligned, else element loads.
__device__ __forceinline__ void load8(const __nv_bfloat16* p, int n, bool vec, float (&out)[8]) {
    if (vec && n >= 8) {
        const uint4 w = __ldg(reinterpret_cast<const uint4*>(p));
        const uint32_t u[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            out[2 * i] = __uint_as_float(u[i] << 16);
            out[2 * i + 1] = __uint_as_float(u[i] & 0xffff0000u);
        }
    } else {
#pragma unroll
        for (int e = 0; e < 8; ++e) out[e] = e < n ? __bfloat162float(p[e]) : 0.0f;
    }
}

__device__ __forceinline__ void load8(const float* p, int n, bool vec, float (&out)[8]) {
    if (vec && n >= 8) {
        const float4 a = __ldg(reinterpret_cast<const float4*>(p));
        const float4 b = __ldg(reinterpret_cast<const float4*>(p) + 1);
        out[0] = a.x; out[1] = a.y; out[2] = a.z; out[3] = a.w;
        out[4] = b.x; out[5] = b.y; out[6] = b.z; out[7] = b.w;
    } else {
#pragma unroll
        for (int e = 0; e < 8; ++e) out[e] = e < n ? __ldg(p + e) : 0.0f;
    }
}

// ---------------------------------------------------------------------------------------------
// Per-row parameters and the transform (bias before temperature; T == 0 greedy; mask -> -inf).
// ---------------------------------------------------------------------------------------------
enum RowFlags : uint32_t { kRowGreedy = 1u, kRowInvalid = 2u };

struct __align__(16) RowParams {
    RowKey key;
    float inv_t;     // 1 / T for sampled rows
    uint32_t flags;  // RowFlags
    uint32_t pad;
};

__device__ __forceinline__ RowParams make_row_params(const float* temperature, const int64_t* seeds,
                                                     const int64_t* positions, uint64_t base_seed,
                                                     uint64_t offset, int64_t row) {
    RowParams p;
    p.key = make_row_key(seeds, positions, base_seed, offset, row);
    const float T = temperature ? temperature[row] : 1.0f;
    p.flags = 0u;
    p.pad = 0u;
    p.inv_t = 1.0f;
    if (!(T >= 0.0f)) {
        p.flags = kRowInvalid;           // T < 0 or NaN
    } else if (T == 0.0f) {
        p.flags = kRowGreedy;
    } else {
        p.inv_t = 1.0f / T;
    }
    return p;
}

__device__ __forceinline__ bool allowed(const uint32_t* mask_row, uint32_t v) {
    return mask_row == nullptr || ((__ldg(mask_row + (v >> 5)) >> (v & 31u)) & 1u);
}

// Perturbed score of one entry from its raw logit y, bias (0 if none), mask bit and noise g
// (ignored on greedy rows).  Bias before temperature; NaN counts as -inf.
__device__ __forceinline__ float perturb(const RowParams& p, float y, float bias, bool is_allowed,
                                         float g) {
    const float t = y + bias;
    const float s = (p.flags & kRowGreedy) ? t : fmaf(t, p.inv_t, g);
    return (is_allowed && s == s) ? s : -CUDART_INF_F;
}

// The same for one entry visited on its own (computes its Philox call).
template <bool kWide>
__device__ __forceinline__ float perturbed_score(const RowParams& p, uint32_t v, float y,
                                                 float bias, bool is_allowed) {
    if (!is_allowed) return -CUDART_INF_F;
    const float g = (p.flags & kRowGreedy) ? 0.0f : gumbel_one<kWide>(p.key, v);
    return perturb(p, y, bias, true, g);
}

// ---------------------------------------------------------------------------------------------
// Lexicographic argmax: larger score, then smaller index.  Index 0x7fffffff marks "nothing yet".
// ---------------------------------------------------------------------------------------------
constexpr int kNoIndex = 0x7fffffff;

__device__ __forceinline__ bool better(float sa, int ia, float sb, int ib) {
    return sa > sb || (sa == sb && ia < ib);
}

__device__ __forceinline__ void warp_argmax(float& s, int& i) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        const float so = __shfl_xor_sync(0xffffffffu, s, off);
        const int io = __shfl_xor_sync(0xffffffffu, i, off);
        if (better(so, io, s, i)) { s = so; i = io; }
    }
}

// Argmax of 16 columns across the 32 lanes of a warp at once ("transposed" reduction): lane l
// holds scores s[j] / indices ix[j] of its own row for columns j = 0..15.  Four halving rounds
// (shuffle offsets 16, 8, 4, 2) each keep half of the columns in every lane, combined with the
// partner lane's values for the same columns; a last xor-1 round finishes.  On return s[0] /
// ix[0] of lane l hold the result for column (l >> 1) & 15 over all 32 rows.  16 shuffle pairs
// instead of 16 x 5 for column-by-column reductions.
template <int kN>
__device__ __forceinline__ void halve_columns(float (&s)[16], int (&ix)[16], int lane) {
    constexpr int kH = kN / 2;
    const bool upper = (lane & kN) != 0;
#pragma unroll
    for (int j = 0; j < kH; ++j) {
        const float keep_s = upper ? s[j + kH] : s[j];
        const int keep_i = upper ? ix[j + kH] : ix[j];
        const float send_s = upper ? s[j] : s[j + kH];
        const int send_i = upper ? ix[j] : ix[j + kH];
        const float rs = __shfl_xor_sync(0xffffffffu, send_s, kN);
        const int ri = __shfl_xor_sync(0xffffffffu, send_i, kN);
        const bool take = better(rs, ri, keep_s, keep_i);
        s[j] = take ? rs : keep_s;
        ix[j] = take ? ri : keep_i;
    }
}

__device__ __forceinline__ void warp_argmax_16_columns(float (&s)[16], int (&ix)[16], int lane) {
    halve_columns<16>(s, ix, lane);
    halve_columns<8>(s, ix, lane);
    halve_columns<4>(s, ix, lane);
    halve_columns<2>(s, ix, lane);
    const float rs = __shfl_xor_sync(0xffffffffu, s[0], 1);
    const int ri = __shfl_xor_sync(0xffffffffu, ix[0], 1);
    if (better(rs, ri, s[0], ix[0])) { s[0] = rs; ix[0] = ri; }
}

// The candidate a tile reports: index -1 when nothing in the tile is above -inf.
__device__ __forceinline__ int candidate_index(float s, int i) {
    return (s > -CUDART_INF_F && i != kNoIndex) ? i : -1;
}

// Index written by a CTA whose device-side wait ran out of time.
constexpr int kPoisonIndex = -2;

// The call's status word: bit s is set when some row of the call ended with row status s != 0.
// Stage 1 of the call's first launch clears it (block 0, thread 0 of the launch that starts at
// row 0: stream order puts it after the previous call's Stage 2); Stage 2 sets the bits.
__device__ __forceinline__ void clear_status_bits(uint32_t* bits, int64_t row0) {
    if (bits != nullptr && row0 == 0 && blockIdx.x == 0 && blockIdx.y == 0 && blockIdx.z == 0 &&
        threadIdx.x == 0)
        *bits = 0u;
}
__device__ __forceinline__ void note_row_status(uint32_t* bits, int status) {
    if (bits != nullptr && status != 0) atomicOr(bits, 1u << status);
}

// Programmatic dependent launch: let the dependent grid start launching / wait for the primary.
__device__ __forceinline__ void pdl_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void pdl_wait_primary() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

}  // namespace lms
