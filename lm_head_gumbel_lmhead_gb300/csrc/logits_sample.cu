// Stage 1 of the Gumbel race over materialised logits: one CTA per (row, tile of tile_v
// entries), the noise generated in registers, one (score, index) candidate per CTA.
// (Megatron-LM PR 8370, "Cost": a fused kernel that generates the noise in registers and reduces
// each row in place, with several blocks per row; FlashSampling steps 2-6 over a logits tile.)
#include <cuda_bf16.h>

#include "lms_device.cuh"
#include "lms_kernels.h"

namespace lms {
namespace {

constexpr int kThreads = 256;

template <typename T>
__device__ __forceinline__ float to_float(T x);
template <>
__device__ __forceinline__ float to_float<float>(float x) { return x; }
template <>
__device__ __forceinline__ float to_float<__nv_bfloat16>(__nv_bfloat16 x) { return __bfloat162float(x); }

// A unit of kUnit consecutive entries per thread and iteration (a multiple of 4, so that whole
// Philox calls cover it): one 16-byte load when the row is 16-byte aligned, else scalar loads.
template <typename T, int kUnit, bool kVector>
__device__ __forceinline__ void load_unit(const T* p, int64_t n_valid, float (&y)[kUnit]) {
    if (kVector && n_valid >= kUnit) {
        static_assert(kUnit * sizeof(T) == 16 || !kVector, "vector units are 16 bytes");
        const uint4 raw = __ldg(reinterpret_cast<const uint4*>(p));
        const T* e = reinterpret_cast<const T*>(&raw);
#pragma unroll
        for (int j = 0; j < kUnit; ++j) y[j] = to_float<T>(e[j]);
    } else {
#pragma unroll
        for (int j = 0; j < kUnit; ++j) y[j] = (j < n_valid) ? to_float<T>(p[j]) : 0.0f;
    }
}

// kPlain: no bias and no mask in this launch.  A sampled row then takes the fast loop: whole
// units with 32-bit indices and no per-entry checks.  NaN needs no test there: a NaN score never
// compares above the running best, so it loses to everything, as -inf does.
template <typename T, int kUnit, bool kVector, bool kWide, bool kPlain>
__global__ void __launch_bounds__(kThreads) logits_stage1_kernel(const T* __restrict__ logits,
                                                                 int64_t ld, int tile_v,
                                                                 SampleArgs a) {
    const int64_t cta = blockIdx.x;
    const int64_t b = cta / a.n_tiles;             // local row
    const int64_t t = cta - b * a.n_tiles;         // tile
    const int64_t row = a.row0 + b;
    clear_status_bits(a.status_bits, a.row0);
    const RowParams p = make_row_params(a.temperature, a.seeds, a.positions, a.base_seed,
                                        a.offset, row);
    float best_s = -CUDART_INF_F;
    int best_i = kNoIndex;
    if (!(p.flags & kRowInvalid)) {
        const T* y_row = logits + row * ld;
        const uint32_t v_tile = static_cast<uint32_t>(t * tile_v);
        const uint32_t v_end = static_cast<uint32_t>((t * tile_v + tile_v < a.V) ? t * tile_v + tile_v : a.V);
        if (kPlain && !(p.flags & kRowGreedy)) {
            // Units are strided by the CTA so that each thread visits its entries in increasing v
            // (strict '>' then keeps the smallest index among equal scores within the thread).
            for (uint32_t v0 = v_tile + threadIdx.x * kUnit; v0 < v_end; v0 += kThreads * kUnit) {
                float y[kUnit];
                load_unit<T, kUnit, kVector>(y_row + v0, v_end - v0, y);
                float g[kUnit];
                gumbel_run<kWide, kUnit>(p.key, v0, g);
                if (v0 + kUnit <= v_end) {
#pragma unroll
                    for (int j = 0; j < kUnit; ++j) {
                        const float s = fmaf(y[j], p.inv_t, g[j]);
                        if (s > best_s) { best_s = s; best_i = static_cast<int>(v0 + j); }
                    }
                } else {
                    const uint32_t n = v_end - v0;
#pragma unroll
                    for (int j = 0; j < kUnit; ++j) {
                        const float s = fmaf(y[j], p.inv_t, g[j]);
                        if (j < n && s > best_s) { best_s = s; best_i = static_cast<int>(v0 + j); }
                    }
                }
            }
        } else if (kPlain) {
            // greedy row, no bias and no mask: the argmax of y itself
            for (uint32_t v0 = v_tile + threadIdx.x * kUnit; v0 < v_end; v0 += kThreads * kUnit) {
                float y[kUnit];
                load_unit<T, kUnit, kVector>(y_row + v0, v_end - v0, y);
                const uint32_t n = v_end - v0;
#pragma unroll
                for (int j = 0; j < kUnit; ++j)
                    if (j < n && y[j] > best_s) { best_s = y[j]; best_i = static_cast<int>(v0 + j); }
            }
        } else {
            const float* bias_row = a.bias ? a.bias + row * a.ld_bias : nullptr;
            const uint32_t* mask_row = a.mask ? a.mask + row * a.ld_mask : nullptr;
            for (uint32_t v0 = v_tile + threadIdx.x * kUnit; v0 < v_end; v0 += kThreads * kUnit) {
                float y[kUnit];
                load_unit<T, kUnit, kVector>(y_row + v0, v_end - v0, y);
                float g[kUnit];
                if (p.flags & kRowGreedy) {
#pragma unroll
                    for (int j = 0; j < kUnit; ++j) g[j] = 0.0f;
                } else {
                    gumbel_run<kWide, kUnit>(p.key, v0, g);
                }
#pragma unroll
                for (int j = 0; j < kUnit; ++j) {
                    const uint32_t v = v0 + j;
                    if (v < v_end) {
                        const float bias = bias_row ? __ldg(bias_row + v) : 0.0f;
                        const float s = perturb(p, y[j], bias, allowed(mask_row, v), g[j]);
                        if (s > best_s) { best_s = s; best_i = static_cast<int>(v); }
                    }
                }
            }
        }
    }
    // Block argmax: shuffles within warps, then across the warps through shared memory.
    warp_argmax(best_s, best_i);
    __shared__ float sh_s[kThreads / 32];
    __shared__ int sh_i[kThreads / 32];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (lane == 0) { sh_s[warp] = best_s; sh_i[warp] = best_i; }
    __syncthreads();
    if (threadIdx.x == 0) {
#pragma unroll
        for (int w = 1; w < kThreads / 32; ++w)
            if (better(sh_s[w], sh_i[w], best_s, best_i)) { best_s = sh_s[w]; best_i = sh_i[w]; }
        a.cand_score[b * a.n_tiles + t] = best_s;
        a.cand_index[b * a.n_tiles + t] = candidate_index(best_s, best_i);
    }
    pdl_launch_dependents();
}

template <typename T, int kUnit, bool kVector, bool kWide>
void launch_noise(const T* y, int64_t ld, int tile_v, bool plain, const SampleArgs& a,
                  unsigned grid, cudaStream_t stream) {
    if (plain) {
        logits_stage1_kernel<T, kUnit, kVector, kWide, true><<<grid, kThreads, 0, stream>>>(y, ld, tile_v, a);
    } else {
        logits_stage1_kernel<T, kUnit, kVector, kWide, false><<<grid, kThreads, 0, stream>>>(y, ld, tile_v, a);
    }
}

template <typename T, int kUnit, bool kVector>
cudaError_t launch_typed(const void* logits, int64_t ld, int tile_v, bool wide, const SampleArgs& a,
                         cudaStream_t stream) {
    const unsigned grid = static_cast<unsigned>(a.B * a.n_tiles);
    const T* y = static_cast<const T*>(logits);
    const bool plain = a.bias == nullptr && a.mask == nullptr;
    if (wide) {
        launch_noise<T, kUnit, kVector, true>(y, ld, tile_v, plain, a, grid, stream);
    } else {
        launch_noise<T, kUnit, kVector, false>(y, ld, tile_v, plain, a, grid, stream);
    }
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_logits_stage1(const void* logits, bool bf16, int64_t ld, int tile_v, bool wide,
                                 const SampleArgs& a, cudaStream_t stream) {
    const size_t esize = bf16 ? 2 : 4;
    const bool aligned = (reinterpret_cast<uintptr_t>(logits) % 16 == 0) &&
                         ((static_cast<size_t>(ld) * esize) % 16 == 0);
    if (bf16) {
        return aligned ? launch_typed<__nv_bfloat16, 8, true>(logits, ld, tile_v, wide, a, stream)
                       : launch_typed<__nv_bfloat16, 4, false>(logits, ld, tile_v, wide, a, stream);
    }
    return aligned ? launch_typed<float, 4, true>(logits, ld, tile_v, wide, a, stream)
                   : launch_typed<float, 4, false>(logits, ld, tile_v, wide, a, stream);
}

}  // namespace lms
