// Fused LM-head + Gumbel-max Stage 1 on CUDA cores, for tiny batches (B <= 8): one CTA per
// vocabulary tile of 128 rows of W.  H sits in shared memory; W streams from HBM with 128-bit
// loads straight into fp32 FMAs; the [128 x B] logits tile stays on chip.
// (FlashSampling "method step details", Stage 1 steps 1-6.)
#include <cuda_bf16.h>

#include "lms_device.cuh"
#include "lms_kernels.h"

namespace lms {
namespace {

constexpr int kTileV = 128;
constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kRowsPerWarp = kTileV / kWarps;   // 16
constexpr int kRowGroup = 4;                    // rows whose loads are in flight together

__device__ __forceinline__ void bf16x8_to_float(const uint4& raw, float (&f)[8]) {
    const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        f[2 * j] = __uint_as_float(w[j] << 16);
        f[2 * j + 1] = __uint_as_float(w[j] & 0xffff0000u);
    }
}

template <int kB, bool kWide>
__global__ void __launch_bounds__(kThreads) lmhead_gemv_kernel(const uint16_t* __restrict__ H,
                                                               int64_t ldh,
                                                               const uint16_t* __restrict__ W,
                                                               int64_t ldw, int D, SampleArgs a) {
    extern __shared__ __align__(16) unsigned char smem_raw[];
    uint16_t* h_s = reinterpret_cast<uint16_t*>(smem_raw);                 // [B][D]
    __shared__ __align__(16) float y_s[kB][kTileV];
    __shared__ RowParams p_s[kB];

    const int B = static_cast<int>(a.B);
    const int tile = blockIdx.x;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    clear_status_bits(a.status_bits, a.row0);

    // Stage H (B rows of D bf16) into shared memory, 16 bytes at a time.
    const int chunks_per_row = D / 8;
    for (int c = threadIdx.x; c < B * chunks_per_row; c += kThreads) {
        const int b = c / chunks_per_row, k = c - b * chunks_per_row;
        reinterpret_cast<uint4*>(h_s)[c] =
            __ldg(reinterpret_cast<const uint4*>(H + (a.row0 + b) * ldh) + k);
    }
    if (threadIdx.x < B) {
        p_s[threadIdx.x] = make_row_params(a.temperature, a.seeds, a.positions, a.base_seed,
                                           a.offset, a.row0 + threadIdx.x);
    }
    __syncthreads();

    // Step 1: y[r][b] = sum_d H[b][d] W[v][d] for this warp's 16 rows, 4 rows at a time.
    const int64_t v_tile0 = static_cast<int64_t>(tile) * kTileV;
    for (int g = 0; g < kRowsPerWarp / kRowGroup; ++g) {
        const int r0 = warp * kRowsPerWarp + g * kRowGroup;
        float acc[kRowGroup][kB];
#pragma unroll
        for (int r = 0; r < kRowGroup; ++r)
#pragma unroll
            for (int b = 0; b < kB; ++b) acc[r][b] = 0.0f;
        const uint4* wrow[kRowGroup];
        bool rvalid[kRowGroup];
#pragma unroll
        for (int r = 0; r < kRowGroup; ++r) {
            const int64_t v = v_tile0 + r0 + r;
            rvalid[r] = v < a.V;
            wrow[r] = reinterpret_cast<const uint4*>(W + (rvalid[r] ? v : 0) * ldw);
        }
#pragma unroll 2
        for (int k = lane; k < chunks_per_row; k += 32) {
            float wf[kRowGroup][8];
#pragma unroll
            for (int r = 0; r < kRowGroup; ++r)
                bf16x8_to_float(rvalid[r] ? __ldcs(wrow[r] + k) : make_uint4(0, 0, 0, 0), wf[r]);
#pragma unroll
            for (int b = 0; b < kB; ++b) {
                if (b < B) {
                    float hf[8];
                    bf16x8_to_float(reinterpret_cast<const uint4*>(h_s + b * D)[k], hf);
#pragma unroll
                    for (int r = 0; r < kRowGroup; ++r)
#pragma unroll
                        for (int j = 0; j < 8; ++j) acc[r][b] = fmaf(hf[j], wf[r][j], acc[r][b]);
                }
            }
        }
#pragma unroll
        for (int r = 0; r < kRowGroup; ++r)
#pragma unroll
            for (int b = 0; b < kB; ++b) {
                float x = acc[r][b];
#pragma unroll
                for (int off = 16; off > 0; off >>= 1) x += __shfl_xor_sync(0xffffffffu, x, off);
                if (lane == 0 && b < B) y_s[b][r0 + r] = x;
            }
    }
    __syncthreads();

    // Steps 2-6: transform, noise, argmax over the tile's 128 entries, one candidate per row.
    // Warp w takes batch row b = w (B <= 8 = warps); lane l the four consecutive entries
    // 4l .. 4l + 3, which one Philox call covers (fp32 noise; two calls for wide noise).
    for (int b = warp; b < B; b += kWarps) {
        const RowParams p = p_s[b];
        const int r0 = 4 * lane;
        const int64_t v0 = v_tile0 + r0;
        float best_s = -CUDART_INF_F;
        int best_i = kNoIndex;
        if (v0 < a.V && !(p.flags & kRowInvalid)) {
            float g[4];
            if (p.flags & kRowGreedy) {
                g[0] = g[1] = g[2] = g[3] = 0.0f;
            } else {
                gumbel_run<kWide, 4>(p.key, static_cast<uint32_t>(v0), g);
            }
            const int64_t row = a.row0 + b;
            const float* brow = a.bias ? a.bias + row * a.ld_bias : nullptr;
            const uint32_t mword = a.mask ? (__ldg(a.mask + row * a.ld_mask + (v0 >> 5)) >> (v0 & 31)) : 0xfu;
            const float4 y = *reinterpret_cast<const float4*>(&y_s[b][r0]);
            const float yv[4] = {y.x, y.y, y.z, y.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int64_t v = v0 + e;
                if (v < a.V) {
                    const float bias = brow ? __ldg(brow + v) : 0.0f;
                    const float sc = perturb(p, yv[e], bias, (mword >> e) & 1u, g[e]);
                    if (sc > best_s) { best_s = sc; best_i = static_cast<int>(v); }
                }
            }
        }
        warp_argmax(best_s, best_i);
        if (lane == 0) {
            a.cand_score[b * a.n_tiles + tile] = best_s;
            a.cand_index[b * a.n_tiles + tile] = candidate_index(best_s, best_i);
        }
    }
    pdl_launch_dependents();
}

template <int kB>
cudaError_t launch_b(const uint16_t* H, int64_t ldh, const uint16_t* W, int64_t ldw, int64_t D,
                     bool wide, const SampleArgs& a, cudaStream_t stream) {
    const size_t smem = static_cast<size_t>(a.B) * D * sizeof(uint16_t);
    const unsigned grid = static_cast<unsigned>(a.n_tiles);
    cudaError_t e;
    if (wide) {
        e = ensure_dynamic_smem(reinterpret_cast<const void*>(lmhead_gemv_kernel<kB, true>), smem);
        if (e != cudaSuccess) return e;
        lmhead_gemv_kernel<kB, true><<<grid, kThreads, smem, stream>>>(H, ldh, W, ldw, static_cast<int>(D), a);
    } else {
        e = ensure_dynamic_smem(reinterpret_cast<const void*>(lmhead_gemv_kernel<kB, false>), smem);
        if (e != cudaSuccess) return e;
        lmhead_gemv_kernel<kB, false><<<grid, kThreads, smem, stream>>>(H, ldh, W, ldw, static_cast<int>(D), a);
    }
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_lmhead_gemv(const uint16_t* H, int64_t ldh, const uint16_t* W, int64_t ldw,
                               int64_t D, bool wide, const SampleArgs& a, cudaStream_t stream) {
    if (a.B <= 1) return launch_b<1>(H, ldh, W, ldw, D, wide, a, stream);
    if (a.B <= 2) return launch_b<2>(H, ldh, W, ldw, D, wide, a, stream);
    if (a.B <= 4) return launch_b<4>(H, ldh, W, ldw, D, wide, a, stream);
    return launch_b<8>(H, ldh, W, ldw, D, wide, a, stream);
}

}  // namespace lms
