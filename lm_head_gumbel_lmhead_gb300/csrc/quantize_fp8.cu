// Per-row FP8 (E4M3) quantisation of bf16 activations for the W8A8 fused path: row b is scaled by
// 2^-e_b, e_b the smallest integer with max_d |H[b][d]| * 2^-e_b <= 448 (0 for an all-zero row),
// and rounded to the nearest E4M3 value (ties to even, saturating).  A power-of-two scale makes the
// scaling exact, so the rounding is the only inexact step.
#include <cuda_bf16.h>
#include <cuda_fp8.h>

#include "lms_device.cuh"
#include "lms_kernels.h"

namespace lms {
namespace {

constexpr int kThreads = 256;

__global__ void __launch_bounds__(kThreads) quantize_rows_e4m3_kernel(
    const __nv_bfloat16* __restrict__ H, int64_t ldh, int64_t D, uint8_t* __restrict__ q,
    int64_t ldq, int32_t* __restrict__ e_out) {
    pdl_launch_dependents();          // the fused kernel may start its prologue now
    const int64_t b = blockIdx.x;
    const __nv_bfloat16* h = H + b * ldh;
    float amax = 0.0f;
    for (int64_t d = threadIdx.x; d < D; d += kThreads) amax = fmaxf(amax, fabsf(__bfloat162float(h[d])));
    for (int off = 16; off > 0; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
    __shared__ float sh[kThreads / 32];
    __shared__ int sh_e;
    if ((threadIdx.x & 31) == 0) sh[threadIdx.x >> 5] = amax;
    __syncthreads();
    if (threadIdx.x == 0) {
        float m = 0.0f;
        for (int w = 0; w < kThreads / 32; ++w) m = fmaxf(m, sh[w]);
        int e = 0;
        if (m > 0.0f) {
            e = ilogbf(m) - 8;                               // m * 2^-e is in [256, 512)
            while (ldexpf(m, -e) > 448.0f) ++e;
            while (ldexpf(m, -(e - 1)) <= 448.0f) --e;
        }
        sh_e = e;
        e_out[b] = e;
    }
    __syncthreads();
    const int e = sh_e;
    for (int64_t d = threadIdx.x; d < D; d += kThreads)
        q[b * ldq + d] = static_cast<uint8_t>(
            __nv_cvt_float_to_fp8(ldexpf(__bfloat162float(h[d]), -e), __NV_SATFINITE, __NV_E4M3));
}

}  // namespace

cudaError_t launch_quantize_rows_e4m3(const uint16_t* H, int64_t ldh, int64_t B, int64_t D,
                                      uint8_t* q, int64_t ldq, int32_t* e_out, cudaStream_t stream) {
    quantize_rows_e4m3_kernel<<<static_cast<unsigned>(B), kThreads, 0, stream>>>(
        reinterpret_cast<const __nv_bfloat16*>(H), ldh, D, q, ldq, e_out);
    return cudaGetLastError();
}

}  // namespace lms
