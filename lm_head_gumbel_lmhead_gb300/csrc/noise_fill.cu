// Noise-fill kernel: the Philox words and the noise the sampling kernels use, written out.
// (Megatron-LM PR 8370, "The change" / "Tests": seeded noise keyed by (request seed, absolute
// position, vocabulary index) that replays bit-exactly.)
#include "lms_device.cuh"
#include "lms_kernels.h"

namespace lms {
namespace {

// One row per blockIdx.y (its key computed once per thread, no division), one thread per Philox
// call: the call serves 4 consecutive entries (fp32 noise) or 2 (wide).  E and g of a whole call
// go out in one 16-byte (fp32 noise) or 8-byte (wide) store when the row start allows it.
template <int kKind, bool kWide>
__global__ void __launch_bounds__(256) noise_fill_kernel(void* __restrict__ out, int64_t row0, int64_t V,
                                                          const int64_t* __restrict__ seeds,
                                                          const int64_t* __restrict__ positions,
                                                          uint64_t base_seed, uint64_t offset) {
    constexpr int kPer = kWide ? 2 : 4;
    const int64_t b = row0 + blockIdx.y;
    const int64_t calls = (V + kPer - 1) / kPer;
    const RowKey k = make_row_key(seeds, positions, base_seed, offset, b);
    const int64_t row_base = b * V;
    // vector stores need the buffer and the row start on the vector boundary (the entry point
    // only guarantees 4-byte alignment of the buffer)
    const bool vec = (row_base % kPer) == 0 &&
                     (reinterpret_cast<uintptr_t>(out) % (kPer * sizeof(float))) == 0;
    for (int64_t n = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; n < calls;
         n += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const Words w = row_call(k, static_cast<uint32_t>(n));
        const uint32_t word[4] = {w.w0, w.w1, w.w2, w.w3};
        const int64_t v0 = n * kPer;
        if constexpr (kKind >= 2) {
            float r[kPer];
#pragma unroll
            for (int e = 0; e < kPer; ++e) {
                const float E = kWide ? exponential_wide(word[2 * e], word[2 * e + 1]) : exponential_fp32(word[e]);
                r[e] = (kKind == 2) ? E : gumbel_from_exponential(E);
            }
            float* o = reinterpret_cast<float*>(out) + row_base + v0;
            if (vec && v0 + kPer <= V) {
                if constexpr (kWide) {
                    *reinterpret_cast<float2*>(o) = make_float2(r[0], r[1]);
                } else {
                    *reinterpret_cast<float4*>(o) = make_float4(r[0], r[1], r[2], r[3]);
                }
            } else {
#pragma unroll
                for (int e = 0; e < kPer; ++e)
                    if (v0 + e < V) o[e] = r[e];
            }
        } else {
#pragma unroll
            for (int e = 0; e < kPer; ++e) {
                const int64_t v = v0 + e;
                if (v >= V) break;
                const int64_t idx = row_base + v;
                if constexpr (kKind == 0) {
                    reinterpret_cast<uint4*>(out)[idx] = make_uint4(w.w0, w.w1, w.w2, w.w3);
                } else {
                    const uint32_t lo = kWide ? word[2 * e] : word[e];
                    const uint32_t hi = kWide ? word[2 * e + 1] : 0u;
                    double u;
                    if (kWide) {
                        const uint64_t kk = ((static_cast<uint64_t>(hi) << 32) | lo) >> 12;
                        u = static_cast<double>((kk << 1) | 1ull) * 0x1p-53;   // exact
                    } else {
                        u = static_cast<double>(((lo >> 8) << 1) | 1u) * 0x1p-25;
                    }
                    reinterpret_cast<double*>(out)[idx] = u;
                }
            }
        }
    }
}

template <int kKind>
cudaError_t launch_kind(void* out, bool wide, int64_t B, int64_t V, const int64_t* seeds,
                        const int64_t* positions, uint64_t base_seed, uint64_t offset,
                        cudaStream_t stream) {
    const int64_t calls = (V + (wide ? 1 : 3)) / (wide ? 2 : 4);
    const int64_t bx = (calls + 4 * 256 - 1) / (4 * 256);   // about four calls per thread
    const unsigned gx = static_cast<unsigned>(bx < 65535 ? bx : 65535);
    for (int64_t r0 = 0; r0 < B; r0 += 65535) {
        const unsigned gy = static_cast<unsigned>(B - r0 < 65535 ? B - r0 : 65535);
        if (wide) {
            noise_fill_kernel<kKind, true><<<dim3(gx, gy), 256, 0, stream>>>(out, r0, V, seeds, positions,
                                                                            base_seed, offset);
        } else {
            noise_fill_kernel<kKind, false><<<dim3(gx, gy), 256, 0, stream>>>(out, r0, V, seeds, positions,
                                                                             base_seed, offset);
        }
        const cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

}  // namespace

cudaError_t launch_noise_fill(void* out, int kind, bool wide, int64_t B, int64_t V,
                              const int64_t* seeds, const int64_t* positions, uint64_t base_seed,
                              uint64_t offset, cudaStream_t stream) {
    switch (kind) {
        case 0: return launch_kind<0>(out, wide, B, V, seeds, positions, base_seed, offset, stream);
        case 1: return launch_kind<1>(out, wide, B, V, seeds, positions, base_seed, offset, stream);
        case 2: return launch_kind<2>(out, wide, B, V, seeds, positions, base_seed, offset, stream);
        default: return launch_kind<3>(out, wide, B, V, seeds, positions, base_seed, offset, stream);
    }
}

}  // namespace lms
