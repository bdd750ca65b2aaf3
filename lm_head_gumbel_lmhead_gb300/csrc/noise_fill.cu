// Noise-fill kernel: the Philox words and the noise the sampling kernels use, written out.
// (Megatron-LM PR 8370, "The change" / "Tests": seeded noise keyed by (request seed, absolute
// position, vocabulary index) that replays bit-exactly.)
#include "lms_device.cuh"
#include "lms_kernels.h"

namespace lms {
namespace {

// One thread per Philox call: the call serves 4 consecutive entries (fp32 noise) or 2 (wide).
template <int kKind, bool kWide>
__global__ void __launch_bounds__(256) noise_fill_kernel(void* __restrict__ out, int64_t B, int64_t V,
                                                          const int64_t* __restrict__ seeds,
                                                          const int64_t* __restrict__ positions,
                                                          uint64_t base_seed, uint64_t offset) {
    constexpr int kPer = kWide ? 2 : 4;
    const int64_t calls_per_row = (V + kPer - 1) / kPer;
    const int64_t total = B * calls_per_row;
    for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < total;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int64_t b = i / calls_per_row;
        const uint32_t n = static_cast<uint32_t>(i - b * calls_per_row);
        const RowKey k = make_row_key(seeds, positions, base_seed, offset, b);
        const Words w = row_call(k, n);
        const uint32_t word[4] = {w.w0, w.w1, w.w2, w.w3};
#pragma unroll
        for (int e = 0; e < kPer; ++e) {
            const int64_t v = static_cast<int64_t>(n) * kPer + e;
            if (v >= V) break;
            const int64_t idx = b * V + v;
            const uint32_t lo = kWide ? word[2 * e] : word[e];
            const uint32_t hi = kWide ? word[2 * e + 1] : 0u;
            if constexpr (kKind == 0) {
                reinterpret_cast<uint4*>(out)[idx] = make_uint4(w.w0, w.w1, w.w2, w.w3);
            } else if constexpr (kKind == 1) {
                double u;
                if (kWide) {
                    const uint64_t kk = ((static_cast<uint64_t>(hi) << 32) | lo) >> 12;
                    u = static_cast<double>((kk << 1) | 1ull) * 0x1p-53;   // exact
                } else {
                    u = static_cast<double>(((lo >> 8) << 1) | 1u) * 0x1p-25;
                }
                reinterpret_cast<double*>(out)[idx] = u;
            } else {
                const float E = kWide ? exponential_wide(lo, hi) : exponential_fp32(lo);
                reinterpret_cast<float*>(out)[idx] = (kKind == 2) ? E : gumbel_from_exponential(E);
            }
        }
    }
}

template <int kKind>
cudaError_t launch_kind(void* out, bool wide, int64_t B, int64_t V, const int64_t* seeds,
                        const int64_t* positions, uint64_t base_seed, uint64_t offset,
                        cudaStream_t stream) {
    const int64_t total = B * ((V + (wide ? 1 : 3)) / (wide ? 2 : 4));
    const int64_t want = (total + 255) / 256;
    const int64_t cap = static_cast<int64_t>(device_sm_count()) * 16;
    const unsigned grid = static_cast<unsigned>(want < cap ? want : cap);
    if (wide) {
        noise_fill_kernel<kKind, true><<<grid, 256, 0, stream>>>(out, B, V, seeds, positions,
                                                                base_seed, offset);
    } else {
        noise_fill_kernel<kKind, false><<<grid, 256, 0, stream>>>(out, B, V, seeds, positions,
                                                                 base_seed, offset);
    }
    return cudaGetLastError();
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
