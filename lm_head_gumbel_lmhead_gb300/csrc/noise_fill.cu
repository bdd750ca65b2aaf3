// Noise-fill kernel: the Philox words and the noise the sampling kernels use, written out.
// (Megatron-LM PR 8370, "The change" / "Tests": seeded noise keyed by (request seed, absolute
// position, vocabulary index) that replays bit-exactly.)
#include "lms_device.cuh"
#include "lms_kernels.h"

namespace lms {
namespace {

template <int kKind, bool kWide>
__global__ void __launch_bounds__(256) noise_fill_kernel(void* __restrict__ out, int64_t B, int64_t V,
                                                          const int64_t* __restrict__ seeds,
                                                          const int64_t* __restrict__ positions,
                                                          uint64_t base_seed, uint64_t offset) {
    const int64_t total = B * V;
    for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < total;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int64_t b = i / V;
        const uint32_t v = static_cast<uint32_t>(i - b * V);
        const RowKey k = make_row_key(seeds, positions, base_seed, offset, b);
        const Words w = row_words(k, v);
        if constexpr (kKind == 0) {
            reinterpret_cast<uint4*>(out)[i] = make_uint4(w.w0, w.w1, w.w2, w.w3);
        } else if constexpr (kKind == 1) {
            double u;
            if (kWide) {
                const uint64_t kk = ((static_cast<uint64_t>(w.w1) << 32) | w.w0) >> 12;
                u = static_cast<double>((kk << 1) | 1ull) * 0x1p-53;
            } else {
                u = static_cast<double>(((w.w0 >> 8) << 1) | 1u) * 0x1p-25;
            }
            reinterpret_cast<double*>(out)[i] = u;
        } else {
            const float E = kWide ? exponential_wide(w) : exponential_fp32(w);
            reinterpret_cast<float*>(out)[i] = (kKind == 2) ? E : gumbel_from_exponential(E);
        }
    }
}

template <int kKind>
cudaError_t launch_kind(void* out, bool wide, int64_t B, int64_t V, const int64_t* seeds,
                        const int64_t* positions, uint64_t base_seed, uint64_t offset,
                        cudaStream_t stream) {
    const int64_t total = B * V;
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
