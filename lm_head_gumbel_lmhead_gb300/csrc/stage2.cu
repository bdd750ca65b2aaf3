// Stage 2 (FlashSampling "method step details", Stage 2): per row, the candidate of the best
// vocabulary tile, t* = argmax_t m_b^(t), output idx_b^(t*).  Ties between tiles go to the
// smaller index, which is the earlier tile.  Also writes the per-row status.
#include "lms_device.cuh"
#include "lms_kernels.h"

namespace lms {
namespace {

constexpr int kStage2Threads = 128;

__global__ void __launch_bounds__(kStage2Threads) stage2_kernel(
    const float* __restrict__ cand_score, const int* __restrict__ cand_index, int64_t n_tiles,
    const float* __restrict__ temperature, int64_t* __restrict__ out, int32_t* __restrict__ row_status) {
    // Wait for Stage 1 when launched as its programmatic dependent.
    pdl_wait_primary();
    const int64_t b = blockIdx.x;
    const float* s_row = cand_score + b * n_tiles;
    const int* i_row = cand_index + b * n_tiles;
    float best_s = -CUDART_INF_F;
    int best_i = kNoIndex;
    int poisoned = 0;
    for (int64_t t = threadIdx.x; t < n_tiles; t += kStage2Threads) {
        const int idx = i_row[t];
        if (idx == kPoisonIndex) {
            poisoned = 1;
        } else if (idx >= 0) {
            const float s = s_row[t];
            if (better(s, idx, best_s, best_i)) { best_s = s; best_i = idx; }
        }
    }
    warp_argmax(best_s, best_i);
    poisoned = __any_sync(0xffffffffu, poisoned);
    __shared__ float sh_s[kStage2Threads / 32];
    __shared__ int sh_i[kStage2Threads / 32];
    __shared__ int sh_p[kStage2Threads / 32];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (lane == 0) { sh_s[warp] = best_s; sh_i[warp] = best_i; sh_p[warp] = poisoned; }
    __syncthreads();
    if (threadIdx.x == 0) {
        for (int w = 1; w < kStage2Threads / 32; ++w) {
            if (better(sh_s[w], sh_i[w], best_s, best_i)) { best_s = sh_s[w]; best_i = sh_i[w]; }
            poisoned |= sh_p[w];
        }
        const float T = temperature ? temperature[b] : 1.0f;
        int32_t status;
        int64_t token;
        if (poisoned) {
            status = 3; token = -1;
        } else if (!(T >= 0.0f)) {
            status = 2; token = -1;
        } else if (candidate_index(best_s, best_i) < 0) {
            status = 1; token = -1;
        } else {
            status = 0; token = best_i;
        }
        out[b] = token;
        if (row_status) row_status[b] = status;
    }
}

}  // namespace

cudaError_t launch_stage2(const float* cand_score, const int* cand_index, int64_t n_tiles,
                          int64_t B, const float* temperature, int64_t* out, int32_t* row_status,
                          cudaStream_t stream) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(B));
    cfg.blockDim = dim3(kStage2Threads);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, stage2_kernel, cand_score, cand_index, n_tiles, temperature,
                              out, row_status);
}

}  // namespace lms
