// Stage 2 (FlashSampling "method step details", Stage 2): per row, the candidate of the best
// vocabulary tile, t* = argmax_t m_b^(t), output idx_b^(t*).  Ties between tiles go to the
// smaller index, which is the earlier tile.  Also writes the per-row status.
#include "lms_device.cuh"
#include "lms_kernels.h"

namespace lms {
namespace {

constexpr int kStage2Threads = 256;
constexpr int kStage2PerThread = 8;   // candidates a thread loads before it compares any

__global__ void __launch_bounds__(kStage2Threads) stage2_kernel(
    const float* __restrict__ cand_score, const int* __restrict__ cand_index, int64_t n_tiles,
    const float* __restrict__ temperature, int64_t* __restrict__ out, int32_t* __restrict__ row_status,
    uint32_t* __restrict__ status_bits) {
    const int64_t b = blockIdx.x;
    // T is an input of the step, not a Stage-1 result: read it before the wait.
    const float T = temperature ? temperature[b] : 1.0f;
    // Wait for Stage 1 when launched as its programmatic dependent.
    pdl_wait_primary();
    const float* s_row = cand_score + b * n_tiles;
    const int* i_row = cand_index + b * n_tiles;
    float best_s = -CUDART_INF_F;
    int best_i = kNoIndex;
    int poisoned = 0;
    // All of a thread's loads of a round are issued before its comparisons, so a round costs one
    // trip to L2 (1187 candidates per row at the Qwen3-8B shape: one round).
    for (int64_t base = threadIdx.x; base < n_tiles; base += kStage2Threads * kStage2PerThread) {
        int idx[kStage2PerThread];
        float sc[kStage2PerThread];
#pragma unroll
        for (int j = 0; j < kStage2PerThread; ++j) {
            const int64_t t = base + j * kStage2Threads;
            idx[j] = t < n_tiles ? i_row[t] : -1;
            sc[j] = t < n_tiles ? s_row[t] : -CUDART_INF_F;
        }
#pragma unroll
        for (int j = 0; j < kStage2PerThread; ++j) {
            if (idx[j] == kPoisonIndex) {
                poisoned = 1;
            } else if (idx[j] >= 0 && better(sc[j], idx[j], best_s, best_i)) {
                best_s = sc[j];
                best_i = idx[j];
            }
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
        note_row_status(status_bits, status);
    }
}

}  // namespace

cudaError_t launch_stage2(const float* cand_score, const int* cand_index, int64_t n_tiles,
                          int64_t B, const float* temperature, int64_t* out, int32_t* row_status,
                          uint32_t* status_bits, cudaStream_t stream) {
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
                              out, row_status, status_bits);
}

}  // namespace lms
