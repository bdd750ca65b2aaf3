// Internal launch interface between the C-ABI layer (lms_api.cu) and the kernels.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include <cstddef>
#include <cstdint>

namespace lms {

// Everything a sampling kernel needs besides its logits / GEMM operands.
struct SampleArgs {
    const float* temperature;
    const int64_t* seeds;
    const int64_t* positions;
    const float* bias;
    int64_t ld_bias;
    const uint32_t* mask;
    int64_t ld_mask;
    uint64_t base_seed;
    uint64_t offset;
    int64_t B;        // rows in this launch
    int64_t row0;     // global row index of the first row (unseeded rows are keyed by it)
    int64_t V;
    int64_t n_tiles;  // candidate columns per row in the workspace
    float* cand_score;  // [B][n_tiles] (already offset to row0)
    int* cand_index;    // [B][n_tiles]
    // FP8 (W8A8) fused path only, else null: logits = acc * 2^h_exp[row] * w_scale[v]
    const int32_t* h_exp;
    const float* w_scale;
    // Gumbel-top-k (topk > 0) only: ordered (score, index) key lists, per tile and TMEM quadrant
    // ([B][n_tiles][4][topk], topk_mode kTopKTileLists) or per Stage-1 CTA and TMEM quadrant
    // ([B][4 grid][topk], kTopKRunning)
    unsigned long long* cand_keys = nullptr;
    int topk = 0;
    int topk_mode = 0;
    // the call's status word (the head of the workspace) or null: Stage 1 of the launch with
    // row0 == 0 clears it, Stage 2 sets bit s for every row that ends with status s != 0
    uint32_t* status_bits = nullptr;
};

// Speculative-decoding verification over materialised logits (see verify.cu).
// A batch row's verification decision.
struct VerifyDecision {
    int j;                     // first rejection (k: none)
    int mode;                  // 0 finished, 1 race at j pending
    float lt, ld;              // log2 normalisers of target and draft at j (ld: j < k)
};

struct VerifyArgs {
    const void* target;        // [B][k + 1] rows of ld elements (fp32 or bf16)
    const void* draft;         // [B][k] rows of ld elements
    int64_t ld;
    int64_t B;
    int k;
    int64_t V;
    const int64_t* tokens;     // [B][k] draft tokens
    const float* temperature;
    const int64_t* seeds;
    const int64_t* positions;
    uint64_t base_seed, offset;
    int64_t nc;                // partials chunks per row
    int64_t ncr;               // race chunks per row
    // workspace
    float* pmax;               // [B (2k + 1)][nc][8] softmax partials, one per warp
    float* psum;
    int* parg;
    VerifyDecision* dec;       // [B]
    float* c_s;                // [B][ncr][2] race candidates: residual, target
    int* c_i;
    int* cnt_r;                // [B] race blocks done (zeroed by the decision kernel)
    // outputs
    int64_t* accept_len;       // [B]
    int64_t* out;              // [B][k + 1]
    int32_t* row_status;       // [B] or null
    uint32_t* status_bits;     // the call's status word (cleared by the first partials launch)
};

void verify_chunks(int64_t V, bool bf16, int64_t* partial_chunks, int64_t* race_chunks);
cudaError_t launch_verify(const VerifyArgs& a, bool bf16, bool wide, cudaStream_t stream);

// The filtered race (a cluster per row; writes tokens and statuses directly).
struct FilterArgs {
    SampleArgs a;
    const int32_t* top_k;
    const float* top_p;
    const float* min_p;
    int k_max;
    int64_t* out;
    int32_t* row_status;
};

cudaError_t launch_filtered_race(const void* logits, bool bf16, int64_t ld, bool wide,
                                 const FilterArgs& f, cudaStream_t stream);

cudaError_t launch_quantize_rows_e4m3(const uint16_t* H, int64_t ldh, int64_t B, int64_t D,
                                      uint8_t* q, int64_t ldq, int32_t* e_out, cudaStream_t stream);

cudaError_t launch_noise_fill(void* out, int kind, bool wide, int64_t B, int64_t V,
                              const int64_t* seeds, const int64_t* positions, uint64_t base_seed,
                              uint64_t offset, cudaStream_t stream);

cudaError_t launch_logits_stage1(const void* logits, bool bf16, int64_t ld, int tile_v, bool wide,
                                 const SampleArgs& a, cudaStream_t stream);

cudaError_t launch_stage2(const float* cand_score, const int* cand_index, int64_t n_tiles,
                          int64_t B, const float* temperature, int64_t* out, int32_t* row_status,
                          uint32_t* status_bits, cudaStream_t stream);

// Stage 2 of Gumbel-top-k: per row, the k best of n_lists ordered key lists of k keys
// (cand_keys [B][n_lists][k]); out [B][k] indices (-1 past the finite ones), scores [B][k] or null.
// part_keys is scratch of stage2_topk_part_bytes(B, k) bytes.
size_t stage2_topk_part_bytes(int64_t B, int k);
cudaError_t launch_stage2_topk(const unsigned long long* cand_keys, int64_t n_lists, int k, int64_t B,
                               const float* temperature, int64_t* out, float* scores,
                               int32_t* row_status, uint32_t* status_bits,
                               unsigned long long* part_keys, cudaStream_t stream);

cudaError_t launch_lmhead_gemv(const uint16_t* H, int64_t ldh, const uint16_t* W, int64_t ldw,
                               int64_t D, bool wide, const SampleArgs& a, cudaStream_t stream);

// The tcgen05 path.  tmW / tmH are TMA descriptors (bf16, 128-byte swizzle, boxes of 64 x 128
// for W and 64 x n_pad for H).  B <= 256 per launch.
// fp8: E4M3 operands (kind::f8f6f4), boxes of 128 x 128 / 128 x n_pad bytes; a.h_exp / a.w_scale set.
cudaError_t launch_lmhead_tc(const CUtensorMap& tmW, const CUtensorMap& tmH, int64_t D, int n_pad,
                             bool wide, uint32_t timeout_ms, uint32_t debug_flags,
                             const SampleArgs& a, cudaStream_t stream, bool fp8 = false);
// (a.topk > 0 selects the Gumbel-top-k epilogue: bf16 only; a.topk_mode says which lists.)

// Batches of 257 .. 1024 rows in one launch (bf16 race only): up to kMaxRowGroups groups of 256
// rows whose CTAs walk the vocabulary tiles together, so W streams from HBM once.  tmH has a box
// of 256 rows; a.B is the launch's row count.
constexpr int kMaxRowGroups = 4;
cudaError_t launch_lmhead_tc_rows(const CUtensorMap& tmW, const CUtensorMap& tmH, int64_t D, bool wide,
                                  uint32_t timeout_ms, uint32_t debug_flags, const SampleArgs& a,
                                  cudaStream_t stream);

// Gumbel-top-k list modes.  Running lists keep, in shared memory, each CTA's k best keys per
// TMEM quadrant and batch column, written out once per CTA; they are used when they fit
// (4 n_pad k keys of 8 bytes within kTopKRunningBytes), else each tile writes its own lists.
constexpr int kTopKTileLists = 1;
constexpr int kTopKRunning = 2;
constexpr uint32_t kTopKRunningBytes = 32u * 1024u;
inline int topk_mode_for(int n_pad, int k) {
    return static_cast<uint32_t>(4 * n_pad) * static_cast<uint32_t>(k) * 8u <= kTopKRunningBytes ? kTopKRunning
                                                                                                  : kTopKTileLists;
}

// The MXFP4-weight path (W4A16).  Wt is the tiled format mxfp4_pack writes (mxfp4_tiled_bytes(V, D)
// bytes: one contiguous 4352-byte block per (128-row tile, 64-element K chunk)); tmH as for
// launch_lmhead_tc.  B <= 128 per launch.
size_t mxfp4_tiled_bytes(int64_t V, int64_t D);
cudaError_t launch_mxfp4_pack(const uint8_t* W4, int64_t ldw4, const uint8_t* S, int64_t lds, int64_t V,
                              int64_t D, uint8_t* out, cudaStream_t stream);
cudaError_t launch_lmhead_mx(const uint8_t* Wt, const CUtensorMap& tmH, int64_t D, int n_pad, bool wide,
                             uint32_t timeout_ms, uint32_t debug_flags, const SampleArgs& a,
                             cudaStream_t stream);

// The CTA-pair tcgen05 path (cta_group::2, M = 256): tmH boxes are 64 x (n_pad / 2).
cudaError_t launch_lmhead_tc_pair(const CUtensorMap& tmW, const CUtensorMap& tmH, int64_t D,
                                  int n_pad, bool wide, uint32_t timeout_ms, uint32_t debug_flags,
                                  const SampleArgs& a, cudaStream_t stream);

int device_sm_count();

// Raises `kernel`'s dynamic shared-memory limit on the current device to at least `bytes`; the
// runtime is called only when the limit cached for (device, kernel) is lower.
cudaError_t ensure_dynamic_smem(const void* kernel, size_t bytes);

// Sets the thread-local message that lms_last_error() returns.
void set_last_error(const char* msg);

}  // namespace lms
