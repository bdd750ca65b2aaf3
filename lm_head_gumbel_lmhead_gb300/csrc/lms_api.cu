// C-ABI entry points (include/lms.h): argument checks, tiling, TMA descriptors, launches.
// Host-detectable errors return before anything is launched; nothing here allocates device
// memory; the only state kept between calls is per-device launch settings (kernel attributes).
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <map>
#include <mutex>
#include <utility>

#include "lms.h"
#include "lms_kernels.h"

namespace {

thread_local char g_last_error[512] = "";

lms_status fail(lms_status st, const char* fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_last_error, sizeof g_last_error, fmt, ap);
    va_end(ap);
    return st;
}

lms_status cuda_fail(cudaError_t e, const char* what) {
    return fail(LMS_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
}

constexpr int64_t kMaxV = (int64_t{1} << 31) - 1;
constexpr int kTcMaxBatchPerLaunch = 256;

size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Every workspace starts with a status block: the call's status word (bit s set when a row ended
// with row status s != 0), then reserved bytes up to a 256-byte boundary.
constexpr size_t kStatusBlock = 256;

struct Tiling {
    int32_t tile_v;
    int64_t n_tiles;
    size_t workspace;
    int32_t path;
};

int pick_logits_tile(int64_t B, int64_t V) {
    // Several CTAs per row: aim for at least ~2 CTAs per SM over the whole grid, with tiles of
    // 1K..8K entries (16 KB..32 KB of fp32 logits).  Measured on GB300 at V = 131072 (bf16, L2
    // flushed): B = 8 takes 10.9 us with 2K tiles against 12.9 us with 1K; B = 1 is fastest with
    // 1K tiles (8.9 us) and B >= 64 with 8K (23.2 us at B = 64).
    const int64_t target_ctas = 152 * 2;
    int64_t t = 8192;
    while (t > 1024 && B * ((V + t - 1) / t) < target_ctas) t >>= 1;
    return static_cast<int>(t);
}

lms_status make_tiling(int32_t op, int64_t B, int64_t D, int64_t V, int32_t tile_req, Tiling* out) {
    if (B <= 0 || V <= 0) return fail(LMS_ERR_INVALID_ARG, "B and V must be positive (B=%lld V=%lld)",
                                      (long long)B, (long long)V);
    if (V > kMaxV) return fail(LMS_ERR_INVALID_ARG, "V must be < 2^31 (V=%lld)", (long long)V);
    if (op == LMS_OP_LMHEAD || op == LMS_OP_LMHEAD_FP8) {
        if (D <= 0) return fail(LMS_ERR_INVALID_ARG, "D must be positive (D=%lld)", (long long)D);
        if (B > 65536) return fail(LMS_ERR_INVALID_ARG, "B must be <= 65536 (B=%lld)", (long long)B);
        if (tile_req != 0 && tile_req != LMS_FUSED_TILE_V)
            return fail(LMS_ERR_UNSUPPORTED, "fused tile_v must be 0 or 128 (got %d)", tile_req);
        out->tile_v = LMS_FUSED_TILE_V;
        // The tcgen05 path streams W at the HBM roofline from B = 1 up (measured on GB300 at the
        // Qwen3-8B shape: 198 us at B = 1 against 201 us for the GEMV path), so it is the
        // automatic choice for every batch; the GEMV path stays available on request.
        out->path = LMS_PATH_TCGEN05;
    } else if (op == LMS_OP_LOGITS) {
        if (B > (int64_t{1} << 31) - 1) return fail(LMS_ERR_INVALID_ARG, "B must be < 2^31");
        if (tile_req == 0) {
            out->tile_v = pick_logits_tile(B, V);
        } else {
            if (tile_req < 256 || tile_req > 65536 || (tile_req & (tile_req - 1)) != 0)
                return fail(LMS_ERR_UNSUPPORTED, "logits tile_v must be a power of two in [256, 65536] (got %d)",
                            tile_req);
            out->tile_v = tile_req;
        }
        out->path = LMS_PATH_AUTO;
    } else {
        return fail(LMS_ERR_INVALID_ARG, "unknown op %d", op);
    }
    out->n_tiles = (V + out->tile_v - 1) / out->tile_v;
    const int64_t grid = B * out->n_tiles;
    if (op == LMS_OP_LOGITS && grid > (int64_t{1} << 31) - 1)
        return fail(LMS_ERR_UNSUPPORTED, "B * n_tiles exceeds the launch grid limit");
    const size_t cand = static_cast<size_t>(B) * static_cast<size_t>(out->n_tiles) * 4;
    out->workspace = kStatusBlock + round_up(cand, 256) + round_up(cand, 256);
    if (op == LMS_OP_LMHEAD_FP8) {
        // + quantised activations [B][round_up(D, 16)] bytes + their exponents [B]
        out->workspace += round_up(static_cast<size_t>(B) * round_up(static_cast<size_t>(D), 16), 256) +
                          round_up(static_cast<size_t>(B) * 4, 256);
        out->path = LMS_PATH_TCGEN05;
    }
    return LMS_OK;
}

lms_status check_params(const lms_sample_params* p, int64_t V) {
    if (p == nullptr) return fail(LMS_ERR_INVALID_ARG, "params is NULL");
    if (p->noise_mode != LMS_NOISE_FP32 && p->noise_mode != LMS_NOISE_WIDE53)
        return fail(LMS_ERR_INVALID_ARG, "unknown noise_mode %d", p->noise_mode);
    if (p->seeds != nullptr && p->positions == nullptr)
        return fail(LMS_ERR_INVALID_ARG, "positions is required when seeds is given");
    if (p->bias != nullptr && p->ld_bias != 0 && p->ld_bias < V)
        return fail(LMS_ERR_INVALID_ARG, "ld_bias must be 0 or >= V");
    if (p->allow_mask != nullptr && p->ld_mask != 0 && p->ld_mask < (V + 31) / 32)
        return fail(LMS_ERR_INVALID_ARG, "ld_mask must be 0 or >= ceil(V/32)");
    if (p->ld_bias < 0 || p->ld_mask < 0) return fail(LMS_ERR_INVALID_ARG, "negative leading dimension");
    if (p->reserved != 0) return fail(LMS_ERR_INVALID_ARG, "reserved must be 0");
    if (p->debug_flags & ~LMS_DEBUG_WITHHOLD_FIRST_LOAD)
        return fail(LMS_ERR_INVALID_ARG, "unknown debug_flags 0x%x", p->debug_flags);
    return LMS_OK;
}

lms::SampleArgs make_args(const lms_sample_params* p, int64_t B, int64_t V, const Tiling& t,
                          void* workspace) {
    lms::SampleArgs a;
    a.temperature = p->temperature;
    a.seeds = p->seeds;
    a.positions = p->positions;
    a.bias = p->bias;
    a.ld_bias = p->ld_bias;
    a.mask = p->allow_mask;
    a.ld_mask = p->ld_mask;
    a.base_seed = p->base_seed;
    a.offset = p->offset;
    a.B = B;
    a.row0 = 0;
    a.V = V;
    a.n_tiles = t.n_tiles;
    const size_t cand = static_cast<size_t>(B) * static_cast<size_t>(t.n_tiles) * 4;
    char* w = static_cast<char*>(workspace);
    a.status_bits = reinterpret_cast<uint32_t*>(w);
    a.cand_score = reinterpret_cast<float*>(w + kStatusBlock);
    a.cand_index = reinterpret_cast<int*>(w + kStatusBlock + round_up(cand, 256));
    a.h_exp = nullptr;
    a.w_scale = nullptr;
    return a;
}

// cuTensorMapEncodeTiled from the driver, found through the runtime (no link to libcuda).
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_tiled_fn() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}

// [rows][ld] row-major -> 2-D map {D, rows}, boxes of 128 bytes x box_rows, 128-byte swizzle,
// out-of-range elements read as zero.  bf16 (ld in elements of 2 bytes) or bytes (E4M3).
lms_status encode_map(CUtensorMap* tm, const void* ptr, int64_t rows, int64_t D, int64_t ld,
                      int box_rows, bool bytes) {
    EncodeTiledFn fn = encode_tiled_fn();
    if (fn == nullptr) return fail(LMS_ERR_CUDA, "cuTensorMapEncodeTiled not available from the driver");
    const int esize = bytes ? 1 : 2;
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(rows)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(ld) * esize};
    const cuuint32_t box[2] = {static_cast<cuuint32_t>(128 / esize), static_cast<cuuint32_t>(box_rows)};
    const cuuint32_t estr[2] = {1, 1};
    const CUresult r = fn(tm, bytes ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
                          2, const_cast<void*>(ptr), dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail(LMS_ERR_CUDA, "cuTensorMapEncodeTiled failed (CUresult %d)", (int)r);
    return LMS_OK;
}

lms_status encode_bf16_map(CUtensorMap* tm, const void* ptr, int64_t rows, int64_t D, int64_t ld,
                           int box_rows) {
    return encode_map(tm, ptr, rows, D, ld, box_rows, false);
}

}  // namespace

namespace lms {
void set_last_error(const char* msg) { snprintf(g_last_error, sizeof g_last_error, "%s", msg); }

cudaError_t ensure_dynamic_smem(const void* kernel, size_t bytes) {
    static std::mutex mu;
    static std::map<std::pair<int, const void*>, size_t> limits;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    std::lock_guard<std::mutex> lock(mu);
    size_t& have = limits[std::make_pair(dev, kernel)];
    if (have >= bytes) return cudaSuccess;
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(bytes));
    if (e == cudaSuccess && bytes > have) have = bytes;
    return e;
}

int device_sm_count() {
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 148;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0)
        return 148;
    return sms;
}
}  // namespace lms

extern "C" {

const char* lms_version(void) { return "lms 0.1 (sm_103a)"; }

const char* lms_last_error(void) { return g_last_error; }

lms_status lms_tile_info(int32_t op, int64_t B, int64_t D, int64_t V, int32_t tile_v_req,
                         int32_t* tile_v_out, int64_t* n_tiles_out, size_t* workspace_bytes_out,
                         int32_t* path_out) {
    Tiling t;
    const lms_status st = make_tiling(op, B, D, V, tile_v_req, &t);
    if (st != LMS_OK) return st;
    if (tile_v_out) *tile_v_out = t.tile_v;
    if (n_tiles_out) *n_tiles_out = t.n_tiles;
    if (workspace_bytes_out) *workspace_bytes_out = t.workspace;
    if (path_out) *path_out = t.path;
    return LMS_OK;
}

size_t lms_workspace_bytes(int32_t op, int64_t B, int64_t D, int64_t V, int32_t tile_v_req) {
    Tiling t;
    return make_tiling(op, B, D, V, tile_v_req, &t) == LMS_OK ? t.workspace : 0;
}

lms_status lms_lmhead_sample(const void* H, int64_t ldh, const void* W, int64_t ldw, int64_t B,
                             int64_t D, int64_t V, const lms_sample_params* params, int64_t* out,
                             void* workspace, size_t workspace_bytes, void* stream) {
    g_last_error[0] = '\0';
    if (H == nullptr || W == nullptr || out == nullptr)
        return fail(LMS_ERR_INVALID_ARG, "H, W and out are required");
    Tiling t;
    lms_status st = make_tiling(LMS_OP_LMHEAD, B, D, V, params ? params->tile_v : 0, &t);
    if (st != LMS_OK) return st;
    if ((st = check_params(params, V)) != LMS_OK) return st;
    if (D % 8 != 0) return fail(LMS_ERR_UNSUPPORTED, "D must be a multiple of 8 (D=%lld)", (long long)D);
    if (D > 65536) return fail(LMS_ERR_UNSUPPORTED, "D must be <= 65536");
    if (ldh < D || ldw < D || ldh % 8 != 0 || ldw % 8 != 0)
        return fail(LMS_ERR_UNSUPPORTED, "ldh/ldw must be >= D and multiples of 8 elements");
    if (reinterpret_cast<uintptr_t>(H) % 16 != 0 || reinterpret_cast<uintptr_t>(W) % 16 != 0)
        return fail(LMS_ERR_UNSUPPORTED, "H and W must be 16-byte aligned");
    if (workspace == nullptr || workspace_bytes < t.workspace)
        return fail(LMS_ERR_WORKSPACE, "workspace of %zu bytes needed", t.workspace);
    int32_t path = params->path == LMS_PATH_AUTO ? t.path : params->path;
    if (path == LMS_PATH_GEMV && (B > LMS_GEMV_MAX_B || static_cast<size_t>(B) * D * 2 > 200 * 1024))
        path = (params->path == LMS_PATH_GEMV) ? -1 : LMS_PATH_TCGEN05;
    if (path == -1) return fail(LMS_ERR_UNSUPPORTED, "GEMV path needs B <= %d and B*D*2 <= 200 KB", LMS_GEMV_MAX_B);
    if (path != LMS_PATH_GEMV && path != LMS_PATH_TCGEN05 && path != LMS_PATH_TCGEN05_PAIR)
        return fail(LMS_ERR_INVALID_ARG, "unknown path %d", params->path);

    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const bool wide = params->noise_mode == LMS_NOISE_WIDE53;
    lms::SampleArgs a = make_args(params, B, V, t, workspace);
    cudaError_t e;
    if (path == LMS_PATH_GEMV) {
        e = lms::launch_lmhead_gemv(static_cast<const uint16_t*>(H), ldh, static_cast<const uint16_t*>(W),
                                    ldw, D, wide, a, s);
        if (e != cudaSuccess) return cuda_fail(e, "GEMV Stage-1 launch");
    } else {
        CUtensorMap tmW;
        if ((st = encode_bf16_map(&tmW, W, V, D, ldw, 128)) != LMS_OK) return st;
        const uint32_t timeout_ms = params->timeout_ms ? params->timeout_ms : 2000u;
        // Batches above 256 rows (one MMA N) run as row-group launches of up to 1024 rows that
        // stream W once each (lmhead_tc_rows.cu); a remainder of <= 256 rows, and the pair path,
        // as launches of <= 256 rows.
        const bool pair = path == LMS_PATH_TCGEN05_PAIR;
        constexpr int64_t kRowGroupLaunch = static_cast<int64_t>(lms::kMaxRowGroups) * kTcMaxBatchPerLaunch;
        for (int64_t r0 = 0, nb = 0; r0 < B; r0 += nb) {
            if (!pair && B - r0 > kTcMaxBatchPerLaunch) {
                nb = (B - r0 < kRowGroupLaunch) ? B - r0 : kRowGroupLaunch;
                CUtensorMap tmH;
                if ((st = encode_bf16_map(&tmH, H, B, D, ldh, static_cast<int>(kTcMaxBatchPerLaunch))) != LMS_OK)
                    return st;
                lms::SampleArgs ac = a;
                ac.B = nb;
                ac.row0 = r0;
                ac.cand_score = a.cand_score + r0 * t.n_tiles;
                ac.cand_index = a.cand_index + r0 * t.n_tiles;
                e = lms::launch_lmhead_tc_rows(tmW, tmH, D, wide, timeout_ms, params->debug_flags, ac, s);
                if (e != cudaSuccess) return cuda_fail(e, "tcgen05 row-group Stage-1 launch");
                continue;
            }
            nb = (B - r0 < kTcMaxBatchPerLaunch) ? B - r0 : kTcMaxBatchPerLaunch;
            const int n_pad = static_cast<int>(nb < 16 ? 16 : (nb + 15) / 16 * 16);
            CUtensorMap tmH;
            if ((st = encode_bf16_map(&tmH, H, B, D, ldh, pair ? n_pad / 2 : n_pad)) != LMS_OK) return st;
            lms::SampleArgs ac = a;
            ac.B = nb;
            ac.row0 = r0;
            ac.cand_score = a.cand_score + r0 * t.n_tiles;
            ac.cand_index = a.cand_index + r0 * t.n_tiles;
            e = pair ? lms::launch_lmhead_tc_pair(tmW, tmH, D, n_pad, wide, timeout_ms,
                                                  params->debug_flags, ac, s)
                     : lms::launch_lmhead_tc(tmW, tmH, D, n_pad, wide, timeout_ms,
                                             params->debug_flags, ac, s);
            if (e != cudaSuccess) return cuda_fail(e, pair ? "tcgen05 pair Stage-1 launch" : "tcgen05 Stage-1 launch");
        }
    }
    e = lms::launch_stage2(a.cand_score, a.cand_index, t.n_tiles, B, params->temperature, out,
                           params->row_status, a.status_bits, s);
    if (e != cudaSuccess) return cuda_fail(e, "Stage-2 launch");
    return LMS_OK;
}

size_t lms_workspace_bytes_topk(int64_t B, int64_t V, int32_t k) {
    if (B <= 0 || V <= 0 || V > kMaxV || k < 1 || k > LMS_TOPK_MAX) return 0;
    const int64_t nt = (V + LMS_FUSED_TILE_V - 1) / LMS_FUSED_TILE_V;
    // per row and tile, one ordered list of k keys per TMEM quadrant (4); then Stage 2's part lists
    return kStatusBlock +
           round_up(static_cast<size_t>(B) * static_cast<size_t>(nt) * 4 * static_cast<size_t>(k) * 8, 256) +
           round_up(lms::stage2_topk_part_bytes(B, k), 256);
}

lms_status lms_lmhead_sample_topk(const void* H, int64_t ldh, const void* W, int64_t ldw, int64_t B,
                                  int64_t D, int64_t V, int32_t k, const lms_sample_params* params,
                                  int64_t* out, float* scores, void* workspace,
                                  size_t workspace_bytes, void* stream) {
    g_last_error[0] = '\0';
    if (H == nullptr || W == nullptr || out == nullptr)
        return fail(LMS_ERR_INVALID_ARG, "H, W and out are required");
    if (k < 1 || k > LMS_TOPK_MAX) return fail(LMS_ERR_INVALID_ARG, "k must be in [1, %d] (k=%d)", LMS_TOPK_MAX, k);
    Tiling t;
    lms_status st = make_tiling(LMS_OP_LMHEAD, B, D, V, params ? params->tile_v : 0, &t);
    if (st != LMS_OK) return st;
    if ((st = check_params(params, V)) != LMS_OK) return st;
    if (D % 8 != 0) return fail(LMS_ERR_UNSUPPORTED, "D must be a multiple of 8 (D=%lld)", (long long)D);
    if (D > 65536) return fail(LMS_ERR_UNSUPPORTED, "D must be <= 65536");
    if (ldh < D || ldw < D || ldh % 8 != 0 || ldw % 8 != 0)
        return fail(LMS_ERR_UNSUPPORTED, "ldh/ldw must be >= D and multiples of 8 elements");
    if (reinterpret_cast<uintptr_t>(H) % 16 != 0 || reinterpret_cast<uintptr_t>(W) % 16 != 0)
        return fail(LMS_ERR_UNSUPPORTED, "H and W must be 16-byte aligned");
    if (params->path != LMS_PATH_AUTO && params->path != LMS_PATH_TCGEN05)
        return fail(LMS_ERR_UNSUPPORTED, "Gumbel-top-k runs on the tcgen05 kernel only");
    const size_t need = lms_workspace_bytes_topk(B, V, k);
    if (workspace == nullptr || workspace_bytes < need)
        return fail(LMS_ERR_WORKSPACE, "workspace of %zu bytes needed", need);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const bool wide = params->noise_mode == LMS_NOISE_WIDE53;
    lms::SampleArgs a = make_args(params, B, V, t, workspace);
    a.cand_score = nullptr;
    a.cand_index = nullptr;
    a.cand_keys = reinterpret_cast<unsigned long long*>(static_cast<char*>(workspace) + kStatusBlock);
    a.topk = k;
    CUtensorMap tmW;
    if ((st = encode_bf16_map(&tmW, W, V, D, ldw, 128)) != LMS_OK) return st;
    const uint32_t timeout_ms = params->timeout_ms ? params->timeout_ms : 2000u;
    // One list mode for the whole call, from the widest launch: running lists (one per row,
    // Stage-1 CTA and TMEM quadrant; the persistent grid is min(n_tiles, SMs) CTAs) when they fit
    // in shared memory, else one list per row, tile and quadrant.
    const int64_t nb0 = B < kTcMaxBatchPerLaunch ? B : kTcMaxBatchPerLaunch;
    a.topk_mode = lms::topk_mode_for(static_cast<int>(nb0 < 16 ? 16 : (nb0 + 15) / 16 * 16), k);
    const int sms = lms::device_sm_count();
    const int64_t n_lists =
        a.topk_mode == lms::kTopKRunning ? 4 * (t.n_tiles < sms ? t.n_tiles : sms) : 4 * t.n_tiles;
    for (int64_t r0 = 0; r0 < B; r0 += kTcMaxBatchPerLaunch) {
        const int64_t nb = (B - r0 < kTcMaxBatchPerLaunch) ? B - r0 : kTcMaxBatchPerLaunch;
        const int n_pad = static_cast<int>(nb < 16 ? 16 : (nb + 15) / 16 * 16);
        CUtensorMap tmH;
        if ((st = encode_bf16_map(&tmH, H, B, D, ldh, n_pad)) != LMS_OK) return st;
        lms::SampleArgs ac = a;
        ac.B = nb;
        ac.row0 = r0;
        ac.cand_keys = a.cand_keys + r0 * n_lists * k;
        const cudaError_t e = lms::launch_lmhead_tc(tmW, tmH, D, n_pad, wide, timeout_ms,
                                                    params->debug_flags, ac, s);
        if (e != cudaSuccess) return cuda_fail(e, "tcgen05 top-k Stage-1 launch");
    }
    unsigned long long* part = reinterpret_cast<unsigned long long*>(
        static_cast<char*>(workspace) + kStatusBlock +
        round_up(static_cast<size_t>(B) * static_cast<size_t>(t.n_tiles) * 4 * static_cast<size_t>(k) * 8, 256));
    const cudaError_t e = lms::launch_stage2_topk(a.cand_keys, n_lists, k, B, params->temperature,
                                                  out, scores, params->row_status, a.status_bits, part, s);
    if (e != cudaSuccess) return cuda_fail(e, "top-k Stage-2 launch");
    return LMS_OK;
}

namespace {
// Workspace of lms_verify_from_logits, region by region (each 256-byte aligned).
// Sized for fp32 logits, whose chunks are the shorter, so one size serves both types.
struct VerifyLayout {
    int64_t nc, ncr;
    size_t part, dec, cand, cnt, total;
    VerifyLayout(int64_t B, int64_t k, int64_t V, bool bf16) {
        int64_t nc32, ncr32;
        lms::verify_chunks(V, false, &nc32, &ncr32);
        lms::verify_chunks(V, bf16, &nc, &ncr);
        const size_t rows = static_cast<size_t>(B) * static_cast<size_t>(2 * k + 1) * static_cast<size_t>(nc32);
        part = round_up(rows * 8 * 4, 256);          // each of pmax, psum, parg: one per warp (8)
        dec = round_up(static_cast<size_t>(B) * sizeof(lms::VerifyDecision), 256);
        cand = round_up(static_cast<size_t>(B) * static_cast<size_t>(ncr32) * 2 * 4, 256);  // c_s, c_i
        cnt = round_up(static_cast<size_t>(B) * 4, 256);                // cnt_r
        total = kStatusBlock + 3 * part + dec + 2 * cand + cnt;
    }
};
constexpr int kVerifyMaxK = 32;
}  // namespace

size_t lms_workspace_bytes_verify(int64_t B, int32_t k, int64_t V) {
    if (B <= 0 || V <= 0 || V > kMaxV || k < 1 || k > kVerifyMaxK) return 0;
    return VerifyLayout(B, k, V, false).total;
}

lms_status lms_verify_from_logits(const void* target, const void* draft, int32_t dtype, int64_t ld,
                                  int64_t B, int32_t k, int64_t V, const int64_t* draft_tokens,
                                  const lms_sample_params* params, int64_t* accept_len, int64_t* out,
                                  void* workspace, size_t workspace_bytes, void* stream) {
    g_last_error[0] = '\0';
    if (target == nullptr || draft == nullptr || draft_tokens == nullptr || accept_len == nullptr ||
        out == nullptr)
        return fail(LMS_ERR_INVALID_ARG, "target, draft, draft_tokens, accept_len and out are required");
    if (dtype != LMS_DTYPE_F32 && dtype != LMS_DTYPE_BF16)
        return fail(LMS_ERR_INVALID_ARG, "unknown dtype %d", dtype);
    if (B <= 0 || V <= 0 || V > kMaxV) return fail(LMS_ERR_INVALID_ARG, "need B > 0 and 0 < V < 2^31");
    if (k < 1 || k > kVerifyMaxK) return fail(LMS_ERR_INVALID_ARG, "k must be in [1, %d] (k=%d)", kVerifyMaxK, k);
    if (ld < V) return fail(LMS_ERR_INVALID_ARG, "ld must be >= V");
    lms_status st = check_params(params, V);
    if (st != LMS_OK) return st;
    if (params->bias != nullptr || params->allow_mask != nullptr || params->tile_v != 0 ||
        params->path != LMS_PATH_AUTO || params->debug_flags != 0)
        return fail(LMS_ERR_INVALID_ARG, "bias, mask, tile_v, path and debug_flags do not apply to verify");
    const VerifyLayout L(B, k, V, dtype == LMS_DTYPE_BF16);
    if (workspace == nullptr || workspace_bytes < L.total)
        return fail(LMS_ERR_WORKSPACE, "workspace of %zu bytes needed", L.total);
    char* w = static_cast<char*>(workspace) + kStatusBlock;
    lms::VerifyArgs a;
    a.status_bits = static_cast<uint32_t*>(workspace);
    a.target = target;
    a.draft = draft;
    a.ld = ld;
    a.B = B;
    a.k = k;
    a.V = V;
    a.tokens = draft_tokens;
    a.temperature = params->temperature;
    a.seeds = params->seeds;
    a.positions = params->positions;
    a.base_seed = params->base_seed;
    a.offset = params->offset;
    a.nc = L.nc;
    a.ncr = L.ncr;
    a.pmax = reinterpret_cast<float*>(w);
    a.psum = reinterpret_cast<float*>(w + L.part);
    a.parg = reinterpret_cast<int*>(w + 2 * L.part);
    a.dec = reinterpret_cast<lms::VerifyDecision*>(w + 3 * L.part);
    char* c = w + 3 * L.part + L.dec;
    a.c_s = reinterpret_cast<float*>(c);
    a.c_i = reinterpret_cast<int*>(c + L.cand);
    a.cnt_r = reinterpret_cast<int*>(c + 2 * L.cand);
    a.accept_len = accept_len;
    a.out = out;
    a.row_status = params->row_status;
    const cudaError_t e = lms::launch_verify(a, dtype == LMS_DTYPE_BF16, params->noise_mode == LMS_NOISE_WIDE53,
                                             static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "verify launch");
    return LMS_OK;
}

lms_status lms_lmhead_sample_fp8(const void* H, int64_t ldh, const void* W8, int64_t ldw8,
                                 const float* w_scale, int64_t B, int64_t D, int64_t V,
                                 const lms_sample_params* params, int64_t* out, void* workspace,
                                 size_t workspace_bytes, void* stream) {
    g_last_error[0] = '\0';
    if (H == nullptr || W8 == nullptr || w_scale == nullptr || out == nullptr)
        return fail(LMS_ERR_INVALID_ARG, "H, W8, w_scale and out are required");
    Tiling t;
    lms_status st = make_tiling(LMS_OP_LMHEAD_FP8, B, D, V, params ? params->tile_v : 0, &t);
    if (st != LMS_OK) return st;
    if ((st = check_params(params, V)) != LMS_OK) return st;
    if (D % 16 != 0) return fail(LMS_ERR_UNSUPPORTED, "D must be a multiple of 16 (D=%lld)", (long long)D);
    if (D > 65536) return fail(LMS_ERR_UNSUPPORTED, "D must be <= 65536");
    if (ldh < D || ldh % 8 != 0 || ldw8 < D || ldw8 % 16 != 0)
        return fail(LMS_ERR_UNSUPPORTED, "ldh must be >= D and a multiple of 8; ldw8 >= D and a multiple of 16");
    if (reinterpret_cast<uintptr_t>(H) % 16 != 0 || reinterpret_cast<uintptr_t>(W8) % 16 != 0)
        return fail(LMS_ERR_UNSUPPORTED, "H and W8 must be 16-byte aligned");
    if (params->path != LMS_PATH_AUTO && params->path != LMS_PATH_TCGEN05)
        return fail(LMS_ERR_UNSUPPORTED, "the FP8 path runs on the tcgen05 kernel only");
    if (workspace == nullptr || workspace_bytes < t.workspace)
        return fail(LMS_ERR_WORKSPACE, "workspace of %zu bytes needed", t.workspace);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    lms::SampleArgs a = make_args(params, B, V, t, workspace);
    const size_t cand = static_cast<size_t>(B) * static_cast<size_t>(t.n_tiles) * 4;
    const int64_t ldq = static_cast<int64_t>(round_up(static_cast<size_t>(D), 16));
    uint8_t* q = static_cast<uint8_t*>(workspace) + kStatusBlock + 2 * round_up(cand, 256);
    int32_t* h_exp = reinterpret_cast<int32_t*>(q + round_up(static_cast<size_t>(B) * ldq, 256));
    a.h_exp = h_exp;
    a.w_scale = w_scale;
    cudaError_t e = lms::launch_quantize_rows_e4m3(static_cast<const uint16_t*>(H), ldh, B, D, q, ldq, h_exp, s);
    if (e != cudaSuccess) return cuda_fail(e, "activation quantisation launch");
    CUtensorMap tmW;
    if ((st = encode_map(&tmW, W8, V, D, ldw8, 128, true)) != LMS_OK) return st;
    const bool wide = params->noise_mode == LMS_NOISE_WIDE53;
    const uint32_t timeout_ms = params->timeout_ms ? params->timeout_ms : 2000u;
    for (int64_t r0 = 0; r0 < B; r0 += kTcMaxBatchPerLaunch) {
        const int64_t nb = (B - r0 < kTcMaxBatchPerLaunch) ? B - r0 : kTcMaxBatchPerLaunch;
        const int n_pad = static_cast<int>(nb < 16 ? 16 : (nb + 15) / 16 * 16);
        CUtensorMap tmH;
        if ((st = encode_map(&tmH, q, B, D, ldq, n_pad, true)) != LMS_OK) return st;
        lms::SampleArgs ac = a;
        ac.B = nb;
        ac.row0 = r0;
        ac.cand_score = a.cand_score + r0 * t.n_tiles;
        ac.cand_index = a.cand_index + r0 * t.n_tiles;
        e = lms::launch_lmhead_tc(tmW, tmH, D, n_pad, wide, timeout_ms, params->debug_flags, ac, s, true);
        if (e != cudaSuccess) return cuda_fail(e, "tcgen05 FP8 Stage-1 launch");
    }
    e = lms::launch_stage2(a.cand_score, a.cand_index, t.n_tiles, B, params->temperature, out,
                           params->row_status, a.status_bits, s);
    if (e != cudaSuccess) return cuda_fail(e, "Stage-2 launch");
    return LMS_OK;
}

size_t lms_mxfp4_tiled_bytes(int64_t V, int64_t D) {
    if (V <= 0 || V > kMaxV || D <= 0 || D > 65536 || D % 32 != 0) return 0;
    return lms::mxfp4_tiled_bytes(V, D);
}

lms_status lms_mxfp4_pack(const void* W4, int64_t ldw4, const void* S, int64_t lds, int64_t V, int64_t D,
                          void* Wt, size_t Wt_bytes, void* stream) {
    g_last_error[0] = '\0';
    if (W4 == nullptr || S == nullptr || Wt == nullptr)
        return fail(LMS_ERR_INVALID_ARG, "W4, S and Wt are required");
    const size_t need = lms_mxfp4_tiled_bytes(V, D);
    if (need == 0)
        return fail(LMS_ERR_INVALID_ARG, "need 0 < V < 2^31 and 0 < D <= 65536 with D a multiple of 32");
    if (ldw4 < D / 2 || lds < V) return fail(LMS_ERR_INVALID_ARG, "ldw4 must be >= D/2 and lds >= V");
    if (reinterpret_cast<uintptr_t>(Wt) % 16 != 0) return fail(LMS_ERR_UNSUPPORTED, "Wt must be 16-byte aligned");
    if (Wt_bytes < need) return fail(LMS_ERR_WORKSPACE, "Wt needs %zu bytes", need);
    const cudaError_t e = lms::launch_mxfp4_pack(static_cast<const uint8_t*>(W4), ldw4,
                                                 static_cast<const uint8_t*>(S), lds, V, D,
                                                 static_cast<uint8_t*>(Wt), static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "MXFP4 pack launch");
    return LMS_OK;
}

lms_status lms_lmhead_sample_mxfp4(const void* H, int64_t ldh, const void* Wt, size_t Wt_bytes, int64_t B,
                                   int64_t D, int64_t V, const lms_sample_params* params, int64_t* out,
                                   void* workspace, size_t workspace_bytes, void* stream) {
    g_last_error[0] = '\0';
    if (H == nullptr || Wt == nullptr || out == nullptr)
        return fail(LMS_ERR_INVALID_ARG, "H, Wt and out are required");
    Tiling t;
    lms_status st = make_tiling(LMS_OP_LMHEAD, B, D, V, params ? params->tile_v : 0, &t);
    if (st != LMS_OK) return st;
    if ((st = check_params(params, V)) != LMS_OK) return st;
    if (D % 32 != 0) return fail(LMS_ERR_UNSUPPORTED, "D must be a multiple of 32 (D=%lld)", (long long)D);
    if (D > 65536) return fail(LMS_ERR_UNSUPPORTED, "D must be <= 65536");
    if (ldh < D || ldh % 8 != 0) return fail(LMS_ERR_UNSUPPORTED, "ldh must be >= D and a multiple of 8");
    if (Wt_bytes < lms::mxfp4_tiled_bytes(V, D))
        return fail(LMS_ERR_INVALID_ARG, "Wt holds %zu bytes, the tiled weights of V x D need %zu", Wt_bytes,
                    lms::mxfp4_tiled_bytes(V, D));
    if (reinterpret_cast<uintptr_t>(H) % 16 != 0 || reinterpret_cast<uintptr_t>(Wt) % 16 != 0)
        return fail(LMS_ERR_UNSUPPORTED, "H and Wt must be 16-byte aligned");
    if (params->path != LMS_PATH_AUTO && params->path != LMS_PATH_TCGEN05)
        return fail(LMS_ERR_UNSUPPORTED, "the MXFP4 path runs on the tcgen05 kernel only");
    if (workspace == nullptr || workspace_bytes < t.workspace)
        return fail(LMS_ERR_WORKSPACE, "workspace of %zu bytes needed", t.workspace);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const bool wide = params->noise_mode == LMS_NOISE_WIDE53;
    lms::SampleArgs a = make_args(params, B, V, t, workspace);
    const uint32_t timeout_ms = params->timeout_ms ? params->timeout_ms : 2000u;
    cudaError_t e;
    // batches above 128 rows run as launches of <= 128 rows: the two accumulators of a launch
    // share TMEM with the rebuilt weight slots
    constexpr int64_t kMxMaxBatchPerLaunch = 128;
    for (int64_t r0 = 0; r0 < B; r0 += kMxMaxBatchPerLaunch) {
        const int64_t nb = (B - r0 < kMxMaxBatchPerLaunch) ? B - r0 : kMxMaxBatchPerLaunch;
        const int n_pad = static_cast<int>(nb < 16 ? 16 : (nb + 15) / 16 * 16);
        CUtensorMap tmH;
        if ((st = encode_bf16_map(&tmH, H, B, D, ldh, n_pad)) != LMS_OK) return st;
        lms::SampleArgs ac = a;
        ac.B = nb;
        ac.row0 = r0;
        ac.cand_score = a.cand_score + r0 * t.n_tiles;
        ac.cand_index = a.cand_index + r0 * t.n_tiles;
        e = lms::launch_lmhead_mx(static_cast<const uint8_t*>(Wt), tmH, D, n_pad, wide, timeout_ms,
                                  params->debug_flags, ac, s);
        if (e != cudaSuccess) return cuda_fail(e, "tcgen05 MXFP4 Stage-1 launch");
    }
    e = lms::launch_stage2(a.cand_score, a.cand_index, t.n_tiles, B, params->temperature, out,
                           params->row_status, a.status_bits, s);
    if (e != cudaSuccess) return cuda_fail(e, "Stage-2 launch");
    return LMS_OK;
}

lms_status lms_sample_from_logits(const void* logits, int32_t dtype, int64_t ld, int64_t B,
                                  int64_t V, const lms_sample_params* params, int64_t* out,
                                  void* workspace, size_t workspace_bytes, void* stream) {
    g_last_error[0] = '\0';
    if (logits == nullptr || out == nullptr) return fail(LMS_ERR_INVALID_ARG, "logits and out are required");
    if (dtype != LMS_DTYPE_F32 && dtype != LMS_DTYPE_BF16)
        return fail(LMS_ERR_INVALID_ARG, "unknown dtype %d", dtype);
    Tiling t;
    lms_status st = make_tiling(LMS_OP_LOGITS, B, 0, V, params ? params->tile_v : 0, &t);
    if (st != LMS_OK) return st;
    if ((st = check_params(params, V)) != LMS_OK) return st;
    if (ld != 0 && ld < V) return fail(LMS_ERR_INVALID_ARG, "ld must be 0 (broadcast) or >= V");
    if (params->path != LMS_PATH_AUTO) return fail(LMS_ERR_INVALID_ARG, "path applies to the fused entry only");
    if (params->debug_flags != 0) return fail(LMS_ERR_INVALID_ARG, "debug_flags apply to the fused entry only");
    if (workspace == nullptr || workspace_bytes < t.workspace)
        return fail(LMS_ERR_WORKSPACE, "workspace of %zu bytes needed", t.workspace);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    lms::SampleArgs a = make_args(params, B, V, t, workspace);
    cudaError_t e = lms::launch_logits_stage1(logits, dtype == LMS_DTYPE_BF16, ld, t.tile_v,
                                              params->noise_mode == LMS_NOISE_WIDE53, a, s);
    if (e != cudaSuccess) return cuda_fail(e, "logits Stage-1 launch");
    e = lms::launch_stage2(a.cand_score, a.cand_index, t.n_tiles, B, params->temperature, out,
                           params->row_status, a.status_bits, s);
    if (e != cudaSuccess) return cuda_fail(e, "Stage-2 launch");
    return LMS_OK;
}

lms_status lms_sample_from_logits_filtered(const void* logits, int32_t dtype, int64_t ld, int64_t B,
                                           int64_t V, const lms_sample_params* params,
                                           const lms_filter_params* filters, int64_t* out,
                                           void* stream) {
    g_last_error[0] = '\0';
    if (logits == nullptr || out == nullptr || filters == nullptr)
        return fail(LMS_ERR_INVALID_ARG, "logits, filters and out are required");
    if (dtype != LMS_DTYPE_F32 && dtype != LMS_DTYPE_BF16)
        return fail(LMS_ERR_INVALID_ARG, "unknown dtype %d", dtype);
    if (B <= 0 || V <= 0 || V > kMaxV || B > kMaxV)
        return fail(LMS_ERR_INVALID_ARG, "need 0 < B < 2^31 and 0 < V < 2^31");
    lms_status st = check_params(params, V);
    if (st != LMS_OK) return st;
    if (ld != 0 && ld < V) return fail(LMS_ERR_INVALID_ARG, "ld must be 0 (broadcast) or >= V");
    if (params->path != LMS_PATH_AUTO || params->debug_flags != 0 || params->tile_v != 0)
        return fail(LMS_ERR_INVALID_ARG, "path, tile_v and debug_flags do not apply to the filtered race");
    if (filters->k_max < 0 || filters->k_max > 1024 || filters->reserved != 0)
        return fail(LMS_ERR_INVALID_ARG, "k_max must be in [0, 1024] and reserved 0");
    lms::FilterArgs f;
    f.a.temperature = params->temperature;
    f.a.seeds = params->seeds;
    f.a.positions = params->positions;
    f.a.bias = params->bias;
    f.a.ld_bias = params->ld_bias;
    f.a.mask = params->allow_mask;
    f.a.ld_mask = params->ld_mask;
    f.a.base_seed = params->base_seed;
    f.a.offset = params->offset;
    f.a.B = B;
    f.a.row0 = 0;
    f.a.V = V;
    f.a.n_tiles = 0;
    f.a.cand_score = nullptr;
    f.a.cand_index = nullptr;
    f.a.h_exp = nullptr;
    f.a.w_scale = nullptr;
    f.top_k = filters->top_k;
    f.top_p = filters->top_p;
    f.min_p = filters->min_p;
    f.k_max = filters->k_max ? filters->k_max : 1024;
    f.out = out;
    f.row_status = params->row_status;
    const cudaError_t e = lms::launch_filtered_race(logits, dtype == LMS_DTYPE_BF16, ld,
                                                    params->noise_mode == LMS_NOISE_WIDE53, f,
                                                    static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "filtered race launch");
    return LMS_OK;
}

lms_status lms_philox_fill_noise(void* out, int32_t kind, int32_t noise_mode, int64_t B, int64_t V,
                                 const int64_t* seeds, const int64_t* positions, uint64_t base_seed,
                                 uint64_t offset, void* stream) {
    g_last_error[0] = '\0';
    if (out == nullptr) return fail(LMS_ERR_INVALID_ARG, "out is required");
    if (kind < LMS_NOISE_OUT_WORDS || kind > LMS_NOISE_OUT_GUMBEL)
        return fail(LMS_ERR_INVALID_ARG, "unknown noise kind %d", kind);
    if (noise_mode != LMS_NOISE_FP32 && noise_mode != LMS_NOISE_WIDE53)
        return fail(LMS_ERR_INVALID_ARG, "unknown noise_mode %d", noise_mode);
    if (B <= 0 || V <= 0 || V > kMaxV) return fail(LMS_ERR_INVALID_ARG, "need B > 0 and 0 < V < 2^31");
    if (seeds != nullptr && positions == nullptr)
        return fail(LMS_ERR_INVALID_ARG, "positions is required when seeds is given");
    const size_t align = kind == LMS_NOISE_OUT_WORDS ? 16 : (kind == LMS_NOISE_OUT_UNIFORM ? 8 : 4);
    if (reinterpret_cast<uintptr_t>(out) % align != 0)
        return fail(LMS_ERR_UNSUPPORTED, "out must be %zu-byte aligned", align);
    const cudaError_t e = lms::launch_noise_fill(out, kind, noise_mode == LMS_NOISE_WIDE53, B, V, seeds,
                                                 positions, base_seed, offset, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "noise-fill launch");
    return LMS_OK;
}

lms_status lms_read_status(const void* workspace, void* stream, uint32_t* status_bits) {
    g_last_error[0] = '\0';
    if (workspace == nullptr) return fail(LMS_ERR_INVALID_ARG, "workspace is required");
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return cuda_fail(e, "lms_read_status: stream synchronisation");
    uint32_t bits = 0;
    e = cudaMemcpy(&bits, workspace, sizeof bits, cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return cuda_fail(e, "lms_read_status: status copy");
    if (status_bits) *status_bits = bits;
    if (bits & (1u << LMS_ROW_DEVICE_TIMEOUT))
        return fail(LMS_ERR_TIMEOUT, "a device-side wait ran out of time (row status 3)");
    return LMS_OK;
}

}  // extern "C"
