// lms_lmhead_sample_noalloc: the fused LM-head + Gumbel-max sampler for callers that cannot
// allocate device memory -- for example code running inside an allocator or a memory-pool
// callback, a host function that must not take the device allocator's lock, or an embedding
// that hands this library only fixed buffers.  Instead of a caller-provided workspace, the
// Stage-1 candidates live in one file-scope device array of fixed size that is part of the
// library image: every GPU that loads the library holds it until the process exits.
//
// Limit: the candidates need 8 bytes per (batch row, vocabulary tile of 128), so the 4 MiB array
// holds B * ceil(V / 128) <= 524288 of them (e.g. B = 256 at V = 262144, or B = 441 at
// V = 151936).  Larger calls are rejected with LMS_ERR_WORKSPACE before anything is launched.
// Nothing in the array has to start at zero: each call's Stage 1 writes every candidate that
// its Stage 2 reads.  Calls whose kernels overlap on the GPU share the array and race.
#include <cuda_runtime.h>

#include <cstdio>
#include <mutex>

#include "lms.h"
#include "lms_kernels.h"

namespace {

constexpr size_t kNoAllocScratchBytes = size_t{4} << 20;   // 4 MiB
constexpr int kMaxDevices = 64;

// The scratch itself.  In host code this name is only a stand-in for the device symbol: its
// device address comes from cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

std::mutex g_setup_mutex;
void* g_scratch_addr[kMaxDevices] = {};

// Device address of the scratch on the current device, looked up once per device.
cudaError_t scratch_address(void** addr) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_setup_mutex);
    if (g_scratch_addr[dev] == nullptr) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess) return e;
        g_scratch_addr[dev] = p;
    }
    *addr = g_scratch_addr[dev];
    return cudaSuccess;
}

}  // namespace

extern "C" {

lms_status lms_lmhead_sample_noalloc(const void* H, int64_t ldh, const void* W, int64_t ldw,
                                     int64_t B, int64_t D, int64_t V,
                                     const lms_sample_params* params, int64_t* out, void* stream) {
    const size_t need = lms_workspace_bytes(LMS_OP_LMHEAD, B, D, V, params ? params->tile_v : 0);
    if (need == 0) {
        // invalid sizes: let the regular entry point produce its own message
        return lms_lmhead_sample(H, ldh, W, ldw, B, D, V, params, out, nullptr, 0, stream);
    }
    if (need > kNoAllocScratchBytes) {
        char msg[256];
        snprintf(msg, sizeof msg,
                 "lms_lmhead_sample_noalloc: B=%lld, V=%lld needs %zu bytes of candidates, more than "
                 "the %zu-byte static scratch (B * ceil(V/128) must be <= %zu); use "
                 "lms_lmhead_sample with a workspace",
                 (long long)B, (long long)V, need, kNoAllocScratchBytes, kNoAllocScratchBytes / 8);
        lms::set_last_error(msg);
        return LMS_ERR_WORKSPACE;
    }
    void* scratch = nullptr;
    const cudaError_t e = scratch_address(&scratch);
    if (e != cudaSuccess) {
        char msg[256];
        snprintf(msg, sizeof msg, "lms_lmhead_sample_noalloc: cudaGetSymbolAddress failed: %s",
                 cudaGetErrorString(e));
        lms::set_last_error(msg);
        return LMS_ERR_CUDA;
    }
    return lms_lmhead_sample(H, ldh, W, ldw, B, D, V, params, out, scratch, kNoAllocScratchBytes,
                             stream);
}

}  // extern "C"
