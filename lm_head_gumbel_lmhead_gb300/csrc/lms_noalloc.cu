// lms_lmhead_sample_noalloc: the fused LM-head + Gumbel-max sampler for callers that cannot
// allocate device memory -- for example code running inside an allocator or a memory-pool
// callback, a host function that must not take the device allocator's lock, or an embedding
// that hands this library only fixed buffers.  Instead of a caller-provided workspace, the
// Stage-1 candidates live in one file-scope device array of fixed size that is part of the
// library image: every GPU that loads the library holds it until the process exits.
//
// Limit: the candidates need 8 bytes per (batch row, vocabulary tile of 128), so the array (the
// 256-byte status block every workspace starts with, then 4 MiB of candidates) holds
// B * ceil(V / 128) <= 524288 of them (e.g. B = 256 at V = 262144, or B = 441 at V = 151936).
// Larger calls are rejected with LMS_ERR_WORKSPACE before anything is launched.
// Nothing in the array has to start at zero: each call's Stage 1 writes every candidate that
// its Stage 2 reads, and clears the status word.  Calls whose kernels overlap on the GPU share
// the array and race.
#include <cuda_runtime.h>

#include <cstdio>
#include <mutex>

#include "lms.h"
#include "lms_kernels.h"

namespace {

constexpr size_t kMaxCandidates = size_t{1} << 19;                 // 524288
constexpr size_t kNoAllocScratchBytes = 256 + kMaxCandidates * 8;   // status block + 4 MiB
constexpr int kMaxDevices = 64;

// The scratch itself.  In host code this name is only a stand-in for the device symbol: its
// device address comes from cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

std::mutex g_setup_mutex;
void* g_scratch_addr[kMaxDevices] = {};

// Device address of the scratch on the current device.  Outside stream capture it is looked up
// on every call (cudaGetSymbolAddress, with the device current), so a module reloaded at another
// address -- after cudaDeviceReset, or in another context -- is seen at once; the address is
// then cached per device for calls made while `stream` is capturing, which use the cache only.
cudaError_t scratch_address(cudaStream_t stream, void** addr, bool* uncached_capture) {
    *uncached_capture = false;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    e = cudaStreamIsCapturing(stream, &cs);
    if (e != cudaSuccess) {
        // (the legacy stream during another stream's global-mode capture): treat as capturing,
        // and consume the error so that no later launch check reports it
        cudaGetLastError();
        cs = cudaStreamCaptureStatusActive;
    }
    std::lock_guard<std::mutex> lock(g_setup_mutex);
    if (cs == cudaStreamCaptureStatusNone) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess) return e;
        g_scratch_addr[dev] = p;
    } else if (g_scratch_addr[dev] == nullptr) {
        *uncached_capture = true;
        return cudaErrorStreamCaptureUnsupported;
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
                 "lms_lmhead_sample_noalloc: B=%lld, V=%lld needs %zu bytes of scratch, more than "
                 "the %zu-byte static scratch (B * ceil(V/128) must be <= %zu); use "
                 "lms_lmhead_sample with a workspace",
                 (long long)B, (long long)V, need, kNoAllocScratchBytes, kMaxCandidates);
        lms::set_last_error(msg);
        return LMS_ERR_WORKSPACE;
    }
    void* scratch = nullptr;
    bool uncached_capture = false;
    const cudaError_t e = scratch_address(static_cast<cudaStream_t>(stream), &scratch, &uncached_capture);
    if (e != cudaSuccess) {
        char msg[256];
        if (uncached_capture)
            snprintf(msg, sizeof msg, "lms_lmhead_sample_noalloc: the first call on a device must "
                                      "come before any stream capture");
        else
            snprintf(msg, sizeof msg, "lms_lmhead_sample_noalloc: scratch address lookup failed: %s",
                     cudaGetErrorString(e));
        lms::set_last_error(msg);
        return LMS_ERR_CUDA;
    }
    return lms_lmhead_sample(H, ldh, W, ldw, B, D, V, params, out, scratch, kNoAllocScratchBytes,
                             stream);
}

}  // extern "C"
