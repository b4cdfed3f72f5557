// ssd_noalloc.cu -- ssd_forward_noalloc: the forward pass for callers that cannot allocate
// device memory (a custom allocator that is not set up yet, a context whose memory is owned
// by someone else, code that must not call cudaMalloc while a graph is being built, and so on).
//
// The scratch that ssd_forward takes from the caller's workspace lives here instead, in a
// file-scope device array of fixed size. Every GPU that loads this library holds that array
// until the process exits. Host code cannot use the array's name as a device address, so
// the address is looked up once per device with cudaGetSymbolAddress and passed on.
#include <cstdio>
#include <mutex>

#include <cuda_runtime.h>

#include "ssd.h"
#include "ssd_internal.cuh"

namespace {

// Largest workspace this entry point can serve (bytes).
constexpr size_t kNoAllocScratchBytes = size_t(16) << 20;

__device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_noalloc_lock;
void* g_noalloc_ptr[kMaxDevices] = {};

// Device address of the scratch array on the current device, looked up on first use.
int scratch_address(void** out) {
    int dev = 0;
    if (ssd::note_cuda_error("cudaGetDevice", cudaGetDevice(&dev)) != cudaSuccess) return SSD_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return SSD_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> guard(g_noalloc_lock);
    if (!g_noalloc_ptr[dev]) {
        void* p = nullptr;
        if (ssd::note_cuda_error("cudaGetSymbolAddress", cudaGetSymbolAddress(&p, g_noalloc_scratch)) != cudaSuccess)
            return SSD_ERR_CUDA;
        g_noalloc_ptr[dev] = p;
    }
    *out = g_noalloc_ptr[dev];
    return SSD_OK;
}

}  // namespace

extern "C" int ssd_forward_noalloc(const ssd_shape* s, ssd_dtype dtype, const void* x, const float* dt,
                                   const float* A, const void* B, const void* C, const float* D, int chunk,
                                   const float* initial_state, const int32_t* cu_seqlens, int nseq, void* y,
                                   float* final_state, void* stream) {
    const size_t need = ssd_workspace_size(s, dtype, chunk, cu_seqlens ? nseq : 0);
    if (need == 0) {
        // invalid or unsupported arguments: let ssd_forward report which
        return ssd_forward(s, dtype, x, dt, A, B, C, D, chunk, initial_state, cu_seqlens, nseq, y, final_state,
                           nullptr, 0, stream);
    }
    if (need > kNoAllocScratchBytes) {
        char msg[160];
        snprintf(msg, sizeof(msg), "problem needs %zu bytes of scratch; the built-in buffer holds %zu", need,
                 kNoAllocScratchBytes);
        ssd::note_cuda_error(msg, cudaErrorMemoryAllocation);
        return SSD_ERR_WORKSPACE;
    }
    void* scratch = nullptr;
    const int rc = scratch_address(&scratch);
    if (rc != SSD_OK) return rc;
    return ssd_forward(s, dtype, x, dt, A, B, C, D, chunk, initial_state, cu_seqlens, nseq, y, final_state,
                       scratch, kNoAllocScratchBytes, stream);
}
