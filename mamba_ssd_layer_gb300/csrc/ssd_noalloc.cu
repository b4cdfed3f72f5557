// ssd_noalloc.cu -- ssd_forward_noalloc: the forward pass for callers that cannot allocate
// device memory (a custom allocator that is not set up yet, a context whose memory is owned
// by someone else, code that must not call cudaMalloc while a graph is being built, and so on).
//
// The scratch that ssd_forward takes from the caller's workspace lives here instead, in a
// file-scope device array of fixed size. Every GPU that loads this library holds that array
// until the process exits. Host code cannot use the array's name as a device address, so
// the address is looked up with cudaGetSymbolAddress (in the current context, on every call) and
// passed on.
#include <cstdio>

#include <cuda_runtime.h>

#include "ssd.h"
#include "ssd_internal.cuh"

namespace {

// Largest workspace this entry point can serve (bytes).
constexpr size_t kNoAllocScratchBytes = size_t(16) << 20;

__device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

// Device address of the scratch array in the current context. Looked up on every call: the lookup does
// not synchronise, and a context that was reset (cudaDeviceReset) and created again may place the
// array elsewhere, so a cached address could point at memory the array no longer occupies.
int scratch_address(void** out) {
    void* p = nullptr;
    if (ssd::note_cuda_error("cudaGetSymbolAddress", cudaGetSymbolAddress(&p, g_noalloc_scratch)) != cudaSuccess)
        return SSD_ERR_CUDA;
    *out = p;
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
