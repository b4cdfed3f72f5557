// ssd_api.cu -- the extern "C" entry points declared in include/ssd.h:
// argument checks, workspace carving, device checks and dispatch to the fp32
// (SIMT) or bf16 (tcgen05) kernels. Nothing here allocates device memory.
#include <cstdint>
#include <cstdio>
#include <cstring>
#include <cuda_runtime.h>

#include <vector>

#include "ssd.h"
#include "ssd_internal.cuh"
#include "ssd_profile.h"

using namespace ssd;

namespace {

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int check_shape(const ssd_shape* s, ssd_dtype dtype, int chunk, int nseq, bool varlen) {
    if (!s) return SSD_ERR_INVALID_ARG;
    if (s->batch < 0 || s->seqlen < 0 || s->nheads <= 0 || s->headdim <= 0 || s->dstate <= 0 || s->ngroups <= 0)
        return SSD_ERR_INVALID_ARG;
    if (s->nheads % s->ngroups != 0) return SSD_ERR_INVALID_ARG;
    if (dtype != SSD_F32 && dtype != SSD_BF16) return SSD_ERR_INVALID_ARG;
    if (varlen && (s->batch != 1 || nseq < 0)) return SSD_ERR_INVALID_ARG;
    if (s->batch * s->seqlen > (int64_t)INT32_MAX / 2) return SSD_ERR_UNSUPPORTED;
    if (chunk != 64 && chunk != 128 && chunk != 256) return SSD_ERR_UNSUPPORTED;
    if (s->nheads > 65535) return SSD_ERR_UNSUPPORTED;
    if (dtype == SSD_F32) {
        if (s->headdim > 256 || s->dstate > 256) return SSD_ERR_UNSUPPORTED;
    } else if (!use_fused_path(*s, dtype)) {
        return SSD_ERR_UNSUPPORTED;
    }
    return SSD_OK;
}

size_t elt(ssd_dtype d) { return d == SSD_F32 ? 4 : 2; }

// The kernels are built for sm_103a only.
int check_device(int* num_sms) {
    int dev = 0;
    if (note_cuda_error("cudaGetDevice", cudaGetDevice(&dev)) != cudaSuccess) return SSD_ERR_CUDA;
    int major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(num_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return SSD_ERR_CUDA;
    if (major != 10 || minor != 3) return SSD_ERR_UNSUPPORTED;
    return SSD_OK;
}

struct ProfState {
    bool on = false;
    std::vector<cudaEvent_t> ev;   // begin/end pairs
    size_t used = 0;               // events recorded since the last read
    long long launches = 0;        // kernels launched since recording was enabled
    const char* kernel = "";       // the kernel the events bracket
};
thread_local ProfState g_prof;
thread_local char g_err_detail[160] = "";

}  // namespace

namespace ssd {
cudaError_t note_cuda_error(const char* step, cudaError_t e) {
    if (e != cudaSuccess) {
        snprintf(g_err_detail, sizeof(g_err_detail), "%s: %s", step, cudaGetErrorName(e));
        (void)cudaGetLastError();
    }
    return e;
}

void prof_launch() {
    if (g_prof.on) ++g_prof.launches;
}

void prof_begin(cudaStream_t s, const char* kernel) {
    if (!g_prof.on) return;
    g_prof.kernel = kernel;
    if (g_prof.used + 2 > g_prof.ev.size()) {
        for (int i = 0; i < 2; ++i) {
            cudaEvent_t e;
            if (cudaEventCreate(&e) != cudaSuccess) { g_prof.on = false; return; }
            g_prof.ev.push_back(e);
        }
    }
    cudaEventRecord(g_prof.ev[g_prof.used], s);
}
void prof_end(cudaStream_t s) {
    if (!g_prof.on || g_prof.used + 2 > g_prof.ev.size()) return;
    cudaEventRecord(g_prof.ev[g_prof.used + 1], s);
    g_prof.used += 2;
}
}  // namespace ssd

extern "C" {

int ssd_profile_enable(int on) {
    if (on && !g_prof.on) { g_prof.used = 0; g_prof.launches = 0; }
    g_prof.on = on != 0;
    return SSD_OK;
}

int ssd_profile_read(double* total_ms, int* launches) {
    double tot = 0.0;
    int n = 0;
    for (size_t i = 0; i + 1 < g_prof.used; i += 2) {
        float ms = 0.f;
        if (cudaEventSynchronize(g_prof.ev[i + 1]) != cudaSuccess ||
            cudaEventElapsedTime(&ms, g_prof.ev[i], g_prof.ev[i + 1]) != cudaSuccess)
            return SSD_ERR_CUDA;
        tot += ms;
        ++n;
    }
    g_prof.used = 0;
    if (total_ms) *total_ms = tot;
    if (launches) *launches = n;
    return SSD_OK;
}

long long ssd_profile_kernel_launches(void) { return g_prof.launches; }

const char* ssd_profile_kernel_name(void) { return g_prof.kernel; }

size_t ssd_workspace_size(const ssd_shape* s, ssd_dtype dtype, int chunk, int nseq) {
    const bool varlen = nseq > 0;
    if (check_shape(s, dtype, chunk, nseq, varlen) != SSD_OK) return 0;
    return ws_layout(*s, dtype, chunk, varlen ? nseq : s->batch, varlen).total;
}

int ssd_forward_ex(const ssd_shape* s, ssd_dtype dtype, unsigned flags, const void* x, const float* dt,
                   const float* A, const void* B, const void* C, const float* D, int chunk,
                   const float* initial_state, const int32_t* cu_seqlens, int nseq, void* y, float* final_state,
                   void* workspace, size_t workspace_bytes, void* stream) {
    const bool varlen = cu_seqlens != nullptr;
    if (flags & ~(SSD_SCALE_X_BY_DT | SSD_DEBUG_FORCE_TIMEOUT)) return SSD_ERR_INVALID_ARG;
    int rc = check_shape(s, dtype, chunk, nseq, varlen);
    if (rc != SSD_OK) return rc;
    const int64_t rows = s->batch * s->seqlen;
    if (rows > 0 && (!x || !dt || !B || !C || !y)) return SSD_ERR_INVALID_ARG;
    if (!A) return SSD_ERR_INVALID_ARG;
    const void* ptrs[] = {x, dt, A, B, C, D, initial_state, cu_seqlens, y, final_state};
    for (const void* p : ptrs)
        if (p && !aligned16(p)) return SSD_ERR_INVALID_ARG;
    if (varlen && nseq <= 0) return SSD_ERR_INVALID_ARG;
    const int64_t nseq_eff = varlen ? nseq : s->batch;
    const WsLayout L = ws_layout(*s, dtype, chunk, nseq_eff, varlen);
    if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u) || workspace_bytes < L.total)
        return SSD_ERR_WORKSPACE;
    int num_sms = 0;
    g_err_detail[0] = '\0';
    rc = check_device(&num_sms);
    if (rc != SSD_OK) return rc;

    Problem p;
    p.s = *s;
    p.dtype = dtype;
    p.chunk = chunk;
    p.varlen = varlen;
    p.scale_x_by_dt = (flags & SSD_SCALE_X_BY_DT) != 0;
    p.force_timeout = (flags & SSD_DEBUG_FORCE_TIMEOUT) != 0;
    p.nseq = nseq_eff;
    p.rows = rows;
    p.x = x; p.dt = dt; p.A = A; p.B = B; p.C = C; p.D = D;
    p.init = initial_state;
    p.cu_seqlens = cu_seqlens;
    p.y = y;
    p.final_state = final_state;
    p.ws = static_cast<char*>(workspace);
    p.L = L;
    p.stream = static_cast<cudaStream_t>(stream);
    p.num_sms = num_sms;

    cudaError_t e;
    if (L.fused) {
        int K = 0;
        int64_t np = 0;
        fused_plan(p, &K, &np);
        // window slots are indexed with 32-bit arithmetic on the device
        if (np > L.max_pieces || np >= (int64_t(1) << 28)) return SSD_ERR_UNSUPPORTED;
        // the header (status, diagnostics) and the window flags start at zero
        e = note_cuda_error("header reset", cudaMemsetAsync(p.status(), 0, L.clear_bytes, p.stream));
        // a packed batch needs its tile and window tables; a dense batch decodes windows arithmetically
        if (e == cudaSuccess && varlen) e = note_cuda_error("prep launch", launch_prep(p, kFusedTile));
        if (e == cudaSuccess) e = note_cuda_error("fused launch", launch_fused(p, K, np, 0));
        if (e == cudaSuccess && p.s.dstate > 128) {
            // second half of the state columns: the window flags start over (an error recorded by the
            // first launch stays in the status word)
            e = note_cuda_error("flag reset", cudaMemsetAsync(p.flags(), 0, L.clear_bytes - L.flags, p.stream));
            if (e == cudaSuccess) e = note_cuda_error("fused launch", launch_fused(p, K, np, 1));
        }
    } else {
        e = note_cuda_error("prep launch", launch_prep(p, chunk));
        if (e == cudaSuccess) e = note_cuda_error("fp32 launch", launch_f32_path(p));
    }
    return e == cudaSuccess ? SSD_OK : SSD_ERR_CUDA;
}

int ssd_forward(const ssd_shape* s, ssd_dtype dtype, const void* x, const float* dt, const float* A,
                const void* B, const void* C, const float* D, int chunk, const float* initial_state,
                const int32_t* cu_seqlens, int nseq, void* y, float* final_state, void* workspace,
                size_t workspace_bytes, void* stream) {
    return ssd_forward_ex(s, dtype, 0u, x, dt, A, B, C, D, chunk, initial_state, cu_seqlens, nseq, y, final_state,
                          workspace, workspace_bytes, stream);
}

size_t ssd_host_buffer_size(const ssd_shape* s, ssd_dtype dtype, int chunk, int nseq) {
    const size_t ws = ssd_workspace_size(s, dtype, chunk, nseq);
    if (!ws) return 0;
    const int64_t rows = s->batch * s->seqlen;
    const int64_t nseq_eff = nseq > 0 ? nseq : s->batch;
    const size_t e = elt(dtype);
    size_t tot = ws;
    tot += align256(rows * s->nheads * s->headdim * e) * 2;                 // x, y
    tot += align256(rows * s->nheads * 4);                                  // dt
    tot += align256(s->nheads * 4) * 2;                                     // A, D
    tot += align256(rows * s->ngroups * s->dstate * e) * 2;                 // B, C
    tot += align256(nseq_eff * s->nheads * s->headdim * s->dstate * 4) * 2; // initial, final
    tot += align256((nseq_eff + 1) * 4);                                    // cu_seqlens
    return tot;
}

int ssd_forward_host_ex(const ssd_shape* s, ssd_dtype dtype, unsigned flags, const void* x, const float* dt,
                        const float* A, const void* B, const void* C, const float* D, int chunk,
                        const float* initial_state, const int32_t* cu_seqlens, int nseq, void* y, float* final_state,
                        void* device_buffer, size_t device_buffer_bytes, void* stream) {
    const bool varlen = cu_seqlens != nullptr;
    if (flags & ~(SSD_SCALE_X_BY_DT | SSD_DEBUG_FORCE_TIMEOUT)) return SSD_ERR_INVALID_ARG;
    int rc = check_shape(s, dtype, chunk, nseq, varlen);
    if (rc != SSD_OK) return rc;
    if (varlen && nseq <= 0) return SSD_ERR_INVALID_ARG;
    const size_t need = ssd_host_buffer_size(s, dtype, chunk, varlen ? nseq : 0);
    if (!device_buffer || (reinterpret_cast<uintptr_t>(device_buffer) & 255u) || device_buffer_bytes < need)
        return SSD_ERR_WORKSPACE;
    const int64_t rows = s->batch * s->seqlen;
    if (rows > 0 && (!x || !dt || !B || !C || !y)) return SSD_ERR_INVALID_ARG;
    if (!A) return SSD_ERR_INVALID_ARG;
    const int64_t nseq_eff = varlen ? nseq : s->batch;
    const size_t e = elt(dtype);
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    char* base = static_cast<char*>(device_buffer);
    size_t off = 0;
    auto carve = [&](size_t bytes) { char* p = base + off; off += align256(bytes); return p; };
    const size_t ws_bytes = ssd_workspace_size(s, dtype, chunk, varlen ? nseq : 0);
    char* ws = carve(ws_bytes);
    const size_t xb = rows * s->nheads * s->headdim * e;
    const size_t dtb = rows * s->nheads * 4;
    const size_t bcb = rows * s->ngroups * s->dstate * e;
    const size_t stb = nseq_eff * s->nheads * s->headdim * s->dstate * 4;
    char* dx = carve(xb);
    char* dy = carve(xb);
    char* ddt = carve(dtb);
    char* dA = carve(s->nheads * 4);
    char* dD = carve(s->nheads * 4);
    char* dB = carve(bcb);
    char* dC = carve(bcb);
    char* dinit = carve(stb);
    char* dfinal = carve(stb);
    char* dcu = carve((nseq_eff + 1) * 4);
    cudaError_t err = cudaSuccess;
    auto h2d = [&](void* dst, const void* src, size_t bytes) {
        if (err == cudaSuccess && src && bytes) err = cudaMemcpyAsync(dst, src, bytes, cudaMemcpyHostToDevice, st);
    };
    h2d(dx, x, xb);
    h2d(ddt, dt, dtb);
    h2d(dA, A, s->nheads * 4);
    h2d(dD, D, s->nheads * 4);
    h2d(dB, B, bcb);
    h2d(dC, C, bcb);
    h2d(dinit, initial_state, stb);
    h2d(dcu, cu_seqlens, (nseq_eff + 1) * 4);
    if (err != cudaSuccess) return SSD_ERR_CUDA;
    rc = ssd_forward_ex(s, dtype, flags, dx, (const float*)ddt, (const float*)dA, dB, dC,
                        D ? (const float*)dD : nullptr, chunk, initial_state ? (const float*)dinit : nullptr,
                        varlen ? (const int32_t*)dcu : nullptr, nseq, dy, final_state ? (float*)dfinal : nullptr, ws,
                        ws_bytes, stream);
    if (rc != SSD_OK) return rc;
    if (cudaMemcpyAsync(y, dy, xb, cudaMemcpyDeviceToHost, st) != cudaSuccess) return SSD_ERR_CUDA;
    if (final_state && cudaMemcpyAsync(final_state, dfinal, stb, cudaMemcpyDeviceToHost, st) != cudaSuccess)
        return SSD_ERR_CUDA;
    if (cudaStreamSynchronize(st) != cudaSuccess) return SSD_ERR_CUDA;
    return ssd_status(ws, stream);
}

int ssd_forward_host(const ssd_shape* s, ssd_dtype dtype, const void* x, const float* dt, const float* A,
                     const void* B, const void* C, const float* D, int chunk, const float* initial_state,
                     const int32_t* cu_seqlens, int nseq, void* y, float* final_state, void* device_buffer,
                     size_t device_buffer_bytes, void* stream) {
    return ssd_forward_host_ex(s, dtype, 0u, x, dt, A, B, C, D, chunk, initial_state, cu_seqlens, nseq, y,
                               final_state, device_buffer, device_buffer_bytes, stream);
}

size_t ssd_slice_workspace_size(const ssd_shape* s) {
    if (!s || s->batch < 0 || s->seqlen < 0 || s->nheads <= 0 || s->headdim <= 0 || s->dstate <= 0 ||
        s->ngroups <= 0 || s->nheads % s->ngroups != 0)
        return 0;
    return slice_ws_bytes(*s);
}

namespace {
int check_slice(const ssd_shape* s, const void* workspace, size_t workspace_bytes, int* num_sms) {
    if (!ssd_slice_workspace_size(s)) return SSD_ERR_INVALID_ARG;
    if (s->batch * s->seqlen > (int64_t)INT32_MAX / 2 || s->nheads > 65535) return SSD_ERR_UNSUPPORTED;
    if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u) || workspace_bytes < slice_ws_bytes(*s))
        return SSD_ERR_WORKSPACE;
    g_err_detail[0] = '\0';
    return check_device(num_sms);
}
}  // namespace

int ssd_slice_decay(const ssd_shape* s, const float* dt, const float* A, float* decay, void* workspace,
                    size_t workspace_bytes, void* stream) {
    if (!s) return SSD_ERR_INVALID_ARG;
    if ((s->batch * s->seqlen > 0 && !dt) || !A || !decay) return SSD_ERR_INVALID_ARG;
    if ((dt && !aligned16(dt)) || !aligned16(A) || !aligned16(decay)) return SSD_ERR_INVALID_ARG;
    int num_sms = 0;
    const int rc = check_slice(s, workspace, workspace_bytes, &num_sms);
    if (rc != SSD_OK) return rc;
    const cudaError_t e = launch_slice_decay(*s, dt, A, decay, static_cast<char*>(workspace),
                                             static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? SSD_OK : SSD_ERR_CUDA;
}

int ssd_slice_correct(const ssd_shape* s, ssd_dtype dtype, const float* dt, const float* A, const void* C,
                      const float* h_in, void* y, float* final_state, void* workspace, size_t workspace_bytes,
                      void* stream) {
    if (!s) return SSD_ERR_INVALID_ARG;
    if (dtype != SSD_F32 && dtype != SSD_BF16) return SSD_ERR_INVALID_ARG;
    const bool any = s->batch * s->seqlen > 0;
    if ((any && (!dt || !C || !y)) || !A || !h_in) return SSD_ERR_INVALID_ARG;
    const void* ptrs[] = {dt, A, C, h_in, y, final_state};
    for (const void* p : ptrs)
        if (p && !aligned16(p)) return SSD_ERR_INVALID_ARG;
    if (!ssd_slice_workspace_size(s)) return SSD_ERR_INVALID_ARG;
    if (!use_fused_path(*s, dtype)) return SSD_ERR_UNSUPPORTED;
    int num_sms = 0;
    const int rc = check_slice(s, workspace, workspace_bytes, &num_sms);
    if (rc != SSD_OK) return rc;
    const cudaError_t e = launch_slice_correct(*s, dt, A, C, h_in, y, final_state, static_cast<char*>(workspace),
                                               static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? SSD_OK : SSD_ERR_CUDA;
}

int ssd_status(const void* workspace, void* stream) {
    if (!workspace) return SSD_ERR_WORKSPACE;
    int v = SSD_ERR_CUDA;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (cudaMemcpyAsync(&v, workspace, sizeof(int), cudaMemcpyDeviceToHost, st) != cudaSuccess) return SSD_ERR_CUDA;
    if (cudaStreamSynchronize(st) != cudaSuccess) return SSD_ERR_CUDA;
    return v;
}

const char* ssd_last_error_detail(void) { return g_err_detail; }

const char* ssd_status_string(int code) {
    switch (code) {
        case SSD_OK: return "ok";
        case SSD_ERR_INVALID_ARG: return "invalid argument";
        case SSD_ERR_UNSUPPORTED: return "unsupported size, chunk or device";
        case SSD_ERR_CUDA: return "CUDA error";
        case SSD_ERR_TIMEOUT: return "device-side wait timed out";
        case SSD_ERR_WORKSPACE: return "workspace missing, misaligned or too small";
        default: return "unknown status";
    }
}

}  // extern "C"
