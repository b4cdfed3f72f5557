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
#include "ssd_norm.cuh"
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

namespace {

// The host entry point on a large dense bf16 batch runs as a pipeline of pieces, so that the copies in
// of piece k + 1, the forward of piece k and the copies out of piece k - 1 overlap (the copy engines
// move both directions at once): batch rows when there are several, else time slices of the one
// sequence, joined by the sequence-parallel hand-off ("LLM(十一)——Mamba" §3.7.2): every slice after the
// first runs from a zero state and is corrected for the state its predecessor ends with.
constexpr int kHostPieces = 4;
constexpr int64_t kHostPipelineBytes = int64_t(32) << 20;   // x bytes below which one piece is used

struct HostPlan {
    int K = 1;                        // pieces; 1: one piece, no pipeline
    bool time = false;                // time slices of one sequence (else groups of batch rows)
    int64_t cut[kHostPieces + 1];     // piece k: batch rows, or tokens, [cut[k], cut[k + 1])
    int64_t len = 0;                  // the largest piece
};

// Time slices end at 30, 60 and 85 % of the sequence (multiples of the 128-token tile): the last piece's
// forward and copies out are what the pipeline cannot overlap, so it is the smallest.
HostPlan host_plan(const ssd_shape& s, ssd_dtype dtype, bool varlen) {
    HostPlan h;
    if (dtype != SSD_BF16 || varlen || !use_fused_path(s, dtype)) return h;
    if (s.batch * s.seqlen * s.nheads * s.headdim * 2 < kHostPipelineBytes) return h;
    if (s.batch >= 2) {
        const int64_t len = (s.batch + kHostPieces - 1) / kHostPieces;
        h.K = (int)((s.batch + len - 1) / len);
        for (int k = 0; k <= h.K; ++k) h.cut[k] = k * len < s.batch ? k * len : s.batch;
    } else if (s.seqlen >= kHostPieces * 1024) {
        static constexpr int kPct[kHostPieces + 1] = {0, 30, 60, 85, 100};
        h.time = true;
        h.K = kHostPieces;
        for (int k = 0; k < kHostPieces; ++k) h.cut[k] = s.seqlen * kPct[k] / 100 / 128 * 128;
        h.cut[kHostPieces] = s.seqlen;
    } else {
        return h;
    }
    for (int k = 0; k < h.K; ++k)
        if (h.cut[k + 1] - h.cut[k] > h.len) h.len = h.cut[k + 1] - h.cut[k];
    return h;
}

// the shape of the largest piece
ssd_shape piece_shape(const ssd_shape& s, const HostPlan& h) {
    ssd_shape p = s;
    if (h.K > 1) {
        if (h.time) p.seqlen = h.len;
        else p.batch = h.len;
    }
    return p;
}

}  // namespace

size_t ssd_host_buffer_size(const ssd_shape* s, ssd_dtype dtype, int chunk, int nseq) {
    const size_t ws1 = ssd_workspace_size(s, dtype, chunk, nseq);
    if (!ws1) return 0;
    const int64_t rows = s->batch * s->seqlen;
    const int64_t nseq_eff = nseq > 0 ? nseq : s->batch;
    const size_t e = elt(dtype);
    const HostPlan h = host_plan(*s, dtype, nseq > 0);
    size_t tot = 0;
    if (h.K > 1) {
        const ssd_shape ps = piece_shape(*s, h);
        tot += align256(ssd_workspace_size(&ps, dtype, chunk, 0)) * h.K;    // one workspace per piece
        if (h.time) {
            tot += align256(ssd_slice_workspace_size(&ps)) * h.K;           // the slices' corrections
            tot += align256(s->nheads * s->headdim * s->dstate * 4) * h.K;  // every slice's final state
        }
        tot += align256(2 * kHostPieces * sizeof(int));                     // the pieces' status words
    } else {
        tot += ws1;
    }
    tot += align256(rows * s->nheads * s->headdim * e) * 2;                 // x, y
    tot += align256(rows * s->nheads * 4);                                  // dt
    tot += align256(s->nheads * 4) * 2;                                     // A, D
    tot += align256(rows * s->ngroups * s->dstate * e) * 2;                 // B, C
    tot += align256(nseq_eff * s->nheads * s->headdim * s->dstate * 4) * 2; // initial, final
    tot += align256((nseq_eff + 1) * 4);                                    // cu_seqlens
    return tot;
}

namespace {

// The pipelined host call (see HostPlan). The caller's stream runs the forwards; one internal stream
// copies in and one copies out, ordered by events; everything is finished when it returns.
int host_pipelined(const ssd_shape* s, const HostPlan& h, unsigned flags, const void* x, const float* dt,
                   const float* A, const void* B, const void* C, const float* D, int chunk,
                   const float* initial_state, void* y, float* final_state, char* base, cudaStream_t st) {
    const int64_t H = s->nheads, P = s->headdim, N = s->dstate, G = s->ngroups, T = s->seqlen;
    const size_t e = 2;
    const size_t xrow = (size_t)H * P * e, dtrow = (size_t)H * 4, bcrow = (size_t)G * N * e;
    const size_t st1 = (size_t)H * P * N * 4;     // one sequence's state
    const int64_t rows = s->batch * T;
    size_t off = 0;
    auto carve = [&](size_t bytes) { char* p = base + off; off += align256(bytes); return p; };
    const ssd_shape ps = piece_shape(*s, h);
    const size_t wsb = ssd_workspace_size(&ps, SSD_BF16, chunk, 0);
    const size_t swsb = h.time ? ssd_slice_workspace_size(&ps) : 0;
    std::vector<char*> ws(h.K), sws(h.K, nullptr), fin(h.K, nullptr);
    for (int k = 0; k < h.K; ++k) ws[k] = carve(wsb);
    if (h.time)
        for (int k = 0; k < h.K; ++k) { sws[k] = carve(swsb); fin[k] = carve(st1); }
    char* dx = carve(rows * xrow);
    char* dy = carve(rows * xrow);
    char* ddt = carve(rows * dtrow);
    char* dA = carve(H * 4);
    char* dD = carve(H * 4);
    char* dB = carve(rows * bcrow);
    char* dC = carve(rows * bcrow);
    char* dinit = carve(s->batch * st1);
    char* dfinal = carve(s->batch * st1);
    int* dstat = reinterpret_cast<int*>(carve(2 * kHostPieces * sizeof(int)));   // every call's status word

    cudaStream_t si = nullptr, so = nullptr;
    std::vector<cudaEvent_t> ev(2 * h.K + 1, nullptr);
    cudaError_t err = cudaStreamCreateWithFlags(&si, cudaStreamNonBlocking);
    if (err == cudaSuccess) err = cudaStreamCreateWithFlags(&so, cudaStreamNonBlocking);
    for (auto& v : ev)
        if (err == cudaSuccess) err = cudaEventCreateWithFlags(&v, cudaEventDisableTiming);
    int rc = SSD_OK;
    auto h2d = [&](void* dst, const void* src, size_t bytes) {
        if (err == cudaSuccess && src && bytes) err = cudaMemcpyAsync(dst, src, bytes, cudaMemcpyHostToDevice, si);
    };
    auto d2h = [&](void* dst, const void* src, size_t bytes) {
        if (err == cudaSuccess && dst && bytes) err = cudaMemcpyAsync(dst, src, bytes, cudaMemcpyDeviceToHost, so);
    };
    // the copies in wait for the caller's earlier work on its stream (it may still use the buffer)
    if (err == cudaSuccess) err = cudaEventRecord(ev[0], st);
    if (err == cudaSuccess) err = cudaStreamWaitEvent(si, ev[0], 0);
    h2d(dA, A, H * 4);
    h2d(dD, D, H * 4);
    h2d(dinit, initial_state, s->batch * st1);
    // piece k: rows [r0, r0 + nr) of the (batch x time) row order, sequences [q0, q0 + nq)
    auto piece = [&](int k, int64_t* r0, int64_t* nr, int64_t* q0, ssd_shape* pk) {
        *pk = *s;
        const int64_t a0 = h.cut[k], n = h.cut[k + 1] - h.cut[k];
        if (h.time) {
            pk->seqlen = n;
            *r0 = a0; *nr = n; *q0 = 0;
        } else {
            pk->batch = n;
            *r0 = a0 * T; *nr = n * T; *q0 = a0;
        }
    };
    for (int k = 0; k < h.K; ++k) {
        int64_t r0, nr, q0;
        ssd_shape pk;
        piece(k, &r0, &nr, &q0, &pk);
        h2d(dx + r0 * xrow, static_cast<const char*>(x) + r0 * xrow, nr * xrow);
        h2d(ddt + r0 * dtrow, reinterpret_cast<const char*>(dt) + r0 * dtrow, nr * dtrow);
        h2d(dB + r0 * bcrow, static_cast<const char*>(B) + r0 * bcrow, nr * bcrow);
        h2d(dC + r0 * bcrow, static_cast<const char*>(C) + r0 * bcrow, nr * bcrow);
        if (err == cudaSuccess) err = cudaEventRecord(ev[1 + k], si);
    }
    for (int k = 0; k < h.K && err == cudaSuccess && rc == SSD_OK; ++k) {
        int64_t r0, nr, q0;
        ssd_shape pk;
        piece(k, &r0, &nr, &q0, &pk);
        err = cudaStreamWaitEvent(st, ev[1 + k], 0);
        if (err != cudaSuccess) break;
        const void* px = dx + r0 * xrow;
        const float* pdt = reinterpret_cast<const float*>(ddt + r0 * dtrow);
        const void* pB = dB + r0 * bcrow;
        const void* pC = dC + r0 * bcrow;
        void* py = dy + r0 * xrow;
        const float* pD = D ? reinterpret_cast<const float*>(dD) : nullptr;
        if (!h.time) {
            rc = ssd_forward_ex(&pk, SSD_BF16, flags, px, pdt, reinterpret_cast<const float*>(dA), pB, pC, pD, chunk,
                                initial_state ? reinterpret_cast<const float*>(dinit + q0 * st1) : nullptr, nullptr, 0,
                                py, final_state ? reinterpret_cast<float*>(dfinal + q0 * st1) : nullptr, ws[k], wsb, st);
        } else {
            const float* h0 = (k == 0 && initial_state) ? reinterpret_cast<const float*>(dinit) : nullptr;
            rc = ssd_forward_ex(&pk, SSD_BF16, flags, px, pdt, reinterpret_cast<const float*>(dA), pB, pC, pD, chunk,
                                h0, nullptr, 0, py, reinterpret_cast<float*>(fin[k]), ws[k], wsb, st);
            if (rc == SSD_OK && k > 0)
                rc = ssd_slice_correct(&pk, SSD_BF16, pdt, reinterpret_cast<const float*>(dA), pC,
                                       reinterpret_cast<const float*>(fin[k - 1]), py, reinterpret_cast<float*>(fin[k]),
                                       sws[k], swsb, st);
        }
        if (rc != SSD_OK) break;
        // the status words of this piece's calls, gathered so that one copy reads them all at the end
        err = cudaMemcpyAsync(dstat + 2 * k, ws[k], sizeof(int), cudaMemcpyDeviceToDevice, st);
        if (err == cudaSuccess)
            err = cudaMemcpyAsync(dstat + 2 * k + 1, h.time && k > 0 ? sws[k] : ws[k], sizeof(int),
                                  cudaMemcpyDeviceToDevice, st);
        if (err != cudaSuccess) break;
        err = cudaEventRecord(ev[1 + h.K + k], st);
        if (err == cudaSuccess) err = cudaStreamWaitEvent(so, ev[1 + h.K + k], 0);
        d2h(static_cast<char*>(y) + r0 * xrow, dy + r0 * xrow, nr * xrow);
        if (final_state && !h.time) d2h(reinterpret_cast<char*>(final_state) + q0 * st1, dfinal + q0 * st1, pk.batch * st1);
    }
    if (final_state && h.time && rc == SSD_OK) d2h(final_state, fin[h.K - 1], st1);
    // everything issued has finished before the buffers are handed back, whatever happened above
    const cudaError_t e1 = si ? cudaStreamSynchronize(si) : cudaSuccess;
    const cudaError_t e2 = cudaStreamSynchronize(st);
    const cudaError_t e3 = so ? cudaStreamSynchronize(so) : cudaSuccess;
    for (auto& v : ev)
        if (v) cudaEventDestroy(v);
    if (si) cudaStreamDestroy(si);
    if (so) cudaStreamDestroy(so);
    if (rc != SSD_OK) return rc;
    if (err != cudaSuccess || e1 != cudaSuccess || e2 != cudaSuccess || e3 != cudaSuccess) {
        note_cuda_error("pipelined host call", err != cudaSuccess ? err : (e1 != cudaSuccess ? e1 : (e2 != cudaSuccess ? e2 : e3)));
        return SSD_ERR_CUDA;
    }
    int stat[2 * kHostPieces];
    if (note_cuda_error("status copy", cudaMemcpy(stat, dstat, 2 * h.K * sizeof(int), cudaMemcpyDeviceToHost)) !=
        cudaSuccess)
        return SSD_ERR_CUDA;
    for (int k = 0; k < 2 * h.K; ++k)
        if (stat[k] != SSD_OK) return stat[k];
    return SSD_OK;
}

}  // namespace

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
    const HostPlan hp = host_plan(*s, dtype, varlen);
    if (hp.K > 1)
        return host_pipelined(s, hp, flags, x, dt, A, B, C, D, chunk, initial_state, y, final_state, base, st);
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

namespace {

// argument checks shared by the device and host forms of the gate and normalization
int check_norm(const ssd_shape* s, float eps, int groups) {
    if (!s || s->batch < 0 || s->seqlen < 0 || s->nheads <= 0 || s->headdim <= 0) return SSD_ERR_INVALID_ARG;
    if (groups <= 0 || !(eps >= 0.f) || !(eps < 3.0e38f)) return SSD_ERR_INVALID_ARG;
    const int64_t channels = s->nheads * s->headdim;
    if (channels % groups != 0) return SSD_ERR_INVALID_ARG;
    if ((channels / groups) % 8 != 0 || channels > norm_max_channels()) return SSD_ERR_UNSUPPORTED;
    return SSD_OK;
}

// The host form on a large block of tokens (y of at least 32 MB) runs as a pipeline over groups of rows,
// which are independent: the copies in of group k + 1, the kernel on group k and the copy out of group
// k - 1 overlap. The caller's stream runs the kernels; one internal stream copies in and one copies out,
// ordered by events. out is written in place over the device copy of y.
constexpr int kNormPieces = 4;
constexpr size_t kNormPipelineBytes = size_t(32) << 20;

int norm_host_run(int64_t rows, int64_t channels, const void* y, const void* z, const float* weight, float eps,
                  int groups, void* out, char* dy, char* dz, char* dw, int num_sms, cudaStream_t st) {
    const size_t rowb = (size_t)channels * 2;
    const bool pipe = rows * rowb >= kNormPipelineBytes && rows >= kNormPieces;
    const int64_t len = pipe ? (rows + kNormPieces - 1) / kNormPieces : rows;
    const int K = (int)((rows + len - 1) / len);
    cudaStream_t si = nullptr, so = nullptr;
    std::vector<cudaEvent_t> ev(2 * K + 1, nullptr);
    cudaError_t err = cudaStreamCreateWithFlags(&si, cudaStreamNonBlocking);
    if (err == cudaSuccess) err = cudaStreamCreateWithFlags(&so, cudaStreamNonBlocking);
    for (auto& v : ev)
        if (err == cudaSuccess) err = cudaEventCreateWithFlags(&v, cudaEventDisableTiming);
    auto h2d = [&](void* dst, const void* src, size_t bytes) {
        if (err == cudaSuccess && bytes) err = cudaMemcpyAsync(dst, src, bytes, cudaMemcpyHostToDevice, si);
    };
    // the copies in wait for the caller's earlier work on its stream (it may still use the buffer)
    if (err == cudaSuccess) err = cudaEventRecord(ev[0], st);
    if (err == cudaSuccess) err = cudaStreamWaitEvent(si, ev[0], 0);
    if (weight) h2d(dw, weight, (size_t)channels * 4);
    for (int k = 0; k < K; ++k) {
        const int64_t r0 = k * len, rk = rows - r0 < len ? rows - r0 : len;
        h2d(dy + r0 * rowb, static_cast<const char*>(y) + r0 * rowb, rk * rowb);
        if (z) h2d(dz + r0 * rowb, static_cast<const char*>(z) + r0 * rowb, rk * rowb);
        if (err == cudaSuccess) err = cudaEventRecord(ev[1 + k], si);
    }
    for (int k = 0; k < K && err == cudaSuccess; ++k) {
        const int64_t r0 = k * len, rk = rows - r0 < len ? rows - r0 : len;
        err = cudaStreamWaitEvent(st, ev[1 + k], 0);
        if (err == cudaSuccess)
            err = launch_gated_rmsnorm(dy + r0 * rowb, z ? dz + r0 * rowb : nullptr,
                                       weight ? reinterpret_cast<const float*>(dw) : nullptr, eps, rk, channels,
                                       groups, dy + r0 * rowb, num_sms, st);
        if (err == cudaSuccess) err = cudaEventRecord(ev[1 + K + k], st);
        if (err == cudaSuccess) err = cudaStreamWaitEvent(so, ev[1 + K + k], 0);
        if (err == cudaSuccess)
            err = cudaMemcpyAsync(static_cast<char*>(out) + r0 * rowb, dy + r0 * rowb, rk * rowb,
                                  cudaMemcpyDeviceToHost, so);
    }
    // everything issued has finished before the buffers are handed back, whatever happened above
    const cudaError_t e1 = si ? cudaStreamSynchronize(si) : cudaSuccess;
    const cudaError_t e2 = cudaStreamSynchronize(st);
    const cudaError_t e3 = so ? cudaStreamSynchronize(so) : cudaSuccess;
    for (auto& v : ev)
        if (v) cudaEventDestroy(v);
    if (si) cudaStreamDestroy(si);
    if (so) cudaStreamDestroy(so);
    const cudaError_t ef = err != cudaSuccess ? err : (e1 != cudaSuccess ? e1 : (e2 != cudaSuccess ? e2 : e3));
    return note_cuda_error("gated rmsnorm host pipeline", ef) == cudaSuccess ? SSD_OK : SSD_ERR_CUDA;
}

}  // namespace

extern "C" {

int ssd_gated_rmsnorm(const ssd_shape* s, const void* y, const void* z, const float* weight, float eps, int groups,
                      void* out, void* stream) {
    int rc = check_norm(s, eps, groups);
    if (rc != SSD_OK) return rc;
    const int64_t rows = s->batch * s->seqlen, channels = s->nheads * s->headdim;
    if (rows > 0 && (!y || !out)) return SSD_ERR_INVALID_ARG;
    const void* ptrs[] = {y, z, weight, out};
    for (const void* p : ptrs)
        if (p && !aligned16(p)) return SSD_ERR_INVALID_ARG;
    if (rows == 0) return SSD_OK;
    int num_sms = 0;
    rc = check_device(&num_sms);
    if (rc != SSD_OK) return rc;
    const cudaError_t e = launch_gated_rmsnorm(y, z, weight, eps, rows, channels, groups, out, num_sms,
                                               static_cast<cudaStream_t>(stream));
    return note_cuda_error("gated rmsnorm launch", e) == cudaSuccess ? SSD_OK : SSD_ERR_CUDA;
}

size_t ssd_gated_rmsnorm_host_buffer_size(const ssd_shape* s, int gated) {
    if (!s || s->batch < 0 || s->seqlen < 0 || s->nheads <= 0 || s->headdim <= 0) return 0;
    const size_t yb = (size_t)(s->batch * s->seqlen) * s->nheads * s->headdim * 2;
    const size_t tot = align256(yb) * (gated ? 2 : 1) + align256((size_t)s->nheads * s->headdim * 4);
    return tot > 0 ? tot : 256;
}

int ssd_gated_rmsnorm_host(const ssd_shape* s, const void* y, const void* z, const float* weight, float eps,
                           int groups, void* out, void* device_buffer, size_t device_buffer_bytes, void* stream) {
    int rc = check_norm(s, eps, groups);
    if (rc != SSD_OK) return rc;
    const size_t need = ssd_gated_rmsnorm_host_buffer_size(s, z != nullptr);
    if (!device_buffer || (reinterpret_cast<uintptr_t>(device_buffer) & 255u) || device_buffer_bytes < need)
        return SSD_ERR_WORKSPACE;
    const int64_t rows = s->batch * s->seqlen, channels = s->nheads * s->headdim;
    if (rows == 0) return SSD_OK;
    if (!y || !out) return SSD_ERR_INVALID_ARG;
    int num_sms = 0;
    rc = check_device(&num_sms);
    if (rc != SSD_OK) return rc;
    const size_t yb = align256((size_t)rows * channels * 2);
    char* dy = static_cast<char*>(device_buffer);
    char* dz = z ? dy + yb : nullptr;
    char* dw = dy + yb * (z ? 2 : 1);
    return norm_host_run(rows, channels, y, z, weight, eps, groups, out, dy, dz, dw, num_sms,
                         static_cast<cudaStream_t>(stream));
}

}  // extern "C"
