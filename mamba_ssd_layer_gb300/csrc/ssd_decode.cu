// ssd_decode.cu -- the one-token recurrent step of the SSD layer on a batch of carried states:
//
//   for every row b and head h (group g = h / (H/G)):
//     a       = exp(dt[b,h] * A[h])
//     S[b,h]  = a * S[b,h] + x[b,h,:] (outer) B[b,g,:]          (P x N, fp32)
//     y[b,h,:] = S[b,h] . C[b,g,:] + D[h] * x[b,h,:]
//
// This is the recurrent (autoregressive inference) mode of the selective SSM with a scalar A
// ("Transformers是SSMs：通过结构化状态空间对偶性的广义模型和高效算法(一)" §2.1; "LLM(十一)——Mamba"
// §3.1.1-3.1.2, and §3.5.3 for its per-token cost; "Mamba-2 状态空间对偶性理论" §1.2).
//
// The step moves the whole state in and out once and does 4 flops per state element, so it is
// bound by HBM bandwidth. The kernel streams the state in 16-byte vectors: a row of the state
// (N / E chunks of E = 16 bytes / element size) is spread over L lanes (L a power of two, the
// smallest that is >= N / E, at most 32), each lane holding one or two chunks, and a warp covers
// 32/L rows at a time.
// The state may be stored as fp32 or as bf16 (then a 16-byte chunk holds 8 elements; the update is
// computed in fp32, y from the unrounded new state, and only the stored state is rounded).
// Every thread loads its four rows before using any of them, so that enough loads are in flight;
// CTAs are small (two warps), so that many are resident per SM and a CTA's set-up is cheap.
// The dot product with C is reduced across the row's L lanes with xor shuffles.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <vector>

#include "ssd.h"
#include "ssd_internal.cuh"

namespace ssd {
namespace {

constexpr int kDecThreads = 64;
constexpr int kDecWarps = kDecThreads / 32;
constexpr int kDecRowsPerThread = 4;

struct DecodeArgs {
    const void* x;          // (batch, H, P) storage type
    const float* dt;        // (batch, H)
    const float* A;         // (H)
    const void* B;          // (batch, G, N) storage type
    const void* C;
    const float* D;         // (H) or null
    const void* state;      // (batch, H, P, N) state type
    void* new_state;        // may alias state
    void* y;                // (batch, H, P) storage type
    int H, P, N, G;
    int heads_per_group;    // H / G
    int L;                  // lanes per state row
    int rows_per_cta;       // kDecWarps * (32 / L) * kDecRowsPerThread
    int row_blocks;         // ceil(P / rows_per_cta)
};

template <typename T>
__device__ __forceinline__ float to_f32(T v);
template <>
__device__ __forceinline__ float to_f32<float>(float v) { return v; }
template <>
__device__ __forceinline__ float to_f32<__nv_bfloat16>(__nv_bfloat16 v) { return __bfloat162float(v); }

template <typename T>
__device__ __forceinline__ T from_f32(float v);
template <>
__device__ __forceinline__ float from_f32<float>(float v) { return v; }
template <>
__device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float v) { return __float2bfloat16_rn(v); }

// E consecutive elements (4 or 8, starting at a multiple of E) as fp32
template <typename T, int E>
__device__ __forceinline__ void load_vec(const T* p, float (&v)[E]) {
    if constexpr (sizeof(T) == 4) {
#pragma unroll
        for (int k = 0; k < E; k += 4) {
            const float4 f = *reinterpret_cast<const float4*>(p + k);
            v[k] = f.x; v[k + 1] = f.y; v[k + 2] = f.z; v[k + 3] = f.w;
        }
    } else if constexpr (E == 4) {
        const uint2 u = *reinterpret_cast<const uint2*>(p);
        const float2 lo = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u.x));
        const float2 hi = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u.y));
        v[0] = lo.x; v[1] = lo.y; v[2] = hi.x; v[3] = hi.y;
    } else {
        const uint4 u = *reinterpret_cast<const uint4*>(p);
        const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w[k]));
            v[2 * k] = f.x; v[2 * k + 1] = f.y;
        }
    }
}

// one 16-byte chunk of a state row (E = 4 fp32 or 8 bf16) as fp32, from its raw bytes (the chunks
// are loaded raw, streamed, and unpacked only when their row is computed: fewer live registers)
template <typename TS, int E>
__device__ __forceinline__ void unpack_state(const uint4 u, float (&v)[E]) {
    if constexpr (sizeof(TS) == 4) {
        v[0] = __uint_as_float(u.x); v[1] = __uint_as_float(u.y); v[2] = __uint_as_float(u.z); v[3] = __uint_as_float(u.w);
    } else {
        const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w[k]));
            v[2 * k] = f.x; v[2 * k + 1] = f.y;
        }
    }
}
template <typename TS, int E>
__device__ __forceinline__ void store_state(TS* p, const float (&v)[E]) {
    uint4 u;
    if constexpr (sizeof(TS) == 4) {
        u = make_uint4(__float_as_uint(v[0]), __float_as_uint(v[1]), __float_as_uint(v[2]), __float_as_uint(v[3]));
    } else {
        uint32_t w[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const __nv_bfloat162 b = __floats2bfloat162_rn(v[2 * k], v[2 * k + 1]);
            w[k] = *reinterpret_cast<const uint32_t*>(&b);
        }
        u = make_uint4(w[0], w[1], w[2], w[3]);
    }
    __stcs(reinterpret_cast<uint4*>(p), u);
}

// T: storage type of x, B, C, y; TS: storage type of the state; CI: 16-byte column chunks per lane
// (N / E <= CI * L, E = 16 / sizeof(TS) state elements per chunk); kScaleX: the input term is dt x
template <typename T, typename TS, int CI, bool kScaleX>
__global__ void __launch_bounds__(kDecThreads) ssd_decode_kernel(const DecodeArgs a) {
    constexpr int E = 16 / (int)sizeof(TS);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int L = a.L;
    const int seg = lane / L, cl = lane % L;          // row slot within the warp, lane within the row
    const int rows_per_pass = kDecWarps * (32 / L);
    const uint32_t unit = blockIdx.x;                 // < 2^31 (checked at launch): 32-bit index math
    const int rb = (int)(unit % (uint32_t)a.row_blocks);
    const uint32_t bh32 = unit / (uint32_t)a.row_blocks;
    const int h = (int)(bh32 % (uint32_t)a.H);
    const int64_t bh = bh32;                          // b * H + h
    const int64_t b = bh32 / (uint32_t)a.H;
    const int g = h / a.heads_per_group;
    const int nch = a.N / E;                          // 16-byte chunks per state row

    const float dtv = a.dt[bh];
    const float decay = expf(dtv * a.A[h]);
    const float in_scale = kScaleX ? dtv : 1.f;           // the skip term keeps the unscaled x
    const float dskip = a.D ? a.D[h] : 0.f;

    const T* Bp = static_cast<const T*>(a.B) + (b * a.G + g) * a.N;
    const T* Cp = static_cast<const T*>(a.C) + (b * a.G + g) * a.N;
    float bv[CI][E], cv[CI][E];
#pragma unroll
    for (int j = 0; j < CI; ++j) {
        const int c = cl + j * L;
        if (c < nch) {
            load_vec<T, E>(Bp + E * c, bv[j]);
            load_vec<T, E>(Cp + E * c, cv[j]);
        } else {
#pragma unroll
            for (int e = 0; e < E; ++e) { bv[j][e] = 0.f; cv[j][e] = 0.f; }
        }
    }

    const int64_t row_base = bh * a.P;                // first state row of (b, h)
    const T* xp = static_cast<const T*>(a.x) + row_base;
    const TS* sp = static_cast<const TS*>(a.state);
    TS* np = static_cast<TS*>(a.new_state);
    int p[kDecRowsPerThread];
    float xv[kDecRowsPerThread];
    uint4 sraw[kDecRowsPerThread][CI];
#pragma unroll
    for (int u = 0; u < kDecRowsPerThread; ++u) {
        p[u] = rb * a.rows_per_cta + u * rows_per_pass + warp * (32 / L) + seg;
        xv[u] = p[u] < a.P ? to_f32<T>(xp[p[u]]) : 0.f;
#pragma unroll
        for (int j = 0; j < CI; ++j) {
            const int c = cl + j * L;
            sraw[u][j] = make_uint4(0u, 0u, 0u, 0u);
            if (p[u] < a.P && c < nch)
                sraw[u][j] = __ldcs(reinterpret_cast<const uint4*>(sp + (row_base + p[u]) * a.N + E * c));
        }
    }
    T* yp = static_cast<T*>(a.y) + row_base;
    const float2 dd = make_float2(decay, decay);
#pragma unroll
    for (int u = 0; u < kDecRowsPerThread; ++u) {
        const float2 xx = make_float2(in_scale * xv[u], in_scale * xv[u]);
        float2 acc2 = make_float2(0.f, 0.f);              // packed fp32 pairs: half the FP instructions
#pragma unroll
        for (int j = 0; j < CI; ++j) {
            const int c = cl + j * L;
            float sv[E], v[E];
            unpack_state<TS, E>(sraw[u][j], sv);
#pragma unroll
            for (int e = 0; e < E; e += 2) {
                const float2 nv = __ffma2_rn(dd, make_float2(sv[e], sv[e + 1]),
                                             __fmul2_rn(xx, make_float2(bv[j][e], bv[j][e + 1])));
                acc2 = __ffma2_rn(nv, make_float2(cv[j][e], cv[j][e + 1]), acc2);
                v[e] = nv.x;
                v[e + 1] = nv.y;
            }
            if (p[u] < a.P && c < nch) store_state<TS, E>(np + (row_base + p[u]) * a.N + E * c, v);
        }
        float acc = acc2.x + acc2.y;
        for (int off = L >> 1; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
        if (cl == 0 && p[u] < a.P) yp[p[u]] = from_f32<T>(fmaf(dskip, xv[u], acc));
    }
}

template <typename T, typename TS>
cudaError_t launch_decode_t(const DecodeArgs& a, int64_t units, bool scale_x, cudaStream_t st) {
    constexpr int E = 16 / (int)sizeof(TS);
    const int ci = (a.N / E + a.L - 1) / a.L;
    prof_launch();
    prof_begin(st, "ssd_decode_kernel");
    if (ci <= 1 && !scale_x)
        ssd_decode_kernel<T, TS, 1, false><<<(unsigned)units, kDecThreads, 0, st>>>(a);
    else if (ci <= 1)
        ssd_decode_kernel<T, TS, 1, true><<<(unsigned)units, kDecThreads, 0, st>>>(a);
    else if (!scale_x)
        ssd_decode_kernel<T, TS, 2, false><<<(unsigned)units, kDecThreads, 0, st>>>(a);
    else
        ssd_decode_kernel<T, TS, 2, true><<<(unsigned)units, kDecThreads, 0, st>>>(a);
    prof_end(st);
    return cudaGetLastError();
}

bool aligned(const void* p, uintptr_t n) { return (reinterpret_cast<uintptr_t>(p) & (n - 1)) == 0; }

int check_decode(const ssd_shape* s, ssd_dtype dtype) {
    if (!s) return SSD_ERR_INVALID_ARG;
    if (s->batch < 0 || s->seqlen != 1 || s->nheads <= 0 || s->headdim <= 0 || s->dstate <= 0 || s->ngroups <= 0)
        return SSD_ERR_INVALID_ARG;
    if (s->nheads % s->ngroups != 0) return SSD_ERR_INVALID_ARG;
    if (dtype != SSD_F32 && dtype != SSD_BF16) return SSD_ERR_INVALID_ARG;
    if (s->headdim > 256 || s->dstate > 256 || (s->dstate & 3) != 0) return SSD_ERR_UNSUPPORTED;
    if (s->batch * s->nheads > (int64_t)INT32_MAX / 2) return SSD_ERR_UNSUPPORTED;
    return SSD_OK;
}

size_t decode_elt(ssd_dtype d) { return d == SSD_F32 ? 4 : 2; }

}  // namespace
}  // namespace ssd

using namespace ssd;

extern "C" {

int ssd_decode_step_ex(const ssd_shape* s, ssd_dtype dtype, ssd_dtype state_dtype, unsigned flags, const void* x,
                       const float* dt, const float* A, const void* B, const void* C, const float* D,
                       const void* state, void* new_state, void* y, void* stream) {
    int rc = check_decode(s, dtype);
    if (rc != SSD_OK) return rc;
    if (flags & ~SSD_SCALE_X_BY_DT) return SSD_ERR_INVALID_ARG;
    if (state_dtype != SSD_F32 && state_dtype != SSD_BF16) return SSD_ERR_INVALID_ARG;
    if (state_dtype == SSD_BF16 && (s->dstate & 7) != 0) return SSD_ERR_UNSUPPORTED;
    if (s->batch == 0) return SSD_OK;
    if (!x || !dt || !A || !B || !C || !state || !new_state || !y) return SSD_ERR_INVALID_ARG;
    if (!aligned(state, 16) || !aligned(new_state, 16) || !aligned(B, 16) || !aligned(C, 16) ||
        !aligned(x, decode_elt(dtype)) || !aligned(y, decode_elt(dtype)) || !aligned(dt, 4) || !aligned(A, 4) ||
        (D && !aligned(D, 4)))
        return SSD_ERR_INVALID_ARG;
    // new_state either is state or does not overlap it
    const size_t stb = (size_t)s->batch * s->nheads * s->headdim * s->dstate * decode_elt(state_dtype);
    const char* s0 = static_cast<const char*>(state);
    const char* s1 = static_cast<const char*>(new_state);
    if (s0 != s1 && s1 < s0 + stb && s0 < s1 + stb) return SSD_ERR_INVALID_ARG;
    int dev = 0, major = 0, minor = 0;
    if (note_cuda_error("cudaGetDevice", cudaGetDevice(&dev)) != cudaSuccess) return SSD_ERR_CUDA;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
        return SSD_ERR_CUDA;
    if (major != 10 || minor != 3) return SSD_ERR_UNSUPPORTED;

    DecodeArgs a;
    a.x = x; a.dt = dt; a.A = A; a.B = B; a.C = C; a.D = D;
    a.state = state; a.new_state = new_state; a.y = y;
    a.H = (int)s->nheads; a.P = (int)s->headdim; a.N = (int)s->dstate; a.G = (int)s->ngroups;
    a.heads_per_group = a.H / a.G;
    const int nch = a.N / (state_dtype == SSD_F32 ? 4 : 8);   // 16-byte chunks per state row
    a.L = 1;
    while (a.L < nch && a.L < 32) a.L <<= 1;
    a.rows_per_cta = kDecWarps * (32 / a.L) * kDecRowsPerThread;
    a.row_blocks = (a.P + a.rows_per_cta - 1) / a.rows_per_cta;
    const int64_t units = s->batch * s->nheads * a.row_blocks;
    if (units > (int64_t)INT32_MAX) return SSD_ERR_UNSUPPORTED;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    cudaError_t e;
    const bool sx = (flags & SSD_SCALE_X_BY_DT) != 0;
    if (state_dtype == SSD_F32)
        e = dtype == SSD_F32 ? launch_decode_t<float, float>(a, units, sx, st)
                             : launch_decode_t<__nv_bfloat16, float>(a, units, sx, st);
    else
        e = dtype == SSD_F32 ? launch_decode_t<float, __nv_bfloat16>(a, units, sx, st)
                             : launch_decode_t<__nv_bfloat16, __nv_bfloat16>(a, units, sx, st);
    return note_cuda_error("decode launch", e) == cudaSuccess ? SSD_OK : SSD_ERR_CUDA;
}

int ssd_decode_step(const ssd_shape* s, ssd_dtype dtype, const void* x, const float* dt, const float* A,
                    const void* B, const void* C, const float* D, const float* state, float* new_state, void* y,
                    void* stream) {
    return ssd_decode_step_ex(s, dtype, SSD_F32, 0u, x, dt, A, B, C, D, state, new_state, y, stream);
}

size_t ssd_decode_host_buffer_size(const ssd_shape* s, ssd_dtype dtype) {
    if (check_decode(s, dtype) != SSD_OK) return 0;
    const size_t e = decode_elt(dtype);
    const size_t rows = (size_t)s->batch * s->nheads;
    size_t tot = 0;
    tot += align256(rows * s->headdim * e) * 2;                    // x, y
    tot += align256(rows * 4);                                     // dt
    tot += align256((size_t)s->nheads * 4) * 2;                    // A, D
    tot += align256((size_t)s->batch * s->ngroups * s->dstate * e) * 2;   // B, C
    tot += align256(rows * s->headdim * s->dstate * 4);            // state (updated in place)
    return tot > 0 ? tot : 256;
}

namespace {

// The host step on many carried states (a state of at least 32 MB) runs as a pipeline over groups of
// batch rows, which are independent: the copies in of group k + 1, the step of group k and the copies
// out of group k - 1 overlap (the copy engines move both directions at once). The caller's stream runs
// the steps; one internal stream copies in and one copies out, ordered by events.
constexpr int kDecodePieces = 4;
constexpr size_t kDecodePipelineBytes = size_t(32) << 20;

int decode_host_pipelined(const ssd_shape* s, ssd_dtype dtype, ssd_dtype state_dtype, unsigned flags, const void* x,
                          const float* dt, const float* A, const void* B, const void* C, const float* D,
                          const void* state, void* new_state, void* y, char* dx, char* dy, char* ddt, char* dA,
                          char* dD, char* dB, char* dC, char* dS, cudaStream_t st) {
    const size_t e = decode_elt(dtype);
    const size_t xrow = (size_t)s->nheads * s->headdim * e, dtrow = (size_t)s->nheads * 4;
    const size_t bcrow = (size_t)s->ngroups * s->dstate * e;
    const size_t srow = (size_t)s->nheads * s->headdim * s->dstate * decode_elt(state_dtype);
    const size_t hb = (size_t)s->nheads * 4;
    const int64_t len = (s->batch + kDecodePieces - 1) / kDecodePieces;
    const int K = (int)((s->batch + len - 1) / len);
    cudaStream_t si = nullptr, so = nullptr;
    std::vector<cudaEvent_t> ev(2 * K + 1, nullptr);
    cudaError_t err = cudaStreamCreateWithFlags(&si, cudaStreamNonBlocking);
    if (err == cudaSuccess) err = cudaStreamCreateWithFlags(&so, cudaStreamNonBlocking);
    for (auto& v : ev)
        if (err == cudaSuccess) err = cudaEventCreateWithFlags(&v, cudaEventDisableTiming);
    auto h2d = [&](void* dst, const void* src, size_t bytes) {
        if (err == cudaSuccess && src && bytes) err = cudaMemcpyAsync(dst, src, bytes, cudaMemcpyHostToDevice, si);
    };
    auto d2h = [&](void* dst, const void* src, size_t bytes) {
        if (err == cudaSuccess && bytes) err = cudaMemcpyAsync(dst, src, bytes, cudaMemcpyDeviceToHost, so);
    };
    // the copies in wait for the caller's earlier work on its stream (it may still use the buffer)
    if (err == cudaSuccess) err = cudaEventRecord(ev[0], st);
    if (err == cudaSuccess) err = cudaStreamWaitEvent(si, ev[0], 0);
    h2d(dA, A, hb);
    h2d(dD, D, hb);
    for (int k = 0; k < K; ++k) {
        const int64_t b0 = k * len, bk = s->batch - b0 < len ? s->batch - b0 : len;
        h2d(dx + b0 * xrow, static_cast<const char*>(x) + b0 * xrow, bk * xrow);
        h2d(ddt + b0 * dtrow, reinterpret_cast<const char*>(dt) + b0 * dtrow, bk * dtrow);
        h2d(dB + b0 * bcrow, static_cast<const char*>(B) + b0 * bcrow, bk * bcrow);
        h2d(dC + b0 * bcrow, static_cast<const char*>(C) + b0 * bcrow, bk * bcrow);
        h2d(dS + b0 * srow, static_cast<const char*>(state) + b0 * srow, bk * srow);
        if (err == cudaSuccess) err = cudaEventRecord(ev[1 + k], si);
    }
    int rc = SSD_OK;
    for (int k = 0; k < K && err == cudaSuccess; ++k) {
        const int64_t b0 = k * len, bk = s->batch - b0 < len ? s->batch - b0 : len;
        ssd_shape pk = *s;
        pk.batch = bk;
        err = cudaStreamWaitEvent(st, ev[1 + k], 0);
        if (err != cudaSuccess) break;
        rc = ssd_decode_step_ex(&pk, dtype, state_dtype, flags, dx + b0 * xrow,
                                reinterpret_cast<const float*>(ddt + b0 * dtrow), reinterpret_cast<const float*>(dA),
                                dB + b0 * bcrow, dC + b0 * bcrow, D ? reinterpret_cast<const float*>(dD) : nullptr,
                                dS + b0 * srow, dS + b0 * srow, dy + b0 * xrow, st);
        if (rc != SSD_OK) break;
        err = cudaEventRecord(ev[1 + K + k], st);
        if (err == cudaSuccess) err = cudaStreamWaitEvent(so, ev[1 + K + k], 0);
        d2h(static_cast<char*>(y) + b0 * xrow, dy + b0 * xrow, bk * xrow);
        d2h(static_cast<char*>(new_state) + b0 * srow, dS + b0 * srow, bk * srow);
    }
    // everything issued has finished before the buffers are handed back, whatever happened above
    const cudaError_t e1 = si ? cudaStreamSynchronize(si) : cudaSuccess;
    const cudaError_t e2 = cudaStreamSynchronize(st);
    const cudaError_t e3 = so ? cudaStreamSynchronize(so) : cudaSuccess;
    for (auto& v : ev)
        if (v) cudaEventDestroy(v);
    if (si) cudaStreamDestroy(si);
    if (so) cudaStreamDestroy(so);
    if (rc != SSD_OK) return rc;
    const cudaError_t ef = err != cudaSuccess ? err : (e1 != cudaSuccess ? e1 : (e2 != cudaSuccess ? e2 : e3));
    return note_cuda_error("decode host pipeline", ef) == cudaSuccess ? SSD_OK : SSD_ERR_CUDA;
}

}  // namespace

int ssd_decode_step_host_ex(const ssd_shape* s, ssd_dtype dtype, ssd_dtype state_dtype, unsigned flags,
                            const void* x, const float* dt, const float* A, const void* B, const void* C,
                            const float* D, const void* state, void* new_state, void* y, void* device_buffer,
                            size_t device_buffer_bytes, void* stream) {
    int rc = check_decode(s, dtype);
    if (rc != SSD_OK) return rc;
    if (flags & ~SSD_SCALE_X_BY_DT) return SSD_ERR_INVALID_ARG;
    if (state_dtype != SSD_F32 && state_dtype != SSD_BF16) return SSD_ERR_INVALID_ARG;
    const size_t need = ssd_decode_host_buffer_size(s, dtype);
    if (!device_buffer || !aligned(device_buffer, 256) || device_buffer_bytes < need) return SSD_ERR_WORKSPACE;
    if (s->batch == 0) return SSD_OK;
    if (!x || !dt || !A || !B || !C || !state || !new_state || !y) return SSD_ERR_INVALID_ARG;
    const size_t e = decode_elt(dtype);
    const size_t rows = (size_t)s->batch * s->nheads;
    const size_t xb = rows * s->headdim * e, dtb = rows * 4, hb = (size_t)s->nheads * 4;
    const size_t bcb = (size_t)s->batch * s->ngroups * s->dstate * e;
    const size_t stb = rows * s->headdim * s->dstate * decode_elt(state_dtype);
    char* base = static_cast<char*>(device_buffer);
    size_t off = 0;
    auto carve = [&](size_t bytes) { char* p = base + off; off += align256(bytes); return p; };
    char* dx = carve(xb);
    char* dy = carve(xb);
    char* ddt = carve(dtb);
    char* dA = carve(hb);
    char* dD = carve(hb);
    char* dB = carve(bcb);
    char* dC = carve(bcb);
    char* dS = carve(stb);
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    cudaError_t err = cudaSuccess;
    if (stb >= kDecodePipelineBytes && s->batch >= kDecodePieces)
        return decode_host_pipelined(s, dtype, state_dtype, flags, x, dt, A, B, C, D, state, new_state, y, dx, dy, ddt,
                                     dA, dD, dB, dC, dS, st);
    auto h2d = [&](void* dst, const void* src, size_t bytes) {
        if (err == cudaSuccess && src && bytes) err = cudaMemcpyAsync(dst, src, bytes, cudaMemcpyHostToDevice, st);
    };
    h2d(dx, x, xb);
    h2d(ddt, dt, dtb);
    h2d(dA, A, hb);
    h2d(dD, D, hb);
    h2d(dB, B, bcb);
    h2d(dC, C, bcb);
    h2d(dS, state, stb);
    if (note_cuda_error("decode host copy in", err) != cudaSuccess) return SSD_ERR_CUDA;
    rc = ssd_decode_step_ex(s, dtype, state_dtype, flags, dx, (const float*)ddt, (const float*)dA, dB, dC,
                            D ? (const float*)dD : nullptr, dS, dS, dy, stream);
    if (rc != SSD_OK) return rc;
    err = cudaMemcpyAsync(y, dy, xb, cudaMemcpyDeviceToHost, st);
    if (err == cudaSuccess) err = cudaMemcpyAsync(new_state, dS, stb, cudaMemcpyDeviceToHost, st);
    if (err == cudaSuccess) err = cudaStreamSynchronize(st);
    return note_cuda_error("decode host copy out", err) == cudaSuccess ? SSD_OK : SSD_ERR_CUDA;
}

int ssd_decode_step_host(const ssd_shape* s, ssd_dtype dtype, const void* x, const float* dt, const float* A,
                         const void* B, const void* C, const float* D, const float* state, float* new_state,
                         void* y, void* device_buffer, size_t device_buffer_bytes, void* stream) {
    return ssd_decode_step_host_ex(s, dtype, SSD_F32, 0u, x, dt, A, B, C, D, state, new_state, y, device_buffer,
                                   device_buffer_bytes, stream);
}

}  // extern "C"
