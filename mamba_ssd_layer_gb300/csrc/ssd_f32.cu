// ssd_f32.cu -- the fp32 path (x, B, C, y in fp32), plain SIMT FMAs.
//
// Tensor-core tf32 cannot hold a 1e-4 relative error, so fp32 inputs are computed
// with CUDA-core fp32 arithmetic. The chunked algorithm is the same as the bf16
// path ("LLM(十一)——Mamba" §3.5):
//   chunk_state_f32: chunk-local cumsum of dt*A, chunk decay a_c = exp(cs_last),
//                    local end state S_c = sum_l exp(cs_last - cs_l) x_l B_l^T
//                    (right factors, §3.5.2);
//   (state pass in ssd_common.cu: center factors);
//   chunk_out_f32:   y_i = sum_{j<=i} exp(cs_i - cs_j) (C_i . B_j) x_j      (diagonal block, §3.5.1)
//                        + exp(cs_i) C_i . h_in                              (left factors, §3.5.2)
//                        + D x_i.
// With the dt-scaled input term every x_j that enters a state or a diagonal block is dt_j x_j; the
// skip term keeps D x_i.
// Cumulative sums are accumulated in fp64 so that differences of large sums do not
// lose digits (the stability concern of §3.5.4); exponentials are fp32.
#include "ssd_internal.cuh"

namespace ssd {

namespace {

constexpr int kMaxQ = 256;

// Chunk-local inclusive cumsum of dt*A in fp64 (one thread; Q <= 256 tokens).
__device__ void chunk_cumsum_f64(const float* __restrict__ dt, const float* __restrict__ A, int h, int H,
                                 int row0, int len, double* cs) {
    if (threadIdx.x == 0) {
        const double a = (double)A[h];
        double acc = 0.0;
        for (int l = 0; l < len; ++l) {
            acc += (double)dt[(int64_t)(row0 + l) * H + h] * a;
            cs[l] = acc;
        }
    }
    __syncthreads();
}

__global__ void __launch_bounds__(256) chunk_state_f32(const int* __restrict__ header, const ChunkDesc* __restrict__ chunks,
                                                       const float* __restrict__ x, const float* __restrict__ dt,
                                                       const float* __restrict__ A, const float* __restrict__ B,
                                                       float* __restrict__ decay, float* __restrict__ states,
                                                       int H, int P, int N, int G, int scale_x_by_dt) {
    __shared__ double cs[kMaxQ];
    __shared__ float w[kMaxQ];
    if (header[0] != SSD_OK || (int)blockIdx.x >= header[1]) return;
    const ChunkDesc d = chunks[blockIdx.x];
    const int h = blockIdx.y;
    const int g = h / (H / G);
    chunk_cumsum_f64(dt, A, h, H, d.row0, d.len, cs);
    const double last = d.len > 0 ? cs[d.len - 1] : 0.0;
    for (int l = threadIdx.x; l < d.len; l += blockDim.x)
        w[l] = (float)exp(last - cs[l]) * (scale_x_by_dt ? dt[(int64_t)(d.row0 + l) * H + h] : 1.f);
    if (threadIdx.x == 0) decay[(int64_t)blockIdx.x * H + h] = (float)exp(last);
    __syncthreads();
    float* S = states + ((int64_t)blockIdx.x * H + h) * P * N;
    for (int e = threadIdx.x; e < P * N; e += blockDim.x) {
        const int p = e / N, n = e % N;
        float acc = 0.f;
        for (int l = 0; l < d.len; ++l) {
            const int64_t r = d.row0 + l;
            acc = fmaf(w[l] * x[(r * H + h) * P + p], B[(r * G + g) * N + n], acc);
        }
        S[e] = acc;
    }
}

// Output of one chunk and head. Rows are processed in tiles of 32; every thread owns
// one row of the tile and a strided set of its P channels.
constexpr int kTile = 32;
constexpr int kThreads = 256;
constexpr int kLanesPerRow = kThreads / kTile;   // 8
constexpr int kMaxPPerThread = 256 / kLanesPerRow;  // P <= 256

__global__ void __launch_bounds__(kThreads) chunk_out_f32(const int* __restrict__ header, const ChunkDesc* __restrict__ chunks,
                                                          const float* __restrict__ x, const float* __restrict__ dt,
                                                          const float* __restrict__ A, const float* __restrict__ B,
                                                          const float* __restrict__ C, const float* __restrict__ D,
                                                          const float* __restrict__ states, float* __restrict__ y,
                                                          int H, int P, int N, int G, int scale_x_by_dt) {
    __shared__ double cs[kMaxQ];
    __shared__ float coef[kTile][kTile + 1];
    if (header[0] != SSD_OK || (int)blockIdx.x >= header[1]) return;
    const ChunkDesc d = chunks[blockIdx.x];
    const int h = blockIdx.y;
    const int g = h / (H / G);
    chunk_cumsum_f64(dt, A, h, H, d.row0, d.len, cs);
    const float Dh = D ? D[h] : 0.f;
    const float* hin = states + ((int64_t)blockIdx.x * H + h) * P * N;   // state entering the chunk
    const int ii = threadIdx.x / kLanesPerRow;   // row within the tile
    const int sub = threadIdx.x % kLanesPerRow;  // channel phase
    const int np = (P + kLanesPerRow - 1) / kLanesPerRow;

    for (int i0 = 0; i0 < d.len; i0 += kTile) {
        float acc[kMaxPPerThread];
#pragma unroll
        for (int m = 0; m < kMaxPPerThread; ++m) acc[m] = 0.f;
        const int i = i0 + ii;
        const int64_t ri = (int64_t)d.row0 + i;
        // diagonal block: causal, decay-masked C B^T times x
        for (int j0 = 0; j0 <= i0; j0 += kTile) {
            __syncthreads();
            for (int e = threadIdx.x; e < kTile * kTile; e += kThreads) {
                const int a = e / kTile, b = e % kTile;
                const int ia = i0 + a, jb = j0 + b;
                float v = 0.f;
                if (jb <= ia && ia < d.len) {
                    const float* Ci = C + (((int64_t)d.row0 + ia) * G + g) * N;
                    const float* Bj = B + (((int64_t)d.row0 + jb) * G + g) * N;
                    float dot = 0.f;
                    for (int n = 0; n < N; ++n) dot = fmaf(Ci[n], Bj[n], dot);
                    v = dot * (float)exp(cs[ia] - cs[jb]);
                    if (scale_x_by_dt) v *= dt[((int64_t)d.row0 + jb) * H + h];
                }
                coef[a][b] = v;
            }
            __syncthreads();
            if (i < d.len) {
                const int jmax = min(kTile, d.len - j0);
                for (int b = 0; b < jmax; ++b) {
                    const float cf = coef[ii][b];
                    const float* xj = x + (((int64_t)d.row0 + j0 + b) * H + h) * P;
#pragma unroll
                    for (int m = 0; m < kMaxPPerThread; ++m) {
                        const int p = sub + m * kLanesPerRow;
                        if (m < np && p < P) acc[m] = fmaf(cf, xj[p], acc[m]);
                    }
                }
            }
        }
        if (i < d.len) {
            // left factor: the state entering the chunk, decayed to token i
            const float* Ci = C + (ri * G + g) * N;
            const float e = (float)exp(cs[i]);
            const float* xi = x + (ri * H + h) * P;
            float* yi = y + (ri * H + h) * P;
#pragma unroll
            for (int m = 0; m < kMaxPPerThread; ++m) {
                const int p = sub + m * kLanesPerRow;
                if (m < np && p < P) {
                    const float* hp = hin + (int64_t)p * N;
                    float dot = 0.f;
                    for (int n = 0; n < N; ++n) dot = fmaf(Ci[n], hp[n], dot);
                    yi[p] = acc[m] + e * dot + Dh * xi[p];
                }
            }
        }
    }
}

}  // namespace

cudaError_t launch_f32_path(const Problem& p) {
    const int H = (int)p.s.nheads, P = (int)p.s.headdim, N = (int)p.s.dstate, G = (int)p.s.ngroups;
    if (p.L.max_chunks == 0) return launch_state_pass(p);
    dim3 grid((unsigned)p.L.max_chunks, (unsigned)H);
    prof_launch();
    chunk_state_f32<<<grid, 256, 0, p.stream>>>(p.status(), p.chunks(), (const float*)p.x, p.dt, p.A,
                                                (const float*)p.B, p.decay(), p.states(), H, P, N, G,
                                                p.scale_x_by_dt ? 1 : 0);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    e = launch_state_pass(p);
    if (e != cudaSuccess) return e;
    prof_launch();
    prof_begin(p.stream, "chunk_out_f32");
    chunk_out_f32<<<grid, kThreads, 0, p.stream>>>(p.status(), p.chunks(), (const float*)p.x, p.dt, p.A,
                                                   (const float*)p.B, (const float*)p.C, p.D, p.states(),
                                                   (float*)p.y, H, P, N, G, p.scale_x_by_dt ? 1 : 0);
    prof_end(p.stream);
    return cudaGetLastError();
}

}  // namespace ssd
