// ssd_handoff.cu -- the device side of the sequence-parallel state hand-off ("LLM(十一)——Mamba"
// §3.7.2 Sequence Parallelism: each worker passes its final state to the next one).
//
// A sequence cut into consecutive slices runs every slice from a zero state (ssd_forward), which
// gives the slice's local outputs and local final state. With h_in the true state entering a slice
// and cs_l = sum of dt*A from the slice's first token to token l (inclusive), linearity of the
// recurrence gives ("LLM(十一)——Mamba" §3.5.2, the center and left factors):
//   final      = local final + exp(cs_last) h_in          (h_in of the next slice)
//   y_l        = local y_l   + exp(cs_l) C_l h_in^T
// Here:
//   slice decay   exp(cs_last) per (sequence row, head)                      tile sums + a scan
//   correction    y_l += exp(cs_l) C_l h_in^T (tcgen05, M = 128 tokens, N = 64 channels per head,
//                 K = state columns), final += exp(cs_last) h_in
// The hand-off itself (h_in of slice k+1 from slice k) is the caller's: it moves one (H, P, N) fp32
// state between devices.
#include <cuda.h>
#include <cuda_runtime.h>

#include "ptx.cuh"
#include "ssd_internal.cuh"

namespace ssd {

namespace {

constexpr int kTileTok = 128;                 // tokens per tile
constexpr int kSliceHeader = 256;             // status word and diagnostics, as in the forward's workspace
constexpr float kLog2eH = 1.4426950408889634f;

__device__ __forceinline__ float ex2h(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Workspace: [header][tile prefix: float (batch, ntiles, H)][decay: float (batch, H)]
struct SliceWs {
    int* status;
    float* prefix;
    float* decay;
};

inline int64_t ntiles_of(const ssd_shape& s) { return (s.seqlen + kTileTok - 1) / kTileTok; }

SliceWs slice_ws(const ssd_shape& s, char* ws) {
    SliceWs w;
    w.status = reinterpret_cast<int*>(ws);
    w.prefix = reinterpret_cast<float*>(ws + kSliceHeader);
    w.decay = reinterpret_cast<float*>(ws + kSliceHeader + align256(s.batch * ntiles_of(s) * s.nheads * 4));
    return w;
}

// Sum of dt over each 128-token tile, per head: one block per (tile, batch row), heads across threads
// (consecutive heads are consecutive addresses), tokens in order.
__global__ void tile_dt_sum_kernel(const float* __restrict__ dt, float* __restrict__ tsum, int T, int H, int ntiles) {
    const int t = blockIdx.x, b = blockIdx.y;
    const int r0 = t * kTileTok;
    const int n = min(kTileTok, T - r0);
    const float* base = dt + ((int64_t)b * T + r0) * H;
    for (int h = threadIdx.x; h < H; h += blockDim.x) {
        float acc = 0.f;
#pragma unroll 8
        for (int r = 0; r < n; ++r) acc += __ldg(base + (int64_t)r * H + h);
        tsum[((int64_t)b * ntiles + t) * H + h] = acc;
    }
}

// Per (batch row, head): the tile sums turned into exclusive prefixes in place, and the slice's decay
// exp(A * sum of dt), in tile order.
__global__ void slice_scan_kernel(const float* __restrict__ A, float* __restrict__ tsum, float* __restrict__ decay,
                                  float* __restrict__ decay_out, int H, int ntiles) {
    const int h = blockIdx.x * blockDim.x + threadIdx.x, b = blockIdx.y;
    if (h >= H) return;
    float acc = 0.f;
    float* p = tsum + (int64_t)b * ntiles * H + h;
    for (int t = 0; t < ntiles; ++t) {
        const float v = p[(int64_t)t * H];
        p[(int64_t)t * H] = acc;
        acc += v;
    }
    const float d = ex2h(acc * (__ldg(A + h) * kLog2eH));
    decay[(int64_t)b * H + h] = d;
    if (decay_out) decay_out[(int64_t)b * H + h] = d;
}

// final[b, h, :, :] += decay[b, h] * h_in[b, h, :, :]
__global__ void final_update_kernel(const float* __restrict__ decay, const float* __restrict__ h_in,
                                    float* __restrict__ fin, int64_t per_head, int64_t n) {
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += stride)
        fin[i] = fmaf(__ldg(decay + i / per_head), __ldg(h_in + i), fin[i]);
}

// y_l += exp(cs_l) C_l h_in^T for one 128-token tile of one batch row and one head pair (both heads of
// a pair share a B/C group). C arrives by TMA in the 128-byte swizzle; h_in of the pair is staged as
// bf16, K-major over the state columns, as the B operand; one elected thread issues two tcgen05 MMAs
// per 16 state columns (M = 128 tokens, N = 64 channels, one per head) into TMEM; eight warps (one per
// head and TMEM lane quadrant) scale the rows by exp(cs_l), add onto y in fp32 and round once.
template <int N>
__global__ void __launch_bounds__(256)
slice_correct_kernel(const __grid_constant__ CUtensorMap mapC, const float* __restrict__ dt,
                     const float* __restrict__ A, const float* __restrict__ prefix, const float* __restrict__ h_in,
                     __nv_bfloat16* __restrict__ y, int* status, int T, int H, int G, int ntiles) {
    constexpr int NB = N / 64;
    constexpr uint32_t kRegion = 16384;        // 128 rows x 128 bytes
    extern __shared__ __align__(1024) uint8_t sm[];
    uint8_t* cbuf = sm;
    uint8_t* hs = sm + NB * kRegion;
    uint64_t* bars = reinterpret_cast<uint64_t*>(sm + 2 * NB * kRegion);   // [0] C landed, [1] MMAs done
    uint32_t* slot = reinterpret_cast<uint32_t*>(bars + 2);
    const int t = blockIdx.x, hp = blockIdx.y, b = blockIdx.z;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int h0 = 2 * hp, g = h0 / (H / G);
    const int64_t row0 = (int64_t)b * T + (int64_t)t * kTileTok;
    if ((smem_u32(sm) & 1023u) != 0) {          // the swizzled layout needs a 1024-byte aligned base
        if (tid == 0) record_status(status, SSD_ERR_UNSUPPORTED);
        return;
    }
    if (tid == 0) {
        mbar_init(bars, 1);
        mbar_init(bars + 1, 1);
        fence_mbar_init();
    }
    if (warp == 0) tmem_alloc(slot, 128);
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem = *slot;
    if (tid == 0) {
        mbar_arrive_expect_tx(bars, NB * kRegion);
        for (int k = 0; k < NB; ++k) tma_load_3d(cbuf + k * kRegion, &mapC, bars, 64 * k, g, (int)row0);
    }
    // h_in of the pair as bf16: row r = 64 hh + p (the (H, P, N) layout makes the pair's 128 rows
    // contiguous), 16-byte chunks of 8 state columns placed by the swizzle
    const float* hsrc = h_in + ((int64_t)b * H + h0) * 64 * N;
    for (int c = tid; c < 128 * (N / 8); c += blockDim.x) {
        const int r = c / (N / 8), n = 8 * (c % (N / 8));
        const float4* src = reinterpret_cast<const float4*>(hsrc + (int64_t)r * N + n);
        const float4 v0 = __ldg(src), v1 = __ldg(src + 1);
        uint4 pk;
        pk.x = pack_bf16x2(v0.x, v0.y);
        pk.y = pack_bf16x2(v0.z, v0.w);
        pk.z = pack_bf16x2(v1.x, v1.y);
        pk.w = pack_bf16x2(v1.z, v1.w);
        *reinterpret_cast<uint4*>(hs + (n / 64) * kRegion + sw128_offset(r, (n % 64) / 8)) = pk;
    }
    fence_proxy_async_smem();
    __syncthreads();
    bool c_landed = true;
    if (tid == 0) {
        c_landed = mbar_wait(bars, 0, status);
        if (c_landed) {
            tc_fence_after_sync();
            const uint32_t idesc = idesc_bf16_f32(128, 64, 0, 0);
#pragma unroll 1
            for (int hh = 0; hh < 2; ++hh)
#pragma unroll 1
                for (int ks = 0; ks < N / 16; ++ks) {
                    const int k = ks / 4, off = (ks % 4) * 32;
                    const uint64_t ad = smem_desc_sw128(smem_u32(cbuf + k * kRegion + off), 0, 1024);
                    const uint64_t bd = smem_desc_sw128(smem_u32(hs + k * kRegion + hh * 8192 + off), 0, 1024);
                    mma_bf16_ss(tmem + 64 * hh, ad, bd, idesc, ks > 0 ? 1u : 0u);
                }
        }
        // committed also when nothing was issued, so that every thread's wait below ends
        mma_commit(bars + 1);
    }
    // this thread's row l (TMEM lane 32 q + lane) and head: cs_l = A (prefix of the earlier tiles plus
    // the sum of dt over the tile's rows 0..l), summed in a fixed order
    const int q = warp & 3, hh = warp >> 2, h = h0 + hh;
    const int l = 32 * q + lane;
    const int tok = t * kTileTok + l;
    float d[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const int tj = t * kTileTok + 32 * j + lane;
        d[j] = tj < T ? __ldg(dt + ((int64_t)b * T + tj) * H + h) : 0.f;
    }
    float below = 0.f;
#pragma unroll
    for (int j = 0; j < 3; ++j) {
        float s = d[j];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
        if (j < q) below += s;
    }
    float sc = d[0];
#pragma unroll
    for (int j = 1; j < 4; ++j) sc = (j == q) ? d[j] : sc;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const float tt = __shfl_up_sync(0xffffffffu, sc, o);
        if (lane >= o) sc += tt;
    }
    const float cs = (__ldg(prefix + ((int64_t)b * ntiles + t) * H + h) + (below + sc)) * (__ldg(A + h) * kLog2eH);
    const float e = ex2h(cs);
    const bool mma_done = mbar_wait(bars + 1, 0, status);
    tc_fence_after_sync();
    if (__all_sync(0xffffffffu, mma_done) && *reinterpret_cast<volatile int*>(status) == SSD_OK) {
        uint32_t v[64];
        const uint32_t col = tmem + ((uint32_t)(32 * q) << 16) + 64 * hh;
        tmem_ld32_nowait(col, v);
        tmem_ld32_nowait(col + 32, v + 32);
        asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
        if (tok < T) {
            uint4* yrow = reinterpret_cast<uint4*>(y + (((int64_t)b * T + tok) * H + h) * 64);
            const float2 ee = make_float2(e, e);
#pragma unroll
            for (int ch = 0; ch < 8; ++ch) {
                uint4 o = yrow[ch];
                uint32_t* ou = reinterpret_cast<uint32_t*>(&o);
#pragma unroll
                for (int m = 0; m < 4; ++m) {
                    const float2 cc = make_float2(__uint_as_float(v[8 * ch + 2 * m]), __uint_as_float(v[8 * ch + 2 * m + 1]));
                    const float2 r = __ffma2_rn(ee, cc, unpack_bf16x2(ou[m]));
                    ou[m] = pack_bf16x2(r.x, r.y);
                }
                yrow[ch] = o;
            }
        }
    }
    // a load that did not land in time is waited for once more (bounded) before the CTA's shared
    // memory goes away
    if (tid == 0 && !c_landed) (void)mbar_wait(bars, 0, status);
    tc_fence_before_sync();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, 128);
}

template <int N>
constexpr size_t correct_smem() {
    // C and h_in regions, the barriers and the TMEM slot; at least 56 KB so that no more than four CTAs
    // (4 x 128 TMEM columns) share an SM
    return (2 * (N / 64) * 16384 + 64) > 57344 ? (2 * (N / 64) * 16384 + 64) : 57344;
}

template <int N>
cudaError_t launch_correct_n(const ssd_shape& s, const CUtensorMap& mapC, const float* dt, const float* A,
                             const SliceWs& w, const float* h_in, void* y, cudaStream_t st) {
    const size_t smem = correct_smem<N>();
    cudaError_t e = note_cuda_error("correct smem attribute",
        cudaFuncSetAttribute(slice_correct_kernel<N>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem));
    if (e != cudaSuccess) return e;
    const dim3 grid((unsigned)ntiles_of(s), (unsigned)(s.nheads / 2), (unsigned)s.batch);
    prof_launch();
    slice_correct_kernel<N><<<grid, 256, smem, st>>>(mapC, dt, A, w.prefix, h_in, static_cast<__nv_bfloat16*>(y),
                                                    w.status, (int)s.seqlen, (int)s.nheads, (int)s.ngroups,
                                                    (int)ntiles_of(s));
    return note_cuda_error("correct launch", cudaGetLastError());
}

// the tile prefixes and the slice decay into the workspace (and into `decay_out` when given)
cudaError_t launch_scan(const ssd_shape& s, const float* dt, const float* A, const SliceWs& w, float* decay_out,
                        cudaStream_t st) {
    const int nt = (int)ntiles_of(s);
    if (s.batch == 0) return cudaSuccess;
    if (nt > 0) {
        prof_launch();
        tile_dt_sum_kernel<<<dim3((unsigned)nt, (unsigned)s.batch), 128, 0, st>>>(dt, w.prefix, (int)s.seqlen,
                                                                                  (int)s.nheads, nt);
        cudaError_t e = note_cuda_error("tile sum launch", cudaGetLastError());
        if (e != cudaSuccess) return e;
    }
    // (an empty slice has no tiles: its decay is exp(0) = 1)
    prof_launch();
    slice_scan_kernel<<<dim3((unsigned)((s.nheads + 127) / 128), (unsigned)s.batch), 128, 0, st>>>(
        A, w.prefix, w.decay, decay_out, (int)s.nheads, nt);
    return note_cuda_error("slice scan launch", cudaGetLastError());
}

}  // namespace

size_t slice_ws_bytes(const ssd_shape& s) {
    return kSliceHeader + align256(s.batch * ntiles_of(s) * s.nheads * 4) + align256(s.batch * s.nheads * 4);
}

cudaError_t launch_slice_decay(const ssd_shape& s, const float* dt, const float* A, float* decay, char* ws,
                               cudaStream_t st) {
    const SliceWs w = slice_ws(s, ws);
    cudaError_t e = note_cuda_error("slice header reset", cudaMemsetAsync(ws, 0, kSliceHeader, st));
    if (e != cudaSuccess) return e;
    return launch_scan(s, dt, A, w, decay, st);
}

cudaError_t launch_slice_correct(const ssd_shape& s, const float* dt, const float* A, const void* C,
                                 const float* h_in, void* y, float* final_state, char* ws, cudaStream_t st) {
    const SliceWs w = slice_ws(s, ws);
    cudaError_t e = note_cuda_error("slice header reset", cudaMemsetAsync(ws, 0, kSliceHeader, st));
    if (e != cudaSuccess) return e;
    e = launch_scan(s, dt, A, w, nullptr, st);
    if (e != cudaSuccess || s.batch == 0) return e;
    if (s.seqlen > 0) {
        CUtensorMap mapC;
        const int64_t N = s.dstate, G = s.ngroups;
        if (!make_map_fused(&mapC, C, N, G, s.batch * s.seqlen, N, N * G))
            return note_cuda_error("correct tensor map", cudaErrorInvalidValue);
        if (N == 64) e = launch_correct_n<64>(s, mapC, dt, A, w, h_in, y, st);
        else if (N == 128) e = launch_correct_n<128>(s, mapC, dt, A, w, h_in, y, st);
        else e = launch_correct_n<256>(s, mapC, dt, A, w, h_in, y, st);
    }
    if (e != cudaSuccess || !final_state) return e;
    const int64_t per_head = (int64_t)s.headdim * s.dstate, n = (int64_t)s.batch * s.nheads * per_head;
    prof_launch();
    final_update_kernel<<<(unsigned)((n + 255) / 256 < 4096 ? (n + 255) / 256 : 4096), 256, 0, st>>>(
        w.decay, h_in, final_state, per_head, n);
    return note_cuda_error("final update launch", cudaGetLastError());
}

}  // namespace ssd
