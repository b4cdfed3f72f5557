// ssd_tc.cu -- the bf16 path on the 5th-generation tensor cores (tcgen05 + TMEM + TMA).
//
// The chunked SSD algorithm ("LLM(十一)——Mamba" §3.5) in three launches after the
// chunk table is built:
//
//   chunk_state_tc  per (chunk, head pair): chunk-local cumsum cs of dt*A, chunk
//                   decay exp(cs_last), and the chunk's local end state
//                     S[(h,p), n] = sum_l exp(cs_last - cs_l) x[l,h,p] B[l,n]
//                   as ONE tcgen05 MMA chain: M = 2 heads x 64 channels = 128,
//                   N = state size, K = chunk tokens ("right factors", §3.5.2).
//   state pass      (ssd_common.cu) h_c = a_c h_{c-1} + S_c ("center factors").
//   chunk_out_tc    per (chunk, head pair), per 128-token tile of the chunk:
//                     G = C B^T                     (M=128 tokens, N=128 tokens, K=N)  shared by both heads
//                     LG_h = L_h o G  -> bf16 smem   (L_ij = exp(cs_i - cs_j), j <= i)   "diagonal blocks", §3.5.1
//                     Yd_h = LG_h X_h               (M=128, N=64, K=128)
//                     Yo = C h_in^T                 (M=128, N=128 = both heads, K=N)    "left factors", §3.5.2
//                     y = Yd + exp(cs_i) Yo + D x   -> bf16
//                   A 256-token chunk is two tiles; the state between them is
//                   exp(cs_127) h_in + S(tile 0), computed on chip with one more MMA.
//
// Operands are staged by TMA with the 128-byte swizzle; x, B and C tiles are used
// both K-major (contraction over state or channel) and MN-major (contraction over
// tokens) straight from the same shared-memory bytes. Accumulation is fp32 in TMEM.
#include <cuda.h>
#include <cuda_runtime.h>

#include "ptx.cuh"
#include "ssd_internal.cuh"

namespace ssd {

namespace {

constexpr int kTileRows = 128;                 // tokens per MMA tile (M)
constexpr int kRegion = kTileRows * 128;       // bytes of one 128-row x 128-byte swizzled box
constexpr int kThreads = 128;

struct TcMaps {
    CUtensorMap x, b, c;
};

// Chunk-local inclusive cumsum of dt*A for one head, by one warp (fp32, len <= 256).
__device__ __forceinline__ void warp_cumsum(const float* __restrict__ dt, float Ah, int h, int H,
                                            int row0, int len, float* cs) {
    const int lane = threadIdx.x & 31;
    float carry = 0.f;
    for (int base = 0; base < len; base += 32) {
        const int l = base + lane;
        float v = (l < len) ? __ldg(dt + (int64_t)(row0 + l) * H + h) * Ah : 0.f;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            float t = __shfl_up_sync(0xffffffffu, v, o);
            if (lane >= o) v += t;
        }
        v += carry;
        if (l < len) cs[l] = v;
        carry = __shfl_sync(0xffffffffu, v, 31);
    }
}

// Scale the rows of a staged x tile in place: row l of every 16-byte chunk is
// multiplied by w[l] (0 beyond `len`). Regions: [head][tile] of kRegion bytes.
__device__ __forceinline__ void scale_rows_inplace(uint8_t* xs, int nheads_local, int ntiles,
                                                   const float* w0, const float* w1, int len) {
    const int chunks = nheads_local * ntiles * kTileRows * 8;
    for (int q = threadIdx.x; q < chunks; q += blockDim.x) {
        const int head = q / (ntiles * kTileRows * 8);
        const int rem = q % (ntiles * kTileRows * 8);
        const int l = rem / 8;                       // token within the chunk (tile-major)
        const float* w = head ? w1 : w0;
        const float s = (l < len) ? w[l] : 0.f;
        uint4* ptr = reinterpret_cast<uint4*>(xs + (size_t)q * 16);
        uint4 v = *ptr;
        uint32_t* u = reinterpret_cast<uint32_t*>(&v);
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            float2 f = unpack_bf16x2(u[k]);
            u[k] = pack_bf16x2(f.x * s, f.y * s);
        }
        *ptr = v;
    }
}

// ----------------------------------------------------------------------------
// chunk_state_tc
// smem: xs [2 heads][ntiles][kRegion], bs [N/64][ntiles][kRegion], cs [2][256], w [2][256]
// ----------------------------------------------------------------------------
__global__ void __launch_bounds__(kThreads, 1)
chunk_state_tc(const __grid_constant__ TcMaps maps, const int* __restrict__ header_in, int* status,
               const ChunkDesc* __restrict__ chunks, const float* __restrict__ dt, const float* __restrict__ A,
               float* __restrict__ decay, float* __restrict__ states, int H, int N, int G, int Q) {
    extern __shared__ uint8_t smem_raw[];
    __shared__ __align__(8) uint64_t bar_tma, bar_mma;
    __shared__ uint32_t tmem_base_sh;
    __shared__ float cs[2][256];
    __shared__ float w[2][256];

    if (header_in[0] != SSD_OK || (int)blockIdx.x >= header_in[1]) return;
    const ChunkDesc d = chunks[blockIdx.x];
    const int h0 = 2 * blockIdx.y;
    const int g = h0 / (H / G);
    const int ntiles = (Q + kTileRows - 1) / kTileRows;
    const int nb = N / 64;
    const int warp = threadIdx.x >> 5;

    uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* xs = base;                                        // 2 * ntiles regions
    uint8_t* bs = base + (size_t)2 * ntiles * kRegion;         // nb * ntiles regions

    if (threadIdx.x == 0) {
        mbar_init(&bar_tma, 1);
        mbar_init(&bar_mma, 1);
        fence_mbar_init();
    }
    if (warp == 0) tmem_alloc(&tmem_base_sh, (uint32_t)(N < 32 ? 32 : N));
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem = tmem_base_sh;

    if (threadIdx.x == 0) {
        const uint32_t bytes = (uint32_t)((2 + nb) * ntiles * kRegion);
        mbar_arrive_expect_tx(&bar_tma, bytes);
        for (int t = 0; t < ntiles; ++t) {
            const int r = d.row0 + t * kTileRows;
            for (int hh = 0; hh < 2; ++hh)
                tma_load_3d(xs + (size_t)(hh * ntiles + t) * kRegion, &maps.x, &bar_tma, 0, h0 + hh, r);
            for (int k = 0; k < nb; ++k)
                tma_load_3d(bs + (size_t)(k * ntiles + t) * kRegion, &maps.b, &bar_tma, 64 * k, g, r);
        }
    }
    if (warp < 2) {
        const int h = h0 + warp;
        warp_cumsum(dt, __ldg(A + h), h, H, d.row0, d.len, cs[warp]);
        __syncwarp();
        const float last = d.len > 0 ? cs[warp][d.len - 1] : 0.f;
        for (int l = threadIdx.x & 31; l < d.len; l += 32) w[warp][l] = __expf(last - cs[warp][l]);
        if ((threadIdx.x & 31) == 0) decay[(int64_t)blockIdx.x * H + h] = __expf(last);
    }
    __syncthreads();
    bool ok = mbar_wait(&bar_tma, 0, status);
    if (ok) {
        scale_rows_inplace(xs, 2, ntiles, w[0], w[1], d.len);
        fence_proxy_async_smem();
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    if (ok && threadIdx.x == 0) {
        const uint32_t idesc = idesc_bf16_f32(128, (uint32_t)N, 1, 1);
        const int ksteps = (Q < ntiles * kTileRows ? Q : ntiles * kTileRows) / 16;
        for (int s = 0; s < ksteps; ++s) {
            const int t = s / 8, sub = s % 8;
            const uint64_t a = smem_desc_sw128(smem_u32(xs + (size_t)t * kRegion + sub * 2048),
                                               (uint32_t)(ntiles * kRegion), 1024);
            const uint64_t b = smem_desc_sw128(smem_u32(bs + (size_t)t * kRegion + sub * 2048),
                                               (uint32_t)(ntiles * kRegion), 1024);
            mma_bf16_ss(tmem, a, b, idesc, s > 0 ? 1u : 0u);
        }
        mma_commit(&bar_mma);
    }
    __syncthreads();
    if (ok) ok = mbar_wait(&bar_mma, 0, status);
    tc_fence_after_sync();
    if (ok) {
        // lane m of the accumulator = (head, channel) row; columns = state index n
        const int m = warp * 32 + (threadIdx.x & 31);
        const int hh = m / 64, p = m % 64;
        float* dst = states + (((int64_t)blockIdx.x * H + h0 + hh) * 64 + p) * N;
        const uint32_t lane_addr = tmem + ((uint32_t)(warp * 32) << 16);
        for (int c0 = 0; c0 < N; c0 += 32) {
            float v[32];
            tmem_ld32(lane_addr + c0, v);
#pragma unroll
            for (int k = 0; k < 32; k += 4)
                *reinterpret_cast<float4*>(dst + c0 + k) = make_float4(v[k], v[k + 1], v[k + 2], v[k + 3]);
        }
    }
    tc_fence_before_sync();
    __syncthreads();
    if (warp == 0) {
        __syncwarp();
        tmem_dealloc(tmem, (uint32_t)(N < 32 ? 32 : N));
    }
}

// ----------------------------------------------------------------------------
// chunk_out_tc
// smem: xs [2][kRegion], bs [nb][kRegion], csm [nb][kRegion], rs [max(2, nb)][kRegion]
// TMEM columns: G [0,128), Yd0 [128,192), Yd1 [192,256), Yo [256,384); the tile-0
// state S aliases [0, N) once G and Yd are consumed.
// ----------------------------------------------------------------------------
constexpr uint32_t kColG = 0, kColYd = 128, kColYo = 256;

// Writes one 128 x N fp32 state (rows = (head, channel), from global) as bf16,
// K-major 128B-swizzled, into `rs` (nb regions of 128 rows).
__device__ __forceinline__ void stage_state_bf16(uint8_t* rs, const float* __restrict__ st0,
                                                 const float* __restrict__ st1, int N) {
    const int m = threadIdx.x;   // 128 threads <-> 128 rows
    const float* src = (m < 64 ? st0 : st1) + (int64_t)(m % 64) * N;
    for (int n0 = 0; n0 < N; n0 += 8) {
        const float4 a = *reinterpret_cast<const float4*>(src + n0);
        const float4 b = *reinterpret_cast<const float4*>(src + n0 + 4);
        uint4 v;
        v.x = pack_bf16x2(a.x, a.y);
        v.y = pack_bf16x2(a.z, a.w);
        v.z = pack_bf16x2(b.x, b.y);
        v.w = pack_bf16x2(b.z, b.w);
        const int k = n0 / 64, c = (n0 % 64) / 8;
        *reinterpret_cast<uint4*>(rs + (size_t)k * kRegion + sw128_offset(m, c)) = v;
    }
}

__global__ void __launch_bounds__(kThreads, 1)
chunk_out_tc(const __grid_constant__ TcMaps maps, const int* __restrict__ header_in, int* status,
             const ChunkDesc* __restrict__ chunks, const float* __restrict__ dt, const float* __restrict__ A,
             const float* __restrict__ D, float* __restrict__ states, __nv_bfloat16* __restrict__ y,
             int H, int N, int G, int Q) {
    // all shared memory is dynamic: swizzled regions first (1024-byte aligned), then the
    // cumsums, barriers and the TMEM address
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    if (header_in[0] != SSD_OK || (int)blockIdx.x >= header_in[1]) return;
    if ((smem_u32(smem_raw) & 1023u) != 0) {
        if (threadIdx.x == 0) record_status(status, SSD_ERR_UNSUPPORTED);
        return;
    }
    const int nb_ = N / 64;
    uint8_t* tail = smem_raw + (size_t)(2 + 2 * nb_ + (nb_ > 2 ? nb_ : 2)) * kRegion;
    float (*cs)[256] = reinterpret_cast<float (*)[256]>(tail);
    uint64_t& bar_tma = *reinterpret_cast<uint64_t*>(tail + 2048);
    uint64_t& bar_mma = *reinterpret_cast<uint64_t*>(tail + 2056);
    uint32_t& tmem_base_sh = *reinterpret_cast<uint32_t*>(tail + 2064);

    const ChunkDesc d = chunks[blockIdx.x];
    const int h0 = 2 * blockIdx.y;
    const int g = h0 / (H / G);
    const int ntiles = (d.len + kTileRows - 1) / kTileRows;
    const int nb = N / 64;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int row = threadIdx.x;   // accumulator lane = tile row (or (head, channel) for S)

    uint8_t* xs = smem_raw;
    uint8_t* bs = xs + 2 * kRegion;
    uint8_t* csm = bs + (size_t)nb * kRegion;
    uint8_t* rs = csm + (size_t)nb * kRegion;

    float* st0 = states + ((int64_t)blockIdx.x * H + h0) * 64 * N;   // entering state, head h0
    float* st1 = st0 + (int64_t)64 * N;                               // head h0 + 1

    if (threadIdx.x == 0) {
        mbar_init(&bar_tma, 1);
        mbar_init(&bar_mma, 1);
        fence_mbar_init();
    }
    if (warp == 0) tmem_alloc(&tmem_base_sh, 512);
    if (warp < 2) {
        const int h = h0 + warp;
        warp_cumsum(dt, __ldg(A + h), h, H, d.row0, d.len, cs[warp]);
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem = tmem_base_sh;
    const uint32_t lane_base = tmem + ((uint32_t)(warp * 32) << 16);
    const float Dh[2] = {D ? __ldg(D + h0) : 0.f, D ? __ldg(D + h0 + 1) : 0.f};

    uint32_t tma_phase = 0, mma_phase = 0;
    bool ok = true;
    for (int t = 0; t < ntiles && ok; ++t) {
        const int r0 = d.row0 + t * kTileRows;
        const int len_t = min(kTileRows, d.len - t * kTileRows);
        const int cbase = t * kTileRows;                        // chunk index of tile row 0
        // 1. loads
        fence_proxy_async_smem();
        __syncthreads();
        if (threadIdx.x == 0) {
            mbar_arrive_expect_tx(&bar_tma, (uint32_t)((2 + 2 * nb) * kRegion));
            tma_load_3d(xs, &maps.x, &bar_tma, 0, h0, r0);
            tma_load_3d(xs + kRegion, &maps.x, &bar_tma, 0, h0 + 1, r0);
            for (int k = 0; k < nb; ++k) {
                tma_load_3d(bs + (size_t)k * kRegion, &maps.b, &bar_tma, 64 * k, g, r0);
                tma_load_3d(csm + (size_t)k * kRegion, &maps.c, &bar_tma, 64 * k, g, r0);
            }
        }
        ok = mbar_wait(&bar_tma, tma_phase, status);
        tma_phase ^= 1u;
        if (!ok) break;
        // 2. G = C B^T
        if (threadIdx.x == 0) {
            tc_fence_after_sync();
            const uint32_t idesc = idesc_bf16_f32(128, 128, 0, 0);
            for (int s = 0; s < N / 16; ++s) {
                const int k = s / 4, off = (s % 4) * 32;
                const uint64_t a = smem_desc_sw128(smem_u32(csm + (size_t)k * kRegion + off), 0, 1024);
                const uint64_t b = smem_desc_sw128(smem_u32(bs + (size_t)k * kRegion + off), 0, 1024);
                mma_bf16_ss(tmem + kColG, a, b, idesc, s > 0 ? 1u : 0u);
            }
            mma_commit(&bar_mma);
        }
        ok = mbar_wait(&bar_mma, mma_phase, status);
        mma_phase ^= 1u;
        tc_fence_after_sync();
        if (!ok) break;
        // 3. per head: LG = L o G (bf16, K-major) then Yd = LG X
        float g_row[128];
        for (int c0 = 0; c0 < 128; c0 += 32) {
            float v[32];
            tmem_ld32(lane_base + kColG + c0, v);
#pragma unroll
            for (int k = 0; k < 32; ++k) g_row[c0 + k] = v[k];
        }
        for (int hh = 0; hh < 2 && ok; ++hh) {
            const float csi = cs[hh][cbase + row];
            const bool rv = row < len_t;
#pragma unroll
            for (int c = 0; c < 16; ++c) {           // 16 chunks of 8 columns
                uint32_t pk[4];
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const int j0 = c * 8 + 2 * k;
                    const float l0 = (rv && j0 <= row) ? __expf(csi - cs[hh][cbase + j0]) : 0.f;
                    const float l1 = (rv && j0 + 1 <= row) ? __expf(csi - cs[hh][cbase + j0 + 1]) : 0.f;
                    pk[k] = pack_bf16x2(g_row[j0] * l0, g_row[j0 + 1] * l1);
                }
                *reinterpret_cast<uint4*>(rs + (size_t)(c / 8) * kRegion + sw128_offset(row, c % 8)) =
                    make_uint4(pk[0], pk[1], pk[2], pk[3]);
            }
            fence_proxy_async_smem();
            tc_fence_before_sync();
            __syncthreads();
            if (threadIdx.x == 0) {
                tc_fence_after_sync();
                const uint32_t idesc = idesc_bf16_f32(128, 64, 0, 1);
                for (int s = 0; s < 8; ++s) {
                    const uint64_t a = smem_desc_sw128(smem_u32(rs + (size_t)(s / 4) * kRegion + (s % 4) * 32), 0, 1024);
                    const uint64_t b = smem_desc_sw128(smem_u32(xs + (size_t)hh * kRegion + s * 2048), kRegion, 1024);
                    mma_bf16_ss(tmem + kColYd + 64 * hh, a, b, idesc, s > 0 ? 1u : 0u);
                }
                mma_commit(&bar_mma);
            }
            ok = mbar_wait(&bar_mma, mma_phase, status);
            mma_phase ^= 1u;
            tc_fence_after_sync();
        }
        if (!ok) break;
        // 4. Yo = C h^T with h the state entering this tile (both heads, N = 128 columns)
        stage_state_bf16(rs, st0, st1, N);
        fence_proxy_async_smem();
        tc_fence_before_sync();
        __syncthreads();
        if (threadIdx.x == 0) {
            tc_fence_after_sync();
            const uint32_t idesc = idesc_bf16_f32(128, 128, 0, 0);
            for (int s = 0; s < N / 16; ++s) {
                const int k = s / 4, off = (s % 4) * 32;
                const uint64_t a = smem_desc_sw128(smem_u32(csm + (size_t)k * kRegion + off), 0, 1024);
                const uint64_t b = smem_desc_sw128(smem_u32(rs + (size_t)k * kRegion + off), 0, 1024);
                mma_bf16_ss(tmem + kColYo, a, b, idesc, s > 0 ? 1u : 0u);
            }
            mma_commit(&bar_mma);
        }
        ok = mbar_wait(&bar_mma, mma_phase, status);
        mma_phase ^= 1u;
        tc_fence_after_sync();
        if (!ok) break;
        // 5. epilogue: y = Yd + exp(cs_i - cs_ref) Yo + D x
        for (int hh = 0; hh < 2; ++hh) {
            const float cs_ref = t > 0 ? cs[hh][cbase - 1] : 0.f;
            const float e = __expf(cs[hh][cbase + row] - cs_ref);
            __nv_bfloat16* yrow = y + ((int64_t)(r0 + row) * H + h0 + hh) * 64;
            for (int c0 = 0; c0 < 64; c0 += 32) {
                float yd[32], yo[32];
                tmem_ld32(lane_base + kColYd + 64 * hh + c0, yd);
                tmem_ld32(lane_base + kColYo + 64 * hh + c0, yo);
                if (row < len_t) {
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        const int cc = c0 / 8 + c;    // 16-byte chunk of the 128-byte row
                        const uint4 xv = *reinterpret_cast<const uint4*>(xs + (size_t)hh * kRegion + sw128_offset(row, cc));
                        const uint32_t* xu = reinterpret_cast<const uint32_t*>(&xv);
                        uint32_t pk[4];
#pragma unroll
                        for (int k = 0; k < 4; ++k) {
                            const float2 xf = unpack_bf16x2(xu[k]);
                            const int j = c * 8 + 2 * k;
                            const float a0 = fmaf(e, yo[j], yd[j]) + Dh[hh] * xf.x;
                            const float a1 = fmaf(e, yo[j + 1], yd[j + 1]) + Dh[hh] * xf.y;
                            pk[k] = pack_bf16x2(a0, a1);
                        }
                        *reinterpret_cast<uint4*>(yrow + cc * 8) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
                    }
                }
            }
        }
        // 6. state entering the next tile: exp(cs_last(tile)) h + S(tile)
        if (t + 1 < ntiles) {
            // decay weights of this tile's tokens to the tile end, scaling x in place
            // (x is no longer needed: Yd and the epilogue are done)
            __syncthreads();
            {
                const int chunks16 = 2 * kTileRows * 8;
                for (int q = threadIdx.x; q < chunks16; q += blockDim.x) {
                    const int hh = q / (kTileRows * 8);
                    const int l = (q % (kTileRows * 8)) / 8;
                    const float s = (l < len_t) ? __expf(cs[hh][cbase + len_t - 1] - cs[hh][cbase + l]) : 0.f;
                    uint4* ptr = reinterpret_cast<uint4*>(xs + (size_t)q * 16);
                    uint4 v = *ptr;
                    uint32_t* u = reinterpret_cast<uint32_t*>(&v);
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        float2 f = unpack_bf16x2(u[k]);
                        u[k] = pack_bf16x2(f.x * s, f.y * s);
                    }
                    *ptr = v;
                }
            }
            fence_proxy_async_smem();
            tc_fence_before_sync();
            __syncthreads();
            if (threadIdx.x == 0) {
                tc_fence_after_sync();
                const uint32_t idesc = idesc_bf16_f32(128, (uint32_t)N, 1, 1);
                for (int s = 0; s < 8; ++s) {
                    const uint64_t a = smem_desc_sw128(smem_u32(xs + s * 2048), kRegion, 1024);
                    const uint64_t b = smem_desc_sw128(smem_u32(bs + s * 2048), kRegion, 1024);
                    mma_bf16_ss(tmem + 0, a, b, idesc, s > 0 ? 1u : 0u);
                }
                mma_commit(&bar_mma);
            }
            ok = mbar_wait(&bar_mma, mma_phase, status);
            mma_phase ^= 1u;
            tc_fence_after_sync();
            if (!ok) break;
            const int hh = row / 64;
            const float a = __expf(cs[hh][cbase + len_t - 1] - (t > 0 ? cs[hh][cbase - 1] : 0.f));
            float* st = (hh ? st1 : st0) + (int64_t)(row % 64) * N;
            for (int c0 = 0; c0 < N; c0 += 32) {
                float v[32];
                tmem_ld32(lane_base + c0, v);
#pragma unroll
                for (int k = 0; k < 32; k += 4) {
                    float4 o = *reinterpret_cast<float4*>(st + c0 + k);
                    o.x = fmaf(a, o.x, v[k]);
                    o.y = fmaf(a, o.y, v[k + 1]);
                    o.z = fmaf(a, o.z, v[k + 2]);
                    o.w = fmaf(a, o.w, v[k + 3]);
                    *reinterpret_cast<float4*>(st + c0 + k) = o;
                }
            }
            __threadfence_block();
        }
        tc_fence_before_sync();
        __syncthreads();
    }
    tc_fence_before_sync();
    __syncthreads();
    if (warp == 0) {
        __syncwarp();
        tmem_dealloc(tmem, 512);
    }
    (void)lane;
}

// ----------------------------------------------------------------------------
// host side
// ----------------------------------------------------------------------------
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn get_encode_fn() {
    static EncodeTiledFn fn = nullptr;
    if (!fn) {
        void* ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
                cudaSuccess && q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(ptr);
    }
    return fn;
}

// Rank-3 bf16 map over (inner, mid, rows) with a (64, 1, 128) box and 128-byte swizzle.
bool make_map(CUtensorMap* m, const void* ptr, int64_t inner, int64_t mid, int64_t rows) {
    EncodeTiledFn enc = get_encode_fn();
    if (!enc) return false;
    cuuint64_t dims[3] = {(cuuint64_t)inner, (cuuint64_t)mid, (cuuint64_t)(rows > 0 ? rows : 1)};
    cuuint64_t strides[2] = {(cuuint64_t)(inner * 2), (cuuint64_t)(inner * mid * 2)};
    cuuint32_t box[3] = {64, 1, (cuuint32_t)kTileRows};
    cuuint32_t estr[3] = {1, 1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(ptr), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

bool bf16_path_supports(const ssd_shape& s, int chunk) {
    return s.headdim == 64 && (s.dstate == 64 || s.dstate == 128 || s.dstate == 256) &&
           ((s.nheads / s.ngroups) % 2 == 0) && (chunk == 64 || chunk == 128 || chunk == 256);
}

cudaError_t launch_bf16_path(const Problem& p) {
    const int H = (int)p.s.nheads, N = (int)p.s.dstate, G = (int)p.s.ngroups, Q = p.chunk;
    if (p.L.max_chunks == 0) return launch_state_pass(p);
    TcMaps maps;
    if (!make_map(&maps.x, p.x, 64, H, p.rows) || !make_map(&maps.b, p.B, N, G, p.rows) ||
        !make_map(&maps.c, p.C, N, G, p.rows))
        return cudaErrorInvalidValue;
    const int ntiles = (Q + kTileRows - 1) / kTileRows;
    const int nb = N / 64;
    dim3 grid((unsigned)p.L.max_chunks, (unsigned)(H / 2));

    const size_t smem_a = 1024 + (size_t)(2 + nb) * ntiles * kRegion;
    cudaFuncSetAttribute(chunk_state_tc, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem_a);
    prof_launch();
    chunk_state_tc<<<grid, kThreads, smem_a, p.stream>>>(maps, p.status(), p.status(), p.chunks(), p.dt, p.A,
                                                         p.decay(), p.states(), H, N, G, Q);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    e = launch_state_pass(p);
    if (e != cudaSuccess) return e;
    // at least 120 KB so that one CTA (and its 512 TMEM columns) owns the SM
    size_t smem_c = (size_t)(2 + 2 * nb + (nb > 2 ? nb : 2)) * kRegion + 2048 + 64;
    if (smem_c < 120 * 1024) smem_c = 120 * 1024;
    cudaFuncSetAttribute(chunk_out_tc, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem_c);
    prof_launch();
    prof_begin(p.stream, "chunk_out_tc");
    chunk_out_tc<<<grid, kThreads, smem_c, p.stream>>>(maps, p.status(), p.status(), p.chunks(), p.dt, p.A, p.D,
                                                       p.states(), (__nv_bfloat16*)p.y, H, N, G, Q);
    prof_end(p.stream);
    return cudaGetLastError();
}

}  // namespace ssd
