// ssd_norm.cu -- the Mamba-2 block's output gate and extra normalization, after the SSD layer:
//     v = y * silu(z),   out = v / sqrt(mean(v^2 over the group) + eps) * weight
// ("LLM(十一)——Mamba" §3.6.1, Block Design: the extra normalization sits after the multiplicative gate,
// before the output projection; RMSNorm over groups of channels of a token, one group by default).
//
// The normalization spans all heads of a token (or of a group of heads), while the fused SSD kernel holds
// two heads per CTA, so it is a pass of its own over y, bound by HBM: 6 bytes per channel (y and z in, out
// back). Two persistent CTAs per SM take every grid-th token. A producer lane streams each token's y and
// z rows into a ring of shared-memory stages with bulk copies (cp.async.bulk, completion on an mbarrier),
// several tokens ahead; two teams of four warps take alternate tokens: a team reads a staged row into
// registers as v, sums v^2 per group (warp sums
// over the lanes of a group, then one shared-memory atomic per group and warp), then write
// out = v * rsqrt(...) * weight with 16-byte stores. Every wait is bounded; on a timeout the CTA
// stops taking tokens (out is then partly written; the call has no device-side status).
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "ptx.cuh"
#include "ssd.h"
#include "ssd_internal.cuh"
#include "ssd_norm.cuh"

namespace ssd {
namespace {

constexpr int kNormWarps = 8;                          // warps that compute; one more produces
constexpr int kNormThreads = 32 * (kNormWarps + 1);
constexpr int kNormMaxStages = 8;
constexpr int kNormCtasPerSm = 2;                      // (two teams each: four tokens in work per SM)
constexpr size_t kNormSmemBudget = 110 * 1024;
constexpr int kNormTeams = 2;                          // teams of compute warps, each on its own tokens
constexpr int kTeamThreads = 32 * kNormWarps / kNormTeams;
constexpr int kNormVecs = 6;                           // 8-channel pieces per compute thread and token
constexpr int64_t kNormMaxChannels = 8 * kNormVecs * kTeamThreads;   // 6144

struct NormArgs {
    const __nv_bfloat16* y;
    const __nv_bfloat16* z;      // null: no gate
    const float* w;              // null: ones
    __nv_bfloat16* out;          // may be y
    int64_t rows;                // tokens
    int C;                       // channels per token (H * P), a multiple of 8
    int gsize;                   // channels per group
    int stages;
    float eps;
};

// shared memory: [stages] x (y row, z row), the weight (C floats), two group-sum buffers per team, the barriers
__host__ __device__ inline size_t norm_stage_bytes(int C) { return ((size_t)4 * C + 127) / 128 * 128; }
__host__ __device__ inline size_t norm_smem_bytes(int C, int groups, int stages) {
    return (size_t)stages * norm_stage_bytes(C) + (size_t)4 * C + (size_t)8 * kNormTeams * ((groups + 1) / 2 * 2) +
           (size_t)16 * stages;
}

// pairs of fp32 in one 64-bit register, with the packed fp32 arithmetic of sm_100 and later (mul/add/fma .f32x2)
__device__ __forceinline__ uint64_t pk2(float a, float b) {
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
    return r;
}
__device__ __forceinline__ float2 upk2(uint64_t r) {
    float2 f;
    asm("mov.b64 {%0, %1}, %2;" : "=f"(f.x), "=f"(f.y) : "l"(r));
    return f;
}
__device__ __forceinline__ uint64_t mul2(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ uint64_t add2(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ uint64_t fma2(uint64_t a, uint64_t b, uint64_t c) {
    uint64_t d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}
// two bf16 (low half first) widened exactly to a pair of fp32
__device__ __forceinline__ uint64_t bf2_to_pair(uint32_t u) {
    return pk2(__uint_as_float(u << 16), __uint_as_float(u & 0xffff0000u));
}
// a pair of fp32 rounded to nearest-even bf16, low half first
__device__ __forceinline__ uint32_t pair_to_bf2(uint64_t p) {
    const float2 f = upk2(p);
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(f.y), "f"(f.x));
    return r;
}
__device__ __forceinline__ float ex2_approx(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
__device__ __forceinline__ float rcp_approx(float x) {
    float y;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// silu of a pair: z * 1 / (1 + 2^(-z log2 e)). For very negative z the power is +inf, its reciprocal 0
// and silu 0 (rcp.approx of +inf is +0); for very positive z the power is 0 and silu z.
__device__ __forceinline__ uint64_t silu2(uint64_t z) {
    const float2 t = upk2(mul2(z, pk2(-1.4426950408889634f, -1.4426950408889634f)));
    const float2 d = upk2(add2(pk2(ex2_approx(t.x), ex2_approx(t.y)), pk2(1.f, 1.f)));
    return mul2(z, pk2(rcp_approx(d.x), rcp_approx(d.y)));
}

// 1-D bulk copy global -> shared, counted on `bar` (16-byte aligned addresses, size a multiple of 16)
__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
                 :: "r"(smem_u32(dst)), "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(smem_u32(bar))
                 : "memory");
}

// the compute threads only (named barrier 1), or one team of them (named barrier 2 + team)
__device__ __forceinline__ void compute_sync() { asm volatile("bar.sync 1, %0;" :: "n"(32 * kNormWarps) : "memory"); }
__device__ __forceinline__ void team_sync(int team) {
    asm volatile("bar.sync %0, %1;" :: "r"(2 + team), "n"(kTeamThreads) : "memory");
}

// bounded wait; false after about two seconds or once `stop` is set
__device__ __forceinline__ bool norm_wait(uint64_t* bar, uint32_t parity, volatile int* stop) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    for (uint32_t it = 1;; ++it) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((it & 7u) != 0) continue;
        if (*stop) return false;
        if (global_timer_ns() - t0 > kWaitLimitNs) { *stop = 1; return false; }
    }
}

// NV: 8-channel pieces a compute thread holds per token (ceil(C / 8 / kTeamThreads)); kGated: z is given
template <int NV, bool kGated>
__global__ void __launch_bounds__(kNormThreads, kNormCtasPerSm) gated_rmsnorm_kernel(const NormArgs a) {
    extern __shared__ __align__(128) uint8_t smem[];
    const int C = a.C, S = a.stages, groups = C / a.gsize;
    const size_t stb = norm_stage_bytes(C);
    float* wsm = reinterpret_cast<float*>(smem + (size_t)S * stb);
    const int gpad = (groups + 1) / 2 * 2;
    float* part = wsm + C;                                   // [team][2][gpad]
    uint64_t* full = reinterpret_cast<uint64_t*>(part + 2 * kNormTeams * gpad);
    uint64_t* empty = full + S;
    __shared__ int stop;
    const int tid = threadIdx.x, warp = tid >> 5;
    if (tid == 0) {
        for (int s = 0; s < S; ++s) { mbar_init(full + s, 1); mbar_init(empty + s, 1); }
        stop = 0;
        fence_mbar_init();
    }
    __syncthreads();
    const uint32_t rowb = (uint32_t)C * 2;
    if (warp == kNormWarps) {
        // ---- producer (one lane): token k of this CTA into stage k % S
        if ((tid & 31) == 0) {
            int k = 0, issued[kNormMaxStages] = {};
            for (int64_t i = blockIdx.x; i < a.rows; i += gridDim.x, ++k) {
                const int s = k % S;
                if (k >= S && !norm_wait(empty + s, (uint32_t)((k / S - 1) & 1), &stop)) break;
                uint8_t* st = smem + (size_t)s * stb;
                mbar_arrive_expect_tx(full + s, kGated ? 2 * rowb : rowb);
                bulk_load(st, a.y + i * C, rowb, full + s);
                if (kGated) bulk_load(st + rowb, a.z + i * C, rowb, full + s);
                ++issued[s];
            }
            // the copies issued land before the CTA's shared memory goes away
            for (int s = 0; s < S; ++s)
                if (issued[s] > 0) {
                    const uint64_t t0 = global_timer_ns();
                    while (!mbar_try_wait(full + s, (uint32_t)((issued[s] - 1) & 1)))
                        if (global_timer_ns() - t0 > kWaitLimitNs) break;
                }
        }
        return;
    }
    // ---- compute warps: the weight into shared memory, both group-sum buffers cleared
    for (int c = tid; c < C; c += 32 * kNormWarps) wsm[c] = a.w ? a.w[c] : 1.f;
    for (int g = tid; g < 2 * kNormTeams * gpad; g += 32 * kNormWarps) part[g] = 0.f;
    compute_sync();
    // team t takes this CTA's tokens k = t, t + kNormTeams, ...; its thread r holds pieces r + m * kTeamThreads
    const int team = tid / kTeamThreads, r = tid % kTeamThreads, lane = tid & 31;
    float* tpart = part + team * 2 * gpad;
    const int nvec = C / 8;
    const float inv_gsize = 1.f / (float)a.gsize;
    // Each thread's pieces, and so their groups, are the same for every token; so is which lanes of the
    // warp share a group. Worked out once: grp[m] (-1 past the row), and per piece the bits of the segmented
    // warp sum: bit o (o = 0..4) adds the partial sum of lane + 2^o (same group, inside the warp and the row),
    // bit 5 marks the first lane of a run of one group, which adds the run's sum to the group's total.
    int grp[NV];
    uint32_t segbits[NV];
#pragma unroll
    for (int m = 0; m < NV; ++m) {
        const int j = r + m * kTeamThreads;
        // the group of piece j: (8 j + 4) / gsize rounded down, in float (exact enough: 8 j + 4 lies at least
        // 4 channels inside its group, and gsize is at most 6144)
        grp[m] = j < nvec ? (int)((float)(8 * j + 4) * inv_gsize) : -1;
        uint32_t bits = 0;
#pragma unroll
        for (int b = 0; b < 5; ++b) {
            const int tg = __shfl_down_sync(0xffffffffu, grp[m], 1 << b);
            if (lane + (1 << b) < 32 && tg == grp[m] && grp[m] >= 0) bits |= 1u << b;
        }
        const int prev = __shfl_up_sync(0xffffffffu, grp[m], 1);
        if (grp[m] >= 0 && (lane == 0 || prev != grp[m])) bits |= 1u << 5;
        segbits[m] = bits;
    }
    int n = 0;                                               // tokens this team has taken
    for (int k = team; blockIdx.x + (int64_t)k * gridDim.x < a.rows; k += kNormTeams, ++n) {
        const int64_t i = blockIdx.x + (int64_t)k * gridDim.x;
        const int s = k % S;
        if (!norm_wait(full + s, (uint32_t)((k / S) & 1), &stop)) break;
        const uint4* yv = reinterpret_cast<const uint4*>(smem + (size_t)s * stb);
        const uint4* zv = reinterpret_cast<const uint4*>(smem + (size_t)s * stb + rowb);
        float* ps = tpart + (n & 1) * gpad;
        // v = y * silu(z) for every piece, kept in registers as fp32 pairs, and each piece's sum of v^2
        uint64_t v[NV][4];
        float ss[NV];
#pragma unroll
        for (int m = 0; m < NV; ++m) {
            const int j = r + m * kTeamThreads;
            uint4 yy = make_uint4(0u, 0u, 0u, 0u), zz = make_uint4(0u, 0u, 0u, 0u);
            if (grp[m] >= 0) {
                yy = yv[j];
                if (kGated) zz = zv[j];
            }
            const uint32_t* uy = reinterpret_cast<const uint32_t*>(&yy);
            const uint32_t* uz = reinterpret_cast<const uint32_t*>(&zz);
            uint64_t acc = pk2(0.f, 0.f);
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                uint64_t f = bf2_to_pair(uy[e]);
                if (kGated) f = mul2(f, silu2(bf2_to_pair(uz[e])));
                v[m][e] = f;
                acc = fma2(f, f, acc);
            }
            const float2 a2 = upk2(acc);
            ss[m] = a2.x + a2.y;
        }
        // segmented warp sums: a warp holds 32 consecutive pieces, and groups are contiguous runs of pieces
#pragma unroll
        for (int b = 0; b < 5; ++b) {
#pragma unroll
            for (int m = 0; m < NV; ++m) {
                const float t = __shfl_down_sync(0xffffffffu, ss[m], 1 << b);
                if (segbits[m] & (1u << b)) ss[m] += t;
            }
        }
#pragma unroll
        for (int m = 0; m < NV; ++m)
            if (segbits[m] & (1u << 5)) atomicAdd(ps + grp[m], ss[m]);
        // (the team's other buffer is cleared for its next token: its sums were last read a token ago)
        for (int g = r; g < groups; g += kTeamThreads) tpart[((n + 1) & 1) * gpad + g] = 0.f;
        team_sync(team);
        // out = v * rsqrt(mean + eps) * weight
        __nv_bfloat16* orow = a.out + i * C;
#pragma unroll
        for (int m = 0; m < NV; ++m) {
            const int j = r + m * kTeamThreads;
            if (grp[m] >= 0) {
                const float rinv = rsqrtf(ps[grp[m]] * inv_gsize + a.eps);
                const uint64_t rr = pk2(rinv, rinv);
                const float4 w0 = reinterpret_cast<const float4*>(wsm)[2 * j];
                const float4 w1 = reinterpret_cast<const float4*>(wsm)[2 * j + 1];
                uint4 o;
                o.x = pair_to_bf2(mul2(v[m][0], mul2(pk2(w0.x, w0.y), rr)));
                o.y = pair_to_bf2(mul2(v[m][1], mul2(pk2(w0.z, w0.w), rr)));
                o.z = pair_to_bf2(mul2(v[m][2], mul2(pk2(w1.x, w1.y), rr)));
                o.w = pair_to_bf2(mul2(v[m][3], mul2(pk2(w1.z, w1.w), rr)));
                reinterpret_cast<uint4*>(orow)[j] = o;
            }
        }
        // the stage and this token's sums have been read by every thread of the team
        team_sync(team);
        if (r == 0) mbar_arrive(empty + s);
    }
}

template <int NV, bool kGated>
cudaError_t launch_norm(const NormArgs& a, size_t smem, unsigned grid, cudaStream_t stream) {
    cudaError_t e = cudaFuncSetAttribute(gated_rmsnorm_kernel<NV, kGated>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    prof_launch();
    prof_begin(stream, "gated_rmsnorm_kernel");
    gated_rmsnorm_kernel<NV, kGated><<<grid, kNormThreads, smem, stream>>>(a);
    const cudaError_t e2 = cudaGetLastError();
    prof_end(stream);
    return e2;
}

template <int NV>
cudaError_t launch_norm_nv(int nv, const NormArgs& a, size_t smem, unsigned grid, cudaStream_t stream) {
    if (nv == NV) return a.z ? launch_norm<NV, true>(a, smem, grid, stream) : launch_norm<NV, false>(a, smem, grid, stream);
    if constexpr (NV < kNormVecs) return launch_norm_nv<NV + 1>(nv, a, smem, grid, stream);
    return cudaErrorInvalidValue;
}

}  // namespace

int64_t norm_max_channels() { return kNormMaxChannels; }

cudaError_t launch_gated_rmsnorm(const void* y, const void* z, const float* weight, float eps, int64_t rows,
                                 int64_t channels, int groups, void* out, int num_sms, cudaStream_t stream) {
    if (rows == 0) return cudaSuccess;
    NormArgs a;
    a.y = static_cast<const __nv_bfloat16*>(y);
    a.z = static_cast<const __nv_bfloat16*>(z);
    a.w = weight;
    a.out = static_cast<__nv_bfloat16*>(out);
    a.rows = rows;
    a.C = (int)channels;
    a.gsize = (int)(channels / groups);
    a.eps = eps;
    int S = kNormMaxStages;
    while (S > 2 && norm_smem_bytes(a.C, groups, S) > kNormSmemBudget) --S;
    a.stages = S;
    const size_t smem = norm_smem_bytes(a.C, groups, S);
    const int64_t grid = rows < (int64_t)kNormCtasPerSm * num_sms ? rows : (int64_t)kNormCtasPerSm * num_sms;
    const int nv = (int)((channels / 8 + kTeamThreads - 1) / kTeamThreads);
    return launch_norm_nv<1>(nv, a, smem, (unsigned)grid, stream);
}

}  // namespace ssd
