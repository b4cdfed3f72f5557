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

__device__ __forceinline__ float2 bf2_to_f2(uint32_t u) {
    return __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u));
}

__device__ __forceinline__ uint32_t f2_to_bf2(float a, float b) {
    const __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<const uint32_t*>(&h);
}

// silu(z) = z * logistic(z), with the fast exponential and division; below -80, where it is smaller than
// 2e-33 in magnitude, it is taken as 0 (the divisor of the quotient would overflow)
__device__ __forceinline__ float silu_f(float z) { return z < -80.f ? 0.f : __fdividef(z, 1.f + __expf(-z)); }

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
                mbar_arrive_expect_tx(full + s, a.z ? 2 * rowb : rowb);
                bulk_load(st, a.y + i * C, rowb, full + s);
                if (a.z) bulk_load(st + rowb, a.z + i * C, rowb, full + s);
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
    const int team = tid / kTeamThreads, r = tid % kTeamThreads;
    float* tpart = part + team * 2 * gpad;
    const int nvec = C / 8;
    // the group of piece j: (8 j + 4) / gsize rounded down, in float (exact enough: 8 j + 4 lies at least 4
    // channels inside its group, and gsize is at most 8192)
    const float inv_gsize = 1.f / (float)a.gsize;
    auto group_of = [&](int j) { return (int)((float)(8 * j + 4) * inv_gsize); };
    int n = 0;                                               // tokens this team has taken
    for (int k = team; blockIdx.x + (int64_t)k * gridDim.x < a.rows; k += kNormTeams, ++n) {
        const int64_t i = blockIdx.x + (int64_t)k * gridDim.x;
        const int s = k % S;
        if (!norm_wait(full + s, (uint32_t)((k / S) & 1), &stop)) break;
        const uint4* yv = reinterpret_cast<const uint4*>(smem + (size_t)s * stb);
        const uint4* zv = reinterpret_cast<const uint4*>(smem + (size_t)s * stb + rowb);
        float* ps = tpart + (n & 1) * gpad;
        // v = y * silu(z), kept in registers; v^2 summed per group: a warp takes 32 consecutive 8-channel
        // pieces, sums each run of lanes in the same group (groups are contiguous), and the run's first lane
        // adds it to the group's total
        const int lane = tid & 31;
        float v[kNormVecs][8];
#pragma unroll
        for (int m = 0; m < kNormVecs; ++m) {
            const int j = r + m * kTeamThreads;
            if (j - lane >= nvec) break;                     // (the whole warp is past the row)
            float ss = 0.f;
            int grp = -1;
            if (j < nvec) {
                const uint4 yy = yv[j];
                const uint32_t* uy = reinterpret_cast<const uint32_t*>(&yy);
                uint4 zz4 = make_uint4(0u, 0u, 0u, 0u);
                if (a.z) zz4 = zv[j];
                const uint32_t* uz = reinterpret_cast<const uint32_t*>(&zz4);
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    float2 f = bf2_to_f2(uy[e]);
                    if (a.z) {
                        const float2 zz = bf2_to_f2(uz[e]);
                        f.x *= silu_f(zz.x);
                        f.y *= silu_f(zz.y);
                    }
                    v[m][2 * e] = f.x;
                    v[m][2 * e + 1] = f.y;
                    ss = fmaf(f.x, f.x, fmaf(f.y, f.y, ss));
                }
                grp = group_of(j);
            }
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const float t = __shfl_down_sync(0xffffffffu, ss, o);
                const int tg = __shfl_down_sync(0xffffffffu, grp, o);
                if (lane + o < 32 && tg == grp) ss += t;
            }
            const int prev = __shfl_up_sync(0xffffffffu, grp, 1);
            if (grp >= 0 && (lane == 0 || prev != grp)) atomicAdd(ps + grp, ss);
        }
        // (the team's other buffer is cleared for its next token: its sums were last read a token ago)
        for (int g = r; g < groups; g += kTeamThreads) tpart[((n + 1) & 1) * gpad + g] = 0.f;
        team_sync(team);
        // out = v * rsqrt(mean + eps) * weight
        __nv_bfloat16* orow = a.out + i * C;
#pragma unroll
        for (int m = 0; m < kNormVecs; ++m) {
            const int j = r + m * kTeamThreads;
            if (j < nvec) {
                const float rinv = rsqrtf(ps[group_of(j)] * inv_gsize + a.eps);
                const float4 w0 = reinterpret_cast<const float4*>(wsm)[2 * j];
                const float4 w1 = reinterpret_cast<const float4*>(wsm)[2 * j + 1];
                uint4 o;
                o.x = f2_to_bf2(v[m][0] * rinv * w0.x, v[m][1] * rinv * w0.y);
                o.y = f2_to_bf2(v[m][2] * rinv * w0.z, v[m][3] * rinv * w0.w);
                o.z = f2_to_bf2(v[m][4] * rinv * w1.x, v[m][5] * rinv * w1.y);
                o.w = f2_to_bf2(v[m][6] * rinv * w1.z, v[m][7] * rinv * w1.w);
                reinterpret_cast<uint4*>(orow)[j] = o;
            }
        }
        // the stage and this token's sums have been read by every thread of the team
        team_sync(team);
        if (r == 0) mbar_arrive(empty + s);
    }
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
    cudaError_t e = cudaFuncSetAttribute(gated_rmsnorm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    const int64_t grid = rows < (int64_t)kNormCtasPerSm * num_sms ? rows : (int64_t)kNormCtasPerSm * num_sms;
    prof_launch();
    gated_rmsnorm_kernel<<<(unsigned)grid, kNormThreads, smem, stream>>>(a);
    return cudaGetLastError();
}

}  // namespace ssd
