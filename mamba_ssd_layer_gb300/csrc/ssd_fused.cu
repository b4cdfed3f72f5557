// ssd_fused.cu -- single-pass fused SSD forward for bf16 (tcgen05 + TMEM + TMA),
// one persistent CTA per SM.
//
// The chunked algorithm ("LLM(十一)——Mamba" §3.5) with every intermediate kept on
// chip except one state per piece of work:
//
//   * Work list: "chains" (sequence s, head pair hp), each a run of 128-token tiles in
//     time order; the list is chain-major and cut into equal pieces, handed out
//     round-robin to the CTAs (balanced, deterministic, no atomics).
//   * Inside a piece the state h (rows = 2 heads x 64 channels, columns = N) is
//     carried in TMEM from tile to tile:  h_t = exp(sum dtA over tile t) h_{t-1} + S_t.
//   * Across pieces: decoupled look-back. A piece whose last chain continues into the
//     next piece first computes that segment's local end state (the "right factors",
//     chunk states B^T X, from a zero start) and publishes it with the segment's decay;
//     a piece whose first chain started earlier combines its predecessors' published
//     states (the "center factors", a scalar 1-SS recurrence over pieces) until it
//     reaches an inclusive state, then publishes its own inclusive state.
//   * Per tile (M = 128 tokens):
//       G  = C B^T                      tcgen05, A = C (K-major), B = B (K-major)
//       LG = L o G (+ D_h on the diagonal), bf16, written back over G in TMEM
//            L_ij = exp(cs_i - cs_j) on the two 64x64 diagonal blocks,
//            exp(cs_i - cs_63) exp(cs_63 - cs_j) on the lower-left block (no
//            subtraction of distant cumsums), 0 above the diagonal  -- §3.5.1, §3.5.4
//       Yd_h = LG_h X_h                 tcgen05, A from TMEM, B = x tile (MN-major)
//       Yo   = C h_{t-1}^T              tcgen05, both heads at once (N = 128)     -- left factors
//       S_t  = (w o X)^T B              tcgen05, M = 2 heads x 64, N = state size -- right factors
//       y    = Yd + exp(cs_i) Yo       (the D skip rides on the LG diagonal)
//
// Warp roles (320 threads): warp 0 = TMA producer, warp 1 = MMA issuer (and TMEM owner),
// warps 2..9 = math (masks, state updates, weights, epilogue, look-back).
// Every wait is bounded; a timeout records SSD_ERR_TIMEOUT and the CTA winds down.
#include <cuda.h>
#include <cuda_runtime.h>

#include "ptx.cuh"
#include "ssd_internal.cuh"

namespace ssd {

namespace {

constexpr int kTile = kFusedTile;
constexpr int kRegion = kTile * 128;          // one 128-row x 128-byte swizzled box (16 KB)
constexpr int kThreads = 320;
constexpr int kMathThreads = 256;
constexpr int kPieceTiles = kFusedPieceTiles;  // target tiles per piece
constexpr float kLog2e = 1.4426950408889634f;

// TMEM column map (512 allocated)
constexpr uint32_t kColST = 0;     // state / aggregate: rows (head, channel), N columns
constexpr uint32_t kColG = 128;    // C B^T (fp32), then L o C B^T (bf16 pairs) in place
constexpr uint32_t kColYD = 256;   // Yd, head 0 then head 1 (64 columns each)
constexpr uint32_t kColYO = 384;   // Yo, rows = tokens, columns = (head, channel)

struct FusedMaps {
    CUtensorMap x, b, c;
};

struct FusedArgs {
    const int* header;          // status word + number of tiles
    int* status;
    const ChunkDesc* tiles;     // tile table (128-token chunks)
    const int32_t* seqoff;      // first tile of each sequence
    const float* dt;
    const float* A;
    const float* D;
    const float* init;
    float* final_state;
    __nv_bfloat16* y;
    int* flags;                 // per piece: 0 none, 1 aggregate, 2 inclusive
    float* decay;               // per piece: [2] per-head decay of the published segment
    float* agg;                 // per piece: [128][N]
    float* incl;                // per piece: [128][N]
    int H, G, nseq, npairs;
    int64_t npieces;
};

// ---------------------------------------------------------------- small helpers
__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}


__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
        "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};"
        :: "r"(taddr), "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
           "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
        : "memory");
}

__device__ __forceinline__ void tmem_st32f(uint32_t taddr, const float (&v)[32]) {
    uint32_t a[16], b[16];
#pragma unroll
    for (int k = 0; k < 16; ++k) { a[k] = __float_as_uint(v[k]); b[k] = __float_as_uint(v[16 + k]); }
    tmem_st16(taddr, a);
    tmem_st16(taddr + 16, b);
}

// TMEM -> registers without waiting; pair with tmem_wait_ld() before using the values
__device__ __forceinline__ void tmem_ld32_nowait(uint32_t taddr, float* v) {
    uint32_t* r = reinterpret_cast<uint32_t*>(v);
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
          "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
          "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr));
}

__device__ __forceinline__ void tmem_wait_ld() {
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_wait_st() {
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// D[tmem] (+)= A[tmem] * B[smem]
__device__ __forceinline__ void mma_bf16_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                            uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}"
        :: "r"(d_tmem), "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate) : "memory");
}

__device__ __forceinline__ int ld_acquire(const int* p) {
    int v;
    asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ void st_release(int* p, int v) {
    asm volatile("st.release.gpu.global.b32 [%0], %1;" :: "l"(p), "r"(v) : "memory");
}

// Barrier slots in shared memory
enum {
    kBarFull0 = 0, kBarFull1, kBarEmpty0, kBarEmpty1,
    kBarG, kBarLG, kBarYD, kBarST, kBarYO, kBarWX, kBarWX1a, kBarWX1b, kBarS, kBarYFree, kBarAgg, kBarMath,
    kBarGrpL, kBarGrpS,
    kNumBars
};

// Pass-1 weights use one barrier per stage (kBarWX1a + stage): the math warps may weight the
// next stage's tile before the MMA warp has consumed this one, and a second arrival on the same
// barrier before the first was waited for would make the waiter miss a phase.
// Expected arrivals per phase: full = producer's expect_tx + its "cumsum written" arrival;
// pass-2 signals from one math group (4 warps); pass-1 weights and the shared barrier from
// both groups (8 warps); MMA commits 1.
__device__ __forceinline__ uint32_t bar_count(int i) {
    switch (i) {
        case kBarFull0: case kBarFull1: return 2;
        case kBarLG: case kBarST: case kBarWX: case kBarYFree: case kBarGrpL: case kBarGrpS: return 4;
        case kBarWX1a: case kBarWX1b: case kBarMath: return 8;
        default: return 1;
    }
}

struct Smem {
    uint8_t* base;
    int N;
    __device__ uint32_t stage_bytes() const { return 2 * kRegion + 2 * (N / 64) * kRegion; }
    __device__ uint8_t* x(int s, int h) const { return base + s * stage_bytes() + h * kRegion; }
    __device__ uint8_t* b(int s) const { return base + s * stage_bytes() + 2 * kRegion; }
    __device__ uint8_t* c(int s) const { return base + s * stage_bytes() + 2 * kRegion + (N / 64) * kRegion; }
    __device__ uint8_t* hs() const { return base + 2 * stage_bytes(); }
    // per stage: tile-local cumsum of dt*A (x log2 e) for both heads [2][128] (pass 1: relative to
    // the segment start) and 4 floats of per-tile values (pass 1: the segment totals)
    __device__ float* cs(int s) const { return reinterpret_cast<float*>(hs() + (N / 64) * kRegion) + s * 260; }
    __device__ float* stage_misc(int s) const { return cs(s) + 256; }
    __device__ float* vtab() const { return cs(0) + 520; }                                            // [2][64]
    __device__ float* misc() const { return vtab() + 128; }                                           // [8]
    __device__ uint64_t* bars() const { return reinterpret_cast<uint64_t*>(misc() + 8); }           // [kNumBars]
    __device__ uint32_t* tmem_slot() const { return reinterpret_cast<uint32_t*>(bars() + kNumBars); }
    __device__ int* abort_flag() const { return reinterpret_cast<int*>(tmem_slot() + 1); }
};

// misc[] layout
enum { kMiscA0 = 0, kMiscA1, kMiscTot0, kMiscTot1, kMiscCarry0, kMiscCarry1, kMiscD0, kMiscD1 };

// Bounded mbarrier wait that also gives up once the CTA is aborting.
// `phases` holds one parity bit per barrier (bit idx), kept in a register.
__device__ __forceinline__ bool wait_bar(const Smem& sm, int idx, uint32_t& phases, const FusedArgs& a) {
    uint64_t* bar = sm.bars() + idx;
    const uint32_t par = (phases >> idx) & 1u;
    phases ^= 1u << idx;
    if (mbar_try_wait(bar, par)) return true;
    const uint64_t t0 = global_timer_ns();
    while (true) {
        if (mbar_try_wait(bar, par)) return true;
        if (*reinterpret_cast<volatile int*>(sm.abort_flag())) return false;
        if (global_timer_ns() - t0 > kWaitLimitNs) {
            record_status(a.status, SSD_ERR_TIMEOUT);
            atomicCAS(a.status + 2, 0, 0x100 + idx);     // which barrier gave up first (diagnostic)
            *reinterpret_cast<volatile int*>(sm.abort_flag()) = 1;
            return false;
        }
    }
}

// Math-warp version: every lane waits, then the warp agrees on the outcome, so later
// warp-collective instructions (tcgen05.ld/st, shuffles) never run diverged.
__device__ __forceinline__ bool wait_bar_warp(const Smem& sm, int idx, uint32_t& phases, const FusedArgs& a) {
    const bool ok = wait_bar(sm, idx, phases, a);
    return __all_sync(0xffffffffu, ok);
}

// Arrive once per math warp (lane 0 after the warp's work is done).
__device__ __forceinline__ void warp_arrive(const Smem& sm, int idx) {
    __syncwarp();
    if ((threadIdx.x & 31) == 0) mbar_arrive(sm.bars() + idx);
}

// ---------------------------------------------------------------- work decomposition
// A cursor over the chain-major tile list: sequence s, head pair hp, tile t of the sequence,
// the sequence's first row and length, and how many tiles of this chain the piece still holds.
struct Cursor {
    int s, hp, t, nt;
    int64_t run;
    int32_t seq_row0, seq_len;
};

__device__ __forceinline__ int64_t piece_begin(int64_t q, int64_t L, int64_t np) { return (q * L) / np; }

__device__ __forceinline__ Cursor locate(int64_t g, int64_t g_end, const int32_t* seqoff, const ChunkDesc* tiles,
                                         int nseq, int npairs) {
    // the sequence s with npairs*seqoff[s] <= g < npairs*seqoff[s+1]; empty sequences share the next
    // sequence's offset, so the largest such s is the non-empty one holding g
    int lo = 0, hi = nseq - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if ((int64_t)npairs * seqoff[mid] <= g) lo = mid; else hi = mid - 1;
    }
    Cursor c;
    c.s = lo;
    const int32_t f0 = seqoff[lo], f1 = seqoff[lo + 1];
    c.nt = f1 - f0;
    const int64_t local = g - (int64_t)npairs * f0;
    c.hp = (int)(local / c.nt);
    c.t = (int)(local % c.nt);
    const int64_t left = c.nt - c.t;
    c.run = (g_end - g) < left ? (g_end - g) : left;
    const ChunkDesc first = tiles[f0], last = tiles[f1 - 1];
    c.seq_row0 = first.row0;
    c.seq_len = last.row0 + last.len - first.row0;
    return c;
}

__device__ __forceinline__ int tile_row0(const Cursor& c, int t) { return c.seq_row0 + kTile * t; }
__device__ __forceinline__ int tile_len(const Cursor& c, int t) {
    const int rem = c.seq_len - kTile * t;
    return rem < kTile ? rem : kTile;
}

// The last chain segment of a piece (the one whose state may continue into the next piece).
__device__ __forceinline__ Cursor last_segment(int64_t g0, int64_t g1, const FusedArgs& a) {
    int64_t g = g0;
    Cursor last{};
    while (g < g1) { last = locate(g, g1, a.seqoff, a.tiles, a.nseq, a.npairs); g += last.run; }
    return last;
}

// ---------------------------------------------------------------- the kernel
template <int N>
__global__ void __launch_bounds__(kThreads, 1)
ssd_fused_kernel(const __grid_constant__ FusedMaps maps, const FusedArgs a) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    Smem sm;
    sm.base = smem_raw;
    sm.N = N;
    constexpr int NB = N / 64;
    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;

    if (a.header[0] != SSD_OK) return;
    const int total_tiles = a.header[1];
    const int64_t L = (int64_t)a.npairs * total_tiles;

    // sequences without tokens: the final state is the initial state (or zero)
    if (a.final_state) {
        for (int s = blockIdx.x; s < a.nseq; s += gridDim.x) {
            if (a.seqoff[s + 1] != a.seqoff[s]) continue;
            const int64_t n = (int64_t)a.H * 64 * N;
            for (int64_t e = tid; e < n; e += blockDim.x)
                a.final_state[(int64_t)s * n + e] = a.init ? a.init[(int64_t)s * n + e] : 0.f;
        }
    }
    if (L == 0) return;

    if ((smem_u32(smem_raw) & 1023u) != 0) {      // layout needs a 1024-byte aligned base
        if (tid == 0) record_status(a.status, SSD_ERR_UNSUPPORTED);
        return;
    }
    if (tid == 0) {
        for (int i = 0; i < kNumBars; ++i) mbar_init(sm.bars() + i, bar_count(i));
        *sm.abort_flag() = 0;
        fence_mbar_init();
    }
    if (warp == 1) {
        __syncwarp();
        tmem_alloc(sm.tmem_slot(), 512);
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem = *sm.tmem_slot();
    const int64_t np = a.npieces;

    if (warp == 0) {
        // ============================================================ producer warp
        // TMA for x (both heads), B and C (lane 0); dt for both heads -> the tile-local cumsum of
        // dt*A (x log2 e), plus the segment carry in pass 1 (all lanes), written into the stage.
        uint32_t ph = 0;
        uint32_t issued = 0;
        int stage = 0;
        bool ok = true;
        auto load_tile = [&](const Cursor& c, int t, bool pass1, float tot0, float tot1, float& carry0,
                             float& carry1) -> bool {
            if ((issued >> stage) & 1u) {
                const bool w = wait_bar(sm, kBarEmpty0 + stage, ph, a);
                if (!__all_sync(0xffffffffu, w)) return false;
            }
            issued |= 1u << stage;
            const int row0 = tile_row0(c, t), len = tile_len(c, t);
            const int h0 = 2 * c.hp;
            uint64_t* full = sm.bars() + kBarFull0 + stage;
            if (lane == 0) {
                const int g = h0 / (a.H / a.G);
                mbar_arrive_expect_tx(full, (uint32_t)((2 + (pass1 ? 1 : 2) * NB) * kRegion));
                tma_load_3d(sm.x(stage, 0), &maps.x, full, 0, h0, row0);
                tma_load_3d(sm.x(stage, 1), &maps.x, full, 0, h0 + 1, row0);
                for (int k = 0; k < NB; ++k) {
                    tma_load_3d(sm.b(stage) + k * kRegion, &maps.b, full, 64 * k, g, row0);
                    if (!pass1) tma_load_3d(sm.c(stage) + k * kRegion, &maps.c, full, 64 * k, g, row0);
                }
            }
            float v[2][4];
#pragma unroll
            for (int hh = 0; hh < 2; ++hh)
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const int l = 4 * lane + k;
                    v[hh][k] = (l < len) ? __ldg(a.dt + (int64_t)(row0 + l) * a.H + h0 + hh) : 0.f;
                }
            float* cs = sm.cs(stage);
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
                const float A2 = __ldg(a.A + h0 + hh) * kLog2e;
                float p[4];
                p[0] = v[hh][0] * A2;
#pragma unroll
                for (int k = 1; k < 4; ++k) p[k] = p[k - 1] + v[hh][k] * A2;
                float sc = p[3];
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) {
                    const float tt = __shfl_up_sync(0xffffffffu, sc, o);
                    if (lane >= o) sc += tt;
                }
                const float base = sc - p[3] + (pass1 ? (hh ? carry1 : carry0) : 0.f);
                float4 o4 = make_float4(base + p[0], base + p[1], base + p[2], base + p[3]);
                *reinterpret_cast<float4*>(cs + hh * 128 + 4 * lane) = o4;
                const float tile_total = __shfl_sync(0xffffffffu, sc, 31);
                if (pass1) { if (hh) carry1 += tile_total; else carry0 += tile_total; }
            }
            if (lane == 0) {
                float* m = sm.stage_misc(stage);
                m[0] = tot0;
                m[1] = tot1;
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(full);
            stage ^= 1;
            return true;
        };
        for (int64_t q = blockIdx.x; q < np && ok; q += gridDim.x) {
            const int64_t g0 = piece_begin(q, L, np), g1 = piece_begin(q + 1, L, np);
            if (g0 >= g1) continue;
            const Cursor last = last_segment(g0, g1, a);
            if (last.t + last.run < last.nt) {
                // pass 1: the segment's total dt*A first (its tokens' weights are decays to its end)
                const int h0 = 2 * last.hp;
                const int r0 = tile_row0(last, last.t);
                const int ntok = tile_row0(last, last.t + (int)last.run - 1) + tile_len(last, last.t + (int)last.run - 1) - r0;
                float s0 = 0.f, s1 = 0.f;
#pragma unroll 4
                for (int l = lane; l < ntok; l += 32) {
                    const float2 d2 = *reinterpret_cast<const float2*>(a.dt + (int64_t)(r0 + l) * a.H + h0);
                    s0 += d2.x;
                    s1 += d2.y;
                }
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) {
                    s0 += __shfl_xor_sync(0xffffffffu, s0, o);
                    s1 += __shfl_xor_sync(0xffffffffu, s1, o);
                }
                const float tot0 = s0 * __ldg(a.A + h0) * kLog2e, tot1 = s1 * __ldg(a.A + h0 + 1) * kLog2e;
                float c0 = 0.f, c1 = 0.f;
                for (int t = last.t; t < last.t + last.run && ok; ++t) ok = load_tile(last, t, true, tot0, tot1, c0, c1);
            }
            for (int64_t g = g0; g < g1 && ok;) {
                const Cursor c = locate(g, g1, a.seqoff, a.tiles, a.nseq, a.npairs);
                float c0 = 0.f, c1 = 0.f;
                for (int t = c.t; t < c.t + c.run && ok; ++t) ok = load_tile(c, t, false, 0.f, 0.f, c0, c1);
                g += c.run;
            }
        }
    } else if (warp == 1) {
        // ============================================================ MMA issuer (lane 0)
        if (lane == 0) {
            uint32_t ph = 0;
            int stage = 0;
            bool have_prev_tile = false;   // a pass-2 tile's Y regions are still being read
            const uint32_t id_g = idesc_bf16_f32(128, 128, 0, 0);
            const uint32_t id_yo = idesc_bf16_f32(128, 128, 0, 0);
            const uint32_t id_yd = idesc_bf16_f32(128, 64, 0, 1);
            const uint32_t id_s = idesc_bf16_f32(128, N, 1, 1);
            bool ok = true;
            auto issue_s = [&](int st, bool accumulate_first) {
                for (int ks = 0; ks < 8; ++ks) {
                    const uint64_t ad = smem_desc_sw128(smem_u32(sm.x(st, 0) + ks * 2048), kRegion, 1024);
                    const uint64_t bd = smem_desc_sw128(smem_u32(sm.b(st) + ks * 2048), kRegion, 1024);
                    mma_bf16_ss(tmem + kColST, ad, bd, id_s, (ks > 0 || accumulate_first) ? 1u : 0u);
                }
            };
            auto issue_g = [&](int st) {
                for (int ks = 0; ks < N / 16; ++ks) {
                    const int k = ks / 4, off = (ks % 4) * 32;
                    const uint64_t ad = smem_desc_sw128(smem_u32(sm.c(st) + k * kRegion + off), 0, 1024);
                    const uint64_t bd = smem_desc_sw128(smem_u32(sm.b(st) + k * kRegion + off), 0, 1024);
                    mma_bf16_ss(tmem + kColG, ad, bd, id_g, ks > 0 ? 1u : 0u);
                }
                mma_commit(sm.bars() + kBarG);
            };
            for (int64_t q = blockIdx.x; q < np && ok; q += gridDim.x) {
                const int64_t g0 = piece_begin(q, L, np), g1 = piece_begin(q + 1, L, np);
                if (g0 >= g1) continue;
                const Cursor last = last_segment(g0, g1, a);
                if (last.t + last.run < last.nt) {
                    for (int i = 0; i < last.run && ok; ++i) {
                        ok = wait_bar(sm, kBarFull0 + stage, ph, a) && wait_bar(sm, kBarWX1a + stage, ph, a);
                        if (!ok) break;
                        tc_fence_after_sync();
                        issue_s(stage, i > 0);
                        mma_commit(sm.bars() + kBarEmpty0 + stage);
                        stage ^= 1;
                    }
                    if (ok) mma_commit(sm.bars() + kBarAgg);
                }
                // pass 2, per tile t (tcgen05.mma runs in issue order, so a later MMA never overtakes an
                // earlier one's reads of the same TMEM):
                //   Yd(t), both heads interleaved       needs L o G(t), Y regions free
                //   G(t+1)                              needs the next stage; runs while the S warps
                //                                       stage the state and weight x
                //   Yo(t) and S(t), interleaved         needs the staged state and the weights
                const int64_t ntiles = g1 - g0;
                for (int64_t k = 0; k < ntiles && ok; ++k) {
                    const int st = stage;
                    if (k == 0) {
                        ok = wait_bar(sm, kBarFull0 + st, ph, a);
                        if (!ok) break;
                        tc_fence_after_sync();
                        issue_g(st);
                    }
                    ok = wait_bar(sm, kBarLG, ph, a);
                    if (ok && have_prev_tile) ok = wait_bar(sm, kBarYFree, ph, a);
                    if (!ok) break;
                    tc_fence_after_sync();
                    for (int ks = 0; ks < 8; ++ks) {
                        for (int h = 0; h < 2; ++h) {
                            const uint32_t acol = kColG + 32 * (ks / 2) + 16 * h + 8 * (ks % 2);
                            const uint64_t bd = smem_desc_sw128(smem_u32(sm.x(st, h) + ks * 2048), kRegion, 1024);
                            mma_bf16_ts(tmem + kColYD + 64 * h, tmem + acol, bd, id_yd, ks > 0 ? 1u : 0u);
                        }
                    }
                    mma_commit(sm.bars() + kBarYD);
                    if (k + 1 < ntiles) {
                        ok = wait_bar(sm, kBarFull0 + (st ^ 1), ph, a);
                        if (!ok) break;
                        tc_fence_after_sync();
                        issue_g(st ^ 1);
                    }
                    ok = wait_bar(sm, kBarST, ph, a) && wait_bar(sm, kBarWX, ph, a);
                    if (!ok) break;
                    tc_fence_after_sync();
                    for (int ks = 0; ks < 8; ++ks) {
                        if (ks < N / 16) {
                            const int kk = ks / 4, off = (ks % 4) * 32;
                            const uint64_t ad = smem_desc_sw128(smem_u32(sm.c(st) + kk * kRegion + off), 0, 1024);
                            const uint64_t bd = smem_desc_sw128(smem_u32(sm.hs() + kk * kRegion + off), 0, 1024);
                            mma_bf16_ss(tmem + kColYO, ad, bd, id_yo, ks > 0 ? 1u : 0u);
                        }
                        const uint64_t ad = smem_desc_sw128(smem_u32(sm.x(st, 0) + ks * 2048), kRegion, 1024);
                        const uint64_t bd = smem_desc_sw128(smem_u32(sm.b(st) + ks * 2048), kRegion, 1024);
                        mma_bf16_ss(tmem + kColST, ad, bd, id_s, 1u);
                    }
                    mma_commit(sm.bars() + kBarYO);
                    mma_commit(sm.bars() + kBarS);
                    mma_commit(sm.bars() + kBarEmpty0 + st);
                    stage ^= 1;
                    have_prev_tile = true;
                }
            }
        }
    } else {
        // ============================================================ math warps
        // warps 2-5 ("L" group): L o G in pass 2; warps 6-9 ("S" group): state steps, weights and
        // the epilogue in pass 2. Both groups share pass 1, publishing and the look-back.
        const int mt = tid - 64;                 // 0..255
        const bool grpL = warp < 6;
        const int gt = mt & 127;                 // thread index within its group
        const int qd = warp & 3;                 // TMEM lane quadrant this warp may access
        const int ch = grpL ? 0 : 1;             // column half in the shared phases
        const int row = 32 * qd + lane;          // TMEM lane = tile row / (head, channel) row
        const uint32_t lane_base = tmem + ((uint32_t)(32 * qd) << 16);
        const int hrow = row >> 6, prow = row & 63;
        constexpr int NH = N / 2;
        const int n0 = ch * NH;
        uint32_t ph = 0;
        int stage = 0;
        float* vt = sm.vtab();
        float* misc = sm.misc();
        bool ok = true;
        auto math_bar = [&]() {    // all 8 math warps
            warp_arrive(sm, kBarMath);
            if (!wait_bar_warp(sm, kBarMath, ph, a)) ok = false;
        };
        auto group_bar = [&]() {   // the 4 warps of this group
            warp_arrive(sm, grpL ? kBarGrpL : kBarGrpS);
            if (!wait_bar_warp(sm, grpL ? kBarGrpL : kBarGrpS, ph, a)) ok = false;
        };
        // x of stage st scaled in place: row l of head h times exp2(last_h - cs_h(l)) (0 past len)
        auto weight_x = [&](int st, int len, float last0, float last1, int first, int stride) {
            const float* cs = sm.cs(st);
            for (int qq = first; qq < 2 * kTile * 8; qq += stride) {
                const int hh = qq >> 10;
                const int l = (qq & 1023) >> 3;
                const float w = (l < len) ? ex2((hh ? last1 : last0) - cs[hh * 128 + l]) : 0.f;
                uint4* p = reinterpret_cast<uint4*>(sm.x(st, 0) + (size_t)qq * 16);
                uint4 v = *p;
                uint32_t* u = reinterpret_cast<uint32_t*>(&v);
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const float2 f = unpack_bf16x2(u[k]);
                    u[k] = pack_bf16x2(f.x * w, f.y * w);
                }
                *p = v;
            }
        };
        float hreg[NH];

        for (int64_t q = blockIdx.x; q < np && ok; q += gridDim.x) {
            const int64_t g0 = piece_begin(q, L, np), g1 = piece_begin(q + 1, L, np);
            if (g0 >= g1) continue;
            const Cursor first = locate(g0, g1, a.seqoff, a.tiles, a.nseq, a.npairs);
            const Cursor last = last_segment(g0, g1, a);
            const bool first_cont = first.t > 0;
            const bool last_cont = last.t + last.run < last.nt;
            const bool single = (first.s == last.s && first.hp == last.hp);

            // ------------------------------------------------ pass 1 (both groups)
            if (last_cont) {
                const int h0 = 2 * last.hp;
                for (int t = last.t; t < last.t + last.run && ok; ++t) {
                    ok = wait_bar_warp(sm, kBarFull0 + stage, ph, a);
                    if (!ok) break;
                    const float* m = sm.stage_misc(stage);
                    const float tot0 = m[0], tot1 = m[1];
                    if (t == last.t && mt == 0) { misc[kMiscTot0] = tot0; misc[kMiscTot1] = tot1; }
                    weight_x(stage, tile_len(last, t), tot0, tot1, mt, kMathThreads);
                    fence_proxy_async_smem();
                    warp_arrive(sm, kBarWX1a + stage);
                    stage ^= 1;
                }
                if (!ok) break;
                ok = wait_bar_warp(sm, kBarAgg, ph, a);
                if (!ok) break;
                tc_fence_after_sync();
                const float dec = ex2(misc[kMiscTot0 + hrow]);
                const int64_t slot = (q * 128 + row) * N + n0;
                const bool starts_chain = last.t == 0;
                const float* ip = (starts_chain && a.init)
                                      ? a.init + (((int64_t)last.s * a.H + h0 + hrow) * 64 + prow) * N + n0
                                      : nullptr;
                float* dst = (starts_chain ? a.incl : a.agg) + slot;
#pragma unroll
                for (int c0 = 0; c0 < NH; c0 += 32) {
                    float v[32];
                    tmem_ld32(lane_base + kColST + n0 + c0, v);
#pragma unroll
                    for (int k = 0; k < 32; k += 4) {
                        float4 o = make_float4(v[k], v[k + 1], v[k + 2], v[k + 3]);
                        if (ip) {
                            const float4 i4 = *reinterpret_cast<const float4*>(ip + c0 + k);
                            o.x = fmaf(dec, i4.x, o.x); o.y = fmaf(dec, i4.y, o.y);
                            o.z = fmaf(dec, i4.z, o.z); o.w = fmaf(dec, i4.w, o.w);
                        }
                        __stcg(reinterpret_cast<float4*>(dst + c0 + k), o);
                    }
                }
                if (!starts_chain && mt < 2) a.decay[q * 2 + mt] = ex2(misc[kMiscTot0 + mt]);
                __threadfence();
                math_bar();
                if (mt == 0) st_release(a.flags + q, starts_chain ? 2 : 1);
                tc_fence_before_sync();
            }

            // ------------------------------------------------ look-back (both groups)
            if (first_cont) {
#pragma unroll
                for (int k = 0; k < NH; ++k) hreg[k] = 0.f;
                float mult = 1.f;
                for (int64_t qq = q - 1; qq >= 0; --qq) {
                    if (piece_begin(qq, L, np) == piece_begin(qq + 1, L, np)) continue;   // empty pieces publish nothing
                    int f = 0;
                    const uint64_t t0 = global_timer_ns();
                    while (true) {
                        int verdict = 0;   // lane 0 polls and decides; the warp follows (no divergence)
                        if (lane == 0) {
                            f = ld_acquire(a.flags + qq);
                            if (f != 0) verdict = 1;
                            else if (*reinterpret_cast<volatile const int*>(a.status) != SSD_OK) verdict = 2;
                            else if (global_timer_ns() - t0 > kWaitLimitNs) {
                                record_status(a.status, SSD_ERR_TIMEOUT);
                                atomicCAS(a.status + 2, 0, 0x200);
                                verdict = 2;
                            }
                        }
                        verdict = __shfl_sync(0xffffffffu, verdict, 0);
                        f = __shfl_sync(0xffffffffu, f, 0);
                        if (verdict == 1) break;
                        if (verdict == 2) { ok = false; break; }
                    }
                    if (!ok) break;
                    const float* src = (f == 2 ? a.incl : a.agg) + (qq * 128 + row) * N + n0;
#pragma unroll
                    for (int k = 0; k < NH; k += 4) {
                        const float4 v = __ldcg(reinterpret_cast<const float4*>(src + k));
                        hreg[k] = fmaf(mult, v.x, hreg[k]);
                        hreg[k + 1] = fmaf(mult, v.y, hreg[k + 1]);
                        hreg[k + 2] = fmaf(mult, v.z, hreg[k + 2]);
                        hreg[k + 3] = fmaf(mult, v.w, hreg[k + 3]);
                    }
                    if (f == 2) break;
                    mult *= __ldcg(a.decay + qq * 2 + hrow);
                }
                if (!ok) break;
                tc_fence_after_sync();
                if (last_cont && single) {
                    // the piece lies inside one chain: inclusive = dec * h_in + aggregate (still in TMEM)
                    const float dec = ex2(misc[kMiscTot0 + hrow]);
                    float* dst = a.incl + (q * 128 + row) * N + n0;
#pragma unroll
                    for (int c0 = 0; c0 < NH; c0 += 32) {
                        float v[32];
                        tmem_ld32(lane_base + kColST + n0 + c0, v);
#pragma unroll
                        for (int k = 0; k < 32; k += 4) {
                            const float4 o = make_float4(fmaf(dec, hreg[c0 + k], v[k]), fmaf(dec, hreg[c0 + k + 1], v[k + 1]),
                                                         fmaf(dec, hreg[c0 + k + 2], v[k + 2]), fmaf(dec, hreg[c0 + k + 3], v[k + 3]));
                            __stcg(reinterpret_cast<float4*>(dst + c0 + k), o);
                        }
                    }
                    __threadfence();
                }
                // park h_in in the TMEM state columns for the first segment
#pragma unroll
                for (int c0 = 0; c0 < NH; c0 += 32) {
                    float v[32];
#pragma unroll
                    for (int k = 0; k < 32; ++k) v[k] = hreg[c0 + k];
                    tmem_st32f(lane_base + kColST + n0 + c0, v);
                }
                tmem_wait_st();
                tc_fence_before_sync();
                math_bar();
                if (last_cont && single && mt == 0) st_release(a.flags + q, 2);
            } else if (last_cont) {
                math_bar();   // the aggregate was read by both groups before the S group parks a state
            }
            if (!ok) break;

            // ------------------------------------------------ pass 2, L group: L o G (+ D on the diagonal)
            if (grpL) {
                for (int64_t g = g0; g < g1 && ok;) {
                    const Cursor c = locate(g, g1, a.seqoff, a.tiles, a.nseq, a.npairs);
                    const int h0 = 2 * c.hp;
                    const float Dlg0 = a.D ? __ldg(a.D + h0) : 0.f;
                    const float Dlg1 = a.D ? __ldg(a.D + h0 + 1) : 0.f;
                    for (int t = c.t; t < c.t + c.run && ok; ++t) {
                        const int len = tile_len(c, t);
                        ok = wait_bar_warp(sm, kBarFull0 + stage, ph, a);
                        if (!ok) break;
                        const float* cs = sm.cs(stage);
                        group_bar();   // everyone is done with the previous tile's vt
                        {
                            const int hh = gt >> 6, j = gt & 63;
                            vt[hh * 64 + j] = ex2(cs[hh * 128 + 63] - cs[hh * 128 + j]);   // exp(cs_63 - cs_j)
                        }
                        group_bar();
                        ok = ok && wait_bar_warp(sm, kBarG, ph, a);
                        if (!ok) break;
                        tc_fence_after_sync();
                        const int i = row;
                        const bool rv = i < len;
                        const float csi0 = cs[i], csi1 = cs[128 + i];
                        const float u0 = ex2(csi0 - cs[63]), u1 = ex2(csi1 - cs[128 + 63]);
#pragma unroll
                        for (int b = 0; b < 4; ++b) {
                            const int jb = 32 * b;
                            uint32_t p0[16], p1[16];
                            const bool need = rv && jb <= i;   // tcgen05.ld is warp-collective
                            if (!__any_sync(0xffffffffu, need)) {
#pragma unroll
                                for (int k = 0; k < 16; ++k) { p0[k] = 0u; p1[k] = 0u; }
                            } else {
                                float gv[32];
                                tmem_ld32(lane_base + kColG + jb, gv);
                                if (!need) {
#pragma unroll
                                    for (int k = 0; k < 32; ++k) gv[k] = 0.f;
                                }
                                if (jb < 64 && i >= 64) {
                                    // lower-left block: exp(cs_i - cs_63) exp(cs_63 - cs_j)
#pragma unroll
                                    for (int k = 0; k < 16; ++k) {
                                        const int j = jb + 2 * k;
                                        p0[k] = pack_bf16x2(gv[2 * k] * u0 * vt[j], gv[2 * k + 1] * u0 * vt[j + 1]);
                                        p1[k] = pack_bf16x2(gv[2 * k] * u1 * vt[64 + j], gv[2 * k + 1] * u1 * vt[64 + j + 1]);
                                    }
                                } else {
                                    // diagonal block: exp(cs_i - cs_j) for j <= i
#pragma unroll
                                    for (int k = 0; k < 16; ++k) {
                                        const int j = jb + 2 * k;
                                        float l00 = 0.f, l01 = 0.f, l10 = 0.f, l11 = 0.f;
                                        if (j <= i) { l00 = ex2(csi0 - cs[j]); l10 = ex2(csi1 - cs[128 + j]); }
                                        if (j + 1 <= i) { l01 = ex2(csi0 - cs[j + 1]); l11 = ex2(csi1 - cs[128 + j + 1]); }
                                        float a0 = gv[2 * k] * l00, a1 = gv[2 * k + 1] * l01;
                                        float b0 = gv[2 * k] * l10, b1 = gv[2 * k + 1] * l11;
                                        if (j == i) { a0 += Dlg0; b0 += Dlg1; }
                                        if (j + 1 == i) { a1 += Dlg0; b1 += Dlg1; }
                                        p0[k] = pack_bf16x2(a0, a1);
                                        p1[k] = pack_bf16x2(b0, b1);
                                    }
                                }
                            }
                            tmem_st16(lane_base + kColG + jb, p0);
                            tmem_st16(lane_base + kColG + jb + 16, p1);
                        }
                        tmem_wait_st();
                        tc_fence_before_sync();
                        warp_arrive(sm, kBarLG);
                        stage ^= 1;
                    }
                    g += c.run;
                }
            } else {
                // ------------------------------------------------ pass 2, S group: state, weights, epilogue
                for (int64_t g = g0; g < g1 && ok;) {
                    const Cursor c = locate(g, g1, a.seqoff, a.tiles, a.nseq, a.npairs);
                    const int h0 = 2 * c.hp;
                    if (!(g == g0 && first_cont)) {
                        // the segment starts its chain: initial state (or zero) into the TMEM state columns
                        const float* ip = (c.t == 0 && a.init) ? a.init + (((int64_t)c.s * a.H + h0 + hrow) * 64 + prow) * N : nullptr;
#pragma unroll
                        for (int c0 = 0; c0 < N; c0 += 32) {
                            float v[32];
#pragma unroll
                            for (int k = 0; k < 32; k += 4) {
                                const float4 i4 = ip ? *reinterpret_cast<const float4*>(ip + c0 + k) : make_float4(0.f, 0.f, 0.f, 0.f);
                                v[k] = i4.x; v[k + 1] = i4.y; v[k + 2] = i4.z; v[k + 3] = i4.w;
                            }
                            tmem_st32f(lane_base + kColST + c0, v);
                        }
                        tmem_wait_st();
                    }
                    for (int t = c.t; t < c.t + c.run && ok; ++t) {
                        const int len = tile_len(c, t);
                        const int row0 = tile_row0(c, t);
                        ok = wait_bar_warp(sm, kBarFull0 + stage, ph, a);
                        if (!ok) break;
                        const float* cs = sm.cs(stage);
                        const float at = ex2(cs[hrow * 128 + len - 1]);     // decay of this row's head over the tile
                        const float e0 = ex2(cs[row]), e1 = ex2(cs[128 + row]);   // exp(cs_i) for both heads
                        const float last0 = cs[len - 1], last1 = cs[128 + len - 1];
                        // ---- state step: stage h_{t-1} (bf16) for Yo and leave a_t h_{t-1} in TMEM for S
                        if (t != c.t) {
                            ok = wait_bar_warp(sm, kBarS, ph, a);
                            if (!ok) break;
                        }
                        tc_fence_after_sync();
#pragma unroll
                        for (int c0 = 0; c0 < N; c0 += 64) {
                            float v[64];
                            tmem_ld32_nowait(lane_base + kColST + c0, v);
                            tmem_ld32_nowait(lane_base + kColST + c0 + 32, v + 32);
                            tmem_wait_ld();
#pragma unroll
                            for (int k = 0; k < 64; k += 8) {
                                const int n = c0 + k;
                                uint4 pk;
                                pk.x = pack_bf16x2(v[k], v[k + 1]);
                                pk.y = pack_bf16x2(v[k + 2], v[k + 3]);
                                pk.z = pack_bf16x2(v[k + 4], v[k + 5]);
                                pk.w = pack_bf16x2(v[k + 6], v[k + 7]);
                                *reinterpret_cast<uint4*>(sm.hs() + (n / 64) * kRegion + sw128_offset(row, (n % 64) / 8)) = pk;
                            }
#pragma unroll
                            for (int k = 0; k < 64; ++k) v[k] *= at;
                            tmem_st32f(lane_base + kColST + c0, *reinterpret_cast<float(*)[32]>(v));
                            tmem_st32f(lane_base + kColST + c0 + 32, *reinterpret_cast<float(*)[32]>(v + 32));
                        }
                        tmem_wait_st();
                        fence_proxy_async_smem();
                        tc_fence_before_sync();
                        warp_arrive(sm, kBarST);
                        // ---- weights for S: x scaled in place once Yd has read it
                        ok = wait_bar_warp(sm, kBarYD, ph, a);
                        if (!ok) break;
                        weight_x(stage, len, last0, last1, gt, 128);
                        fence_proxy_async_smem();
                        warp_arrive(sm, kBarWX);
                        // ---- epilogue: y = Yd + exp(cs_i) Yo for both heads of row i
                        ok = wait_bar_warp(sm, kBarYO, ph, a);
                        if (!ok) break;
                        tc_fence_after_sync();
                        {
                            const int i = row;
#pragma unroll
                            for (int hh = 0; hh < 2; ++hh) {
                                const float e = hh ? e1 : e0;
                                __nv_bfloat16* yrow = a.y + ((int64_t)(row0 + i) * a.H + h0 + hh) * 64;
#pragma unroll
                                for (int c0 = 0; c0 < 64; c0 += 32) {
                                    float yd[32], yo[32];
                                    tmem_ld32_nowait(lane_base + kColYD + 64 * hh + c0, yd);
                                    tmem_ld32_nowait(lane_base + kColYO + 64 * hh + c0, yo);
                                    tmem_wait_ld();
                                    if (i < len) {
#pragma unroll
                                        for (int k = 0; k < 32; k += 8) {
                                            uint4 v;
                                            v.x = pack_bf16x2(fmaf(e, yo[k], yd[k]), fmaf(e, yo[k + 1], yd[k + 1]));
                                            v.y = pack_bf16x2(fmaf(e, yo[k + 2], yd[k + 2]), fmaf(e, yo[k + 3], yd[k + 3]));
                                            v.z = pack_bf16x2(fmaf(e, yo[k + 4], yd[k + 4]), fmaf(e, yo[k + 5], yd[k + 5]));
                                            v.w = pack_bf16x2(fmaf(e, yo[k + 6], yd[k + 6]), fmaf(e, yo[k + 7], yd[k + 7]));
                                            *reinterpret_cast<uint4*>(yrow + c0 + k) = v;
                                        }
                                    }
                                }
                            }
                        }
                        tc_fence_before_sync();
                        warp_arrive(sm, kBarYFree);
                        stage ^= 1;
                    }
                    if (!ok) break;
                    // end of segment: the last S, then the final state at a chain end
                    ok = wait_bar_warp(sm, kBarS, ph, a);
                    if (!ok) break;
                    tc_fence_after_sync();
                    if (c.t + c.run == c.nt && a.final_state) {
                        float* fp = a.final_state + (((int64_t)c.s * a.H + h0 + hrow) * 64 + prow) * N;
#pragma unroll
                        for (int c0 = 0; c0 < N; c0 += 32) {
                            float v[32];
                            tmem_ld32(lane_base + kColST + c0, v);
#pragma unroll
                            for (int k = 0; k < 32; k += 4)
                                *reinterpret_cast<float4*>(fp + c0 + k) = make_float4(v[k], v[k + 1], v[k + 2], v[k + 3]);
                        }
                    }
                    tc_fence_before_sync();
                    g += c.run;
                }
            }
            // both groups finish the piece before the next one's shared phases
            math_bar();
        }
        if (!ok) *reinterpret_cast<volatile int*>(sm.abort_flag()) = 1;
    }

    tc_fence_before_sync();
    __syncthreads();
    if (warp == 1) {
        __syncwarp();   // lane 0 ran the MMA loop alone: reconverge before the warp-collective dealloc
        tmem_dealloc(tmem, 512);
    }
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

bool make_map_fused(CUtensorMap* m, const void* ptr, int64_t inner, int64_t mid, int64_t rows) {
    static EncodeTiledFn enc = nullptr;
    if (!enc) {
        void* fp = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fp, 12000, cudaEnableDefault, &q) !=
                cudaSuccess || q != cudaDriverEntryPointSuccess)
            return false;
        enc = reinterpret_cast<EncodeTiledFn>(fp);
    }
    cuuint64_t dims[3] = {(cuuint64_t)inner, (cuuint64_t)mid, (cuuint64_t)(rows > 0 ? rows : 1)};
    cuuint64_t strides[2] = {(cuuint64_t)(inner * 2), (cuuint64_t)(inner * mid * 2)};
    cuuint32_t box[3] = {64, 1, (cuuint32_t)kTile};
    cuuint32_t estr[3] = {1, 1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(ptr), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int N>
size_t fused_smem_bytes() {
    const size_t stage = 2 * kRegion + 2 * (N / 64) * kRegion;
    return 2 * stage + (N / 64) * kRegion + (520 + 128 + 8) * 4 + kNumBars * 8 + 16;
}

template <int N>
cudaError_t launch_fused_n(const Problem& p, const FusedArgs& fa, const FusedMaps& maps, int grid) {
    const size_t smem = fused_smem_bytes<N>();
    cudaError_t e = note_cuda_error("fused smem attribute",
        cudaFuncSetAttribute(ssd_fused_kernel<N>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem));
    if (e != cudaSuccess) return e;
    int per_sm = 0;
    e = note_cuda_error("fused occupancy",
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, ssd_fused_kernel<N>, kThreads, smem));
    if (e != cudaSuccess) return e;
    if (per_sm < 1) return note_cuda_error("fused occupancy is zero", cudaErrorLaunchOutOfResources);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = p.stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return note_cuda_error("fused cooperative launch", cudaLaunchKernelEx(&cfg, ssd_fused_kernel<N>, maps, fa));
}

}  // namespace


int64_t fused_pieces(const Problem& p) {
    const int64_t npairs = p.s.nheads / 2;
    const int grid = p.num_sms < kFusedMaxGrid ? p.num_sms : kFusedMaxGrid;
    const int64_t L = npairs * p.L.max_chunks;
    int64_t rounds = L / ((int64_t)grid * kPieceTiles);
    if (rounds < 1) rounds = 1;
    return rounds * grid;
}

cudaError_t launch_fused(const Problem& p) {
    const int H = (int)p.s.nheads, N = (int)p.s.dstate, G = (int)p.s.ngroups;
    const int64_t npairs = H / 2;
    FusedMaps maps;
    if (!make_map_fused(&maps.x, p.x, 64, H, p.rows) || !make_map_fused(&maps.b, p.B, N, G, p.rows) ||
        !make_map_fused(&maps.c, p.C, N, G, p.rows))
        return note_cuda_error("fused tensor maps", cudaErrorInvalidValue);
    const int grid = p.num_sms < kFusedMaxGrid ? p.num_sms : kFusedMaxGrid;
    // pieces: ~kPieceTiles tiles each (sized from the tile-count bound; the kernel cuts the
    // actual list), a whole number of rounds over the grid
    const int64_t np = fused_pieces(p);
    FusedArgs fa;
    fa.header = p.status();
    fa.status = p.status();
    fa.tiles = p.chunks();
    fa.seqoff = p.seqoff();
    fa.dt = p.dt;
    fa.A = p.A;
    fa.D = p.D;
    fa.init = p.init;
    fa.final_state = p.final_state;
    fa.y = (__nv_bfloat16*)p.y;
    if (np > p.L.max_pieces) return cudaErrorInvalidValue;
    fa.flags = p.flags();
    fa.decay = reinterpret_cast<float*>(p.ws + p.L.pdecay);
    fa.agg = reinterpret_cast<float*>(p.ws + p.L.agg);
    fa.incl = reinterpret_cast<float*>(p.ws + p.L.incl);
    fa.H = H;
    fa.G = G;
    fa.nseq = (int)p.nseq;
    fa.npairs = (int)npairs;
    fa.npieces = np;
    cudaError_t e;
    prof_begin(p.stream);
    e = (N == 64) ? launch_fused_n<64>(p, fa, maps, grid) : launch_fused_n<128>(p, fa, maps, grid);
    prof_end(p.stream);
    return e;
}

}  // namespace ssd
