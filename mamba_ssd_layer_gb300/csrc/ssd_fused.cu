// ssd_fused.cu -- fused SSD forward for bf16 (tcgen05 + TMEM + TMA), one persistent CTA per SM,
// launched cooperatively.
//
// The chunked algorithm ("LLM(十一)——Mamba" §3.5) over 128-token tiles, with every intermediate kept on
// chip except one state per window of tiles:
//
//   * Work: "chains" (sequence s, head pair hp), each a run of tiles in time order, cut into windows
//     of K tiles; windows are dispatched window-rank-major (all chains' first windows, then the second
//     ones, ...), round-robin over the CTAs.
//   * Phase A (right factors): every window with a successor computes its aggregate, the state at its
//     end from a zero start, sum_t decay(t -> end) (w o X_t)^T B_t, on the tensor core (M = 2 heads x
//     64 channels, N = state size), and the decay over it.
//   * Phase B (center factors): a scan over each chain's windows, h(w+1) = decay(w) h(w) + agg(w) from
//     the initial state, gives the state entering every window.
//   * Phase C: each window's tiles in time order, the state carried in TMEM from tile to tile:
//       G  = C B^T                      tcgen05, A = C (K-major), B = B (K-major)
//       LG = L o G (+ D_h on the diagonal), bf16, written back over G in TMEM; L_ij = exp(cs_i - cs_j)
//            on the diagonal 32-blocks, exp(cs_i - cs_p) exp(cs_p - cs_j) (p the last token of j's
//            32-block, both factors <= 1) left of them, 0 above -- §3.5.1, §3.5.4
//       Yd_h = LG_h X_h                 tcgen05, A from TMEM, B = x tile (MN-major)
//       Yo   = C h_{t-1}^T              tcgen05, both heads at once (N = 128)     -- left factors
//       S_t  = (w o X)^T B              tcgen05, accumulated onto a_t h_{t-1}     -- right factors
//       y    = Yd + exp(cs_i) Yo       (the D skip rides on the L o G diagonal)
//     Two C B^T buffers in TMEM alternate between tiles (a tile's buffer later takes its Yo), so the
//     next tile's C B^T and mask overlap this tile's MMAs.
//
// Roles (576 threads): warp 0 = TMA producer (and the dt cumsums), warp 1 = MMA issuer (and TMEM
// owner), warps 2..17 = math (weights, masks, state steps, epilogue, aggregates, the scan).
// Every wait is bounded; a timeout records SSD_ERR_TIMEOUT and the CTA winds down.
#include <cuda.h>
#include <cuda_runtime.h>

#include <type_traits>

#include "ptx.cuh"
#include "ssd_internal.cuh"

namespace ssd {

namespace {

constexpr int kTile = kFusedTile;
constexpr int kRegion = kTile * 128;          // one 128-row x 128-byte swizzled box (16 KB)
constexpr int kThreads = 576;        // producer warp, MMA warp, 16 math warps
constexpr int kMathThreads = 512;
constexpr float kLog2e = 1.4426950408889634f;

// TMEM column map (512 allocated)
constexpr uint32_t kColST = 0;     // state / aggregate: rows (head, channel), N columns
constexpr uint32_t kColYD = 128;   // Yd, head 0 then head 1 (64 columns each)
constexpr uint32_t kColGB = 256;   // two 128-column buffers, alternating per tile: C B^T (fp32), then
                                   // L o C B^T (bf16 pairs) in place -- the 16 fp32 columns 16c..16c+15
                                   // become 8 packed columns of head 0 followed by 8 of head 1, both for
                                   // tokens j = 16c..16c+15 -- then that tile's Yo (rows = tokens, columns =
                                   // (head, channel))

struct FusedMaps {
    CUtensorMap x, b, c;
    CUtensorMap y;              // y as (64, H, rows), 64 x 1 x 32 boxes: one row quadrant of one head
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
    float* decay;               // per piece: [2] per-head decay of the window
    // Per piece, 128 x N fp32 in column-chunk-major order: the float4 holding row r, columns
    // 4c .. 4c + 3 is unit c * 128 + r, so that a warp (32 consecutive rows) reads or writes 512
    // contiguous bytes per column chunk.
    float* agg;                 // the window's end state from a zero entering state
    float* incl;                // the state entering the window
    const int32_t* woff;        // packed batch: first window of each sequence
    int H, G, nseq, npairs;
    int64_t npieces;            // pieces to dispatch (exact for a dense batch, a bound for a packed one)
    int K;                      // tiles per window
    int dense;                  // 1: batch of equal sequences (pieces decoded arithmetically)
    int64_t seqlen;             // dense: tokens per sequence
    int nt_dense;               // dense: tiles per sequence
    int W_dense;                // dense: windows per sequence
    // Split state: this launch covers state columns [n_off, n_off + N) of n_full (B, C, the initial
    // and final states); with y_accum its y is added onto the y already there (the other columns'
    // share), and D is left to the first launch.
    int n_off, n_full, y_accum;
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

// TMEM -> registers without waiting; pair with tmem_wait_ld() before using the values
__device__ __forceinline__ void tmem_ld16_nowait(uint32_t taddr, float* v) {
    uint32_t* r = reinterpret_cast<uint32_t*>(v);
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
}

__device__ __forceinline__ void tmem_st8(uint32_t taddr, const uint32_t* r) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};"
        :: "r"(taddr), "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7])
        : "memory");
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

// Barrier slots in shared memory
enum {
    kBarFullX0 = 0, kBarFullX1, kBarFullBC0, kBarFullBC1, kBarEmpty0, kBarEmpty1,
    kBarG, kBarLG, kBarYD, kBarST, kBarYO, kBarWX, kBarS, kBarYFree,
    kBarPair0,                       // + qd + 4 * (kq / 2): the two warps that stage one head of a row quadrant
    kNumBars = kBarPair0 + 8
};

// Expected arrivals per phase: the x barrier = producer's expect_tx + its "cumsum written"
// arrival; the B/C barrier = the expect_tx alone; math-warp signals one per math warp (16); MMA
// commits 1; a warp-pair barrier one per warp.
__device__ __forceinline__ uint32_t bar_count(int i) {
    if (i >= kBarPair0) return 2;
    switch (i) {
        case kBarFullX0: case kBarFullX1: return 2;
        case kBarLG: case kBarST: case kBarWX: case kBarYFree:
            return 16;
        default: return 1;
    }
}

// Phase A barriers (re-initialised for phase C): per stage a full barrier (expect_tx + cumsum
// arrival), an empty barrier (MMA commit) and a weights barrier (one arrival per math warp), plus
// the aggregate barrier (MMA commit after a window's last tile).
constexpr int kBarAFull0 = 0;   // + s: full, + 3 + s: empty, + 6 + s: weights, + 9: aggregate
static_assert(kBarAFull0 + 10 <= kNumBars, "phase A reuses the first ten barrier slots");
// Phase-A windows per CTA whose totals are precomputed together (more fall back to the producer)
constexpr int kMaxWinA = 96;
// phase-C cumsum table per stage: [2][128] plus 8 row-side values
constexpr int kCsStride = 264;
// floor of dt in log2(dt): dt = 0 contributes exp(-99.7) ~ 0 instead of an infinity
constexpr float kMinDt = 1e-30f;

struct Smem;
__device__ void init_bars_a(const Smem& sm);
__device__ void init_bars_c(const Smem& sm);

struct Smem {
    uint8_t* base;
    int N;
    __device__ uint32_t stage_bytes() const { return 2 * kRegion + 2 * (N / 64) * kRegion; }
    __device__ uint8_t* x(int s, int h) const { return base + s * stage_bytes() + h * kRegion; }
    __device__ uint8_t* b(int s) const { return base + s * stage_bytes() + 2 * kRegion; }
    __device__ uint8_t* c(int s) const { return base + s * stage_bytes() + 2 * kRegion + (N / 64) * kRegion; }
    __device__ uint8_t* hs() const { return base + 2 * stage_bytes(); }
    // y staging for the epilogue (x layout, one 16 KB region per head): the state staging area for
    // N = 128 (free between Yo and the next state step, both of which each warp orders for its own
    // bytes), separate regions for N = 64
    __device__ uint8_t* ystage(int h) const {
        return N >= 128 ? hs() + h * kRegion : hs() + (N / 64) * kRegion + h * kRegion;
    }
    // phase A: three stages of x (both heads) and B; their cumsums in a region phase A leaves unused
    __device__ uint8_t* xa(int s, int h) const { return base + s * (2 + N / 64) * kRegion + h * kRegion; }
    __device__ uint8_t* ba(int s) const { return xa(s, 2); }
    __device__ float* csa(int s) const {
        return reinterpret_cast<float*>(N >= 128 ? hs() : ystage(0)) + s * 260;
    }
    // phase A window totals (and their per-warp partial sums): behind the phase-A cumsums in the same
    // unused area (32 KB for either state size)
    __device__ float* tota() const { return csa(0) + 1024; }
    __device__ uint8_t* small() const { return hs() + (N / 64) * kRegion + (N >= 128 ? 0 : 2 * kRegion); }
    // per stage: the tile-local cumsum of dt*A (x log2 e) as seen from a column (token j), [2][128]:
    // cs_j, minus log2(dt_j) when the input term is dt x (exp(cs_i - table_j) is then L_ij dt_j);
    // then 8 floats per stage: per head (4 h + k) the plain cumsum at the last tokens of the first three
    // 32-token blocks (k = 0..2) and at the tile's last token (k = 3)
    __device__ float* cs(int s) const { return reinterpret_cast<float*>(small()) + s * kCsStride; }
    // exp(cs_p - table_j) per head and token j < 96, p = last token of j's 32-token block: [2][96]
    __device__ float* vt() const { return cs(0) + 2 * kCsStride; }
    __device__ uint64_t* bars() const { return reinterpret_cast<uint64_t*>(vt() + 192); }           // [kNumBars]
    __device__ uint32_t* tmem_slot() const { return reinterpret_cast<uint32_t*>(bars() + kNumBars); }
    __device__ int* abort_flag() const { return reinterpret_cast<int*>(tmem_slot() + 1); }
};

__device__ void init_bars_a(const Smem& sm) {
    for (int s = 0; s < 3; ++s) {
        mbar_init(sm.bars() + kBarAFull0 + s, 2);
        mbar_init(sm.bars() + kBarAFull0 + 3 + s, 1);
        mbar_init(sm.bars() + kBarAFull0 + 6 + s, 16);
    }
    mbar_init(sm.bars() + kBarAFull0 + 9, 1);
}

__device__ void init_bars_c(const Smem& sm) {
    for (int i = 0; i < kNumBars; ++i) mbar_init(sm.bars() + i, bar_count(i));
}

// Grid-wide barrier number k (1, 2, ...) of this launch over the arrival counter in the workspace
// header (zeroed by the preparation kernel): every CTA arrives, then waits, bounded, for all of them.
// A CTA that is already aborting, or sees another CTA's error, does not wait. Returns true if the CTA
// may go on.
__device__ bool grid_sync(const Smem& sm, const FusedArgs& a, int k);


// Bounded mbarrier wait that also gives up once the CTA is aborting.
// `phases` holds one parity bit per barrier (bit idx), kept in a register.
__device__ __forceinline__ bool wait_bar(const Smem& sm, int idx, uint32_t& phases, const FusedArgs& a) {
    uint64_t* bar = sm.bars() + idx;
    const uint32_t par = (phases >> idx) & 1u;
    phases ^= 1u << idx;
    if (mbar_try_wait(bar, par)) return true;
    const uint64_t t0 = global_timer_ns();
    for (uint32_t it = 1;; ++it) {
        if (mbar_try_wait(bar, par)) return true;   // may block for a short, hardware-chosen time
        if ((it & 63u) != 0) continue;
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

// Non-blocking: true (and the phase consumed) if the phase is already complete.
__device__ __forceinline__ bool test_bar(const Smem& sm, int idx, uint32_t& phases) {
    const uint32_t par = (phases >> idx) & 1u;
    if (!mbar_try_wait(sm.bars() + idx, par)) return false;
    phases ^= 1u << idx;
    return true;
}

// Arrive once per math warp (lane 0 after the warp's work is done).
__device__ __forceinline__ void warp_arrive(const Smem& sm, int idx) {
    __syncwarp();
    if ((threadIdx.x & 31) == 0) mbar_arrive(sm.bars() + idx);
}

__device__ bool grid_sync(const Smem& sm, const FusedArgs& a, int k) {
    __syncthreads();
    if (threadIdx.x == 0) {
        int* ctr = a.status + 4;
        __threadfence();
        atomicAdd(ctr, 1);
        volatile int* abort = sm.abort_flag();
        if (!*abort) {
            const int target = k * (int)gridDim.x;
            const uint64_t t0 = global_timer_ns();
            for (uint32_t it = 1; ld_acquire(ctr) < target; ++it) {
                if ((it & 63u) != 0) continue;
                if (*reinterpret_cast<volatile const int*>(a.status) != SSD_OK) { *abort = 1; break; }
                if (global_timer_ns() - t0 > kWaitLimitNs) {
                    record_status(a.status, SSD_ERR_TIMEOUT);
                    atomicCAS(a.status + 2, 0, 0x300 + k);
                    *abort = 1;
                    break;
                }
            }
        }
        __threadfence();
    }
    __syncthreads();
    return !*reinterpret_cast<volatile int*>(sm.abort_flag());
}

// The same among the 16 math warps only (named barrier 1 over their 512 threads): the producer and the
// MMA warp are busy with phase C meanwhile.
__device__ bool grid_sync_math(const Smem& sm, const FusedArgs& a, int k) {
    asm volatile("bar.sync 1, %0;" :: "n"(kMathThreads) : "memory");
    if (threadIdx.x == 64) {
        int* ctr = a.status + 4;
        __threadfence();
        atomicAdd(ctr, 1);
        volatile int* abort = sm.abort_flag();
        if (!*abort) {
            const int target = k * (int)gridDim.x;
            const uint64_t t0 = global_timer_ns();
            for (uint32_t it = 1; ld_acquire(ctr) < target; ++it) {
                if ((it & 63u) != 0) continue;
                if (*reinterpret_cast<volatile const int*>(a.status) != SSD_OK) { *abort = 1; break; }
                if (global_timer_ns() - t0 > kWaitLimitNs) {
                    record_status(a.status, SSD_ERR_TIMEOUT);
                    atomicCAS(a.status + 2, 0, 0x300 + k);
                    *abort = 1;
                    break;
                }
            }
        }
        __threadfence();
    }
    asm volatile("bar.sync 1, %0;" :: "n"(kMathThreads) : "memory");
    return !*reinterpret_cast<volatile int*>(sm.abort_flag());
}

// ---------------------------------------------------------------- work decomposition
// A piece is one window of K consecutive 128-token tiles of one chain (sequence s, head pair hp).
// Pieces are numbered chain-major (q = first window of the chain + w) for the published states;
// a dense batch is dispatched window-major (all chains' window 0, then window 1, ...), so that the
// pieces of one chain that run at the same time are few and a look-back stays short.
struct Piece {
    int64_t q;                 // published-state slot
    int s, hp, w;              // sequence, head pair, window
    int t0, t1, nt;            // tiles [t0, t1) of the sequence's nt tiles
    int32_t seq_row0, seq_len; // first packed row and length of the sequence
    bool valid;
};

__device__ __forceinline__ Piece decode_piece(int64_t d, const FusedArgs& a) {
    Piece p;
    p.valid = true;
    if (a.dense) {
        const int64_t nchains = (int64_t)a.nseq * a.npairs;
        const int64_t w = d / nchains, c = d % nchains;
        p.w = (int)w;
        p.s = (int)(c / a.npairs);
        p.hp = (int)(c % a.npairs);
        p.q = c * a.W_dense + w;
        p.nt = a.nt_dense;
        p.seq_row0 = (int32_t)(p.s * a.seqlen);
        p.seq_len = (int32_t)a.seqlen;
    } else {
        const int64_t total = (int64_t)a.header[3] * a.npairs;
        if (d >= total) { p.valid = false; return p; }
        int lo = 0, hi = a.nseq - 1;
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if ((int64_t)a.npairs * a.woff[mid] <= d) lo = mid; else hi = mid - 1;
        }
        const int32_t w0 = a.woff[lo], w1 = a.woff[lo + 1];
        const int64_t local = d - (int64_t)a.npairs * w0;
        const int Ws = w1 - w0;
        p.s = lo;
        p.hp = (int)(local / Ws);
        p.w = (int)(local % Ws);
        p.q = d;
        const int32_t f0 = a.seqoff[lo], f1 = a.seqoff[lo + 1];
        p.nt = f1 - f0;
        const ChunkDesc first = a.tiles[f0], last = a.tiles[f1 - 1];
        p.seq_row0 = first.row0;
        p.seq_len = last.row0 + last.len - first.row0;
    }
    p.t0 = p.w * a.K;
    p.t1 = p.t0 + a.K < p.nt ? p.t0 + a.K : p.nt;
    return p;
}

__device__ __forceinline__ int tile_row0(const Piece& c, int t) { return c.seq_row0 + kTile * t; }
__device__ __forceinline__ int tile_len(const Piece& c, int t) {
    const int rem = c.seq_len - kTile * t;
    return rem < kTile ? rem : kTile;
}

// ---------------------------------------------------------------- the kernel
// Three phases separated by grid-wide barriers (the launch is cooperative, so every CTA is resident):
//   A  right factors: every window that has a successor computes its aggregate -- the state at its
//      end from a zero start, sum_t decay(t -> end) (w o X_t)^T B_t -- and the decay over it;
//   B  center factors: a scan over each chain's windows turns the aggregates into the state entering
//      every window (starting from the initial state);
//   C  the window's tiles in time order from its entering state: diagonal blocks, left factors, the
//      state carried on chip from tile to tile, y.
// kScaleX: the input term is dt x B^T (a separate instantiation, so that the plain one carries none of it).
// kAccum: y is added onto the y already in memory (the second state-column half of N = 256).
template <int N, bool kScaleX, bool kAccum>
__global__ void __launch_bounds__(kThreads)
ssd_fused_kernel(const __grid_constant__ FusedMaps maps, const FusedArgs a) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    Smem sm;
    sm.base = smem_raw;
    sm.N = N;
    constexpr int NB = N / 64;
    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;

    if (a.header[0] != SSD_OK) return;

    // sequences without tokens: the final state is the initial state (or zero)
    if (a.final_state) {
        for (int s = blockIdx.x; s < a.nseq; s += gridDim.x) {
            if (a.dense ? a.seqlen > 0 : a.seqoff[s + 1] != a.seqoff[s]) continue;
            const int64_t n = (int64_t)a.H * 64 * N;       // (head, channel) rows x this launch's columns
            for (int64_t e = tid; e < n; e += blockDim.x) {
                const int64_t g = ((int64_t)s * a.H * 64 + e / N) * a.n_full + a.n_off + e % N;
                a.final_state[g] = a.init ? a.init[g] : 0.f;
            }
        }
    }
    const int64_t np = a.npieces;
    if (np == 0 || (a.dense && a.nt_dense == 0)) return;
    // phase C visits this CTA's windows in the reverse of phase A's order: its first tiles are then the
    // ones it aggregated last, whose x and B may still be in L2
    const int64_t pc_count = np > (int64_t)blockIdx.x ? (np - blockIdx.x + gridDim.x - 1) / gridDim.x : 0;
    // phase A visits the windows with a successor: for a dense batch the first W - 1 window ranks of
    // every chain (the dispatch order puts them first), for a packed batch every window, skipping ends
    const int64_t nA = a.dense ? (int64_t)a.nseq * a.npairs * (a.W_dense - 1) : np;

    if ((smem_u32(smem_raw) & 1023u) != 0) {      // layout needs a 1024-byte aligned base
        if (tid == 0) record_status(a.status, SSD_ERR_UNSUPPORTED);
        return;
    }
    if (tid == 0) {
        init_bars_a(sm);
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

    // math-warp geometry (warps 2..17): four per TMEM lane quadrant qd (the rows 32 qd .. 32 qd + 31
    // a warp may access); kq (0..3) picks the warp's share of the columns in every phase:
    //   L o G       16-column groups kq and 7 - kq (both heads)
    //   state       state columns kq N/4 .. (kq + 1) N/4
    //   epilogue    head kq / 2, channels 32 (kq % 2) .. + 31
    const int mt = tid - 64;                 // 0..511
    const int qd = warp & 3;
    const int kq = (warp - 2) >> 2;
    const int row = 32 * qd + lane;          // TMEM lane = tile row / (head, channel) row
    const uint32_t lane_base = tmem + ((uint32_t)(32 * qd) << 16);
    const int hrow = row >> 6, prow = row & 63;
    constexpr int NQ = N / 4;                // state columns per thread
    const int nq0 = kq * NQ;

    // TMEM state columns [c0, c0 + cnt) of this thread's row, cnt a multiple of 16
    auto st_load = [&](int c0, int cnt, float* v) {
        for (int k = 0; k < cnt; k += 16) tmem_ld16_nowait(lane_base + kColST + c0 + k, v + k);
        tmem_wait_ld();
    };
    auto st_store = [&](int c0, int cnt, const float* v) {
        for (int k = 0; k < cnt; k += 16) {
            uint32_t r[16];
#pragma unroll
            for (int e = 0; e < 16; ++e) r[e] = __float_as_uint(v[k + e]);
            tmem_st16(lane_base + kColST + c0 + k, r);
        }
    };
    // x of a stage (head regions x0 and x0 + 16 KB) scaled in place: row l of head h times
    // exp2(last_h - cs_h(l)), 0 past len (bf16 products of the bf16 inputs and the weight rounded to
    // bf16). Thread mt (0..511) takes half a row; its four 16-byte chunks are visited in a row-rotated
    // order so that a warp's accesses spread over all banks.
    auto weight_x = [&](uint8_t* x0, const float* cs, int len, float last0, float last1) {
        const int pr = mt >> 1, hh = pr >> 7, l = pr & 127, hf = mt & 1;
        const float w = (l < len) ? ex2((hh ? last1 : last0) - cs[hh * 128 + l]) : 0.f;
        const __nv_bfloat162 ww = __float2bfloat162_rn(w);
        uint8_t* rowp = x0 + hh * kRegion + l * 128 + 64 * hf;
        uint4 v[4];
#pragma unroll
        for (int cc = 0; cc < 4; ++cc) v[cc] = *reinterpret_cast<const uint4*>(rowp + 16 * ((cc + l) & 3));
#pragma unroll
        for (int cc = 0; cc < 4; ++cc) {
            __nv_bfloat162* b = reinterpret_cast<__nv_bfloat162*>(&v[cc]);
#pragma unroll
            for (int k = 0; k < 4; ++k) b[k] = __hmul2(b[k], ww);
            *reinterpret_cast<uint4*>(rowp + 16 * ((cc + l) & 3)) = v[cc];
        }
    };
    // producer: dt of a tile's tokens for both heads of the pair, 4 per lane (issued early)
    auto load_dt = [&](int row0, int len, int h0, float (&v)[2][4]) {
#pragma unroll
        for (int hh = 0; hh < 2; ++hh)
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const int l = 4 * lane + k;
                v[hh][k] = (l < len) ? __ldg(a.dt + (int64_t)(row0 + l) * a.H + h0 + hh) : 0.f;
            }
    };
    // producer: tile-local inclusive cumsum of dt*A (x log2 e) plus `carry`; cv gets this lane's four
    // values per head, carry advances by the tile's total, and cs[2][128] gets the column-side table
    // (minus log2(dt) when the input term is dt x)
    auto cumsum = [&](const float (&v)[2][4], const float (&Al)[2], float* cs, float (&carry)[2], float (&cv)[2][4]) {
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
            const float A2 = Al[hh];
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
            const float base = sc - p[3] + carry[hh];
#pragma unroll
            for (int k = 0; k < 4; ++k) cv[hh][k] = base + p[k];
            float4 col = make_float4(cv[hh][0], cv[hh][1], cv[hh][2], cv[hh][3]);
            if constexpr (kScaleX) {
                col.x -= __log2f(fmaxf(v[hh][0], kMinDt));
                col.y -= __log2f(fmaxf(v[hh][1], kMinDt));
                col.z -= __log2f(fmaxf(v[hh][2], kMinDt));
                col.w -= __log2f(fmaxf(v[hh][3], kMinDt));
            }
            *reinterpret_cast<float4*>(cs + hh * 128 + 4 * lane) = col;
            carry[hh] += __shfl_sync(0xffffffffu, sc, 31);
        }
    };

    // Totals of dt*A (x log2 e) over this CTA's phase-A windows, by every thread at once: the weights of
    // a window's tiles are decays to its end, so the producer needs them before its first tile. Each warp
    // reduces its share, then one thread per window adds the warps' partial sums in a fixed order (the
    // result must not depend on timing).
    float* totA = sm.tota();
    float* partA = totA + 2 * kMaxWinA;           // [window][warp][2]
    const int64_t myA = nA > (int64_t)blockIdx.x ? (nA - blockIdx.x + gridDim.x - 1) / gridDim.x : 0;
    const bool totA_fits = myA <= kMaxWinA;
    if (totA_fits) {
        for (int64_t k = 0; k < myA; ++k) {
            const Piece c = decode_piece(blockIdx.x + k * gridDim.x, a);
            if (!c.valid || c.t1 >= c.nt) continue;
            const int h0 = 2 * c.hp;
            const int r0 = tile_row0(c, c.t0);
            const int ntok = tile_row0(c, c.t1 - 1) + tile_len(c, c.t1 - 1) - r0;
            float s0 = 0.f, s1 = 0.f;
            for (int l = tid; l < ntok; l += blockDim.x) {
                const float2 d2 = *reinterpret_cast<const float2*>(a.dt + (int64_t)(r0 + l) * a.H + h0);
                s0 += d2.x;
                s1 += d2.y;
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
                s0 += __shfl_xor_sync(0xffffffffu, s0, o);
                s1 += __shfl_xor_sync(0xffffffffu, s1, o);
            }
            if (lane == 0) {
                partA[(k * (kThreads / 32) + warp) * 2] = s0;
                partA[(k * (kThreads / 32) + warp) * 2 + 1] = s1;
            }
        }
        __syncthreads();
        if (tid < myA) {
            const Piece c = decode_piece(blockIdx.x + (int64_t)tid * gridDim.x, a);
            if (c.valid && c.t1 < c.nt) {
                float s0 = 0.f, s1 = 0.f;
                for (int w = 0; w < kThreads / 32; ++w) {
                    s0 += partA[(tid * (kThreads / 32) + w) * 2];
                    s1 += partA[(tid * (kThreads / 32) + w) * 2 + 1];
                }
                totA[2 * tid] = s0 * __ldg(a.A + 2 * c.hp) * kLog2e;
                totA[2 * tid + 1] = s1 * __ldg(a.A + 2 * c.hp + 1) * kLog2e;
            }
        }
        __syncthreads();
    }

    // ==================================================================== phase A
    if (warp == 0) {
        // producer: per window its total dt*A first (the weights are decays to the window's end), then
        // every tile: x (both heads) and B by TMA (lane 0), the cumsum with the window carry (all lanes)
        uint32_t ph = 0, issued = 0;
        int stage = 0;
        bool ok = true;
        for (int64_t d = blockIdx.x; d < nA && ok; d += gridDim.x) {
            const Piece c = decode_piece(d, a);
            if (!c.valid) break;
            if (c.t1 >= c.nt) continue;
            const int h0 = 2 * c.hp;
            float tot0, tot1;
            if (totA_fits) {
                const int64_t k = (d - blockIdx.x) / gridDim.x;
                tot0 = totA[2 * k];
                tot1 = totA[2 * k + 1];
            } else {
                const int r0 = tile_row0(c, c.t0);
                const int ntok = tile_row0(c, c.t1 - 1) + tile_len(c, c.t1 - 1) - r0;
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
                tot0 = s0 * __ldg(a.A + h0) * kLog2e;
                tot1 = s1 * __ldg(a.A + h0 + 1) * kLog2e;
            }
            const float Al[2] = {__ldg(a.A + h0) * kLog2e, __ldg(a.A + h0 + 1) * kLog2e};
            float carry[2] = {0.f, 0.f};
            // dt of the next two tiles, loaded two tiles ahead (a load takes longer than a tile here)
            float vn[2][4], vn2[2][4];
            load_dt(tile_row0(c, c.t0), tile_len(c, c.t0), h0, vn);
            if (c.t0 + 1 < c.t1) load_dt(tile_row0(c, c.t0 + 1), tile_len(c, c.t0 + 1), h0, vn2);
            for (int t = c.t0; t < c.t1 && ok; ++t) {
                const int row0 = tile_row0(c, t), len = tile_len(c, t);
                float v[2][4], cv[2][4];
#pragma unroll
                for (int hh = 0; hh < 2; ++hh)
#pragma unroll
                    for (int k = 0; k < 4; ++k) { v[hh][k] = vn[hh][k]; vn[hh][k] = vn2[hh][k]; }
                if (t + 2 < c.t1) load_dt(tile_row0(c, t + 2), tile_len(c, t + 2), h0, vn2);
                if ((issued >> stage) & 1u) {
                    const bool w = wait_bar(sm, kBarAFull0 + 3 + stage, ph, a);   // the stage's empty barrier
                    if (!__all_sync(0xffffffffu, w)) { ok = false; break; }
                }
                issued |= 1u << stage;
                uint64_t* full = sm.bars() + kBarAFull0 + stage;
                if (lane == 0) {
                    const int g = h0 / (a.H / a.G);
                    mbar_arrive_expect_tx(full, (uint32_t)((2 + NB) * kRegion));
                    tma_load_3d(sm.xa(stage, 0), &maps.x, full, 0, h0, row0);
                    tma_load_3d(sm.xa(stage, 1), &maps.x, full, 0, h0 + 1, row0);
                    for (int k = 0; k < NB; ++k)
                        tma_load_3d(sm.ba(stage) + k * kRegion, &maps.b, full, 64 * k, g, row0);
                }
                float* cs = sm.csa(stage);
                cumsum(v, Al, cs, carry, cv);
                if (lane == 0) { cs[256] = tot0; cs[257] = tot1; }
                __syncwarp();
                if (lane == 0) mbar_arrive(full);
                stage = stage == 2 ? 0 : stage + 1;
            }
        }
        // drain: every stage's last tile consumed, so no arrival is pending when the barriers are reset
        for (int s = 0; s < 3 && ok; ++s)
            if ((issued >> s) & 1u) ok = __all_sync(0xffffffffu, wait_bar(sm, kBarAFull0 + 3 + s, ph, a));
        if (!ok) *reinterpret_cast<volatile int*>(sm.abort_flag()) = 1;
    } else if (warp == 1) {
        // MMA: S_agg += (w o X_t)^T B_t over the window's tiles (M = 2 heads x 64, N = state size)
        if (lane == 0) {
            uint32_t ph = 0;
            int stage = 0;
            bool ok = true;
            const uint32_t id_s = idesc_bf16_f32(128, N, 1, 1);
            for (int64_t d = blockIdx.x; d < nA && ok; d += gridDim.x) {
                const Piece c = decode_piece(d, a);
                if (!c.valid) break;
                if (c.t1 >= c.nt) continue;
                for (int t = c.t0; t < c.t1 && ok; ++t) {
                    ok = wait_bar(sm, kBarAFull0 + stage, ph, a) && wait_bar(sm, kBarAFull0 + 6 + stage, ph, a);
                    if (!ok) break;
                    tc_fence_after_sync();
                    for (int ks = 0; ks < 8; ++ks) {
                        const uint64_t ad = smem_desc_sw128(smem_u32(sm.xa(stage, 0) + ks * 2048), kRegion, 1024);
                        const uint64_t bd = smem_desc_sw128(smem_u32(sm.ba(stage) + ks * 2048), kRegion, 1024);
                        mma_bf16_ss(tmem + kColST, ad, bd, id_s, (ks > 0 || t > c.t0) ? 1u : 0u);
                    }
                    mma_commit(sm.bars() + kBarAFull0 + 3 + stage);
                    stage = stage == 2 ? 0 : stage + 1;
                }
                if (ok) mma_commit(sm.bars() + kBarAFull0 + 9);
            }
            if (!ok) *reinterpret_cast<volatile int*>(sm.abort_flag()) = 1;
        }
    } else {
        // math warps: weights of every tile; the window's aggregate and decay to global memory
        uint32_t ph = 0;
        int stage = 0;
        bool ok = true;
        for (int64_t d = blockIdx.x; d < nA && ok; d += gridDim.x) {
            const Piece c = decode_piece(d, a);
            if (!c.valid) break;
            if (c.t1 >= c.nt) continue;
            float tot0 = 0.f, tot1 = 0.f;
            for (int t = c.t0; t < c.t1 && ok; ++t) {
                ok = wait_bar_warp(sm, kBarAFull0 + stage, ph, a);
                if (!ok) break;
                const float* cs = sm.csa(stage);
                tot0 = cs[256];
                tot1 = cs[257];
                weight_x(sm.xa(stage, 0), cs, tile_len(c, t), tot0, tot1);
                fence_proxy_async_smem();
                warp_arrive(sm, kBarAFull0 + 6 + stage);
                stage = stage == 2 ? 0 : stage + 1;
            }
            if (!ok) break;
            ok = wait_bar_warp(sm, kBarAFull0 + 9, ph, a);
            if (!ok) break;
            tc_fence_after_sync();
            float v[NQ];
            st_load(nq0, NQ, v);
            float4* dst = reinterpret_cast<float4*>(a.agg + c.q * 128 * N) + (nq0 / 4) * 128 + row;
#pragma unroll
            for (int k = 0; k < NQ; k += 4) __stcg(dst + (k / 4) * 128, make_float4(v[k], v[k + 1], v[k + 2], v[k + 3]));
            if (mt < 2) a.decay[c.q * 2 + mt] = ex2(mt ? tot1 : tot0);
            tc_fence_before_sync();
        }
        if (!ok) *reinterpret_cast<volatile int*>(sm.abort_flag()) = 1;
    }

    // ==================================================================== phase B
    bool run = grid_sync(sm, a, 1);
    // phase C's barriers now: the producer and the MMA warp start phase C right away (its inputs do not
    // depend on phase B), while the math warps run the scan and a second grid-wide barrier of their own
    if (tid == 0) {
        init_bars_c(sm);
        fence_mbar_init();
    }
    __syncthreads();
    if (warp >= 2) {
        if (run) {
            // chain ch = (sequence s, head pair hp) with windows q0 .. q0 + W - 1; item = 4 floats of the
            // (head, channel) x state matrix: h(w + 1) = decay(w) h(w) + agg(w), h(0) = initial state
            constexpr int per_chain = 32 * N;     // float4 units in 128 x N
            const int64_t nch = (int64_t)a.nseq * a.npairs;
            for (int64_t it = (int64_t)blockIdx.x * kMathThreads + mt; it < nch * per_chain;
                 it += (int64_t)gridDim.x * kMathThreads) {
                const int64_t ch = it / per_chain;
                const int e4 = (int)(it % per_chain);
                const int s = (int)(ch / a.npairs), hp = (int)(ch % a.npairs);
                int64_t q0;
                int W;
                if (a.dense) {
                    W = a.W_dense;
                    q0 = ch * W;
                } else {
                    const int32_t w0 = a.woff[s];
                    W = a.woff[s + 1] - w0;
                    q0 = (int64_t)a.npairs * w0 + (int64_t)hp * W;
                }
                if (W <= 1) continue;
                const int r = e4 & 127, n = 4 * (e4 >> 7);     // column-chunk-major unit e4
                const int hr = r >> 6, pr = r & 63;
                float4 h = make_float4(0.f, 0.f, 0.f, 0.f);
                if (a.init)
                    h = *reinterpret_cast<const float4*>(a.init + (((int64_t)s * a.H + 2 * hp + hr) * 64 + pr) * a.n_full + a.n_off + n);
                for (int w0 = 0; w0 + 1 < W; w0 += 8) {
                    // eight windows' loads first, then the dependent updates
                    float dcy[8];
                    float4 g[8];
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        if (w0 + j + 1 < W) {
                            dcy[j] = __ldcg(a.decay + (q0 + w0 + j) * 2 + hr);
                            g[j] = __ldcg(reinterpret_cast<const float4*>(a.agg + (q0 + w0 + j) * 128 * N) + e4);
                        }
                    }
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        if (w0 + j + 1 < W) {
                            h = make_float4(fmaf(dcy[j], h.x, g[j].x), fmaf(dcy[j], h.y, g[j].y),
                                            fmaf(dcy[j], h.z, g[j].z), fmaf(dcy[j], h.w, g[j].w));
                            __stcg(reinterpret_cast<float4*>(a.incl + (q0 + w0 + j + 1) * 128 * N) + e4, h);
                        }
                    }
                }
            }
        }
        run = grid_sync_math(sm, a, 2) && run;
    }

    // ==================================================================== phase C
    if (run && warp == 0) {
        // producer: every window's tiles in time order -- B and C by TMA on the B/C barrier (they feed
        // C B^T first), x on the x barrier; the tile-local cumsum of dt*A (x log2 e); the table
        // v_j = exp(cs_p - cs_j), p the last token of j's 32-token block (j < 96), once the previous
        // tile's L o G (its only reader) is done
        uint32_t ph = 0, issued = 0, p2 = 0;
        int stage = 0;
        bool ok = true;
        for (int64_t kd = pc_count - 1; kd >= 0 && ok; --kd) {
            const int64_t d = blockIdx.x + kd * gridDim.x;
            const Piece c = decode_piece(d, a);
            if (!c.valid) continue;
            const int h0 = 2 * c.hp;
            const float Al[2] = {__ldg(a.A + h0) * kLog2e, __ldg(a.A + h0 + 1) * kLog2e};
            for (int t = c.t0; t < c.t1 && ok; ++t) {
                const int row0 = tile_row0(c, t), len = tile_len(c, t);
                float v[2][4], cv[2][4];
                load_dt(row0, len, h0, v);
                if ((issued >> stage) & 1u) {
                    const bool w = wait_bar(sm, kBarEmpty0 + stage, ph, a);
                    if (!__all_sync(0xffffffffu, w)) { ok = false; break; }
                }
                issued |= 1u << stage;
                uint64_t* fullx = sm.bars() + kBarFullX0 + stage;
                if (lane == 0) {
                    const int g = h0 / (a.H / a.G);
                    uint64_t* fullbc = sm.bars() + kBarFullBC0 + stage;
                    mbar_arrive_expect_tx(fullbc, (uint32_t)(2 * NB * kRegion));
                    for (int k = 0; k < NB; ++k) {
                        tma_load_3d(sm.b(stage) + k * kRegion, &maps.b, fullbc, 64 * k, g, row0);
                        tma_load_3d(sm.c(stage) + k * kRegion, &maps.c, fullbc, 64 * k, g, row0);
                    }
                    mbar_arrive_expect_tx(fullx, (uint32_t)(2 * kRegion));
                    tma_load_3d(sm.x(stage, 0), &maps.x, fullx, 0, h0, row0);
                    tma_load_3d(sm.x(stage, 1), &maps.x, fullx, 0, h0 + 1, row0);
                }
                float carry[2] = {0.f, 0.f};
                float* cst = sm.cs(stage);
                cumsum(v, Al, cst, carry, cv);
                // row-side values: the cumsum at tokens 31, 63, 95 and at the tile's last token (the
                // plain table already holds them)
#pragma unroll
                for (int hh = 0; hh < 2 && kScaleX; ++hh) {
                    if (lane == 7 || lane == 15 || lane == 23) cst[256 + 4 * hh + (lane >> 3)] = cv[hh][3];
                    if (lane == ((len - 1) >> 2)) {
                        const int k = (len - 1) & 3;
                        cst[256 + 4 * hh + 3] = k == 0 ? cv[hh][0] : k == 1 ? cv[hh][1] : k == 2 ? cv[hh][2] : cv[hh][3];
                    }
                }
                if (p2 > 0) {
                    const bool w = wait_bar(sm, kBarLG, ph, a);
                    if (!__all_sync(0xffffffffu, w)) { ok = false; break; }
                }
                ++p2;
                float* vt = sm.vt();
#pragma unroll
                for (int hh = 0; hh < 2; ++hh) {
                    const float piv = __shfl_sync(0xffffffffu, cv[hh][3], lane | 7);
                    float4 col = make_float4(cv[hh][0], cv[hh][1], cv[hh][2], cv[hh][3]);
                    if constexpr (kScaleX) {    // the same column-side values as the table
                        col.x -= __log2f(fmaxf(v[hh][0], kMinDt));
                        col.y -= __log2f(fmaxf(v[hh][1], kMinDt));
                        col.z -= __log2f(fmaxf(v[hh][2], kMinDt));
                        col.w -= __log2f(fmaxf(v[hh][3], kMinDt));
                    }
                    if (lane < 24)
                        *reinterpret_cast<float4*>(vt + hh * 96 + 4 * lane) =
                            make_float4(ex2(piv - col.x), ex2(piv - col.y), ex2(piv - col.z), ex2(piv - col.w));
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(fullx);
                stage ^= 1;
            }
        }
        if (!ok) *reinterpret_cast<volatile int*>(sm.abort_flag()) = 1;
    } else if (run && warp == 1) {
        // ============================================================ MMA issuer (lane 0)
        if (lane == 0) {
            uint32_t ph = 0;
            int stage = 0;
            uint32_t kt = 0;               // tiles issued so far (selects the C B^T buffer)
            const uint32_t id_g = idesc_bf16_f32(128, 128, 0, 0);
            const uint32_t id_yo = idesc_bf16_f32(128, 128, 0, 0);
            const uint32_t id_yd = idesc_bf16_f32(128, 64, 0, 1);
            const uint32_t id_s = idesc_bf16_f32(128, N, 1, 1);
            bool ok = true;
            auto issue_g = [&](int st, uint32_t gcol) {
                for (int ks = 0; ks < N / 16; ++ks) {
                    const int k = ks / 4, off = (ks % 4) * 32;
                    const uint64_t ad = smem_desc_sw128(smem_u32(sm.c(st) + k * kRegion + off), 0, 1024);
                    const uint64_t bd = smem_desc_sw128(smem_u32(sm.b(st) + k * kRegion + off), 0, 1024);
                    mma_bf16_ss(tmem + gcol, ad, bd, id_g, ks > 0 ? 1u : 0u);
                }
                mma_commit(sm.bars() + kBarG);
            };
            for (int64_t kd = pc_count - 1; kd >= 0 && ok; --kd) {
                const int64_t d = blockIdx.x + kd * gridDim.x;
                const Piece c = decode_piece(d, a);
                if (!c.valid) continue;
                // per tile t (tcgen05.mma runs in issue order, so a later MMA never overtakes an earlier
                // one's reads of the same TMEM). The tile's C B^T buffer gb holds C B^T, then L o C B^T,
                // then Yo; the other buffer gn takes C B^T of the next tile.
                //   Yd(t), both heads interleaved     needs L o G(t) in gb, the previous epilogue done
                //   G(t+1) into gn                    as soon as the next stage's B and C are there
                //   Yo(t) into gb                     needs the staged state h_{t-1}
                //   S(t)                              needs the weighted x
                for (int t = c.t0; t < c.t1 && ok; ++t) {
                    const int st = stage;
                    const uint32_t gb = kColGB + 128 * (kt & 1), gn = kColGB + 128 * ((kt + 1) & 1);
                    if (t == c.t0) {
                        ok = wait_bar(sm, kBarFullBC0 + st, ph, a);
                        if (!ok) break;
                        tc_fence_after_sync();
                        issue_g(st, gb);
                    }
                    ok = wait_bar(sm, kBarLG, ph, a) && wait_bar(sm, kBarFullX0 + st, ph, a);
                    if (ok && kt > 0) ok = wait_bar(sm, kBarYFree, ph, a);
                    if (!ok) break;
                    tc_fence_after_sync();
                    for (int ks = 0; ks < 8; ++ks) {
                        for (int h = 0; h < 2; ++h) {
                            const uint32_t acol = gb + 32 * (ks / 2) + 16 * (ks % 2) + 8 * h;
                            const uint64_t bd = smem_desc_sw128(smem_u32(sm.x(st, h) + ks * 2048), kRegion, 1024);
                            mma_bf16_ts(tmem + kColYD + 64 * h, tmem + acol, bd, id_yd, ks > 0 ? 1u : 0u);
                        }
                    }
                    mma_commit(sm.bars() + kBarYD);
                    const bool more = t + 1 < c.t1;
                    bool g_done = false;
                    if (more && test_bar(sm, kBarFullBC0 + (st ^ 1), ph)) {
                        tc_fence_after_sync();
                        issue_g(st ^ 1, gn);
                        g_done = true;
                    }
                    ok = wait_bar(sm, kBarST, ph, a);
                    if (!ok) break;
                    tc_fence_after_sync();
                    for (int ks = 0; ks < N / 16; ++ks) {
                        const int kk = ks / 4, off = (ks % 4) * 32;
                        const uint64_t ad = smem_desc_sw128(smem_u32(sm.c(st) + kk * kRegion + off), 0, 1024);
                        const uint64_t bd = smem_desc_sw128(smem_u32(sm.hs() + kk * kRegion + off), 0, 1024);
                        mma_bf16_ss(tmem + gb, ad, bd, id_yo, ks > 0 ? 1u : 0u);
                    }
                    mma_commit(sm.bars() + kBarYO);
                    if (more && !g_done) {
                        ok = wait_bar(sm, kBarFullBC0 + (st ^ 1), ph, a);
                        if (!ok) break;
                        tc_fence_after_sync();
                        issue_g(st ^ 1, gn);
                    }
                    ok = wait_bar(sm, kBarWX, ph, a);
                    if (!ok) break;
                    tc_fence_after_sync();
                    for (int ks = 0; ks < 8; ++ks) {
                        const uint64_t ad = smem_desc_sw128(smem_u32(sm.x(st, 0) + ks * 2048), kRegion, 1024);
                        const uint64_t bd = smem_desc_sw128(smem_u32(sm.b(st) + ks * 2048), kRegion, 1024);
                        mma_bf16_ss(tmem + kColST, ad, bd, id_s, 1u);
                    }
                    mma_commit(sm.bars() + kBarS);
                    mma_commit(sm.bars() + kBarEmpty0 + st);
                    stage ^= 1;
                    ++kt;
                }
            }
            if (!ok) *reinterpret_cast<volatile int*>(sm.abort_flag()) = 1;
        }
    } else if (run) {
        // ============================================================ math warps
        uint32_t ph = 0;
        int stage = 0;
        uint32_t kt = 0;                         // tiles done (selects the C B^T buffer)
        bool ok = true;
        // L o G (+ D on the diagonal) of stage st, in place over C B^T in the TMEM buffer gcol, by groups
        // of 16 columns. This thread: row i; group g holds columns j = 16 g .. 16 g + 15 and is written as
        // packed bf16 (8 columns of head 0, then 8 of head 1). A group above the diagonal block of the
        // thread's row quadrant is zero; a group left of it takes exp(cs_i - cs_p) exp(cs_p - cs_j) with p
        // the last token of the 32-token block the group lies in (both factors <= 1, no subtraction of
        // distant cumsums); the two groups of the diagonal block take exp(cs_i - cs_j) directly.
        // The causal work grows with the row quadrant, and a quadrant's rows can only be reached from the
        // warps of its own SM sub-partition. Each of those four warps takes groups kq and 7 - kq, so that
        // the two costly diagonal groups of a quadrant go to different warps.
        auto lg_group = [&](const float* cs, int g, const float* gv, bool rv, float ci0, float ci1, uint32_t col,
                            float D0, float D1) {
            uint32_t p0[8], p1[8];
            if (g < 2 * qd) {
                // the row-side cumsum at p = 32 (g / 2) + 31
                const int p = 32 * (g >> 1) + 31;
                const float cp0 = kScaleX ? cs[256 + (g >> 1)] : cs[p], cp1 = kScaleX ? cs[256 + 4 + (g >> 1)] : cs[128 + p];
                const float u0 = ex2(ci0 - cp0), u1 = ex2(ci1 - cp1);
                const float2 uu0 = make_float2(u0, u0), uu1 = make_float2(u1, u1);
                const float4* v0 = reinterpret_cast<const float4*>(sm.vt() + 16 * g);
                const float4* v1 = reinterpret_cast<const float4*>(sm.vt() + 96 + 16 * g);
#pragma unroll
                for (int k4 = 0; k4 < 4; ++k4) {
                    const float4 a4 = v0[k4], b4 = v1[k4];
                    const int e = 4 * k4;
                    const float2 g0 = make_float2(gv[e], gv[e + 1]), g1 = make_float2(gv[e + 2], gv[e + 3]);
                    const float2 ra = __fmul2_rn(g0, __fmul2_rn(uu0, make_float2(a4.x, a4.y)));
                    const float2 rb = __fmul2_rn(g1, __fmul2_rn(uu0, make_float2(a4.z, a4.w)));
                    const float2 rc = __fmul2_rn(g0, __fmul2_rn(uu1, make_float2(b4.x, b4.y)));
                    const float2 rd = __fmul2_rn(g1, __fmul2_rn(uu1, make_float2(b4.z, b4.w)));
                    p0[2 * k4] = pack_bf16x2(ra.x, ra.y);
                    p0[2 * k4 + 1] = pack_bf16x2(rb.x, rb.y);
                    p1[2 * k4] = pack_bf16x2(rc.x, rc.y);
                    p1[2 * k4 + 1] = pack_bf16x2(rd.x, rd.y);
                }
            } else if (g <= 2 * qd + 1) {
                const float4* c0p = reinterpret_cast<const float4*>(cs + 16 * g);
                const float4* c1p = reinterpret_cast<const float4*>(cs + 128 + 16 * g);
                const float2 cc0 = make_float2(ci0, ci0), cc1 = make_float2(ci1, ci1), m1 = make_float2(-1.f, -1.f);
                const int jb0 = 16 * (g - 2 * qd);      // first column relative to the diagonal block
#pragma unroll
                for (int k4 = 0; k4 < 4; ++k4) {
                    const float4 a4 = c0p[k4], b4 = c1p[k4];
                    const int e = 4 * k4;
                    const int jl = jb0 + e;               // row within the diagonal block = lane
                    const float2 da = __ffma2_rn(make_float2(a4.x, a4.y), m1, cc0);
                    const float2 db = __ffma2_rn(make_float2(a4.z, a4.w), m1, cc0);
                    const float2 dc = __ffma2_rn(make_float2(b4.x, b4.y), m1, cc1);
                    const float2 dd = __ffma2_rn(make_float2(b4.z, b4.w), m1, cc1);
                    float2 ra = __fmul2_rn(make_float2(gv[e], gv[e + 1]), make_float2(ex2(da.x), ex2(da.y)));
                    float2 rb = __fmul2_rn(make_float2(gv[e + 2], gv[e + 3]), make_float2(ex2(db.x), ex2(db.y)));
                    float2 rc = __fmul2_rn(make_float2(gv[e], gv[e + 1]), make_float2(ex2(dc.x), ex2(dc.y)));
                    float2 rd = __fmul2_rn(make_float2(gv[e + 2], gv[e + 3]), make_float2(ex2(dd.x), ex2(dd.y)));
                    if (jl > lane) { ra.x = 0.f; rc.x = 0.f; }
                    if (jl + 1 > lane) { ra.y = 0.f; rc.y = 0.f; }
                    if (jl + 2 > lane) { rb.x = 0.f; rd.x = 0.f; }
                    if (jl + 3 > lane) { rb.y = 0.f; rd.y = 0.f; }
                    if (jl == lane) { ra.x += D0; rc.x += D1; }
                    if (jl + 1 == lane) { ra.y += D0; rc.y += D1; }
                    if (jl + 2 == lane) { rb.x += D0; rd.x += D1; }
                    if (jl + 3 == lane) { rb.y += D0; rd.y += D1; }
                    p0[2 * k4] = pack_bf16x2(ra.x, ra.y);
                    p0[2 * k4 + 1] = pack_bf16x2(rb.x, rb.y);
                    p1[2 * k4] = pack_bf16x2(rc.x, rc.y);
                    p1[2 * k4 + 1] = pack_bf16x2(rd.x, rd.y);
                }
            } else {
#pragma unroll
                for (int e = 0; e < 8; ++e) { p0[e] = 0u; p1[e] = 0u; }
            }
            if (!rv) {
#pragma unroll
                for (int e = 0; e < 8; ++e) { p0[e] = 0u; p1[e] = 0u; }
            }
            tmem_st8(col, p0);
            tmem_st8(col + 8, p1);
        };
        // this warp's two column groups of L o G for stage st into buffer gcol
        // lgd: log2(dt) of this thread's row per head when the input term is dt x (else 0), turning the
        // column-side table entry of the row into its row-side cumsum. Returns exp(cs_i) of the row for
        // head kq / 2, which the tile's epilogue needs.
        auto lg_tile = [&](int st, int len, uint32_t gcol, float D0, float D1, const float (&lgd)[2]) {
            const float* cs = sm.cs(st);
            const bool rv = row < len;
            float ci0 = 0.f, ci1 = 0.f, e_out = 0.f;
            if constexpr (kScaleX) {
                ci0 = cs[row] + lgd[0];
                ci1 = cs[128 + row] + lgd[1];
                e_out = ex2((kq >> 1) ? ci1 : ci0);
            }
            const uint32_t ca = lane_base + gcol + 16 * kq, cb = lane_base + gcol + 16 * (7 - kq);
            if (!__any_sync(0xffffffffu, rv)) {
                uint32_t z[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) z[e] = 0u;
                tmem_st8(ca, z);
                tmem_st8(ca + 8, z);
                tmem_st8(cb, z);
                tmem_st8(cb + 8, z);
            } else {
                float gv[32];
                tmem_ld16_nowait(ca, gv);
                tmem_ld16_nowait(cb, gv + 16);
                if constexpr (!kScaleX) {
                    ci0 = cs[row];
                    ci1 = cs[128 + row];
                }
                tmem_wait_ld();
                lg_group(cs, kq, gv, rv, ci0, ci1, ca, D0, D1);
                lg_group(cs, 7 - kq, gv + 16, rv, ci0, ci1, cb, D0, D1);
            }
            tmem_wait_st();
            tc_fence_before_sync();
            warp_arrive(sm, kBarLG);
            return e_out;
        };
        // dt of this thread's row of a tile, per head (only needed when the input term is dt x)
        auto load_row_dt = [&](int row0, int len, int h0, float (&d)[2]) {
            d[0] = d[1] = 1.f;
            if (kScaleX && row < len) {
                const float2 v = *reinterpret_cast<const float2*>(a.dt + (int64_t)(row0 + row) * a.H + h0);
                d[0] = v.x;
                d[1] = v.y;
            }
        };
        auto log2_row_dt = [&](const float (&d)[2], float (&lgd)[2]) {
            lgd[0] = kScaleX ? __log2f(fmaxf(d[0], kMinDt)) : 0.f;
            lgd[1] = kScaleX ? __log2f(fmaxf(d[1], kMinDt)) : 0.f;
        };
        // state step of stage st: h_{t-1} (this thread's state columns) to bf16 in the staging area for
        // Yo, and a_t h_{t-1} back into TMEM for S(t) to accumulate onto
        // The two warps (kq = 2 hh, 2 hh + 1) of a row quadrant that stage head hh's rows meet on their
        // own barrier (bounded like every wait, so an aborting partner cannot leave the other stuck).
        // Both take every meeting point in the same order, so its phases stay in step.
        auto pair_sync = [&]() {
            const int idx = kBarPair0 + qd + 4 * (kq >> 1);
            warp_arrive(sm, idx);
            return wait_bar_warp(sm, idx, ph, a);
        };
        // the staging bytes of this warp pair's last bulk store may be overwritten once the store has
        // read them: the issuing lane waits for that, then the pair meets
        auto ystage_release = [&]() {
            if ((kq & 1) == 0 && lane == 0) bulk_wait_read_all();
            return pair_sync();
        };
        auto state_step = [&](int st, int len) {
            // the state's TMEM load is in flight while the warp pair meets (it touches no shared memory)
            float v[NQ];
            for (int k = 0; k < NQ; k += 16) tmem_ld16_nowait(lane_base + kColST + nq0 + k, v + k);
            const bool released = ystage_release();
            tmem_wait_ld();
            if (!released) return false;
            const float* cs = sm.cs(st);
            // the tile's decay (row-side cumsum at its last token)
            const float at = ex2(kScaleX ? cs[256 + 4 * hrow + 3] : cs[hrow * 128 + len - 1]);
            const float2 aa = make_float2(at, at);
#pragma unroll
            for (int cc = 0; cc < NQ; cc += 8) {
                const int n = nq0 + cc;
                uint4 pk;
                pk.x = pack_bf16x2(v[cc], v[cc + 1]);
                pk.y = pack_bf16x2(v[cc + 2], v[cc + 3]);
                pk.z = pack_bf16x2(v[cc + 4], v[cc + 5]);
                pk.w = pack_bf16x2(v[cc + 6], v[cc + 7]);
                *reinterpret_cast<uint4*>(sm.hs() + (n / 64) * kRegion + sw128_offset(row, (n % 64) / 8)) = pk;
            }
#pragma unroll
            for (int e = 0; e < NQ; e += 2) {
                const float2 s2 = __fmul2_rn(make_float2(v[e], v[e + 1]), aa);
                v[e] = s2.x;
                v[e + 1] = s2.y;
            }
            st_store(nq0, NQ, v);
            tmem_wait_st();
            return true;
        };
        // y = Yd + e Yo for row i, head kq / 2, channels 32 (kq % 2) .. + 31, with e = exp(cs_i) (read
        // from the stage before it was released: the stage may be refilled by now) and Yo in buffer gcol.
        // The warp stages its 32 rows x 64 bytes (x layout). A row quadrant that lies wholly inside the
        // sequence goes out as one bulk tensor store per head; otherwise (and when adding onto y) the
        // warp writes its rows back four lanes per row, so that each store instruction covers eight
        // whole 64-byte row pieces. For N = 128 the staging bytes are exactly those this warp's state
        // step writes (state columns kq N/4 .. = head kq / 2's region, chunks 4 (kq % 2) ..); the state
        // step first waits until the bulk store has read them (ystage_release).
        auto epilogue = [&](float e, int len, int row0, int h0, uint32_t gcol) {
            const int hh = kq >> 1, c0 = 32 * (kq & 1);
            const int i = row;
            const float2 ee = make_float2(e, e);
            uint8_t* stg = sm.ystage(hh);
            float yd[32], yo[32];
            tmem_ld16_nowait(lane_base + kColYD + 64 * hh + c0, yd);
            tmem_ld16_nowait(lane_base + gcol + 64 * hh + c0, yo);
            tmem_ld16_nowait(lane_base + kColYD + 64 * hh + c0 + 16, yd + 16);
            tmem_ld16_nowait(lane_base + gcol + 64 * hh + c0 + 16, yo + 16);
            tmem_wait_ld();
#pragma unroll
            for (int k = 0; k < 32; k += 8) {
                uint4 v;
                uint32_t* vu = reinterpret_cast<uint32_t*>(&v);
#pragma unroll
                for (int m = 0; m < 4; ++m) {
                    const float2 r = __ffma2_rn(ee, make_float2(yo[k + 2 * m], yo[k + 2 * m + 1]),
                                                make_float2(yd[k + 2 * m], yd[k + 2 * m + 1]));
                    vu[m] = pack_bf16x2(r.x, r.y);
                }
                *reinterpret_cast<uint4*>(stg + sw128_offset(i, (c0 + k) / 8)) = v;
            }
            if (kAccum ? 32 * qd + 32 <= len : (!a.y_accum && 32 * qd + 32 <= len)) {
                // the quadrant's 32 rows all belong to the sequence: the two warps holding its two halves
                // of the head's 64 channels meet, and one bulk tensor store writes the 4 KB (with kAccum
                // a bulk reduction adds them onto the y in memory: the bf16 sum of two bf16 values, as
                // in the loop below)
                fence_proxy_async_smem();
                if (!pair_sync()) return false;
                if ((kq & 1) == 0 && lane == 0) {
                    if constexpr (kAccum)
                        tma_reduce_add_3d(&maps.y, stg + 32 * qd * 128, 0, h0 + hh, row0 + 32 * qd);
                    else
                        tma_store_3d(&maps.y, stg + 32 * qd * 128, 0, h0 + hh, row0 + 32 * qd);
                    bulk_commit_group();
                }
                return true;
            }
            __syncwarp();
            const int cl = (c0 >> 3) + (lane & 3);          // 16-byte chunk of the row this lane writes
            if constexpr (kAccum) {
                // add onto the other state columns' share, in fp32; the four old pieces are loaded
                // before any store (as far as the compiler knows a store could alias a later load,
                // which would serialise the loads)
                uint4 old[4];
#pragma unroll
                for (int pass = 0; pass < 4; ++pass) {
                    const int r = 32 * qd + 8 * pass + (lane >> 2);
                    old[pass] = make_uint4(0u, 0u, 0u, 0u);
                    if (r < len)
                        old[pass] = __ldcs(reinterpret_cast<const uint4*>(
                            a.y + ((int64_t)(row0 + r) * a.H + h0 + hh) * 64 + 8 * cl));
                }
#pragma unroll
                for (int pass = 0; pass < 4; ++pass) {
                    const int r = 32 * qd + 8 * pass + (lane >> 2);
                    if (r < len) {
                        uint4 v = *reinterpret_cast<const uint4*>(stg + sw128_offset(r, cl));
                        const uint32_t* ov = reinterpret_cast<const uint32_t*>(&old[pass]);
                        uint32_t* nv = reinterpret_cast<uint32_t*>(&v);
#pragma unroll
                        for (int m = 0; m < 4; ++m) {
                            const float2 f = __fadd2_rn(unpack_bf16x2(nv[m]), unpack_bf16x2(ov[m]));
                            nv[m] = pack_bf16x2(f.x, f.y);
                        }
                        *reinterpret_cast<uint4*>(a.y + ((int64_t)(row0 + r) * a.H + h0 + hh) * 64 + 8 * cl) = v;
                    }
                }
            } else {
                // the general loop: it also handles a.y_accum, although the accumulating launches take
                // the kAccum instantiation (this text keeps the plain instantiations' code unchanged)
#pragma unroll
                for (int pass = 0; pass < 4; ++pass) {
                    const int r = 32 * qd + 8 * pass + (lane >> 2);
                    if (r < len) {
                        uint4 v = *reinterpret_cast<const uint4*>(stg + sw128_offset(r, cl));
                        uint4* dst = reinterpret_cast<uint4*>(a.y + ((int64_t)(row0 + r) * a.H + h0 + hh) * 64 + 8 * cl);
                        if (a.y_accum) {
                            // add onto the other state columns' share, in fp32
                            const uint4 o = *dst;
                            const uint32_t* ov = reinterpret_cast<const uint32_t*>(&o);
                            uint32_t* nv = reinterpret_cast<uint32_t*>(&v);
#pragma unroll
                            for (int m = 0; m < 4; ++m) {
                                const float2 f = __fadd2_rn(unpack_bf16x2(nv[m]), unpack_bf16x2(ov[m]));
                                nv[m] = pack_bf16x2(f.x, f.y);
                            }
                        }
                        *dst = v;
                    }
                }
            }
            __syncwarp();
            return true;
        };

        for (int64_t kd = pc_count - 1; kd >= 0 && ok; --kd) {
            const int64_t d = blockIdx.x + kd * gridDim.x;
            const Piece c = decode_piece(d, a);
            if (!c.valid) continue;
            const int h0 = 2 * c.hp;
            const float Dlg0 = a.D ? __ldg(a.D + h0) : 0.f;
            const float Dlg1 = a.D ? __ldg(a.D + h0 + 1) : 0.f;

            // L o G of the window's first tile (it does not need the entering state)
            float dnext[2], lgd[2];
            load_row_dt(tile_row0(c, c.t0), tile_len(c, c.t0), h0, dnext);
            ok = wait_bar_warp(sm, kBarFullX0 + stage, ph, a) && wait_bar_warp(sm, kBarG, ph, a);
            if (!ok) break;
            tc_fence_after_sync();
            log2_row_dt(dnext, lgd);
            float e_next = lg_tile(stage, tile_len(c, c.t0), kColGB + 128 * (kt & 1), Dlg0, Dlg1, lgd);

            // the entering state into this thread's state columns: the initial state (or zero) at a
            // chain's start, else the scan's result
            {
                // the initial state is (row, column) row-major; the scan's result is column-chunk-major
                const float* src = c.w == 0
                    ? (a.init ? a.init + (((int64_t)c.s * a.H + h0 + hrow) * 64 + prow) * a.n_full + a.n_off + nq0 : nullptr)
                    : a.incl + c.q * 128 * N;
                const int step = c.w == 0 ? 4 : 512;
                const float* s0 = c.w == 0 ? src : src + ((nq0 / 4) * 128 + row) * 4;
                float v[NQ];
#pragma unroll
                for (int k = 0; k < NQ; k += 4) {
                    const float4 i4 = src ? __ldcg(reinterpret_cast<const float4*>(s0 + (k / 4) * step)) : make_float4(0.f, 0.f, 0.f, 0.f);
                    v[k] = i4.x; v[k + 1] = i4.y; v[k + 2] = i4.z; v[k + 3] = i4.w;
                }
                st_store(nq0, NQ, v);
                tmem_wait_st();
            }

            for (int t = c.t0; t < c.t1 && ok; ++t) {
                const int st = stage;
                const int len = tile_len(c, t);
                const int row0 = tile_row0(c, t);
                const float* cs = sm.cs(st);
                if (t != c.t0) {
                    ok = wait_bar_warp(sm, kBarS, ph, a);
                    if (!ok) break;
                }
                tc_fence_after_sync();
                // exp(cs_i) for this tile's epilogue (read before the stage can be refilled)
                const float e_row = kScaleX ? e_next : ex2(cs[(kq >> 1) * 128 + row]);
                if (kScaleX && t + 1 < c.t1) load_row_dt(tile_row0(c, t + 1), tile_len(c, t + 1), h0, dnext);
                ok = state_step(st, len);
                if (!ok) break;
                fence_proxy_async_smem();
                tc_fence_before_sync();
                warp_arrive(sm, kBarST);
                ok = wait_bar_warp(sm, kBarYD, ph, a);
                if (!ok) break;
                if constexpr (kScaleX)
                    weight_x(sm.x(st, 0), cs, len, cs[256 + 3], cs[256 + 7]);
                else
                    weight_x(sm.x(st, 0), cs, len, cs[len - 1], cs[128 + len - 1]);
                fence_proxy_async_smem();
                warp_arrive(sm, kBarWX);
                if (t + 1 < c.t1) {
                    ok = wait_bar_warp(sm, kBarFullX0 + (st ^ 1), ph, a) && wait_bar_warp(sm, kBarG, ph, a);
                    if (!ok) break;
                    tc_fence_after_sync();
                    log2_row_dt(dnext, lgd);
                    e_next = lg_tile(st ^ 1, tile_len(c, t + 1), kColGB + 128 * ((kt + 1) & 1), Dlg0, Dlg1, lgd);
                }
                ok = wait_bar_warp(sm, kBarYO, ph, a);
                if (!ok) break;
                tc_fence_after_sync();
                ok = epilogue(e_row, len, row0, h0, kColGB + 128 * (kt & 1));
                if (!ok) break;
                fence_proxy_async_smem();
                tc_fence_before_sync();
                warp_arrive(sm, kBarYFree);
                stage ^= 1;
                ++kt;
            }
            if (!ok) break;
            // end of the window: the last S, then the final state at a chain end (each thread only
            // touches its own state columns, so the next window may park its state right after)
            ok = wait_bar_warp(sm, kBarS, ph, a);
            if (!ok) break;
            tc_fence_after_sync();
            if (c.t1 == c.nt && a.final_state) {
                float* fp = a.final_state + (((int64_t)c.s * a.H + h0 + hrow) * 64 + prow) * a.n_full + a.n_off + nq0;
                float v[NQ];
                st_load(nq0, NQ, v);
#pragma unroll
                for (int k = 0; k < NQ; k += 4)
                    *reinterpret_cast<float4*>(fp + k) = make_float4(v[k], v[k + 1], v[k + 2], v[k + 3]);
            }
            tc_fence_before_sync();
        }
        // the bulk stores of y issued by this lane complete before the CTA's shared memory goes away
        if ((kq & 1) == 0 && lane == 0) bulk_wait_all();
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

// 3-D view (inner, mid, rows) of a bf16 tensor whose mid and row strides are mid_stride and row_stride
// elements (inner is contiguous), boxes of 64 x 1 x box_rows with the 128-byte swizzle
bool make_map_fused(CUtensorMap* m, const void* ptr, int64_t inner, int64_t mid, int64_t rows, int64_t mid_stride,
                    int64_t row_stride, int box_rows = kTile) {
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
    cuuint64_t strides[2] = {(cuuint64_t)(mid_stride * 2), (cuuint64_t)(row_stride * 2)};
    cuuint32_t box[3] = {64, 1, (cuuint32_t)box_rows};
    cuuint32_t estr[3] = {1, 1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(ptr), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int N>
size_t fused_smem_bytes() {
    const size_t stage = 2 * kRegion + 2 * (N / 64) * kRegion;
    return 2 * stage + (N / 64) * kRegion + (N >= 128 ? 0 : 2 * kRegion) + (2 * kCsStride + 192) * 4 + kNumBars * 8 + 16;
}

template <int N, bool kScaleX, bool kAccum>
cudaError_t launch_fused_n(const Problem& p, const FusedArgs& fa, const FusedMaps& maps, int grid) {
    const size_t smem = fused_smem_bytes<N>();
    cudaError_t e = note_cuda_error("fused smem attribute",
        cudaFuncSetAttribute(ssd_fused_kernel<N, kScaleX, kAccum>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem));
    if (e != cudaSuccess) return e;
    int per_sm = 0;
    e = note_cuda_error("fused occupancy",
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, ssd_fused_kernel<N, kScaleX, kAccum>, kThreads, smem));
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
    prof_launch();
    return note_cuda_error("fused cooperative launch", cudaLaunchKernelEx(&cfg, ssd_fused_kernel<N, kScaleX, kAccum>, maps, fa));
}

}  // namespace


void fused_plan(const Problem& p, int* K_out, int64_t* np_out) {
    const int64_t npairs = p.s.nheads / 2;
    const int grid = p.num_sms < kFusedMaxGrid ? p.num_sms : kFusedMaxGrid;
    if (!p.varlen) {
        // dense: pick the window K (tiles per piece) with the lowest estimated time, in units of one
        // tile of phase C (measured on GB300): the busiest CTA's phase-C windows, K tiles plus about
        // one tile of fixed work each; its phase-A windows at about 0.27 of a tile per tile; and the
        // scan over all windows with a successor, about 0.008 of a tile per window
        const int64_t nt = (p.s.seqlen + kFusedTile - 1) / kFusedTile;
        const int64_t nchains = p.s.batch * npairs;
        int bestK = kFusedMinWindow;
        double best = 1e300;
        for (int K = kFusedMinWindow; K <= kFusedMaxWindow; ++K) {
            const int64_t W = (nt + K - 1) / K;
            const int64_t np = nchains * W, nA = nchains * (W - 1);
            const int64_t rounds = (np + grid - 1) / grid, rounds_a = (nA + grid - 1) / grid;
            const double cost = (double)rounds * (K + 1.0) + 0.27 * (double)rounds_a * K + 0.008 * (double)nA;
            if (cost < best - 1e-9) { best = cost; bestK = K; }
        }
        *K_out = bestK;
        *np_out = nchains * ((nt + bestK - 1) / bestK);
    } else {
        // packed batch: windows of 8 tiles; the piece count is bounded here, exact on the device
        const int K = 8;
        *K_out = K;
        const int64_t max_tiles = p.L.max_chunks;
        *np_out = npairs * ((max_tiles - p.nseq + K - 1) / K + p.nseq);
    }
}

cudaError_t launch_fused(const Problem& p, int K, int64_t np, int part) {
    const int H = (int)p.s.nheads, Nf = (int)p.s.dstate, G = (int)p.s.ngroups;
    const int N = Nf > 128 ? 128 : Nf;            // state columns per launch
    const int64_t npairs = H / 2;
    FusedMaps maps;
    const __nv_bfloat16* Bp = static_cast<const __nv_bfloat16*>(p.B) + (int64_t)part * N;
    const __nv_bfloat16* Cp = static_cast<const __nv_bfloat16*>(p.C) + (int64_t)part * N;
    if (!make_map_fused(&maps.x, p.x, 64, H, p.rows, 64, (int64_t)64 * H) ||
        !make_map_fused(&maps.b, Bp, N, G, p.rows, Nf, (int64_t)Nf * G) ||
        !make_map_fused(&maps.c, Cp, N, G, p.rows, Nf, (int64_t)Nf * G) ||
        !make_map_fused(&maps.y, p.y, 64, H, p.rows, 64, (int64_t)64 * H, 32))
        return note_cuda_error("fused tensor maps", cudaErrorInvalidValue);
    const int grid = p.num_sms < kFusedMaxGrid ? p.num_sms : kFusedMaxGrid;
    FusedArgs fa;
    fa.header = p.status();
    fa.status = p.status();
    fa.tiles = p.chunks();
    fa.seqoff = p.seqoff();
    fa.woff = p.varlen ? p.woff() : nullptr;
    fa.dt = p.dt;
    fa.A = p.A;
    fa.D = part == 0 ? p.D : nullptr;
    fa.init = p.init;
    fa.final_state = p.final_state;
    fa.y = (__nv_bfloat16*)p.y;
    fa.decay = reinterpret_cast<float*>(p.ws + p.L.pdecay);
    fa.agg = reinterpret_cast<float*>(p.ws + p.L.agg);
    fa.incl = reinterpret_cast<float*>(p.ws + p.L.incl);
    fa.H = H;
    fa.G = G;
    fa.nseq = (int)p.nseq;
    fa.npairs = (int)npairs;
    fa.npieces = np;
    fa.K = K;
    fa.dense = p.varlen ? 0 : 1;
    fa.seqlen = p.s.seqlen;
    fa.nt_dense = (int)((p.s.seqlen + kFusedTile - 1) / kFusedTile);
    fa.W_dense = (fa.nt_dense + K - 1) / K;
    fa.n_off = part * N;
    fa.n_full = Nf;
    fa.y_accum = part > 0 ? 1 : 0;
    cudaError_t e;
    prof_begin(p.stream, "ssd_fused_kernel");
    if (fa.y_accum)      // only the second half of N = 256, which runs the N = 128 kernel
        e = p.scale_x_by_dt ? launch_fused_n<128, true, true>(p, fa, maps, grid)
                            : launch_fused_n<128, false, true>(p, fa, maps, grid);
    else if (p.scale_x_by_dt)
        e = (N == 64) ? launch_fused_n<64, true, false>(p, fa, maps, grid) : launch_fused_n<128, true, false>(p, fa, maps, grid);
    else
        e = (N == 64) ? launch_fused_n<64, false, false>(p, fa, maps, grid) : launch_fused_n<128, false, false>(p, fa, maps, grid);
    prof_end(p.stream);
    return e;
}

}  // namespace ssd
