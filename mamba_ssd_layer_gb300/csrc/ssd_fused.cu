// ssd_fused.cu -- fused SSD forward for bf16 (tcgen05 + TMEM + TMA), one persistent CTA per SM,
// launched cooperatively (every CTA is resident, so CTAs may wait on one another).
//
// The chunked algorithm ("LLM(十一)——Mamba" §3.5) over 128-token tiles, with every intermediate kept on
// chip except one state per window of tiles:
//
//   * Work: "chains" (sequence s, head pair hp), each a run of tiles in time order, cut into windows
//     of K tiles. A CTA takes windows d = blockIdx.x, blockIdx.x + grid, ... of the dispatch order
//     (window-rank-major for a dense batch: every chain's first window, then the second ones, ...);
//     "iteration" d / grid is the round in which a window runs.
//   * Right factors: a window with a successor first computes its aggregate, the state at its end from a
//     zero start, sum_t decay(t -> end) (w o X_t)^T B_t (tcgen05, M = 2 heads x 64 channels, N = state
//     columns), and publishes it. The same CTA then reads the window's x again for its tiles, while it
//     is still in L2.
//   * Center factors (look-back): the state entering a window is the published end state of the last
//     predecessor that ran in an earlier iteration (or the initial state), carried through the
//     aggregates of the predecessors in this iteration: h = decay(w') h + agg(w'). A window whose
//     successor runs in a later iteration publishes its end state as the same fold, decay(w) h_in +
//     agg(w), as soon as it has h_in, long before its last tile. The order of every sum is fixed by the
//     dispatch alone, so results do not depend on timing.
//   * Tiles, in time order from the entering state, the state carried in TMEM:
//       G  = C B^T                      tcgen05, A = C (K-major), B = B (K-major)
//       LG = L o G, bf16, written back over G in TMEM; L_ij = exp(cs_i - cs_j) on the diagonal
//            32-blocks, exp(cs_i - cs_p) exp(cs_p - cs_j) (p the last token of j's 32-block, both
//            factors <= 1) left of them, 0 above -- §3.5.1, §3.5.4
//       Yd_h = LG_h X_h                 tcgen05, A from TMEM, B = x tile (MN-major)
//       S_t  = (w o X)^T B              tcgen05, accumulated onto a_t h_{t-1}     -- right factors
//       Yo   = C h_{t-1}^T              tcgen05, both heads at once (N = 128)     -- left factors
//       y    = Yd + D_h x + exp(cs_i) Yo, in fp32, rounded once to bf16
//
// Roles (640 threads, 20 warps), each working on its own tile of the stream so that they overlap. A
// warp reaches the TMEM lanes of quadrant warp & 3 only, so each TMEM role is a warpgroup (four
// consecutive warps, one per quadrant):
//   warp 0        TMA producer (x, B, C into a two-stage ring)
//   warp 1        MMA issuer and TMEM owner
//   warp 2        tables: per-tile cumsums of dt*A (x log2 e), the factored-mask column table,
//                 the window totals
//   warp 3        L o G of lane quadrant 3, its right two 32-column blocks (with warp 7)
//   warps 4..7    L o G, one warp per TMEM lane quadrant
//   warps 8..15   epilogue, one warpgroup per head: drains Yd (plus D x) into registers as soon as it
//                 is there, weights x in place for S, then combines with Yo and stores y
//   warps 16..19  state: the per-tile state step, window aggregates out, the look-back in, end states
// Every wait is bounded; a timeout records SSD_ERR_TIMEOUT and the CTA winds down after letting its
// copies and MMAs in flight finish.
#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "ptx.cuh"
#include "ssd_internal.cuh"

namespace ssd {

namespace {

constexpr int kTile = kFusedTile;
constexpr int kRegion = kTile * 128;          // one 128-row x 128-byte swizzled box (16 KB)
constexpr int kThreads = 640;                 // 20 warps
constexpr float kLog2e = 1.4426950408889634f;
// floor of dt in log2(dt): dt = 0 contributes exp(-99.7) ~ 0 instead of an infinity
constexpr float kMinDt = 1e-30f;
// cumsum table per stage: [2][128] plus 8 row-side values
constexpr int kCsStride = 264;
// columns of the factored-mask table (tokens of the first three 32-blocks)
constexpr int kVtCols = 96;

constexpr int kWarpProducer = 0, kWarpMMA = 1, kWarpTables = 2;
constexpr int kWarpMask = 4, kWarpEpi = 8, kWarpState = 16;   // TMEM lane quadrant = warp & 3
constexpr int kWarpMaskQ3 = 3;    // the second L o G warp of lane quadrant 3 (the quadrant with the most work)

// TMEM column map (512 allocated)
constexpr uint32_t kColST = 0;     // state / aggregate: rows (head, channel), N columns
constexpr uint32_t kColYD = 128;   // Yd, head 0 then head 1 (64 columns each)
constexpr uint32_t kColGB = 256;   // two 128-column buffers, alternating per tile: C B^T (fp32), then
                                   // L o C B^T (bf16 pairs) in place -- the 16 fp32 columns 16c..16c+15
                                   // become 8 packed columns of head 0 followed by 8 of head 1, both for
                                   // tokens j = 16c..16c+15 -- then that tile's Yo (rows = tokens, columns =
                                   // (head, channel))

// mbarriers. [2]: one per stage of the ring (by stream position p & 1) or per C B^T buffer (by the
// count of tiles c & 1). Expected arrivals in bar_count.
enum : int {
    kFullBC = 0,     // [2] B and C of the stage landed (a correction tile: C only) (TMA bytes)
    kFullX = 2,      // [2] x of the stage landed (TMA bytes)
    kTblRead = 4,    // [2] the stage's tables and record read: 8 epilogue, 5 mask and 4 state warps
    kTblAny = 6,     // [2] the stage's tables and tile record written (every position, and the end record)
    kBCFree = 8,     // [2] MMA done with the stage's B and C
    kXFree = 10,     // [2] the tile's y (staged in the stage's x) stored: 8 epilogue warps
    kGFull = 12,     // [2] C B^T in the buffer
    kLGFull = 14,    // [2] L o G in the buffer: 5 mask warps
    kGBFree = 16,    // [2] the buffer's Yo read: 8 epilogue warps
    kDrained = 18,   // [2] the stage's Yd read and x weighted (a correction tile: begun): 8 epilogue warps
    kYDFull = 20,    // Yd in TMEM
    kState = 21,     // h_{t-1} staged as bf16, a_t h_{t-1} back in TMEM (correction: h_in staged): 4 state warps
    kSO = 22,        // S(t) and Yo(t) done (correction: the correction product done)
    kVTFree = 23,    // the factored-mask table read (off-diagonal blocks done): 5 mask warps
    kNcorr = 24,     // the correction tile count written (table warp, once)
    kMmaDone = 25,   // the MMA warp's final drain
    kYDFree = 26,    // the tile's z (held in the Yd columns) read by the combine: 8 epilogue warps
    kNumBars = 27
};

__host__ __device__ constexpr uint32_t bar_count(int i) {
    return ((i >= kXFree && i < kXFree + 2) || (i >= kGBFree && i < kGBFree + 2) || (i >= kDrained && i < kDrained + 2) ||
            i == kYDFree)
               ? 8u
         : (i >= kTblRead && i < kTblRead + 2) ? 17u
         : ((i >= kLGFull && i < kLGFull + 2) || i == kVTFree) ? 5u
         : i == kState ? 4u
         : 1u;
}

// tile record flags: a correction tile; the end of this CTA's stream (no tile)
constexpr int kRecCorr = 1, kRecEnd = 2;

// Timeout location codes (workspace header word 2): 0x100 + barrier for an mbarrier wait, 0x300 for a
// look-back wait on another CTA's published state.
constexpr int kLocLookback = 0x300;

struct FusedMaps {
    CUtensorMap x, b, c;
    CUtensorMap y;              // y as (64, H, rows), 64 x 1 x 32 boxes: one row quadrant of one head
};

struct FusedArgs {
    int* status;                // workspace header: [0] status word, [2] first timeout location
    const ChunkDesc* tiles;     // tile table (packed batch)
    const int32_t* seqoff;      // first tile of each sequence (packed batch)
    const int32_t* cu;          // sequence offsets in rows (packed batch)
    const float* dt;
    const float* A;
    const float* D;
    const float* init;
    float* final_state;
    __nv_bfloat16* y;
    // Published states of a CTA's last window when it ends inside its chain (slot = the CTA):
    int* flags;                 // per slot and lane quadrant: 1 aggregate, 2 end state published
    float* decay;               // per slot and lane quadrant: decay over the window
    // Per slot, 128 x N fp32 in column-chunk-major order: the float4 holding row r, columns
    // 4c .. 4c + 3 is unit c * 128 + r, so that a warp (32 consecutive rows) reads or writes 512
    // contiguous bytes per column chunk.
    float* agg;                 // the window's end state from a zero entering state
    float* incl;                // the window's true end state
    int H, G, nseq, npairs;
    int dense;                  // 1: batch of equal sequences (chains decoded arithmetically)
    int seqlen;                 // dense: tokens per sequence
    int nt_dense;               // dense: tiles per sequence
    // Split state: this launch covers state columns [n_off, n_off + N) of n_full (B, C, the initial
    // and final states); with y_accum its y is added onto the y already there (the other columns'
    // share), and D is left to the first launch.
    int n_off, n_full, y_accum;
    uint64_t lookback_limit_ns; // limit of a wait on another CTA's published state
    int force_timeout;          // failure-detection test: every look-back waits for a state that never comes
};

// ---------------------------------------------------------------- small helpers
__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ void tmem_st8(uint32_t taddr, const uint32_t* r) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};"
        :: "r"(taddr), "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7])
        : "memory");
}

__device__ __forceinline__ void tmem_ld16_nowait(uint32_t taddr, uint32_t* r) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
}

__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t* r) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
        "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};"
        :: "r"(taddr), "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
           "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
        : "memory");
}

__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// D[tmem] (+)= A[tmem] * B[smem]
__device__ __forceinline__ void mma_bf16_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                            uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}"
        :: "r"(d_tmem), "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate) : "memory");
}

__device__ __forceinline__ float2 fmul2(float2 a, float2 b) { return __fmul2_rn(a, b); }

// Per-warpgroup register budgets (setmaxnreg): the launch gives every thread kLaunchRegs; the
// producer / MMA / tables / quadrant-3 mask warpgroup and the mask warpgroup hand some back and the two
// epilogue warpgroups take them: 128 (88 + 88 + 96) + 256 * 96 <= 640 * 96. The first warpgroup's budget
// equals the mask warpgroup's, since warp 3 runs the mask code.
constexpr uint32_t kLaunchRegs = 96, kRegsWG0 = 88, kRegsMask = 88, kRegsEpi = 96;
static_assert(128 * (kRegsWG0 + kRegsMask + kLaunchRegs) + 256 * kRegsEpi <= 640 * kLaunchRegs, "register split");
template <uint32_t R> __device__ __forceinline__ void regs_dec() { asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" :: "n"(R)); }
template <uint32_t R> __device__ __forceinline__ void regs_inc() { asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" :: "n"(R)); }

// ---------------------------------------------------------------- shared memory layout
template <int N>
struct Lay {
    static constexpr int NB = N / 64;                                  // 64-column regions of B, C, HS
    static constexpr uint32_t kStage = (2 + 2 * NB) * kRegion;         // x (2 heads), B, C
    static constexpr uint32_t kHS = 2 * kStage;                        // h_{t-1} in bf16 for Yo
    static constexpr uint32_t kCs = kHS + NB * kRegion;                // [2][kCsStride] floats
    static constexpr uint32_t kVt = kCs + 2 * kCsStride * 4;           // [2 heads][kVtCols] halves
    static constexpr uint32_t kRec = kVt + 2 * kVtCols * 2;            // [2] tile records (int4)
    static constexpr uint32_t kBars = kRec + 2 * 16;                   // [kNumBars] u64
    static constexpr uint32_t kMisc = kBars + kNumBars * 8;            // tmem slot, abort flag, correction count
    static constexpr uint32_t kFold = kMisc + 16;                      // [4][8] slots, [4][8] decays
    static constexpr uint32_t kTotal = kFold + 256;
    static_assert(kBars % 8 == 0, "barriers are 8-byte aligned");
    static_assert(kTotal <= 232448, "shared memory per CTA");
};

template <int N>
struct Smem {
    uint8_t* base;
    __device__ uint8_t* x(int s, int h) const { return base + s * Lay<N>::kStage + h * kRegion; }
    __device__ uint8_t* b(int s) const { return base + s * Lay<N>::kStage + 2 * kRegion; }
    __device__ uint8_t* c(int s) const { return base + s * Lay<N>::kStage + (2 + Lay<N>::NB) * kRegion; }
    __device__ uint8_t* hs() const { return base + Lay<N>::kHS; }
    // per stage: the tile-local cumsum of dt*A (x log2 e) as seen from a column (token j), [2][128]:
    // cs_j, minus log2(dt_j) when the input term is dt x (exp(cs_i - table_j) is then L_ij dt_j);
    // then 8 floats: per head hh, [4 hh + k] = the plain cumsum at tokens 31, 63, 95 (k = 0..2) and,
    // k = 3, at the tile's last token (a tile) or the window's total (an aggregate tile)
    __device__ float* cs(int s) const { return reinterpret_cast<float*>(base + Lay<N>::kCs) + s * kCsStride; }
    // exp(cs_p - table_j) per head and token j < 96, p = last token of j's 32-token block: [2][96]
    __device__ __half* vt() const { return reinterpret_cast<__half*>(base + Lay<N>::kVt); }
    // per stage: the tile record {first row, tokens, first head, flags} (flags: kRecCorr, kRecEnd)
    __device__ int4* rec(int s) const { return reinterpret_cast<int4*>(base + Lay<N>::kRec) + s; }
    __device__ uint64_t* bars() const { return reinterpret_cast<uint64_t*>(base + Lay<N>::kBars); }
    __device__ uint32_t* tmem_slot() const { return reinterpret_cast<uint32_t*>(base + Lay<N>::kMisc); }
    __device__ int* abort_flag() const { return reinterpret_cast<int*>(base + Lay<N>::kMisc + 4); }
    // the number of correction tiles (written once by the table warp, see Stream)
    __device__ volatile int* ncorr() const { return reinterpret_cast<volatile int*>(base + Lay<N>::kMisc + 8); }
    // a state warp's look-back: the slots folded onto the base and their decays, per lane quadrant
    __device__ int* fold_slot(int q) const { return reinterpret_cast<int*>(base + Lay<N>::kFold) + 8 * q; }
    __device__ float* fold_dec(int q) const { return reinterpret_cast<float*>(base + Lay<N>::kFold + 128) + 8 * q; }
};

// ---------------------------------------------------------------- bounded waits
struct Waiter {
    uint64_t* bars;
    volatile int* abort;
    int* status;
};

// Bounded wait for the phase of `idx` whose parity is bit idx of `ph` (then flipped). Gives up when
// the CTA is aborting (honor_abort) or after the limit; returns false then.
// The loop of a wait that did not complete at once.
__device__ __forceinline__ bool wait_par_slow(uint64_t* bars, volatile int* abort, int* status, int idx, uint32_t par,
                                              bool honor_abort) {
    const Waiter w{bars, abort, status};
    uint64_t* bar = bars + idx;
    const uint64_t t0 = global_timer_ns();
    for (uint32_t it = 1;; ++it) {
        // try_wait lets the hardware suspend the thread briefly while the phase is pending (with the
        // default time limit: a long sleep hint made every hand-off wake later, a spin on test_wait took
        // issue slots from the warps that work; both measured slower)
        if (mbar_try_wait(bar, par)) return true;
        if ((it & 7u) != 0) continue;
        if (honor_abort && *w.abort) return false;
        if (global_timer_ns() - t0 > kWaitLimitNs) {
            record_status(w.status, SSD_ERR_TIMEOUT);
            atomicCAS(w.status + 2, 0, 0x100 + idx);
            *w.abort = 1;
            return false;
        }
    }
}

__device__ __forceinline__ bool wait_par(const Waiter& w, int idx, uint32_t par, bool honor_abort = true) {
    if (mbar_try_wait(w.bars + idx, par)) return true;
    return wait_par_slow(w.bars, w.abort, w.status, idx, par, honor_abort);
}

__device__ __forceinline__ bool wait_bar(const Waiter& w, int idx, uint32_t& ph) {
    const uint32_t par = (ph >> idx) & 1u;
    ph ^= 1u << idx;
    return wait_par(w, idx, par);
}

// Bounded wait like wait_bar that, while the phase is pending, keeps calling `side` (which returns true
// once it has nothing left to do) between brief hardware suspensions; the single-thread MMA issuer uses
// it to issue independent work as soon as that work's inputs are there.
template <class F>
__device__ __forceinline__ bool poll_bar(const Waiter& w, int idx, uint32_t& ph, F&& side) {
    const uint32_t par = (ph >> idx) & 1u;
    uint64_t* bar = w.bars + idx;
    if (!mbar_try_wait(bar, par)) {
        const uint64_t t0 = global_timer_ns();
        for (uint32_t it = 1;; ++it) {
            if (side()) {
                if (!wait_par_slow(w.bars, w.abort, w.status, idx, par, true)) return false;
                break;
            }
            if (mbar_try_wait(bar, par)) break;
            if ((it & 7u) != 0) continue;
            if (*w.abort) return false;
            if (global_timer_ns() - t0 > kWaitLimitNs) {
                record_status(w.status, SSD_ERR_TIMEOUT);
                atomicCAS(w.status + 2, 0, 0x100 + idx);
                *w.abort = 1;
                return false;
            }
        }
    }
    ph ^= 1u << idx;
    return true;
}

// Every lane waits, then the warp agrees on the outcome, so later warp-collective instructions
// (tcgen05.ld/st, shuffles) never run diverged.
__device__ __forceinline__ bool wait_warp(const Waiter& w, int idx, uint32_t& ph) {
    const bool ok = wait_bar(w, idx, ph);
    return __all_sync(0xffffffffu, ok);
}

// Non-blocking: true (and the phase consumed) if the phase is already complete.
__device__ __forceinline__ bool test_bar(const Waiter& w, int idx, uint32_t& ph) {
    const uint32_t par = (ph >> idx) & 1u;
    if (!mbar_try_wait(w.bars + idx, par)) return false;
    ph ^= 1u << idx;
    return true;
}

// Lane 0 arrives once for the warp (after the warp's work is done).
__device__ __forceinline__ void warp_arrive(const Waiter& w, int idx) {
    __syncwarp();
    if ((threadIdx.x & 31) == 0) mbar_arrive(w.bars + idx);
}

// ---------------------------------------------------------------- work decomposition
// Chains (sequence s, head pair hp) are laid end to end, chain-major (sequence major, head pair minor),
// as one run of 128-token tiles; CTA b takes the contiguous range [range_start(b), range_start(b + 1))
// of it. The range is cut at chain boundaries into windows: the first may start inside a chain (it
// looks back at the CTAs before it for its entering state), the last may end inside one (its successor,
// on the next CTA, needs its aggregate), the ones between are whole chains.

// total tiles of all chains: dense, arithmetic; packed, from the tile table the prep kernel built
__device__ __forceinline__ int total_tiles(const FusedArgs& a) {
    return a.dense ? a.nseq * a.npairs * a.nt_dense : a.npairs * a.status[1];
}
__device__ __forceinline__ int range_start(int b, const FusedArgs& a) {
    return (int)(((long long)b * total_tiles(a)) / (long long)gridDim.x);
}
// The published-state slot of CTA b: b itself, or, when there are fewer tiles than CTAs, the run
// index of its first tile (distinct for every CTA that has tiles), so that min(grid, tiles) slots do.
__device__ __forceinline__ int slot_of(int b, const FusedArgs& a) {
    const int r = range_start(b, a);
    return r < b ? r : b;
}

// The chain holding global tile g, and g's tile index in it.
struct ChainPos {
    int s, hp, t, nt;           // sequence, head pair, tile in the chain, tiles of the chain
    int32_t seq_row0, seq_len;  // first packed row and length of the sequence
};

__device__ __forceinline__ ChainPos decode_at(int g, const FusedArgs& a) {
    ChainPos c;
    if (a.dense) {
        const int ch = g / a.nt_dense;
        c.t = g - ch * a.nt_dense;
        c.nt = a.nt_dense;
        c.s = ch / a.npairs;
        c.hp = ch - c.s * a.npairs;
        c.seq_row0 = (int32_t)(c.s * a.seqlen);
        c.seq_len = (int32_t)a.seqlen;
    } else {
        // The chains of sequence s hold run indices [npairs f0, npairs f1), f0..f1 its tiles in the
        // sequence-major tile table, so tile g / npairs of the table is one of g's sequence (an empty
        // sequence has no tile). Its record gives the sequence, its first tile and its first row, and the
        // sequence's end offset its length: two dependent loads.
        const int f = g / a.npairs;
        const ChunkDesc d = a.tiles[f];
        c.s = d.seq;
        const int f0 = f - d.ci;
        c.seq_row0 = d.row0 - kTile * d.ci;
        c.seq_len = __ldg(a.cu + c.s + 1) - c.seq_row0;
        c.nt = (c.seq_len + kTile - 1) / kTile;
        const int local = g - a.npairs * f0;
        c.hp = local / c.nt;
        c.t = local - c.hp * c.nt;
    }
    return c;
}

// The tile stream of this CTA, walked identically by every role: every window's tiles in time order
// (the first window from a zero state when it starts inside its chain, the others from their chain's
// initial state), then, when the first window starts inside its chain, its correction tiles: its first
// tiles again, for y += exp(cs_l) C_l h_in^T once the entering state h_in is known. The count of
// correction tiles comes from the table warp (through shared memory): the tiles before the decay from
// the window's start underflows in fp32 (after that the correction is exactly zero).
struct Stream {
    int g0, g1;           // this CTA's range of the chain-major tile run
    int gw;               // run index of the current window's first tile
    int t, t0, t1;        // tile, the window's tiles [t0, t1) of its chain (correction: [t0, t0 + count))
    int hp;               // head pair
    int32_t row0, len;    // first packed row and length of the sequence
    bool corr;            // a correction tile
    bool valid;
    __device__ int tile_row0() const { return row0 + kTile * t; }
    __device__ int tile_len() const {
        const int rem = len - kTile * t;
        return rem < kTile ? rem : kTile;
    }
    __device__ void load_at(int g, const FusedArgs& a) {
        const ChainPos c = decode_at(g, a);
        gw = g;
        t0 = t = c.t;
        t1 = c.t + (g1 - g) < c.nt ? c.t + (g1 - g) : c.nt;
        hp = c.hp;
        row0 = c.seq_row0;
        len = c.seq_len;
    }
    __device__ void start(const FusedArgs& a) {
        g0 = range_start((int)blockIdx.x, a);
        g1 = range_start((int)blockIdx.x + 1, a);
        valid = g1 > g0;
        corr = false;
        if (valid) load_at(g0, a);
    }
    // ncorr: the correction tile count, read once the window tiles are done and the table warp has
    // published it (`ready` waits for that; false on timeout or abort)
    template <class Ready>
    __device__ void next(const FusedArgs& a, const volatile int* ncorr, Ready&& ready) {
        if (++t < t1) return;
        if (corr) { valid = false; return; }
        const int g = gw + (t1 - t0);
        if (g < g1) { load_at(g, a); return; }
        // the window tiles are done: the correction tiles of the first window, if any
        load_at(g0, a);
        if (t0 == 0 || !ready()) { valid = false; return; }
        const int n = *ncorr;
        if (n <= 0) { valid = false; return; }
        corr = true;
        t1 = t0 + n;
    }
};

// ---------------------------------------------------------------- epilogue helpers (cold paths kept out
// of line so that they do not add to the registers of the per-tile path)
// 16-byte chunk ch of a 128-byte row of a swizzled region (row pointer, row & 7)
__device__ __forceinline__ uint8_t* chunk_ptr(uint8_t* rowp, int ix, int ch) { return rowp + ((ch ^ ix) << 4); }

// one staged y row (64 bf16 channels) to global memory; with `accum` added in fp32 onto the y there
__device__ __noinline__ void store_row(uint8_t* rowp, int ix, __nv_bfloat16* yrow, bool accum) {
#pragma unroll
    for (int ch = 0; ch < 8; ++ch) {
        uint4 v = *reinterpret_cast<const uint4*>(chunk_ptr(rowp, ix, ch));
        if (accum) {
            const uint4 o = *reinterpret_cast<const uint4*>(yrow + 8 * ch);
            const uint32_t* ov = reinterpret_cast<const uint32_t*>(&o);
            uint32_t* nv = reinterpret_cast<uint32_t*>(&v);
#pragma unroll
            for (int m = 0; m < 4; ++m) {
                const float2 f = __fadd2_rn(unpack_bf16x2(nv[m]), unpack_bf16x2(ov[m]));
                nv[m] = pack_bf16x2(f.x, f.y);
            }
        }
        *reinterpret_cast<uint4*>(yrow + 8 * ch) = v;
    }
}

// ---------------------------------------------------------------- the kernel
// kScaleX: the input term is dt x B^T (a separate instantiation, so that the plain one carries none of it).
// kAccum: y is added onto the y already in memory (the second state-column half of N = 256).
template <int N, bool kScaleX, bool kAccum>
__global__ void __launch_bounds__(kThreads, 1)
ssd_fused_kernel(const __grid_constant__ FusedMaps maps, const FusedArgs a) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    using L = Lay<N>;
    constexpr int NB = L::NB;
    Smem<N> sm;
    sm.base = smem_raw;
    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;

    if (a.status[0] != SSD_OK) return;

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
    if (a.dense && a.nt_dense == 0) return;
    if ((smem_u32(smem_raw) & 1023u) != 0) {      // the swizzled layout needs a 1024-byte aligned base
        if (tid == 0) record_status(a.status, SSD_ERR_UNSUPPORTED);
        return;
    }
    if (tid == 0) {
        for (int i = 0; i < kNumBars; ++i) mbar_init(sm.bars() + i, bar_count(i));
        *sm.abort_flag() = 0;
        fence_mbar_init();
    }
    if (warp == kWarpMMA) {
        __syncwarp();
        tmem_alloc(sm.tmem_slot(), 512);
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem = *sm.tmem_slot();
    const Waiter wt{sm.bars(), sm.abort_flag(), a.status};
    auto set_abort = [&]() { *reinterpret_cast<volatile int*>(sm.abort_flag()) = 1; };

    if (warp == kWarpProducer) {
        // ============================================================ TMA producer (lane 0)
        // Stage s = p & 1 of stream position p holds x (both heads), B and C (a correction tile: C only).
        // A stage is reloaded once the MMA warp is done with its B and C and, for x, once the tile's y
        // (staged in its x region) has been stored.
        regs_dec<kRegsWG0>();
        if (lane == 0) {
            uint32_t ph = 0;
            bool ok = true;
            int nbc[2] = {0, 0}, nx[2] = {0, 0};
            Stream it;
            it.start(a);
            auto ready = [&]() { return wait_par(wt, kNcorr, 0u); };
            for (int p = 0; it.valid && ok; it.next(a, sm.ncorr(), ready), ++p) {
                const int s = p & 1;
                const int h0 = 2 * it.hp, g = h0 / (a.H / a.G);
                const int row0 = it.tile_row0();
                if (p >= 2 && !(ok = wait_bar(wt, kBCFree + s, ph))) break;
                uint64_t* fbc = sm.bars() + kFullBC + s;
                mbar_arrive_expect_tx(fbc, (uint32_t)((it.corr ? NB : 2 * NB) * kRegion));
                if (!it.corr)
                    for (int k = 0; k < NB; ++k) tma_load_3d(sm.b(s) + k * kRegion, &maps.b, fbc, 64 * k, g, row0);
                for (int k = 0; k < NB; ++k) tma_load_3d(sm.c(s) + k * kRegion, &maps.c, fbc, 64 * k, g, row0);
                ++nbc[s];
                if (it.corr) continue;        // (correction tiles come last: no x load follows)
                if (p >= 2 && !(ok = wait_bar(wt, kXFree + s, ph))) break;
                uint64_t* fx = sm.bars() + kFullX + s;
                mbar_arrive_expect_tx(fx, (uint32_t)(2 * kRegion));
                tma_load_3d(sm.x(s, 0), &maps.x, fx, 0, h0, row0);
                tma_load_3d(sm.x(s, 1), &maps.x, fx, 0, h0 + 1, row0);
                ++nx[s];
            }
            if (!ok) set_abort();
            // every load issued has landed before the CTA's shared memory goes away
            for (int s = 0; s < 2; ++s) {
                if (nbc[s] > 0) wait_par(wt, kFullBC + s, (uint32_t)(nbc[s] - 1) & 1u, false);
                if (nx[s] > 0) wait_par(wt, kFullX + s, (uint32_t)(nx[s] - 1) & 1u, false);
            }
        }
    } else if (warp == kWarpMMA) {
        // ============================================================ MMA issuer (lane 0)
        regs_dec<kRegsWG0>();
        if (lane == 0) {
            uint32_t ph = 0;
            bool ok = true, any = false;
            int cC = 0;                          // tiles so far (correction tiles too): TMEM buffer cC & 1
            bool corr_started = false;
            bool g_next = false;                 // C B^T of the tile cC already issued
            const uint32_t id_g = idesc_bf16_f32(128, 128, 0, 0);
            const uint32_t id_yo = idesc_bf16_f32(128, 128, 0, 0);
            const uint32_t id_yd = idesc_bf16_f32(128, 64, 0, 1);
            const uint32_t id_s = idesc_bf16_f32(128, N, 1, 1);
            auto issue_g = [&](int st, int buf) {
#pragma unroll 1
                for (int ks = 0; ks < N / 16; ++ks) {
                    const int k = ks / 4, off = (ks % 4) * 32;
                    const uint64_t ad = smem_desc_sw128(smem_u32(sm.c(st) + k * kRegion + off), 0, 1024);
                    const uint64_t bd = smem_desc_sw128(smem_u32(sm.b(st) + k * kRegion + off), 0, 1024);
                    mma_bf16_ss(tmem + kColGB + 128 * buf, ad, bd, id_g, ks > 0 ? 1u : 0u);
                }
                mma_commit(sm.bars() + kGFull + buf);
            };
            // S += (w o X)^T B over the stage (M = 2 heads x 64 channels, N = state columns), onto a_t h_{t-1}
            auto issue_s = [&](int st) {
#pragma unroll 1
                for (int ks = 0; ks < 8; ++ks) {
                    const uint64_t ad = smem_desc_sw128(smem_u32(sm.x(st, 0) + ks * 2048), kRegion, 1024);
                    const uint64_t bd = smem_desc_sw128(smem_u32(sm.b(st) + ks * 2048), kRegion, 1024);
                    mma_bf16_ss(tmem + kColST, ad, bd, id_s, 1u);
                }
            };
            // C h^T into the buffer's columns (M = tokens, N = 2 heads x 64 channels): Yo, or the correction
            auto issue_yo = [&](int st, uint32_t gb) {
#pragma unroll 1
                for (int ks = 0; ks < N / 16; ++ks) {
                    const int kk = ks / 4, off = (ks % 4) * 32;
                    const uint64_t ad = smem_desc_sw128(smem_u32(sm.c(st) + kk * kRegion + off), 0, 1024);
                    const uint64_t bd = smem_desc_sw128(smem_u32(sm.hs() + kk * kRegion + off), 0, 1024);
                    mma_bf16_ss(tmem + gb, ad, bd, id_yo, ks > 0 ? 1u : 0u);
                }
            };
            Stream it;
            it.start(a);
            auto ready = [&]() { return wait_par(wt, kNcorr, 0u); };
            for (int p = 0; it.valid && ok; it.next(a, sm.ncorr(), ready), ++p) {
                const int s = p & 1;
                any = true;
                const int buf = cC & 1;
                if (it.corr) {
                    // the correction product C(t) h_in^T: h_in staged by the state warps (once). The epilogue
                    // has taken the previous product (Drained: it signals each correction tile as it starts
                    // on it), so that its waits on SO never fall two phases behind.
                    ok = wait_bar(wt, kFullBC + s, ph) && (cC < 2 || wait_bar(wt, kGBFree + buf, ph)) &&
                         wait_bar(wt, kDrained + s, ph) && (corr_started || wait_bar(wt, kState, ph));
                    if (!ok) break;
                    corr_started = true;
                    tc_fence_after_sync();
                    issue_yo(s, kColGB + 128 * buf);
                    mma_commit(sm.bars() + kSO);
                    mma_commit(sm.bars() + kBCFree + s);
                    ++cC;
                    continue;
                }
                if (!g_next) {
                    ok = wait_bar(wt, kFullBC + s, ph) && (cC < 2 || wait_bar(wt, kGBFree + buf, ph));
                    if (!ok) break;
                    tc_fence_after_sync();
                    issue_g(s, buf);
                }
                g_next = false;
                // C B^T of the stream's next tile (of this window or the next one; it needs only the stage and
                // the buffer) goes out as soon as its B and C are there and its buffer is free, also while
                // this tile waits for its L o G, so that the mask warps can go on
                const bool next_tile = it.t + 1 < it.t1 || it.gw + (it.t1 - it.t0) < it.g1;
                bool bc_ok = false, gb_ok = false;
                auto try_g_next = [&]() -> bool {
                    if (!next_tile || g_next) return true;
                    if (!bc_ok) bc_ok = test_bar(wt, kFullBC + (s ^ 1), ph);
                    if (bc_ok && !gb_ok) gb_ok = (cC + 1 < 2) || test_bar(wt, kGBFree + (buf ^ 1), ph);
                    if (!(bc_ok && gb_ok)) return false;
                    tc_fence_after_sync();
                    issue_g(s ^ 1, buf ^ 1);
                    g_next = true;
                    return true;
                };
                // Yd(t), both heads interleaved: needs L o G(t) and x(t); the previous tile's Yd has been
                // drained (its Drained phase was waited for before its S)
                ok = poll_bar(wt, kLGFull + buf, ph, try_g_next) && wait_bar(wt, kFullX + s, ph) &&
                     (cC == 0 || wait_bar(wt, kYDFree, ph));
                if (!ok) break;
                tc_fence_after_sync();
                const uint32_t gb = kColGB + 128 * buf;
#pragma unroll 1
                for (int ks = 0; ks < 8; ++ks) {
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        const uint64_t bd = smem_desc_sw128(smem_u32(sm.x(s, h) + ks * 2048), kRegion, 1024);
                        mma_bf16_ts(tmem + kColYD + 64 * h, tmem + gb + 16 * ks + 8 * h, bd, id_yd, ks > 0 ? 1u : 0u);
                    }
                }
                mma_commit(sm.bars() + kYDFull);
                // S(t) onto a_t h_{t-1}, then Yo(t) into the buffer that held L o G(t)
                ok = poll_bar(wt, kDrained + s, ph, try_g_next) && wait_bar(wt, kState, ph);
                if (!ok) break;
                tc_fence_after_sync();
                issue_s(s);
                issue_yo(s, gb);
                mma_commit(sm.bars() + kSO);
                mma_commit(sm.bars() + kBCFree + s);
                if (next_tile && !g_next) {
                    ok = (bc_ok || wait_bar(wt, kFullBC + (s ^ 1), ph)) &&
                         (gb_ok || cC + 1 < 2 || wait_bar(wt, kGBFree + (buf ^ 1), ph));
                    if (!ok) break;
                    tc_fence_after_sync();
                    issue_g(s ^ 1, buf ^ 1);
                    g_next = true;
                }
                ++cC;
            }
            if (!ok) set_abort();
            // every MMA issued has completed before TMEM is freed
            if (any) {
                mma_commit(sm.bars() + kMmaDone);
                wait_par(wt, kMmaDone, 0u, false);
            }
        }
    } else if (warp == kWarpTables) {
        // ============================================================ tables (whole warp)
        // Per stream position: dt of the tile for both heads of the pair (prefetched one position
        // ahead), the cumsum of dt*A (x log2 e) -- tile-local for a tile, from the first window's start
        // for a correction tile -- and, for a tile, the factored-mask column table (once the mask warps are
        // done with the previous one). While walking the first window it counts the correction tiles.
        regs_dec<kRegsWG0>();
        uint32_t ph = 0;
        bool ok = true;
        bool vt_used = false;
        float carry[2] = {0.f, 0.f};
        float ccarry[2] = {0.f, 0.f};    // correction tiles: cumsum of the first window's earlier tiles
        float wcarry[2] = {0.f, 0.f};    // first window: cumsum before the current tile
        int ncount = 0;                  // first window: tiles whose correction is not all zero
        Stream it;
        it.start(a);
        auto load_dt = [&](const Stream& st, float (&v)[2][4]) {
            if (!st.valid) return;
            const int row0 = st.tile_row0(), len = st.tile_len(), h0 = 2 * st.hp;
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const int l = 4 * lane + k;
                float2 d2 = make_float2(0.f, 0.f);
                if (l < len) d2 = __ldg(reinterpret_cast<const float2*>(a.dt + (int64_t)(row0 + l) * a.H + h0));
                v[0][k] = d2.x;
                v[1][k] = d2.y;
            }
        };
        auto ready = [&]() { return __all_sync(0xffffffffu, wait_par(wt, kNcorr, 0u)); };
        float vn[2][4] = {};
        int np_done = 0;
        load_dt(it, vn);
        for (int p = 0; it.valid && ok; ++p) {
            const int s = p & 1;
            // this tile's dt (loaded one tile ahead) and place in the stream; then the next tile's dt
            float v[2][4];
#pragma unroll
            for (int hh = 0; hh < 2; ++hh)
#pragma unroll
                for (int k = 0; k < 4; ++k) v[hh][k] = vn[hh][k];
            const bool corr = it.corr;
            const bool first_win = !corr && it.gw == it.g0;
            const int h0 = 2 * it.hp, len = it.tile_len(), row0 = it.tile_row0();
            if (first_win) {
                // the correction of tile t is exactly zero once exp2 of the cumsum before it underflows
                // (ex2.approx.ftz gives 0 below 2^-126), for both heads
                if (fmaxf(wcarry[0], wcarry[1]) > -126.f) ncount = it.t - it.t0 + 1;
                if (it.t + 1 == it.t1) {
                    // the first window's last tile: the count is final (zero when the window starts its chain)
                    if (lane == 0) *sm.ncorr() = it.t0 > 0 ? ncount : 0;
                    __syncwarp();
                    if (lane == 0) mbar_arrive(sm.bars() + kNcorr);
                }
            }
            it.next(a, sm.ncorr(), ready);
            load_dt(it, vn);
            carry[0] = corr ? ccarry[0] : 0.f;
            carry[1] = corr ? ccarry[1] : 0.f;
            if (p >= 2) {
                // every role has read the tables this stage held two positions ago
                ok = __all_sync(0xffffffffu, wait_bar(wt, kTblRead + s, ph));
                if (!ok) break;
            }
            float* cs = sm.cs(s);
            float cv[2][4];
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
                const float A2 = __ldg(a.A + h0 + hh) * kLog2e;
                float pz[4];
                pz[0] = v[hh][0] * A2;
#pragma unroll
                for (int k = 1; k < 4; ++k) pz[k] = pz[k - 1] + v[hh][k] * A2;
                float sc = pz[3];
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) {
                    const float tt = __shfl_up_sync(0xffffffffu, sc, o);
                    if (lane >= o) sc += tt;
                }
                const float base = sc - pz[3] + carry[hh];
#pragma unroll
                for (int k = 0; k < 4; ++k) cv[hh][k] = base + pz[k];
                float4 col = make_float4(cv[hh][0], cv[hh][1], cv[hh][2], cv[hh][3]);
                if constexpr (kScaleX) {
                    if (!corr) {
                        col.x -= __log2f(fmaxf(v[hh][0], kMinDt));
                        col.y -= __log2f(fmaxf(v[hh][1], kMinDt));
                        col.z -= __log2f(fmaxf(v[hh][2], kMinDt));
                        col.w -= __log2f(fmaxf(v[hh][3], kMinDt));
                    }
                }
                *reinterpret_cast<float4*>(cs + hh * 128 + 4 * lane) = col;
                // the tile's total (dt is zero past the sequence)
                const float ttot = __shfl_sync(0xffffffffu, sc, 31);
                if (corr) ccarry[hh] += ttot;
                if (first_win) wcarry[hh] += ttot;
                // row-side values: the plain cumsum at tokens 31, 63, 95, and the last value
                if (lane == 7 || lane == 15 || lane == 23) cs[256 + 4 * hh + (lane >> 3)] = cv[hh][3];
                if (lane == ((len - 1) >> 2)) {
                    const int k = (len - 1) & 3;
                    cs[256 + 4 * hh + 3] = k == 0 ? cv[hh][0] : k == 1 ? cv[hh][1] : k == 2 ? cv[hh][2] : cv[hh][3];
                }
            }
            if (!corr) {
                // v_j = exp(cs_p - table_j), p the last token of j's 32-token block (j < 96), computed before
                // the mask warps release the table (after their off-diagonal blocks) so that only the
                // stores follow the release
                __half2 vv[2][2];
#pragma unroll
                for (int hh = 0; hh < 2; ++hh) {
                    const float piv = __shfl_sync(0xffffffffu, cv[hh][3], lane | 7);
                    float4 col = make_float4(cv[hh][0], cv[hh][1], cv[hh][2], cv[hh][3]);
                    if constexpr (kScaleX) {
                        col.x -= __log2f(fmaxf(v[hh][0], kMinDt));
                        col.y -= __log2f(fmaxf(v[hh][1], kMinDt));
                        col.z -= __log2f(fmaxf(v[hh][2], kMinDt));
                        col.w -= __log2f(fmaxf(v[hh][3], kMinDt));
                    }
                    vv[hh][0] = __floats2half2_rn(ex2(piv - col.x), ex2(piv - col.y));
                    vv[hh][1] = __floats2half2_rn(ex2(piv - col.z), ex2(piv - col.w));
                }
                if (vt_used) {
                    ok = __all_sync(0xffffffffu, wait_bar(wt, kVTFree, ph));
                    if (!ok) break;
                }
                vt_used = true;
                if (lane < 24) {
#pragma unroll
                    for (int hh = 0; hh < 2; ++hh) {
                        __half2* dst = reinterpret_cast<__half2*>(sm.vt() + hh * kVtCols + 4 * lane);
                        dst[0] = vv[hh][0];
                        dst[1] = vv[hh][1];
                    }
                }
            }
            if (lane == 0) *sm.rec(s) = make_int4(row0, len, h0, corr ? kRecCorr : 0);
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(sm.bars() + kTblAny + s);
            }
            np_done = p + 1;
        }
        // the end record after the last tile, once its stage is free
        if (ok) {
            const int s = np_done & 1;
            if (np_done >= 2) ok = __all_sync(0xffffffffu, wait_bar(wt, kTblRead + s, ph));
            if (ok && lane == 0) {
                *sm.rec(s) = make_int4(0, 0, 0, kRecEnd);
                mbar_arrive(sm.bars() + kTblAny + s);
            }
        }
        if (!ok) set_abort();
    } else if ((warp >= kWarpMask && warp < kWarpMask + 4) || warp == kWarpMaskQ3) {
        // ============================================================ L o G (one warp per lane quadrant)
        // Row i = 32 q + lane of the tile; 16-column group g holds tokens j = 16 g .. 16 g + 15 and is
        // written as packed bf16 (8 columns of head 0, then 8 of head 1). 32-block b = g / 2:
        //   b < q   exp(cs_i - cs_p) exp(cs_p - cs_j), p the block's last token (both factors <= 1)
        //   b = q   exp(cs_i - cs_j), zero where j > i
        //   b > q   zero
        // Quadrant 3 has the most: its four blocks are split between warp 7 (blocks 0, 1) and warp 3
        // (blocks 2, 3), which write disjoint columns. (Warp 3 belongs to the first warpgroup, whose
        // register budget equals the mask warpgroup's.)
        regs_dec<kRegsMask>();
        const int q = warp & 3, i = 32 * q + lane;
        const int b_lo = warp == kWarpMaskQ3 ? 2 : 0, b_hi = warp == kWarpMask + 3 ? 2 : 4;
        const uint32_t lane_base = tmem + ((uint32_t)(32 * q) << 16);
        uint32_t ph = 0;
        bool ok = true;
        int cC = 0;
        // causal masks of the diagonal block for the packed pairs (2m, 2m + 1): keep the low half when
        // 2m <= lane, the high half when 2m + 1 <= lane
        float lgd[2] = {0.f, 0.f};
        Stream it;
        it.start(a);
        auto ready = [&]() { return __all_sync(0xffffffffu, wait_par(wt, kNcorr, 0u)); };
        for (int p = 0; it.valid && ok; it.next(a, sm.ncorr(), ready), ++p) {
            if (it.corr) {
                // nothing to do for a correction tile but to take part in the release of its tables
                const int s = p & 1;
                ok = wait_warp(wt, kTblAny + s, ph);
                if (ok) warp_arrive(wt, kTblRead + s);
                continue;
            }
            const int s = p & 1, buf = cC & 1;
            const int len = it.tile_len();
            if constexpr (kScaleX) {
                // log2(dt) of this row per head: the table holds the column side, cs_j - log2(dt_j)
                float2 d2 = make_float2(1.f, 1.f);
                if (i < len)
                    d2 = __ldg(reinterpret_cast<const float2*>(a.dt + (int64_t)(it.tile_row0() + i) * a.H + 2 * it.hp));
                lgd[0] = __log2f(fmaxf(d2.x, kMinDt));
                lgd[1] = __log2f(fmaxf(d2.y, kMinDt));
            }
            ok = wait_warp(wt, kGFull + buf, ph) && wait_warp(wt, kTblAny + s, ph);
            if (!ok) break;
            tc_fence_after_sync();
            const float* cs = sm.cs(s);
            const __half* vt = sm.vt();
            const uint32_t gcol = lane_base + kColGB + 128 * buf;
            const bool rv = i < len;
            const float ci0 = cs[i] + lgd[0], ci1 = cs[128 + i] + lgd[1];
            uint32_t zero[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) zero[e] = 0u;
            if (!__any_sync(0xffffffffu, rv)) {
                if (lane == 0) mbar_arrive(sm.bars() + kVTFree);
#pragma unroll 1
                for (int g = 2 * b_lo; g < 2 * b_hi; ++g) { tmem_st8(gcol + 16 * g, zero); tmem_st8(gcol + 16 * g + 8, zero); }
            } else {
#pragma unroll 1
                for (int b = b_lo; b < b_hi; ++b) {
                    if (b > q) {
                        tmem_st8(gcol + 32 * b, zero);
                        tmem_st8(gcol + 32 * b + 8, zero);
                        tmem_st8(gcol + 32 * b + 16, zero);
                        tmem_st8(gcol + 32 * b + 24, zero);
                        continue;
                    }
                    if (b == q) {
                        // the off-diagonal blocks are done: the next tile's column table may be written
                        __syncwarp();
                        if (lane == 0) mbar_arrive(sm.bars() + kVTFree);
                    }
                    uint32_t gr[32];
                    tmem_ld16_nowait(gcol + 32 * b, gr);
                    tmem_ld16_nowait(gcol + 32 * b + 16, gr + 16);
                    tmem_wait_ld();
                    float2 uu0, uu1;
                    if (b < q) {
                        const float u0 = ex2(ci0 - cs[256 + b]), u1 = ex2(ci1 - cs[256 + 4 + b]);
                        uu0 = make_float2(u0, u0);
                        uu1 = make_float2(u1, u1);
                    }
#pragma unroll
                    for (int gg = 0; gg < 2; ++gg) {     // the block's two 16-column groups
#pragma unroll 1  // (a rolled loop: the code of every role's per-tile path shares the instruction cache)
                        for (int hh = 0; hh < 2; ++hh) {  // head 0's 8 packed columns, then head 1's
                            uint32_t pk[8];
                            const float ci = hh ? ci1 : ci0;
                            if (b < q) {
                                const float2 uu = hh ? uu1 : uu0;
                                const uint4* vp = reinterpret_cast<const uint4*>(vt + hh * kVtCols + 32 * b + 16 * gg);
#pragma unroll
                                for (int k8 = 0; k8 < 2; ++k8) {
                                    const uint4 a8 = vp[k8];
                                    const __half2* ah = reinterpret_cast<const __half2*>(&a8);
#pragma unroll
                                    for (int m = 0; m < 4; ++m) {
                                        const int e = 16 * gg + 8 * k8 + 2 * m;
                                        const float2 g2 = make_float2(__uint_as_float(gr[e]), __uint_as_float(gr[e + 1]));
                                        const float2 r = fmul2(g2, fmul2(uu, __half22float2(ah[m])));
                                        pk[4 * k8 + m] = pack_bf16x2(r.x, r.y);
                                    }
                                }
                            } else {
                                const float4* cp = reinterpret_cast<const float4*>(cs + hh * 128 + 32 * b + 16 * gg);
                                const float2 cc = make_float2(ci, ci), m1 = make_float2(-1.f, -1.f);
#pragma unroll
                                for (int k4 = 0; k4 < 4; ++k4) {
                                    const float4 a4 = cp[k4];
                                    const float2 da = __ffma2_rn(make_float2(a4.x, a4.y), m1, cc);
                                    const float2 db = __ffma2_rn(make_float2(a4.z, a4.w), m1, cc);
                                    const int e = 16 * gg + 4 * k4;      // column within the block
                                    const float2 ra = fmul2(make_float2(__uint_as_float(gr[e]), __uint_as_float(gr[e + 1])),
                                                            make_float2(ex2(da.x), ex2(da.y)));
                                    const float2 rb = fmul2(make_float2(__uint_as_float(gr[e + 2]), __uint_as_float(gr[e + 3])),
                                                            make_float2(ex2(db.x), ex2(db.y)));
                                    // columns e .. e + 3 of the block against row `lane` of it: keep j <= i
                                    const uint32_t m01 = (e + 1 <= lane) ? 0xffffffffu : (e <= lane ? 0x0000ffffu : 0u);
                                    const uint32_t m23 = (e + 3 <= lane) ? 0xffffffffu : (e + 2 <= lane ? 0x0000ffffu : 0u);
                                    pk[2 * k4] = pack_bf16x2(ra.x, ra.y) & m01;
                                    pk[2 * k4 + 1] = pack_bf16x2(rb.x, rb.y) & m23;
                                }
                            }
                            if (!rv) {
#pragma unroll
                                for (int e = 0; e < 8; ++e) pk[e] = 0u;
                            }
                            tmem_st8(gcol + 32 * b + 16 * gg + 8 * hh, pk);
                        }
                    }
                }
                if (b_hi <= q) {
                    // (this warp's blocks are all off-diagonal: done with the column table)
                    __syncwarp();
                    if (lane == 0) mbar_arrive(sm.bars() + kVTFree);
                }
            }
            tmem_wait_st();
            tc_fence_before_sync();
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(sm.bars() + kLGFull + buf);
                mbar_arrive(sm.bars() + kTblRead + s);
            }
            ++cC;
        }
        if (!ok) set_abort();
    } else if (warp >= kWarpEpi && warp < kWarpEpi + 8) {
        // ============================================================ epilogue (one warpgroup per head)
        // Row i = 32 q + lane of the tile, head hh of the pair, its 64 channels.
        //   tile:  drain -- z = Yd + D x (fp32, back into the Yd columns), x row times exp(last - cs_i)
        //          in place
        //          combine -- y = z + exp(cs_i) Yo, rounded once to bf16, staged in the x region of the
        //          stage (free once S and Yo are done), and stored: a row quadrant wholly inside the
        //          sequence as one bulk tensor store (kAccum: a bulk reduce-add), otherwise row by row
        //   correction tile: the same combine with z = 0, exp(cs_i) (cs from the first window's start)
        //          and the correction product, added onto the stored y (a bulk reduce-add, or row by row)
        regs_inc<kRegsEpi>();
        const int hh = (warp - kWarpEpi) >> 2, q = warp & 3, i = 32 * q + lane, ix = i & 7;
        const uint32_t lane_base = tmem + ((uint32_t)(32 * q) << 16);
        uint32_t ph = 0;
        bool ok = true;
        int cC = 0;
        bool y_visible = false;     // this warp's own y stores of the window pass are complete
        for (int p = 0; ok; ++p) {
            const int s = p & 1;
            // the tile record tells what the stage holds (or that the stream has ended)
            ok = wait_warp(wt, kTblAny + s, ph);
            if (!ok) break;
            const int4 rc = *sm.rec(s);
            if (rc.w & kRecEnd) break;
            const bool is_corr = (rc.w & kRecCorr) != 0;
            const int row0 = rc.x, len = rc.y, h0 = rc.z;
            const float tab = sm.cs(s)[hh * 128 + i], last = sm.cs(s)[256 + 4 * hh + 3];
            warp_arrive(wt, kTblRead + s);
            float lgd = 0.f;
            if constexpr (kScaleX) {
                if (!is_corr) {
                    float dti = 1.f;
                    if (i < len) dti = __ldg(a.dt + (int64_t)(row0 + i) * a.H + h0 + hh);
                    lgd = __log2f(fmaxf(dti, kMinDt));
                }
            }
            uint8_t* const xr = sm.x(s, hh);
            uint8_t* const xrow = xr + i * 128;
            const int buf = cC & 1;
            // z = Yd + D x of this row (64 columns), kept in TMEM in place of Yd until the combine
            const uint32_t zcol = lane_base + kColYD + 64 * hh;
            float e_row;
            if (is_corr) {
                // (this warp is done with the previous position, its SO wait included)
                warp_arrive(wt, kDrained + s);
                // the correction is added onto the y of the window pass where it is stored (a bulk tensor
                // reduce-add, or an fp32 add per row of a partial quadrant), so z is zero. This warp stored
                // those rows: its bulk stores are waited for, and made visible to ordinary loads, once.
                if (!y_visible) {
                    if (lane == 0) {
                        bulk_wait_all();
                        fence_proxy_async_global();
                    }
                    __syncwarp();
                    y_visible = true;
                }
                {
                    uint32_t f[16];
#pragma unroll
                    for (int m = 0; m < 16; ++m) f[m] = 0u;
#pragma unroll
                    for (int c16 = 0; c16 < 4; ++c16) tmem_st16(zcol + 16 * c16, f);
                }
                tmem_wait_st();
                e_row = (i < len) ? ex2(tab) : 0.f;
            } else {
                ok = wait_warp(wt, kFullX + s, ph);
                if (!ok) break;
                const float w = (i < len) ? ex2(last - tab) : 0.f;
                e_row = ex2(tab + lgd);
                const float Dh = a.D ? __ldg(a.D + h0 + hh) : 0.f;
                // ---- drain: z = Yd + D x back into the Yd columns, the x row times w in place
                ok = wait_warp(wt, kYDFull, ph);
                if (!ok) break;
                tc_fence_after_sync();
                const float2 dd = make_float2(Dh, Dh), ww = make_float2(w, w);
#pragma unroll 1  // (rolled: the code of every role's per-tile path shares the instruction cache)
                for (int c16 = 0; c16 < 4; ++c16) {
                    uint32_t zv[16];
                    tmem_ld16_nowait(zcol + 16 * c16, zv);
                    tmem_wait_ld();
#pragma unroll
                    for (int cc = 0; cc < 2; ++cc) {
                        uint4* pv = reinterpret_cast<uint4*>(chunk_ptr(xrow, ix, 2 * c16 + cc));
                        uint4 v = *pv;
                        uint32_t* u = reinterpret_cast<uint32_t*>(&v);
#pragma unroll
                        for (int m = 0; m < 4; ++m) {
                            const int e = 8 * cc + 2 * m;
                            const float2 xf = unpack_bf16x2(u[m]);
                            const float2 zz = __ffma2_rn(dd, xf, make_float2(__uint_as_float(zv[e]), __uint_as_float(zv[e + 1])));
                            zv[e] = __float_as_uint(zz.x);
                            zv[e + 1] = __float_as_uint(zz.y);
                            const float2 f = fmul2(xf, ww);
                            u[m] = pack_bf16x2(f.x, f.y);
                        }
                        *pv = v;
                    }
                    tmem_st16(zcol + 16 * c16, zv);
                }
                tmem_wait_st();
                fence_proxy_async_smem();
                tc_fence_before_sync();
                warp_arrive(wt, kDrained + s);
            }
            // ---- combine
            ok = wait_warp(wt, kSO, ph);
            if (!ok) break;
            tc_fence_after_sync();
            {
                const float2 ee = make_float2(e_row, e_row);
                const uint32_t yo_col = lane_base + kColGB + 128 * buf + 64 * hh;
#pragma unroll 1
                for (int c16 = 0; c16 < 4; ++c16) {
                    uint32_t zv[16], yo[16];
                    tmem_ld16_nowait(zcol + 16 * c16, zv);
                    tmem_ld16_nowait(yo_col + 16 * c16, yo);
                    tmem_wait_ld();
#pragma unroll
                    for (int cc = 0; cc < 2; ++cc) {
                        uint4 v;
                        uint32_t* vu = reinterpret_cast<uint32_t*>(&v);
#pragma unroll
                        for (int m = 0; m < 4; ++m) {
                            const int e = 8 * cc + 2 * m;
                            const float2 r = __ffma2_rn(ee, make_float2(__uint_as_float(yo[e]), __uint_as_float(yo[e + 1])),
                                                        make_float2(__uint_as_float(zv[e]), __uint_as_float(zv[e + 1])));
                            vu[m] = pack_bf16x2(r.x, r.y);
                        }
                        *reinterpret_cast<uint4*>(chunk_ptr(xrow, ix, 2 * c16 + cc)) = v;
                    }
                }
            }
            tc_fence_before_sync();
            fence_proxy_async_smem();
            warp_arrive(wt, kGBFree + buf);
            if (!is_corr) warp_arrive(wt, kYDFree);
            // (a correction tile adds its product onto the stored y, which holds every other share)
            const bool accum = is_corr || kAccum || a.y_accum;
            if (32 * q + 32 <= len && (is_corr || !(a.y_accum && !kAccum))) {
                // the quadrant's 32 rows all belong to the sequence: one bulk tensor store of 4 KB
                if (lane == 0) {
                    if (accum)
                        tma_reduce_add_3d(&maps.y, xr + 32 * q * 128, 0, h0 + hh, row0 + 32 * q);
                    else
                        tma_store_3d(&maps.y, xr + 32 * q * 128, 0, h0 + hh, row0 + 32 * q);
                    bulk_commit_group();
                    bulk_wait_read_all();
                }
            } else if (i < len) {
                // a partial quadrant: each row from the staging (added in fp32 onto the other state
                // columns' share when accumulating)
                store_row(xrow, ix, a.y + ((int64_t)(row0 + i) * a.H + h0 + hh) * 64, accum);
            }
            warp_arrive(wt, kXFree + s);
            ++cC;
        }
        if (!ok) set_abort();
        // the bulk stores issued by this lane complete before the CTA's shared memory goes away
        if (lane == 0) bulk_wait_all();
    } else if (warp >= kWarpState && warp < kWarpState + 4) {
        // ============================================================ state (one warp per lane quadrant)
        // TMEM row r = 32 q + lane of the state: head hr of the pair, channel pr; N state columns.
        // Each warp publishes and reads only its own quadrant's rows, with its own flag, so the four
        // warps never wait on one another.
        const int q = warp & 3, r = 32 * q + lane, hr = r >> 6, pr = r & 63;
        const uint32_t lane_base = tmem + ((uint32_t)(32 * q) << 16);
        uint32_t ph = 0;
        bool ok = true;
        auto pub_ptr = [&](float* base, int slot, int chunk) {
            // the 4 float4 units of row r, columns 16 chunk .. + 15 (column-chunk-major)
            return reinterpret_cast<float4*>(base + (int64_t)slot * (128 * N)) + (4 * chunk) * 128 + r;
        };
        auto publish = [&](float* base, int slot, int flag, float dec) {
#pragma unroll 1
            for (int k = 0; k < N / 16; ++k) {
                uint32_t v[16];
                tmem_ld16_nowait(lane_base + kColST + 16 * k, v);
                tmem_wait_ld();
                float4* dst = pub_ptr(base, slot, k);
#pragma unroll
                for (int j = 0; j < 4; ++j)
                    __stcg(dst + j * 128, make_float4(__uint_as_float(v[4 * j]), __uint_as_float(v[4 * j + 1]),
                                                      __uint_as_float(v[4 * j + 2]), __uint_as_float(v[4 * j + 3])));
            }
            // every lane's stores are performed at GPU scope before the flag is released (the release
            // of one lane would not order the other lanes' stores)
            if (lane == 0 && flag == 1) a.decay[slot * 4 + q] = dec;
            __threadfence();
            __syncwarp();
            if (lane == 0) st_release_gpu(a.flags + slot * 4 + q, flag);
        };
        // bounded wait of lane 0 until another CTA's quadrant flag is at least `want`; returns the flag
        // value seen (1 aggregate, 2 end state), 0 on timeout or abort
        auto wait_flag = [&](int slot, int want) -> int {
            bool good = true;
            int seen = 0;
            if (lane == 0) {
                const int* fp = a.flags + slot * 4 + q;
                const int target = a.force_timeout ? 3 : want;
                if (ld_acquire_gpu(fp) < target) {
                    const uint64_t t0 = global_timer_ns();
                    for (uint32_t it2 = 1; ld_acquire_gpu(fp) < target; ++it2) {
                        if ((it2 & 31u) != 0) continue;
                        if (*reinterpret_cast<volatile int*>(sm.abort_flag()) ||
                            *reinterpret_cast<volatile const int*>(a.status) != SSD_OK) { good = false; break; }
                        if (global_timer_ns() - t0 > a.lookback_limit_ns) {
                            record_status(a.status, SSD_ERR_TIMEOUT);
                            atomicCAS(a.status + 2, 0, kLocLookback);
                            good = false;
                            break;
                        }
                    }
                }
            }
            good = __shfl_sync(0xffffffffu, good ? 1 : 0, 0) != 0;
            // each lane acquires the flag itself, so its later loads of the published state are ordered
            // after the publisher's stores (and the warp agrees on the value lane 0 saw)
            if (good) {
                seen = ld_acquire_gpu(a.flags + slot * 4 + q);
                seen = __shfl_sync(0xffffffffu, seen, 0);
            }
            return good ? seen : 0;
        };
        // this window's end state decay(w) h_in + agg(w) out, chunk k of it (the aggregate rows are this
        // thread's own stores)
        const int my_slot = slot_of((int)blockIdx.x, a);
        // the initial state's row r of sequence s, head pair hp (this launch's columns), or null
        auto init_row_of = [&](int s_, int hp_) -> const float* {
            return a.init ? a.init + (((int64_t)s_ * a.H + 2 * hp_ + hr) * 64 + pr) * a.n_full + a.n_off : nullptr;
        };
        auto final_row_of = [&](int s_, int hp_) -> float* {
            return a.final_state + (((int64_t)s_ * a.H + 2 * hp_ + hr) * 64 + pr) * a.n_full + a.n_off;
        };
        const int g0 = range_start((int)blockIdx.x, a), g1 = range_start((int)blockIdx.x + 1, a);
        int p = 0;                       // stream position
        if (g1 > g0) {
            // ---- pass 1: the windows, each from its chain's initial state, or from zero when it starts
            // inside its chain (the first window only; corrected below)
            ChainPos cf{};
            int f_t0 = 0, f_t1 = 0;      // the first window's tiles
            float f_log = 0.f;           // its decay, log2
            for (int g = g0; g < g1 && ok;) {
                const ChainPos c = decode_at(g, a);
                const int t0 = c.t, t1 = c.t + (g1 - g) < c.nt ? c.t + (g1 - g) : c.nt;
                const bool first = g == g0, last = g + (t1 - t0) == g1;
                {
                    const float* irow = t0 == 0 ? init_row_of(c.s, c.hp) : nullptr;
#pragma unroll 1
                    for (int k = 0; k < N / 16; ++k) {
                        float4 h[4];
#pragma unroll
                        for (int j = 0; j < 4; ++j)
                            h[j] = irow ? __ldg(reinterpret_cast<const float4*>(irow + 16 * k) + j) : make_float4(0.f, 0.f, 0.f, 0.f);
                        tmem_st16(lane_base + kColST + 16 * k, reinterpret_cast<const uint32_t*>(h));
                    }
                    tmem_wait_st();
                }
                float wlog = 0.f;        // the window's decay, log2 (sum of its tiles' totals, in order)
                // ---- the tiles: h_{t-1} to bf16 for Yo, a_t h_{t-1} back for S(t) to accumulate onto
                for (int t = t0; t < t1 && ok; ++t, ++p) {
                    const int s = p & 1;
                    ok = wait_warp(wt, kTblAny + s, ph);
                    if (!ok) break;
                    const float tl = sm.cs(s)[256 + 4 * hr + 3];
                    warp_arrive(wt, kTblRead + s);
                    wlog += tl;
                    const float at = ex2(tl);
                    ok = t == t0 || wait_warp(wt, kSO, ph);
                    if (!ok) break;
                    tc_fence_after_sync();
                    const float2 aa = make_float2(at, at);
#pragma unroll 1
                    for (int k = 0; k < N / 16; ++k) {
                        uint32_t v[16];
                        tmem_ld16_nowait(lane_base + kColST + 16 * k, v);
                        tmem_wait_ld();
#pragma unroll
                        for (int cc = 0; cc < 2; ++cc) {
                            const int n = 16 * k + 8 * cc;
                            uint4 pk;
                            pk.x = pack_bf16x2(__uint_as_float(v[8 * cc]), __uint_as_float(v[8 * cc + 1]));
                            pk.y = pack_bf16x2(__uint_as_float(v[8 * cc + 2]), __uint_as_float(v[8 * cc + 3]));
                            pk.z = pack_bf16x2(__uint_as_float(v[8 * cc + 4]), __uint_as_float(v[8 * cc + 5]));
                            pk.w = pack_bf16x2(__uint_as_float(v[8 * cc + 6]), __uint_as_float(v[8 * cc + 7]));
                            *reinterpret_cast<uint4*>(sm.hs() + (n / 64) * kRegion + sw128_offset(r, (n % 64) / 8)) = pk;
                        }
#pragma unroll
                        for (int e = 0; e < 16; e += 2) {
                            const float2 s2 = fmul2(make_float2(__uint_as_float(v[e]), __uint_as_float(v[e + 1])), aa);
                            v[e] = __float_as_uint(s2.x);
                            v[e + 1] = __float_as_uint(s2.y);
                        }
                        tmem_st16(lane_base + kColST + 16 * k, v);
                    }
                    tmem_wait_st();
                    fence_proxy_async_smem();
                    tc_fence_before_sync();
                    warp_arrive(wt, kState);
                }
                if (!ok) break;
                // ---- the window's end: the last S, then its end state out -- a chain's final state, and
                // the state the next CTA looks back for when the window ends inside its chain (1: from a
                // zero start, to be folded; 2: from the chain's start, the true state)
                ok = wait_warp(wt, kSO, ph);
                if (!ok) break;
                tc_fence_after_sync();
                if (t1 == c.nt && a.final_state) {
                    float* fp = final_row_of(c.s, c.hp);
#pragma unroll 1
                    for (int k = 0; k < N / 16; ++k) {
                        uint32_t v[16];
                        tmem_ld16_nowait(lane_base + kColST + 16 * k, v);
                        tmem_wait_ld();
#pragma unroll
                        for (int j = 0; j < 4; ++j)
                            *reinterpret_cast<float4*>(fp + 16 * k + 4 * j) =
                                make_float4(__uint_as_float(v[4 * j]), __uint_as_float(v[4 * j + 1]),
                                            __uint_as_float(v[4 * j + 2]), __uint_as_float(v[4 * j + 3]));
                    }
                }
                if (last && t1 < c.nt) {
                    if (t0 > 0) publish(a.agg, my_slot, 1, ex2(wlog));
                    else publish(a.incl, my_slot, 2, 0.f);
                }
                if (first) { cf = c; f_t0 = t0; f_t1 = t1; f_log = wlog; }
                // (the next window's entering state overwrites the state columns: its S waits for it)
                tc_fence_before_sync();
                g += t1 - t0;
            }
            // ---- the first window's entering state, when it starts inside its chain: the look-back over
            // the CTAs before this one, whose last windows are the chain's previous pieces, nearest first:
            // stop at the nearest with its true end state published, or at the one whose window starts the
            // chain (its entering state is the initial state), then fold their zero-start end states onto
            // that base, oldest first. Every path gives the same bits, since a published true end state is
            // this same fold, done by its window. h_in then goes to shared memory (bf16) for the correction
            // products, onto the final state when the window ends its chain, and, when the window also ends
            // this range inside its chain, into this window's own true end state.
            if (ok && f_t0 > 0) {
                constexpr int kMaxFold = 8;
                int* fold = sm.fold_slot(q);  // (shared memory: read in the loop below without a round trip)
                int nf = 0, base = -1;       // base: the slot whose end state starts the fold, -1 the initial state
                const int cg0 = g0 - f_t0;   // run index of the chain's first tile
                for (int j = (int)blockIdx.x - 1;; --j) {
                    if (range_start(j, a) == range_start(j + 1, a)) continue;   // a CTA without tiles
                    const int sj = slot_of(j, a);
                    const int f = wait_flag(sj, 1);
                    if (f == 0) { ok = false; break; }
                    if (f >= 2) { base = sj; break; }
                    if (lane == 0) fold[nf] = sj;
                    ++nf;
                    if (range_start(j, a) <= cg0) break;
                    if (nf == kMaxFold) {
                        // a long chain: wait for this one's true end state rather than walking further
                        --nf;
                        if (wait_flag(sj, 2) == 0) ok = false;
                        base = sj;
                        break;
                    }
                }
                if (ok) {
                    // the folded slots' decays, once
                    __syncwarp();
                    if (lane < nf) sm.fold_dec(q)[lane] = __ldcg(a.decay + fold[lane] * 4 + q);
                    __syncwarp();
                    const float* fdecs = sm.fold_dec(q);
                    const float* irow = init_row_of(cf.s, cf.hp);
                    const bool fin = f_t1 == cf.nt && a.final_state;
                    const bool out_incl = f_t1 < cf.nt;      // (then the first window is also the last)
                    const float fdec = ex2(f_log);
                    float* frow = fin ? final_row_of(cf.s, cf.hp) : nullptr;
                    // 16 state columns at a time. Every load of a column group (the base, up to two folded
                    // states, this thread's own final-state or zero-start end-state values: never both) goes
                    // out before any of them is used, so that a group costs about one round trip to L2.
#pragma unroll 1
                    for (int ck = 0; ck < N / 16; ++ck) {
                        float4 h[4], ot[4];
                        if (base >= 0) {
                            const float4* src = pub_ptr(a.incl, base, ck);
#pragma unroll
                            for (int j = 0; j < 4; ++j) h[j] = __ldcg(src + j * 128);
                        } else if (irow) {
#pragma unroll
                            for (int j = 0; j < 4; ++j) h[j] = __ldg(reinterpret_cast<const float4*>(irow + 16 * ck) + j);
                        } else {
#pragma unroll
                            for (int j = 0; j < 4; ++j) h[j] = make_float4(0.f, 0.f, 0.f, 0.f);
                        }
                        if (fin) {
#pragma unroll
                            for (int j = 0; j < 4; ++j) ot[j] = __ldcg(reinterpret_cast<const float4*>(frow + 16 * ck) + j);
                        } else if (out_incl) {
                            const float4* ag = pub_ptr(a.agg, my_slot, ck);
#pragma unroll
                            for (int j = 0; j < 4; ++j) ot[j] = __ldcg(ag + j * 128);
                        }
                        for (int f0 = nf - 1; f0 >= 0; f0 -= 2) {
                            float dcy[2];
                            float4 gg[2][4];
#pragma unroll
                            for (int u = 0; u < 2; ++u) {
                                if (f0 - u >= 0) {
                                    dcy[u] = fdecs[f0 - u];
                                    const float4* src = pub_ptr(a.agg, fold[f0 - u], ck);
#pragma unroll
                                    for (int j = 0; j < 4; ++j) gg[u][j] = __ldcg(src + j * 128);
                                }
                            }
#pragma unroll
                            for (int u = 0; u < 2; ++u) {
                                if (f0 - u >= 0) {
#pragma unroll
                                    for (int jj = 0; jj < 4; ++jj)
                                        h[jj] = make_float4(fmaf(dcy[u], h[jj].x, gg[u][jj].x), fmaf(dcy[u], h[jj].y, gg[u][jj].y),
                                                            fmaf(dcy[u], h[jj].z, gg[u][jj].z), fmaf(dcy[u], h[jj].w, gg[u][jj].w));
                                }
                            }
                        }
                        // h_in as bf16 for the correction products
#pragma unroll
                        for (int hf = 0; hf < 2; ++hf) {
                            const int n = 16 * ck + 8 * hf;
                            uint4 pk;
                            pk.x = pack_bf16x2(h[2 * hf].x, h[2 * hf].y);
                            pk.y = pack_bf16x2(h[2 * hf].z, h[2 * hf].w);
                            pk.z = pack_bf16x2(h[2 * hf + 1].x, h[2 * hf + 1].y);
                            pk.w = pack_bf16x2(h[2 * hf + 1].z, h[2 * hf + 1].w);
                            *reinterpret_cast<uint4*>(sm.hs() + (n / 64) * kRegion + sw128_offset(r, (n % 64) / 8)) = pk;
                        }
                        if (fin) {
                            // the chain's final state from its zero-start value (this thread's own stores)
#pragma unroll
                            for (int jj = 0; jj < 4; ++jj)
                                reinterpret_cast<float4*>(frow + 16 * ck)[jj] =
                                    make_float4(fmaf(fdec, h[jj].x, ot[jj].x), fmaf(fdec, h[jj].y, ot[jj].y),
                                                fmaf(fdec, h[jj].z, ot[jj].z), fmaf(fdec, h[jj].w, ot[jj].w));
                        } else if (out_incl) {
                            // this window's true end state, decay * h_in + its zero-start end state
                            float4* dst = pub_ptr(a.incl, my_slot, ck);
#pragma unroll
                            for (int jj = 0; jj < 4; ++jj)
                                __stcg(dst + jj * 128, make_float4(fmaf(fdec, h[jj].x, ot[jj].x), fmaf(fdec, h[jj].y, ot[jj].y),
                                                                   fmaf(fdec, h[jj].z, ot[jj].z), fmaf(fdec, h[jj].w, ot[jj].w)));
                        }
                    }
                    if (out_incl) {
                        __threadfence();
                        __syncwarp();
                        if (lane == 0) st_release_gpu(a.flags + my_slot * 4 + q, 2);
                    }
                    fence_proxy_async_smem();
                    tc_fence_before_sync();
                    warp_arrive(wt, kState);
                    // the correction tiles' tables are not read here, but every role takes part in their
                    // release
                    ok = __all_sync(0xffffffffu, wait_par(wt, kNcorr, 0u));
                    const int nc = ok ? *sm.ncorr() : 0;
                    for (int j = 0; j < nc && ok; ++j, ++p) {
                        ok = wait_warp(wt, kTblAny + (p & 1), ph);
                        if (ok) warp_arrive(wt, kTblRead + (p & 1));
                    }
                }
            }
        }
        if (!ok) set_abort();
    }

    tc_fence_before_sync();
    __syncthreads();
    if (warp == kWarpMMA) {
        __syncwarp();   // lane 0 ran the MMA loop alone: reconverge before the warp-collective dealloc
        tmem_dealloc(tmem, 512);
    }
}

}  // namespace

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// 3-D view (inner, mid, rows) of a bf16 tensor whose mid and row strides are mid_stride and row_stride
// elements (inner is contiguous), boxes of 64 x 1 x box_rows with the 128-byte swizzle
bool make_map_fused(CUtensorMap* m, const void* ptr, int64_t inner, int64_t mid, int64_t rows, int64_t mid_stride,
                    int64_t row_stride, int box_rows) {
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

namespace {

template <int N, bool kScaleX, bool kAccum>
cudaError_t launch_fused_n(const Problem& p, const FusedArgs& fa, const FusedMaps& maps, int grid) {
    const size_t smem = Lay<N>::kTotal;
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

// CTAs of the fused launch. Each takes one contiguous range of the chain-major tile run. A range that
// starts inside its chain pays a tail at the end (the look-back, the fold and the correction tiles),
// worth about kTailTiles tiles (measured on GB300). When a dense batch has at most one chain per SM and
// a chain is not longer than an even range plus that tail, one CTA per chain does without any tail (and
// with fewer CTAs its tiles run a little faster): the Mamba-2-130M-shaped layer, 96 chains of 16 tiles,
// takes 80 us that way against 86 us on 152 ranges of 10 or 11 tiles.
constexpr int64_t kTailTiles = 6;
static int fused_grid(const Problem& p) {
    const int grid = p.num_sms < kFusedMaxGrid ? p.num_sms : kFusedMaxGrid;
    if (p.varlen) return grid;
    const int64_t chains = p.s.batch * (p.s.nheads / 2);
    const int64_t nt = (p.s.seqlen + kFusedTile - 1) / kFusedTile;
    if (chains > 0 && chains <= grid && nt <= (chains * nt + grid - 1) / grid + kTailTiles) return (int)chains;
    return grid;
}

void fused_plan(const Problem& p, int* K_out, int64_t* np_out) {
    // one contiguous range of the chain-major tile run per CTA; one published-state slot per CTA
    *K_out = 0;
    const int64_t grid = fused_grid(p);
    const int64_t all_tiles = (p.s.nheads / 2) * p.L.max_chunks;
    *np_out = all_tiles < grid ? (all_tiles > 0 ? all_tiles : 1) : grid;
}

cudaError_t launch_fused(const Problem& p, int, int64_t, int part) {
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
    const int grid = fused_grid(p);
    FusedArgs fa;
    fa.status = p.status();
    fa.tiles = p.chunks();
    fa.seqoff = p.seqoff();
    fa.cu = p.varlen ? p.cu_seqlens : nullptr;
    fa.dt = p.dt;
    fa.A = p.A;
    fa.D = part == 0 ? p.D : nullptr;
    fa.init = p.init;
    fa.final_state = p.final_state;
    fa.y = (__nv_bfloat16*)p.y;
    fa.flags = p.flags();
    fa.decay = reinterpret_cast<float*>(p.ws + p.L.pdecay);
    fa.agg = reinterpret_cast<float*>(p.ws + p.L.agg);
    fa.incl = reinterpret_cast<float*>(p.ws + p.L.incl);
    fa.H = H;
    fa.G = G;
    fa.nseq = (int)p.nseq;
    fa.npairs = (int)npairs;
    fa.dense = p.varlen ? 0 : 1;
    fa.seqlen = (int)p.s.seqlen;
    fa.nt_dense = (int)((p.s.seqlen + kFusedTile - 1) / kFusedTile);
    fa.n_off = part * N;
    fa.n_full = Nf;
    fa.y_accum = part > 0 ? 1 : 0;
    fa.force_timeout = p.force_timeout ? 1 : 0;
    fa.lookback_limit_ns = p.force_timeout ? 1000000ull : kWaitLimitNs;
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
