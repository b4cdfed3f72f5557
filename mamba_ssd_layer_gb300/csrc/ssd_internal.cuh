// ssd_internal.cuh -- shared definitions of the SSD library: workspace layout,
// the chunk table, and the launchers each translation unit provides.
#pragma once
#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "ssd.h"

namespace ssd {

// One chunk of the decomposition: `len` (<= Q) consecutive tokens of one sequence,
// starting at packed row `row0`; `seq` is the sequence and `ci` the chunk's index in it.
struct ChunkDesc {
    int32_t row0, len, seq, ci;
};

// Workspace layout (byte offsets, every section 256-byte aligned except the flags, which follow the
// header directly so that one memset clears both).
//   header  : int32 status, int32 number of chunks (tiles) actually built, int32 location
//             code of the first device-side timeout (0 = none), int32 number of windows (packed
//             batch, fused path), int32 spare x 4
//   flags   : (fused path) int32[max_pieces * 4], per CTA slot and TMEM lane quadrant: 1 = the aggregate of
//             the CTA's last window is published, 2 = the state at its end is too, 0 = neither yet
//   chunks  : ChunkDesc[max_chunks]  (chunks of `chunk` tokens; 128-token tiles on the fused path)
//   seqoff  : int32[nseq + 1], first chunk of every sequence
// fp32 path (three kernels):
//   decay   : float[max_chunks * H], exp(sum of dt*A over the chunk)
//   states  : float[max_chunks * H * P * N]; the chunk-state kernel writes each chunk's
//             local end state here and the state pass overwrites it in place with the
//             true state entering the chunk
// fused path (bf16, P = 64, N in {64, 128, 256}; 128 state columns per launch):
//   pdecay  : float[max_pieces * 4], decay of each slot's window over its tiles, per lane quadrant (the
//             head of quadrants 0, 1 is the pair's first head, of quadrants 2, 3 its second)
//   agg     : float[max_pieces * 128 * Nl], the window's end state from a zero entering state
//   incl    : float[max_pieces * 128 * Nl], the true state at the window's end
//   (Nl = min(N, 128), the state columns of one launch)
constexpr int kFusedTile = 128;
constexpr int kFusedMaxGrid = 160;    // CTAs of the fused kernel, at most (one per SM)

struct WsLayout {
    size_t header, flags, chunks, seqoff, decay, states, pdecay, agg, incl, total;
    size_t clear_bytes;          // bytes from the header on that every call clears before its kernels
    int64_t max_chunks, nseq, max_pieces;
    bool fused;
};

inline size_t align256(size_t v) { return (v + 255) & ~size_t(255); }

// The fused kernel holds up to 128 state columns; N = 256 runs as two launches over the two column
// halves (the state columns evolve independently and add up in y).
inline bool use_fused_path(const ssd_shape& s, ssd_dtype dtype) {
    return dtype == SSD_BF16 && s.headdim == 64 && (s.dstate == 64 || s.dstate == 128 || s.dstate == 256) &&
           ((s.nheads / s.ngroups) % 2 == 0);
}

inline WsLayout ws_layout(const ssd_shape& s, ssd_dtype dtype, int chunk, int64_t nseq_eff, bool varlen) {
    WsLayout w{};
    w.fused = use_fused_path(s, dtype);
    const int q = w.fused ? kFusedTile : chunk;
    const int64_t rows = s.batch * s.seqlen;
    w.nseq = nseq_eff;
    if (varlen)
        w.max_chunks = (rows + q - 1) / q + nseq_eff;
    else
        w.max_chunks = s.batch * ((s.seqlen + q - 1) / q);
    size_t off = 0;
    w.header = off; off += 32;
    if (w.fused) {
        // one published-state slot per CTA that has tiles (its last window, when it ends inside its
        // chain): min(grid, tiles of all chains) slots
        const int64_t all_tiles = (s.nheads / 2) * w.max_chunks;
        w.max_pieces = all_tiles < kFusedMaxGrid ? (all_tiles > 0 ? all_tiles : 1) : kFusedMaxGrid;
        w.flags = off; off += sizeof(int32_t) * 4 * (size_t)w.max_pieces;
    }
    w.clear_bytes = off;
    off = align256(off);
    w.chunks = off; off = align256(off + sizeof(ChunkDesc) * (size_t)(w.max_chunks > 0 ? w.max_chunks : 1));
    w.seqoff = off; off = align256(off + sizeof(int32_t) * (size_t)(nseq_eff + 1));
    if (w.fused) {
        const int64_t ncol = s.dstate > 128 ? 128 : s.dstate;   // state columns of one launch
        w.pdecay = off; off = align256(off + sizeof(float) * 4 * (size_t)w.max_pieces);
        w.agg = off;    off = align256(off + sizeof(float) * (size_t)(w.max_pieces * 128 * ncol));
        w.incl = off;   off = align256(off + sizeof(float) * (size_t)(w.max_pieces * 128 * ncol));
    } else {
        w.decay = off;  off = align256(off + sizeof(float) * (size_t)(w.max_chunks * s.nheads));
        w.states = off; off = align256(off + sizeof(float) * (size_t)(w.max_chunks * s.nheads * s.headdim * s.dstate));
    }
    w.total = off;
    return w;
}

// Everything a launcher needs, resolved by the API layer.
struct Problem {
    ssd_shape s;
    ssd_dtype dtype;
    int chunk;
    bool varlen;
    bool scale_x_by_dt;    // the input term is dt x B^T (SSD_SCALE_X_BY_DT)
    bool force_timeout;    // SSD_DEBUG_FORCE_TIMEOUT: every cross-CTA wait of the fused kernel is made to
                           // run out after about a millisecond (failure-detection tests)
    int64_t nseq;          // sequences: batch (dense) or segments (varlen)
    int64_t rows;          // packed rows = batch * seqlen
    const void* x;
    const float* dt;
    const float* A;
    const void* B;
    const void* C;
    const float* D;
    const float* init;
    const int32_t* cu_seqlens;
    void* y;
    float* final_state;
    char* ws;
    WsLayout L;
    cudaStream_t stream;
    int num_sms;

    int* status() const { return reinterpret_cast<int*>(ws + L.header); }
    int* nchunks() const { return reinterpret_cast<int*>(ws + L.header) + 1; }
    ChunkDesc* chunks() const { return reinterpret_cast<ChunkDesc*>(ws + L.chunks); }
    int32_t* seqoff() const { return reinterpret_cast<int32_t*>(ws + L.seqoff); }
    float* decay() const { return reinterpret_cast<float*>(ws + L.decay); }
    float* states() const { return reinterpret_cast<float*>(ws + L.states); }
    int32_t* flags() const { return reinterpret_cast<int32_t*>(ws + L.flags); }
};

// ssd_api.cu: records the failing step of an SSD_ERR_CUDA for ssd_last_error_detail
// and clears the runtime's sticky "last error" so later calls do not inherit it.
cudaError_t note_cuda_error(const char* step, cudaError_t e);
// ssd_api.cu: optional event pair around the dominant kernel (see ssd_profile.h), and a count
// of every kernel launch (each launcher calls prof_launch once per launch it makes)
void prof_launch();
void prof_begin(cudaStream_t s, const char* kernel);
void prof_end(cudaStream_t s);

// ssd_common.cu: chunk (tile) table of `q` tokens
cudaError_t launch_prep(const Problem& p, int q);
cudaError_t launch_state_pass(const Problem& p);
// ssd_f32.cu
cudaError_t launch_f32_path(const Problem& p);
// ssd_fused.cu (single-pass tcgen05 path): K is unused (0); npieces = the published-state slots (one per CTA)
void fused_plan(const Problem& p, int* K, int64_t* npieces);
// part: which 128-column half of an N = 256 state (0 for N <= 128)
cudaError_t launch_fused(const Problem& p, int K, int64_t npieces, int part);

// A TMA map of a 3-D view (inner, mid, rows) of a bf16 tensor whose mid and row strides are mid_stride
// and row_stride elements (inner contiguous): boxes of 64 x 1 x box_rows with the 128-byte swizzle.
bool make_map_fused(CUtensorMap* m, const void* ptr, int64_t inner, int64_t mid, int64_t rows, int64_t mid_stride,
                    int64_t row_stride, int box_rows = kFusedTile);

// The sequence-slice hand-off (ssd_handoff.cu).
size_t slice_ws_bytes(const ssd_shape& s);
cudaError_t launch_slice_decay(const ssd_shape& s, const float* dt, const float* A, float* decay, char* ws,
                               cudaStream_t st);
cudaError_t launch_slice_correct(const ssd_shape& s, const float* dt, const float* A, const void* C,
                                 const float* h_in, void* y, float* final_state, char* ws, cudaStream_t st);

}  // namespace ssd
