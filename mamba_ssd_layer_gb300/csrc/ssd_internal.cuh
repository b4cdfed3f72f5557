// ssd_internal.cuh -- shared definitions of the SSD library: workspace layout,
// the chunk table, and the launchers each translation unit provides.
#pragma once
#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

#include "ssd.h"

namespace ssd {

// One chunk of the decomposition: `len` (<= Q) consecutive tokens of one sequence,
// starting at packed row `row0`; `seq` is the sequence and `ci` the chunk's index in it.
struct ChunkDesc {
    int32_t row0, len, seq, ci;
};

// Workspace layout (byte offsets, every section 256-byte aligned).
//   header  : int32 status, int32 number of chunks actually built
//   chunks  : ChunkDesc[max_chunks]
//   seqoff  : int32[nseq + 1], first chunk of every sequence
//   decay   : float[max_chunks * H], exp(sum of dt*A over the chunk)
//   states  : float[max_chunks * H * P * N]; the chunk-state kernel writes each chunk's
//             local end state here and the state pass overwrites it in place with the
//             true state entering the chunk
struct WsLayout {
    size_t header, chunks, seqoff, decay, states, total;
    int64_t max_chunks, nseq;
};

inline size_t align256(size_t v) { return (v + 255) & ~size_t(255); }

inline WsLayout ws_layout(const ssd_shape& s, int chunk, int64_t nseq_eff, bool varlen) {
    WsLayout w{};
    const int64_t rows = s.batch * s.seqlen;
    w.nseq = nseq_eff;
    if (varlen)
        w.max_chunks = (rows + chunk - 1) / chunk + nseq_eff;
    else
        w.max_chunks = s.batch * ((s.seqlen + chunk - 1) / chunk);
    size_t off = 0;
    w.header = off; off = align256(off + 16);
    w.chunks = off; off = align256(off + sizeof(ChunkDesc) * (size_t)(w.max_chunks > 0 ? w.max_chunks : 1));
    w.seqoff = off; off = align256(off + sizeof(int32_t) * (size_t)(nseq_eff + 1));
    w.decay = off;  off = align256(off + sizeof(float) * (size_t)(w.max_chunks * s.nheads));
    w.states = off; off = align256(off + sizeof(float) * (size_t)(w.max_chunks * s.nheads * s.headdim * s.dstate));
    w.total = off;
    return w;
}

// Everything a launcher needs, resolved by the API layer.
struct Problem {
    ssd_shape s;
    ssd_dtype dtype;
    int chunk;
    bool varlen;
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
};

// ssd_api.cu: optional event pair around the dominant kernel (see ssd_profile.h)
void prof_begin(cudaStream_t s);
void prof_end(cudaStream_t s);

// ssd_common.cu
cudaError_t launch_prep(const Problem& p);
cudaError_t launch_state_pass(const Problem& p);
// ssd_f32.cu
cudaError_t launch_f32_path(const Problem& p);
// ssd_tc.cu
cudaError_t launch_bf16_path(const Problem& p);
bool bf16_path_supports(const ssd_shape& s, int chunk);

}  // namespace ssd
