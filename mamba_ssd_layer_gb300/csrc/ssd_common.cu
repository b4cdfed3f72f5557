// ssd_common.cu -- kernels shared by the fp32 and bf16 paths:
//   * chunk-table construction (dense batch or packed variable-length row), and
//   * the inter-chunk state pass (the "center factors" of the low-rank blocks).
//
// The state pass is the scalar-decay recurrence over chunk states,
//   h_c = a_c * h_{c-1} + S_c,  h_{-1} = initial state,
// i.e. multiplication by the 1-semiseparable matrix built from the chunk decays
// ("LLM(十一)——Mamba" §3.5.2, Center Factors; step 3 of the chunking-and-state-
// passing description). It runs sequentially over chunks (fp32, no cumsum
// differences, so long sequences do not lose precision) and in parallel over
// (sequence, head, state element), with 16-byte vector loads and stores.
#include <type_traits>

#include "ssd_internal.cuh"

namespace ssd {

// Builds the chunk table: every sequence is cut into chunks of Q tokens from its
// start (the last one may be shorter). Sequence s is [cu[s], cu[s+1]) when
// cu != nullptr, else [s*seqlen, (s+1)*seqlen). Invalid offsets (decreasing, or
// past the row) record SSD_ERR_INVALID_ARG and build an empty table.

__global__ void __launch_bounds__(1024) prep_kernel(const int32_t* __restrict__ cu, int64_t nseq,
                                                    int64_t seqlen, int64_t rows, int Q,
                                                    int* header, ChunkDesc* chunks, int32_t* seqoff,
                                                    int64_t max_chunks) {
    __shared__ int32_t warp_tot[32];
    __shared__ int32_t carry;
    __shared__ int bad;
    const int tid = threadIdx.x;
    if (tid == 0) { carry = 0; bad = 0; }
    __syncthreads();
    // pass 1: validate
    for (int64_t s = tid; s < nseq; s += blockDim.x) {
        if (cu) {
            int64_t a = cu[s], b = cu[s + 1];
            if (a < 0 || b < a || b > rows || (s == 0 && a != 0) || (s == nseq - 1 && b != rows)) bad = 1;
        }
    }
    __syncthreads();
    if (bad) {
        if (tid == 0) { header[0] = SSD_ERR_INVALID_ARG; header[1] = 0; seqoff[0] = 0; }
        for (int64_t s = tid; s < nseq; s += blockDim.x) seqoff[s + 1] = 0;
        return;
    }
    // pass 3: exclusive scan of chunk counts, block-wide, in tiles of blockDim
    for (int64_t base = 0; base < nseq; base += blockDim.x) {
        const int64_t s = base + tid;
        int64_t start = 0, len = 0;
        if (s < nseq) {
            start = cu ? (int64_t)cu[s] : s * seqlen;
            len = cu ? (int64_t)cu[s + 1] - cu[s] : seqlen;
        }
        const int32_t n = (s < nseq) ? (int32_t)((len + Q - 1) / Q) : 0;
        // inclusive warp scan
        int32_t v = n;
        const int lane = tid & 31, warp = tid >> 5;
        for (int o = 1; o < 32; o <<= 1) {
            int32_t t = __shfl_up_sync(0xffffffffu, v, o);
            if (lane >= o) v += t;
        }
        if (lane == 31) warp_tot[warp] = v;
        __syncthreads();
        if (warp == 0) {
            int32_t w = (lane < (int)(blockDim.x >> 5)) ? warp_tot[lane] : 0;
            for (int o = 1; o < 32; o <<= 1) {
                int32_t t = __shfl_up_sync(0xffffffffu, w, o);
                if (lane >= o) w += t;
            }
            warp_tot[lane] = w;   // inclusive prefix over warps
        }
        __syncthreads();
        const int32_t excl = carry + (warp > 0 ? warp_tot[warp - 1] : 0) + v - n;
        if (s < nseq) {
            seqoff[s] = excl;
            for (int32_t c = 0; c < n && excl + c < max_chunks; ++c) {
                ChunkDesc d;
                d.row0 = (int32_t)(start + (int64_t)c * Q);
                d.len = (int32_t)(len - (int64_t)c * Q < Q ? len - (int64_t)c * Q : Q);
                d.seq = (int32_t)s;
                d.ci = c;
                chunks[excl + c] = d;
            }
        }
        __syncthreads();
        if (tid == 0) carry += warp_tot[(blockDim.x >> 5) - 1];
        __syncthreads();
    }
    if (tid == 0) {
        seqoff[nseq] = carry;
        header[0] = SSD_OK;
        header[1] = carry;
        header[2] = 0;   // first device-side timeout location (diagnostic), 0 = none
        header[3] = 0;
        header[4] = 0;   // arrival counter of the fused kernel's grid-wide barriers
        header[5] = 0;
    }
}

cudaError_t launch_prep(const Problem& p, int q) {
    prof_launch();
    prep_kernel<<<1, 1024, 0, p.stream>>>(p.varlen ? p.cu_seqlens : nullptr, p.nseq, p.s.seqlen, p.rows,
                                          q, p.status(), p.chunks(), p.seqoff(), p.L.max_chunks);
    return cudaGetLastError();
}

// State pass. Grid: (element blocks, H, nseq). Each thread owns VEC consecutive
// floats of one (sequence, head) state and walks the sequence's chunks in order:
// it swaps the chunk's local end state S_c for the entering state h_{c-1}, then
// advances h_c = a_c h_{c-1} + S_c. The final state of the sequence is written out.
template <int VEC>
__global__ void __launch_bounds__(256) state_pass_kernel(const int* __restrict__ header,
                                                         const int32_t* __restrict__ seqoff,
                                                         const float* __restrict__ decay,
                                                         float* __restrict__ states,
                                                         const float* __restrict__ init,
                                                         float* __restrict__ final_state,
                                                         int H, int64_t PN) {
    if (header[0] != SSD_OK) return;
    const int h = blockIdx.y;
    const int64_t s = blockIdx.z;
    const int64_t e = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) * VEC;
    if (e >= PN) return;
    using V = typename std::conditional<VEC == 4, float4, float>::type;
    float hv[VEC];
    if (init) {
        V t = *reinterpret_cast<const V*>(init + ((int64_t)s * H + h) * PN + e);
        const float* tp = reinterpret_cast<const float*>(&t);
#pragma unroll
        for (int i = 0; i < VEC; ++i) hv[i] = tp[i];
    } else {
#pragma unroll
        for (int i = 0; i < VEC; ++i) hv[i] = 0.f;
    }
    const int32_t c0 = seqoff[s], c1 = seqoff[s + 1];
    // software pipeline: the next chunk's local state is loaded before the current update
    V nxt;
    if (c0 < c1) nxt = __ldcs(reinterpret_cast<const V*>(states + ((int64_t)c0 * H + h) * PN + e));
    for (int32_t c = c0; c < c1; ++c) {
        V cur = nxt;
        if (c + 1 < c1) nxt = __ldcs(reinterpret_cast<const V*>(states + ((int64_t)(c + 1) * H + h) * PN + e));
        const float a = decay[(int64_t)c * H + h];
        V out;
        float* op = reinterpret_cast<float*>(&out);
        const float* cp = reinterpret_cast<const float*>(&cur);
#pragma unroll
        for (int i = 0; i < VEC; ++i) {
            op[i] = hv[i];
            hv[i] = fmaf(a, hv[i], cp[i]);
        }
        *reinterpret_cast<V*>(states + ((int64_t)c * H + h) * PN + e) = out;
    }
    if (final_state) {
        V out;
        float* op = reinterpret_cast<float*>(&out);
#pragma unroll
        for (int i = 0; i < VEC; ++i) op[i] = hv[i];
        *reinterpret_cast<V*>(final_state + ((int64_t)s * H + h) * PN + e) = out;
    }
}

cudaError_t launch_state_pass(const Problem& p) {
    const int64_t PN = p.s.headdim * p.s.dstate;
    if (p.nseq == 0) return cudaSuccess;
    const bool vec4 = (PN % 4) == 0;
    const int64_t units = vec4 ? PN / 4 : PN;
    dim3 grid((unsigned)((units + 255) / 256), (unsigned)p.s.nheads, (unsigned)p.nseq);
    prof_launch();
    if (vec4)
        state_pass_kernel<4><<<grid, 256, 0, p.stream>>>(p.status(), p.seqoff(), p.decay(), p.states(),
                                                         p.init, p.final_state, (int)p.s.nheads, PN);
    else
        state_pass_kernel<1><<<grid, 256, 0, p.stream>>>(p.status(), p.seqoff(), p.decay(), p.states(),
                                                         p.init, p.final_state, (int)p.s.nheads, PN);
    return cudaGetLastError();
}

}  // namespace ssd
