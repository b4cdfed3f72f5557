/*
 * ssd.h -- C ABI of the GB300 (sm_103a) SSD layer forward pass.
 *
 * The operation (one call = one layer forward over a batch):
 *
 *   for every sequence s, head h (group g = h / (H/G)) and token t of s:
 *     a_t = exp(dt[t,h] * A[h])
 *     S   = a_t * S + x[t,h,:] (outer) B[t,g,:]          S: (P, N), starts at initial_state[s,h] or 0
 *     y[t,h,:] = S . C[t,g,:] + D[h] * x[t,h,:]
 *   final_state[s,h] = S after the last token of s
 *
 * equivalently Y = (L o C B^T) X + D X with the 1-semiseparable mask
 * L_ij = exp(sum_{k=j+1..i} dt_k A) (i >= j). It is computed with the chunked block
 * decomposition: per-chunk cumulative sums of dt*A, diagonal blocks in the
 * quadratic (masked attention) form, chunk states B^T X, an inter-chunk
 * scalar-decay recurrence over the states, and C . state outputs plus the D skip.
 *
 * Sources: recurrence and scalar-identity A -- "Mamba-2 状态空间对偶性理论" §1.2
 * and "LLM(十一)——Mamba" §3.1.1-3.1.2; quadratic form -- "LLM(十一)——Mamba"
 * §3.1.3; the chunked algorithm (diagonal blocks, right/center/left factors) --
 * "LLM(十一)——Mamba" §3.5 (3.5.1 Diagonal Blocks, 3.5.2 Low-Rank Blocks, the ssd
 * listing in 3.5.3); variable length by state reset -- "LLM(十一)——Mamba" §3.7.3;
 * grouped B/C heads -- "LLM(十一)——Mamba" §3.6.
 *
 * Conventions for every entry point:
 *   - All tensor pointers are DEVICE pointers (except in ssd_forward_host), row-major
 *     and contiguous, 16-byte aligned. The caller owns every buffer and the stream.
 *   - The library allocates no device memory. Scratch lives in the caller's workspace.
 *   - Work is enqueued on `stream`; no call synchronises the stream except
 *     ssd_status and ssd_forward_host.
 *   - Return value: SSD_OK or one of the SSD_ERR_* codes below; nothing is launched
 *     when an argument check fails. Errors raised on the device (a bounded wait that
 *     timed out) are recorded in the workspace and read back by ssd_status.
 */
#ifndef SSD_GB300_H
#define SSD_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Storage type of x, B, C and y. dt, A, D and the states are always fp32. */
typedef enum { SSD_F32 = 0, SSD_BF16 = 1 } ssd_dtype;

#define SSD_OK               0
#define SSD_ERR_INVALID_ARG  1  /* bad shape, NULL pointer, misalignment, H % G, cu_seqlens with batch != 1 */
#define SSD_ERR_UNSUPPORTED  2  /* chunk or head/state size outside the kernel set, or not an sm_103 device */
#define SSD_ERR_CUDA         3  /* a CUDA runtime call or launch failed */
#define SSD_ERR_TIMEOUT      4  /* a bounded device-side wait gave up (reported by ssd_status) */
#define SSD_ERR_WORKSPACE    5  /* workspace NULL, misaligned or smaller than ssd_workspace_size() */

/*
 * Problem shape. batch rows of seqlen tokens each (dense), or, with cu_seqlens,
 * batch == 1 and seqlen = total number of packed tokens.
 *   nheads  H  -- heads; headdim P -- channels per head; dstate N -- state size;
 *   ngroups G  -- B/C groups, G divides H, heads [g*H/G, (g+1)*H/G) share group g.
 */
typedef struct {
    int64_t batch, seqlen, nheads, headdim, dstate, ngroups;
} ssd_shape;

/*
 * Bytes of device workspace ssd_forward needs for this shape, dtype, chunk and
 * number of sequences (nseq = number of cu_seqlens segments, or 0 for a dense batch).
 * Returns 0 when the arguments are invalid or unsupported.
 */
size_t ssd_workspace_size(const ssd_shape *shape, ssd_dtype dtype, int chunk, int nseq);

/*
 * One forward pass, enqueued on `stream` (a cudaStream_t; NULL = legacy default stream).
 *
 *   x             (batch, seqlen, H, P)  dtype
 *   dt            (batch, seqlen, H)     fp32, expected > 0 (used as given: no softplus, no bias)
 *   A             (H)                    fp32, expected < 0
 *   B, C          (batch, seqlen, G, N)  dtype
 *   D             (H)                    fp32, or NULL for no skip term
 *   chunk         block length Q of the decomposition: 64, 128 or 256. The result does not
 *                 depend on it beyond rounding. The fp32 path uses it as its block length; the
 *                 bf16 path validates it and otherwise ignores it (its tile is always 128 tokens).
 *   initial_state (nseq_or_batch, H, P, N) fp32, or NULL for zero states
 *   cu_seqlens    (nseq + 1) int32 DEVICE array of segment offsets into the packed row
 *                 (first 0, last seqlen, non-decreasing), or NULL for a dense batch.
 *                 Requires batch == 1. No state crosses a segment boundary.
 *   nseq          number of segments when cu_seqlens != NULL, else ignored
 *   y             (batch, seqlen, H, P)  dtype, written
 *   final_state   (nseq_or_batch, H, P, N) fp32, written, or NULL
 *   workspace     device scratch of at least ssd_workspace_size(...) bytes, 256-byte aligned;
 *                 its contents on entry do not matter
 *
 * Supported sizes: dtype SSD_F32 -- any P <= 256, N <= 256 (SIMT fp32 kernels);
 * dtype SSD_BF16 -- P == 64, N in {64, 128, 256}, H/G even (tcgen05 kernels).
 * y must not alias any input. Inputs must be finite.
 */
int ssd_forward(const ssd_shape *shape, ssd_dtype dtype,
                const void *x, const float *dt, const float *A,
                const void *B, const void *C, const float *D,
                int chunk, const float *initial_state,
                const int32_t *cu_seqlens, int nseq,
                void *y, float *final_state,
                void *workspace, size_t workspace_bytes,
                void *stream);

/*
 * Flags of ssd_forward_ex / ssd_forward_host_ex / ssd_decode_step_ex.
 *
 * SSD_SCALE_X_BY_DT: the input term of the recurrence is dt_t * x_t (outer) B_t instead of
 *   x_t (outer) B_t -- the discretization the full model keeps from Mamba, with the input matrix
 *   taken as dt * B ("LLM(十一)——Mamba" §3.5.4: the continuous parameters are transformed before they
 *   enter the SSD code; "Transformers是SSMs (一)" §2.1, Remark 1). The skip term stays D * x_t, and
 *   the decay stays exp(dt_t * A). dt must then be >= 0 (its logarithm is taken on the bf16 path).
 *   Fusing it saves the caller a pass that scales x.
 */
#define SSD_SCALE_X_BY_DT 1u

/*
 * SSD_DEBUG_FORCE_TIMEOUT: a failure-detection test hook of the bf16 (tcgen05) path, not for normal
 *   use. Every wait of a CTA for a window state published by another CTA (the look-back of the
 *   inter-chunk pass) waits for a value that is never written, with a limit of about one millisecond
 *   instead of two seconds. The call then ends with SSD_ERR_TIMEOUT in the workspace (ssd_status
 *   returns it, and the workspace's third int32 holds the location code 0x300), every kernel returns,
 *   and y is only partly written. Nothing is left running on the GPU: copies and tensor-core work
 *   already issued are waited for before each CTA exits. The fp32 path ignores the flag.
 */
#define SSD_DEBUG_FORCE_TIMEOUT 0x80000000u

/*
 * ssd_forward with option flags (0, SSD_SCALE_X_BY_DT, SSD_DEBUG_FORCE_TIMEOUT); other bits give
 * SSD_ERR_INVALID_ARG.
 * Everything else is as for ssd_forward.
 */
int ssd_forward_ex(const ssd_shape *shape, ssd_dtype dtype, unsigned flags,
                   const void *x, const float *dt, const float *A,
                   const void *B, const void *C, const float *D,
                   int chunk, const float *initial_state,
                   const int32_t *cu_seqlens, int nseq,
                   void *y, float *final_state,
                   void *workspace, size_t workspace_bytes,
                   void *stream);

/*
 * The same forward pass on HOST buffers: copies the inputs to device memory
 * carved out of `device_buffer`, runs ssd_forward, copies y and final_state back,
 * and synchronises `stream`. Host buffers should be pinned for full copy speed.
 * cu_seqlens is a HOST array here. device_buffer must hold at least
 * ssd_host_buffer_size(...) bytes (inputs, outputs and workspace).
 */
size_t ssd_host_buffer_size(const ssd_shape *shape, ssd_dtype dtype, int chunk, int nseq);
int ssd_forward_host(const ssd_shape *shape, ssd_dtype dtype,
                     const void *x, const float *dt, const float *A,
                     const void *B, const void *C, const float *D,
                     int chunk, const float *initial_state,
                     const int32_t *cu_seqlens, int nseq,
                     void *y, float *final_state,
                     void *device_buffer, size_t device_buffer_bytes,
                     void *stream);
/* ssd_forward_host with option flags (see ssd_forward_ex). */
int ssd_forward_host_ex(const ssd_shape *shape, ssd_dtype dtype, unsigned flags,
                        const void *x, const float *dt, const float *A,
                        const void *B, const void *C, const float *D,
                        int chunk, const float *initial_state,
                        const int32_t *cu_seqlens, int nseq,
                        void *y, float *final_state,
                        void *device_buffer, size_t device_buffer_bytes,
                        void *stream);

/*
 * ssd_forward for callers that cannot allocate device memory (for example code that runs
 * before its allocator is set up, or inside a context whose memory it does not own). There
 * is no counterpart on the pages: this entry point only changes where scratch comes from.
 *
 * Arguments and results are those of ssd_forward without the workspace: the scratch is a
 * file-scope device array of 16 MiB inside this library, which every GPU that loads the
 * library holds until the process exits. Problems whose ssd_workspace_size exceeds it are
 * rejected with SSD_ERR_WORKSPACE before anything is launched (ssd_last_error_detail gives
 * both sizes). Nothing here calls cudaMalloc, cudaFree or any allocating routine.
 * Nothing in the array has to start at zero: the first kernel of every call clears the
 * status word, counters and look-back flags that the later kernels read.
 *
 * Every call looks up the array's device address in the current context (cudaGetSymbolAddress, which
 * does not synchronise). The first call in a process may also load the library's device code; make it
 * before any stream capture.
 * Every call shares the one array: calls whose work overlaps on the GPU (different
 * streams, or host threads without ordering) race and corrupt each other's results.
 * Errors found on the device are not readable for these calls, because the caller cannot reach the
 * array: a bounded wait that timed out, or malformed cu_seqlens (not starting at 0, decreasing, or not
 * ending at seqlen), which the device-side table builder rejects and which leaves y unwritten. Callers
 * must therefore pass checked segment offsets.
 */
int ssd_forward_noalloc(const ssd_shape *shape, ssd_dtype dtype,
                        const void *x, const float *dt, const float *A,
                        const void *B, const void *C, const float *D,
                        int chunk, const float *initial_state,
                        const int32_t *cu_seqlens, int nseq,
                        void *y, float *final_state,
                        void *stream);

/*
 * One token of the recurrence on a batch of carried states: the recurrent (autoregressive
 * inference) step of the same layer ("Transformers是SSMs (一)" §2.1; "LLM(十一)——Mamba"
 * §3.1.1-3.1.2, with its per-token cost in §3.5.3; "Mamba-2 状态空间对偶性理论" §1.2):
 *
 *   for every row b and head h (group g = h / (H/G)):
 *     a = exp(dt[b,h] * A[h])
 *     new_state[b,h] = a * state[b,h] + x[b,h,:] (outer) B[b,g,:]
 *     y[b,h,:]       = new_state[b,h] . C[b,g,:] + D[h] * x[b,h,:]
 *
 * shape->seqlen must be 1 (one token per row); batch is the number of carried states.
 *   x             (batch, 1, H, P)  dtype
 *   dt            (batch, 1, H)     fp32
 *   A             (H)               fp32
 *   B, C          (batch, 1, G, N)  dtype
 *   D             (H) fp32, or NULL for no skip term
 *   state         (batch, H, P, N)  fp32, read
 *   new_state     (batch, H, P, N)  fp32, written; it may be `state` itself (update in place) but
 *                 must not overlap it otherwise
 *   y             (batch, 1, H, P)  dtype, written
 * All pointers are DEVICE pointers; state, new_state, B and C 16-byte aligned. Supported sizes:
 * P <= 256, N <= 256 with N % 4 == 0, either dtype. No workspace; nothing is synchronised; the
 * same error codes as ssd_forward (nothing is launched when a check fails). batch == 0 is a no-op.
 */
int ssd_decode_step(const ssd_shape *shape, ssd_dtype dtype,
                    const void *x, const float *dt, const float *A,
                    const void *B, const void *C, const float *D,
                    const float *state, float *new_state, void *y,
                    void *stream);

/*
 * ssd_decode_step with the carried state stored as `state_dtype`: SSD_F32 (as above) or SSD_BF16,
 * which halves the bytes the step moves. With a bf16 state the update is computed in fp32 from the
 * stored values, y is taken from the unrounded new state, and only the stored new state is rounded
 * (to nearest even). state and new_state are then (batch, H, P, N) bf16 and N must be a multiple of
 * 8. flags: 0 or SSD_SCALE_X_BY_DT (defined above). Everything else is as for ssd_decode_step.
 */
int ssd_decode_step_ex(const ssd_shape *shape, ssd_dtype dtype, ssd_dtype state_dtype, unsigned flags,
                       const void *x, const float *dt, const float *A,
                       const void *B, const void *C, const float *D,
                       const void *state, void *new_state, void *y,
                       void *stream);

/*
 * The same step on HOST buffers: copies the inputs and the state into `device_buffer` (at least
 * ssd_decode_host_buffer_size bytes, 256-byte aligned), runs ssd_decode_step there in place, copies
 * y and the new state back and synchronises `stream`. new_state may be the host `state` buffer.
 * ssd_decode_host_buffer_size returns 0 for invalid or unsupported shapes.
 */
size_t ssd_decode_host_buffer_size(const ssd_shape *shape, ssd_dtype dtype);
int ssd_decode_step_host(const ssd_shape *shape, ssd_dtype dtype,
                         const void *x, const float *dt, const float *A,
                         const void *B, const void *C, const float *D,
                         const float *state, float *new_state, void *y,
                         void *device_buffer, size_t device_buffer_bytes,
                         void *stream);
/* The host-buffer step with the state stored as `state_dtype` (see ssd_decode_step_ex); the buffer
 * size from ssd_decode_host_buffer_size is enough for either state type. */
int ssd_decode_step_host_ex(const ssd_shape *shape, ssd_dtype dtype, ssd_dtype state_dtype, unsigned flags,
                            const void *x, const float *dt, const float *A,
                            const void *B, const void *C, const float *D,
                            const void *state, void *new_state, void *y,
                            void *device_buffer, size_t device_buffer_bytes,
                            void *stream);

/*
 * Sequence-parallel hand-off ("LLM(十一)——Mamba" §3.7.2 Sequence Parallelism: a worker passes its final
 * state to the next). A sequence cut into consecutive slices runs every slice with ssd_forward from a
 * zero state (on one device each, or one after another); that gives the slice's local y and local
 * final state. With h_in the true state entering a slice and cs_l the sum of dt*A from the slice's
 * first token through token l, linearity gives ("LLM(十一)——Mamba" §3.5.2, center and left factors)
 *     true final = local final + decay * h_in,   decay = exp(cs_last)      (the next slice's h_in)
 *     true y_l   = local y_l   + exp(cs_l) * C_l . h_in^T
 * The caller moves h_in between devices (a copy into local memory; see the Python package's
 * context_parallel module); these calls are the device-side pieces. Dense batches only: each of the
 * `batch` rows of `shape` is a slice of its own sequence (no cu_seqlens).
 *
 * ssd_slice_workspace_size: scratch bytes of either call for `shape` (a 256-byte header whose first
 *   word is read by ssd_status, then per-tile sums of dt and the decays).
 * ssd_slice_decay: decay (batch, H) fp32 = exp(A[h] * sum over the row of dt[., h]); 1 for an empty
 *   slice. Works for both storage types (it reads dt and A only).
 * ssd_slice_correct: y (bf16, (batch, seqlen, H, P), the slice's local outputs) += exp(cs_l) C_l h_in^T,
 *   accumulated in fp32 and rounded to bf16 once more; and, when final_state is not NULL,
 *   final_state (batch, H, P, N) += decay * h_in. h_in: (batch, H, P, N) fp32, read-only (staged as bf16
 *   for the tensor cores, like the chunk states of the forward). bf16 only, with the forward's bf16
 *   shape rules (P = 64, N in {64, 128, 256}, H/G even); C as in ssd_forward.
 * Errors as ssd_forward (argument checks before any launch; SSD_ERR_TIMEOUT through ssd_status).
 */
size_t ssd_slice_workspace_size(const ssd_shape *shape);
int ssd_slice_decay(const ssd_shape *shape, const float *dt, const float *A, float *decay,
                    void *workspace, size_t workspace_bytes, void *stream);
int ssd_slice_correct(const ssd_shape *shape, ssd_dtype dtype, const float *dt, const float *A,
                      const void *C, const float *h_in, void *y, float *final_state,
                      void *workspace, size_t workspace_bytes, void *stream);

/*
 * The Mamba-2 block's output gate and extra normalization, after the SSD layer ("LLM(十一)——Mamba"
 * §3.6.1, Block Design: a normalization layer is added before the output projection, after the
 * multiplicative gate branch). Per token and per group of H*P/groups consecutive channels:
 *     v   = y * silu(z),   silu(z) = z / (1 + exp(-z))        (z NULL: v = y, no gate)
 *     out = v / sqrt(mean over the group of v^2 + eps) * weight
 * The pages print neither formula: the gate's nonlinearity is taken as SiLU, the default nonlinearity of
 * "LLM(十一)——Mamba" §3.6.2, and the normalization as RMSNorm (one group: the whole token; groups > 1:
 * the GroupNorm-style variant).
 *
 *   y, z, out  (batch, seqlen, H, P) bf16 device arrays (shape's dstate and ngroups are ignored); out may
 *              be y itself (in place)
 *   weight     (H*P) fp32, or NULL for ones
 *   eps        >= 0 (silu is computed in fp32 with the hardware approximations of 2^x and 1/x; for very
 *              negative z it is 0)
 *   groups     divides H*P; a group must be a multiple of 8 channels, and H*P at most 6144
 *              (SSD_ERR_UNSUPPORTED otherwise)
 * Enqueued on `stream`; no workspace, no device-side status. Pointers 16-byte aligned. Errors: argument
 * checks before any launch (SSD_ERR_INVALID_ARG, SSD_ERR_UNSUPPORTED), SSD_ERR_CUDA for a failed launch.
 */
int ssd_gated_rmsnorm(const ssd_shape *shape, const void *y, const void *z, const float *weight, float eps,
                      int groups, void *out, void *stream);

/*
 * The same on host buffers: y, z (NULL: no gate), weight (NULL: ones) and out are host arrays (pinned for
 * speed; out may be y). The call copies them through `device_buffer` (device memory the caller owns, 256-byte
 * aligned, at least ssd_gated_rmsnorm_host_buffer_size(shape, z != NULL) bytes), runs the kernel and
 * returns when out holds the result. Tokens of at least 32 MB of y run as a pipeline of four groups of
 * rows whose copies in, kernels and copies out overlap (on the caller's stream and two internal ones).
 * Errors as ssd_gated_rmsnorm, plus SSD_ERR_WORKSPACE for a missing, misaligned or short buffer.
 */
size_t ssd_gated_rmsnorm_host_buffer_size(const ssd_shape *shape, int gated);
int ssd_gated_rmsnorm_host(const ssd_shape *shape, const void *y, const void *z, const float *weight, float eps,
                           int groups, void *out, void *device_buffer, size_t device_buffer_bytes, void *stream);

/*
 * Synchronises `stream`, then returns the device-side status recorded in the
 * workspace by the last ssd_forward (or ssd_slice_* call) that used it: SSD_OK, SSD_ERR_TIMEOUT (a bounded wait gave up),
 * SSD_ERR_INVALID_ARG (malformed cu_seqlens, found by the device-side table builder; y is then not
 * written), or SSD_ERR_CUDA if the copy itself fails.
 */
int ssd_status(const void *workspace, void *stream);

/* Static, NUL-terminated description of a return code. */
const char *ssd_status_string(int code);

/*
 * Detail of the most recent SSD_ERR_CUDA returned to the calling host thread: the
 * failing step and the CUDA runtime's error name (e.g. "fused launch:
 * cudaErrorInvalidValue"), or "" if none. The string stays valid until the next call
 * from the same thread.
 */
const char *ssd_last_error_detail(void);

#ifdef __cplusplus
}
#endif
#endif /* SSD_GB300_H */
