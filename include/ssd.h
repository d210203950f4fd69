/*
 * ssd.h -- C ABI of libssd: the Mamba-2 state-space-duality (SSD) chunked
 * forward pass on NVIDIA GB300 (sm_103a).
 *
 * The operation (one scalar decay per head, "Why SSM and linear-RNN FLOPs do
 * not convert into GPU FLOPs", paragraph 1):
 *
 *     h_t = exp(dt_t * A_h) * h_{t-1} + dt_t * x_t B_t^T      h_t in R^{P x N}
 *     y_t = h_t C_t + D_h * x_t
 *
 * computed chunk-wise ("Mamba-2 in NVIDIA cuTile: Faster Forward Kernels",
 * section "Why Mamba-2 is a useful kernel example": one kernel prepares the
 * cumulative decay values, another the state entering each chunk, a third
 * the outputs, with the intra-chunk interactions kept on-chip).  The
 * quadratic-inside / linear-across split with chunk size Q follows the
 * da_be19 thread, post 5/6.
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * Shapes use the names of the pages' notation:
 *   b = batch, L = seqlen, H = nheads, P = headdim, N = dstate,
 *   G = ngroups (heads h = g*H/G .. (g+1)*H/G - 1 share B and C),
 *   Q = chunk_size, nc = L / Q.
 * Tensor layouts (row-major, contiguous, element type in brackets; "T" is
 * fp32 or bf16 as given by ssd_shape_t.dtype):
 *   x          [b, L, H, P]       T
 *   dt         [b, L, H]          T   (already positive: no softplus/bias here)
 *   A          [H]                fp32 (negative)
 *   B, C       [b, L, G, N]       T
 *   D          [H]                fp32 (skip term; NULL = no skip)
 *   init_state [b, H, P, N]       fp32 (NULL = zero initial state)
 *   y          [b, L, H, P]       ydtype (fp32, or the input dtype)
 *   final_state[b, H, P, N]       fp32 (NULL = not written)
 *   dA_cumsum  [b, H, nc, Q]      fp32 inclusive cumsum of dt*A inside a chunk
 *   states     [b, nc, H, P, N]   fp32 state each chunk produces from zero
 *   states_in  [b, nc, H, P, N]   fp32 state entering each chunk
 * Ownership: every pointer is caller-owned device memory (x, y, ... may come
 * from any allocator); the library allocates nothing and keeps no pointer
 * after a call returns.  Every pointer must be 16-byte aligned.
 * Execution: calls are asynchronous on `stream` (0 = legacy default stream).
 * Errors: argument errors are detected on the host and returned before
 * anything is enqueued (SSD_ERR_INVALID_ARG / SSD_ERR_UNSUPPORTED);
 * a failed launch returns SSD_ERR_CUDA.  Failures the kernels detect while
 * they run (a bounded wait that gave up) cannot be returned by the call that
 * enqueued them: they are latched in a per-device status word that
 * ssd_get_device_status() reads.  No entry point but that one synchronises.
 * Supported on the GPU: chunk_size 64 or 128, any L (nc = ceil(L / Q): a
 * partial last chunk is processed as if padded with dt = 0 steps, which
 * neither decay nor feed the state, and nothing is written for them; the
 * stage layouts below then hold nc chunks, the missing dA_cumsum entries
 * repeating the chunk's last value), H % G == 0, P in {16, 32, 64, 128},
 * N in {16, 32, 64, 128, 256}.
 * Outputs are bitwise reproducible run to run: no floating-point atomics.
 */
#ifndef SSD_H_
#define SSD_H_

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#if defined(__GNUC__)
#define SSD_API __attribute__((visibility("default")))
#else
#define SSD_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    SSD_OK = 0,
    SSD_ERR_INVALID_ARG = 1,   /* null pointer, bad shape, misaligned pointer */
    SSD_ERR_UNSUPPORTED = 2,   /* a valid shape the library has no kernel for */
    SSD_ERR_CUDA = 3,          /* a CUDA launch or query failed */
    SSD_ERR_WORKSPACE = 4,     /* workspace missing or smaller than required */
    SSD_ERR_SCRATCH_LIMIT = 5, /* ssd_fwd_noalloc: shape needs more than its static scratch */
    SSD_ERR_TIMEOUT = 6        /* a kernel's bounded wait gave up (read by ssd_get_device_status) */
} ssd_status_t;

typedef enum { SSD_DTYPE_F32 = 0, SSD_DTYPE_BF16 = 1 } ssd_dtype_t;

/*
 * Problem description.  `dtype` is the element type of x, dt, B, C.
 * `ydtype` is the element type of y: SSD_DTYPE_F32 (the default of a
 * zero-initialised struct; y keeps the fp32 accumulator's precision) or the
 * input dtype (bf16 y: half the output bytes, plus bf16 output rounding of at
 * most 2^-9 relative).
 */
typedef struct {
    int64_t batch, seqlen, nheads, headdim, dstate, ngroups, chunk_size;
    ssd_dtype_t dtype;
    ssd_dtype_t ydtype;
} ssd_shape_t;

/* Human-readable name of a status code (static storage, never NULL). */
SSD_API const char *ssd_status_string(ssd_status_t status);

/* Version of this ABI: (major << 16) | minor. */
SSD_API int ssd_abi_version(void);

/*
 * Device-detected failures.  Every wait inside the tensor-core kernels is
 * bounded in time; a wait that gives up (a producer that never arrives)
 * makes its CTA drain its own copies and MMAs, free its tensor memory and
 * exit, and latches SSD_ERR_TIMEOUT in a status word of the current device
 * that every call of this library shares.  The outputs of the call that
 * timed out are then incomplete.
 * ssd_get_device_status(stream) waits for `stream` (cudaStreamSynchronize),
 * reads the word and clears it: SSD_OK when no wait of any call on this
 * device has given up since the previous read, SSD_ERR_TIMEOUT otherwise,
 * SSD_ERR_CUDA when the stream or the read failed.  The word is sticky
 * across calls and streams (like the CUDA runtime's sticky errors): to pin a
 * failure on one call, read it before and after that call.
 */
SSD_API ssd_status_t ssd_get_device_status(cudaStream_t stream);

/*
 * Bytes of device workspace ssd_fwd needs for `shape` on the current
 * device (0 for an invalid shape).  The workspace holds the ready flags and
 * per-chunk operand packs (masked C B^T with the chunk's B and C, bf16) and
 * the per-segment states of the two-pass chunk scan; how the sequence is cut
 * into segments depends on the device's SM count, so query the size with the
 * device current that will run the call.  It needs no initialisation (every
 * call clears what it reads) and may be reused by later calls on the same
 * stream.
 */
SSD_API size_t ssd_fwd_workspace_size(const ssd_shape_t *shape);

/*
 * Fused SSD forward: y and final_state from x, dt, A, B, C, D, init_state.
 * The whole chunked algorithm -- cumulative decay, chunk states, the pass of
 * states between chunks, chunk outputs -- runs on the GPU with the state and
 * the intra-chunk score matrix kept on-chip; only per-segment states and the
 * per-chunk operand packs touch the workspace.  `workspace` must hold
 * ssd_fwd_workspace_size(shape) bytes (SSD_ERR_WORKSPACE otherwise).  D,
 * init_state, final_state may be NULL.  The result does not depend on
 * chunk_size beyond rounding (a chunked sum is exact in any blocking): on the
 * tensor-core path a chunk of 128 steps runs as two 64-step tiles.
 */
SSD_API ssd_status_t ssd_fwd(const ssd_shape_t *shape, const void *x, const void *dt,
                     const float *A, const void *B, const void *C,
                     const float *D, const float *init_state, void *y,
                     float *final_state, void *workspace, size_t workspace_bytes,
                     cudaStream_t stream);

/*
 * ssd_fwd without a workspace argument, for callers that cannot allocate
 * device memory: code running inside a host application or inference
 * server that owns the whole device memory pool and forbids allocations
 * outside it, or latency-critical paths that must not call cudaMalloc after
 * start-up (it can block on the device and can fail under memory pressure).
 * The pages have no counterpart; it is the same computation as ssd_fwd.
 *
 * Scratch comes from one static device buffer of SSD_NOALLOC_SCRATCH_BYTES
 * that lives in this library (every GPU that loads the library holds it
 * until the process exits).  Shapes whose ssd_fwd_workspace_size() exceeds
 * it return SSD_ERR_SCRATCH_LIMIT before anything is enqueued.  The call
 * itself allocates nothing: no cudaMalloc, no cudaFree.
 * The first call on each device (and the first after that device's context
 * was destroyed and created again) looks up the buffer's device address
 * (cudaGetSymbolAddress) with that device current; make that first call
 * before any stream capture.  Every call shares the one buffer: calls whose
 * GPU work overlaps (different streams, or several host threads) race on
 * it, so serialise them.  Inputs, outputs and errors as for ssd_fwd; a wait
 * that gave up inside its kernels is read with ssd_get_device_status.
 */
#define SSD_NOALLOC_SCRATCH_BYTES (32u << 20)
SSD_API ssd_status_t ssd_fwd_noalloc(const ssd_shape_t *shape, const void *x, const void *dt,
                                     const float *A, const void *B, const void *C,
                                     const float *D, const float *init_state, void *y,
                                     float *final_state, cudaStream_t stream);

/*
 * Packed variable-length batch: nseq independent sequences stored back to
 * back along L (x [1, Ltot, H, P], dt [1, Ltot, H], B, C [1, Ltot, G, N], y
 * [1, Ltot, H, P]; shape->batch must be 1 and shape->seqlen = Ltot).
 * Sequence s covers steps cu_seqlens[s] .. cu_seqlens[s+1] - 1 (a HOST array
 * of nseq + 1 offsets, 0 first and Ltot last, non-decreasing); its state
 * starts from init_states[s] (NULL: zero) and ends in final_states[s] (NULL:
 * not written), both [nseq, H, P, N] fp32.  No state crosses a sequence
 * boundary.  On the tensor-core path (bf16 inputs and a tile shape it
 * covers) the sequences run in launch sets of up to 800: a chunk-scan CTA
 * per (sequence, head block), longest first, with the C B^T pass walking
 * every sequence's chunks; when those CTAs leave SMs free, every sequence is
 * cut into segments of the same chunk count (a segment-state pass forms the
 * earlier segments' local states, as in ssd_fwd); when they would take
 * several waves of CTAs, consecutive short sequences may share a CTA, which
 * runs them one after another.  The longest sequences may instead run the
 * fused forward of ssd_fwd each, whichever a host-side cost model rates
 * faster.  A sequence's partial last chunk then reads the next sequence's
 * first steps and gives them dt = 0, so they add 0 times their values:
 * finite inputs leave no trace across the boundary (a non-finite x or B
 * there would).  Other inputs run the fused forward per sequence.
 * Everything is enqueued on `stream` and shares `workspace`, which must hold
 * ssd_fwd_varlen_workspace_size(shape, cu_seqlens, nseq) bytes (0 for
 * invalid arguments).  Every sequence's start must keep the pointers it
 * derives 16-byte aligned (cu_seqlens[s] * H * sizeof(dtype) a multiple of
 * 16, e.g. H a multiple of 8 for bf16): SSD_ERR_INVALID_ARG otherwise.
 * (The pages are silent on batches of unequal lengths; this packs them the
 * way the chunk split of "Mamba-2 in NVIDIA cuTile", section "Why Mamba-2 is
 * a useful kernel example", extends to.)
 */
SSD_API size_t ssd_fwd_varlen_workspace_size(const ssd_shape_t *shape, const int64_t *cu_seqlens, int64_t nseq);
SSD_API ssd_status_t ssd_fwd_varlen(const ssd_shape_t *shape, const int64_t *cu_seqlens, int64_t nseq,
                                    const void *x, const void *dt, const float *A, const void *B,
                                    const void *C, const float *D, const float *init_states, void *y,
                                    float *final_states, void *workspace, size_t workspace_bytes,
                                    cudaStream_t stream);

/*
 * Stage 1: dA_cumsum[b,h,c,q] = sum_{k<=q} dt[b, c*Q+k, h] * A[h].
 * ("Mamba-2 in NVIDIA cuTile", section "Why Mamba-2 is a useful kernel
 * example": the kernel that prepares the cumulative decay values.)
 */
SSD_API ssd_status_t ssd_chunk_cumsum(const ssd_shape_t *shape, const void *dt,
                              const float *A, float *dA_cumsum,
                              cudaStream_t stream);

/*
 * Stage 2: states[b,c,h,p,n] = sum_q exp(cum[Q-1] - cum[q]) * dt_q *
 *          x[b, cQ+q, h, p] * B[b, cQ+q, g(h), n]   (cum = dA_cumsum[b,h,c,:]),
 * the state chunk c produces from a zero start: a decay-weighted x^T B
 * contraction per chunk (the BMMs for state accumulation of the da_be19
 * thread, post 5/6).
 */
SSD_API ssd_status_t ssd_chunk_state(const ssd_shape_t *shape, const void *x,
                             const void *dt, const void *B,
                             const float *dA_cumsum, float *states,
                             cudaStream_t stream);

/*
 * Stage 3: states_in[b,0] = init_state (zeros when NULL);
 *          states_in[b,c+1] = exp(dA_cumsum[b,h,c,Q-1]) * states_in[b,c] + states[b,c];
 *          final_state = the value after the last chunk (if non-NULL).
 * ("Mamba-2 in NVIDIA cuTile", the kernel that calculates the state
 * entering each chunk.)
 */
SSD_API ssd_status_t ssd_state_passing(const ssd_shape_t *shape, const float *states,
                               const float *dA_cumsum, const float *init_state,
                               float *states_in, float *final_state,
                               cudaStream_t stream);

/*
 * Stage 4: for t in chunk c (cum = dA_cumsum[b,h,c,:], i = t - cQ):
 *   y[b,t,h,:] = sum_{j<=i} (C_t . B_j) exp(cum_i - cum_j) dt_j x_j
 *              + exp(cum_i) * states_in[b,c,h] C_t + D[h] x_t
 * The masked intra-chunk score matrix stays on-chip ("Mamba-2 in NVIDIA
 * cuTile", the output kernel whose intermediate interactions stay in
 * registers).  D may be NULL.
 */
SSD_API ssd_status_t ssd_chunk_scan(const ssd_shape_t *shape, const void *x,
                            const void *dt, const void *B, const void *C,
                            const float *dA_cumsum, const float *states_in,
                            const float *D, void *y, void *workspace,
                            size_t workspace_bytes, cudaStream_t stream);

/*
 * Bytes of device workspace ssd_chunk_scan needs for `shape` (0 for an
 * invalid shape, and 0 where the call needs none; workspace may then be
 * NULL).  On the bf16 tensor-core path it holds the per-chunk operand packs
 * (masked C B^T with the chunk's B and C) and their ready flags; it needs no
 * initialisation and may be reused by later calls on the same stream.
 */
SSD_API size_t ssd_chunk_scan_workspace_size(const ssd_shape_t *shape);

/*
 * Self-test of the failure path (the pages have no counterpart): enqueues
 * the tensor-core chunk-scan stage kernel of ssd_chunk_scan alone, with its
 * operand packs marked "not yet published" and no kernel that publishes
 * them, so the wait of every CTA for its first pack runs out after
 * `wait_ns` nanoseconds of wall time (clamped to [1e5, 1e9]).  Each CTA
 * gives up before it loads any x tile or operand pack or issues any MMA,
 * lets the loads it did issue (its dt boxes) land, frees its tensor memory
 * and exits; SSD_ERR_TIMEOUT is latched for ssd_get_device_status.
 * Arguments as for ssd_chunk_scan; y is left unwritten.  Returns
 * SSD_ERR_UNSUPPORTED for shapes off the tensor-core path.  Nothing here
 * faults, traps or hangs the GPU: the test of the bounded waits.
 */
SSD_API ssd_status_t ssd_selftest_scan_timeout(const ssd_shape_t *shape, const void *x,
                                               const void *dt, const void *B, const void *C,
                                               const float *dA_cumsum, const float *states_in,
                                               const float *D, void *y, void *workspace,
                                               size_t workspace_bytes, uint64_t wait_ns,
                                               cudaStream_t stream);

/*
 * The same recurrence as ssd_fwd, evaluated as a plain sequential scan over
 * t on the fp32 ALUs (no tensor cores): the schedule the scan-versus-matmul
 * comparison of "Why SSM and linear-RNN FLOPs do not convert into GPU
 * FLOPs", paragraph 1, measures.  Same arguments and layouts as ssd_fwd,
 * no workspace.  Requires only H % G == 0 (any L, any chunk_size field).
 */
SSD_API ssd_status_t selective_scan_fwd(const ssd_shape_t *shape, const void *x,
                                const void *dt, const float *A, const void *B,
                                const void *C, const float *D,
                                const float *init_state, void *y,
                                float *final_state, cudaStream_t stream);

/*
 * Quadratic (dual) form for short sequences: the same y and final_state as
 * ssd_fwd, computed without chunks as
 *   y     = (L o C B^T) (dt o x) + (exp(cum) o C) init^T + D x,
 *   L_ts  = exp(cum_t - cum_s) for s <= t (0 above), cum = running sum of dt A,
 *   final = sum_s exp(cum_{L-1} - cum_s) dt_s x_s^T B_s + exp(cum_{L-1}) init
 * (the attention-like form that can beat the chunked algorithm on short
 * sequences: the da_be19 thread, post 5/6).  Work grows with L^2, so it is
 * offered for L <= 1024 only: bf16 inputs, P in {64, 128}, N in {64, 128},
 * heads per group a multiple of 128 / P; SSD_ERR_UNSUPPORTED otherwise.
 * shape->chunk_size is ignored.  No workspace.  D, init_state and
 * final_state may be NULL.  A bounded wait that gives up is latched for
 * ssd_get_device_status.
 */
SSD_API ssd_status_t ssd_fwd_quadratic(const ssd_shape_t *shape, const void *x, const void *dt,
                                       const float *A, const void *B, const void *C, const float *D,
                                       const float *init_state, void *y, float *final_state,
                                       cudaStream_t stream);

/*
 * Recurrent (decode) step: one new token per sequence advances the state in
 * place and gives that token's output -- the recurrence itself for a single
 * step, O(P N) work per head with a state of constant size (the inference
 * mode of the da_be19 thread, post 5/6):
 *   state[b,h] <- exp(dt[b,h] A[h]) state[b,h] + dt[b,h] x[b,h] B[b,g(h)]^T
 *   y[b,h]      = state[b,h] C[b,g(h)] + D[h] x[b,h]
 * Layouts: x [b, H, P], dt [b, H], B, C [b, G, N] (T = shape->dtype), A, D [H]
 * fp32 (D may be NULL), state [b, H, P, N] fp32 (read and written), y
 * [b, H, P] (shape->ydtype).  shape->seqlen and chunk_size are ignored (one
 * step).  Running a sequence token by token through this call gives the
 * same result as ssd_fwd over the whole sequence (up to rounding); a state
 * left by ssd_fwd (final_state) continues directly.
 */
SSD_API ssd_status_t ssd_decode_step(const ssd_shape_t *shape, const void *x, const void *dt,
                                     const float *A, const void *B, const void *C, const float *D,
                                     float *state, void *y, cudaStream_t stream);

/*
 * Launch timing (instrumentation; the pages have no counterpart).  While
 * enabled, every entry point records a CUDA event on its stream before each
 * kernel it launches and one after the last, so a caller can read the device
 * time of each launch of the most recent call.  Disabled by default; the
 * events cost a few microseconds of host time per launch.
 *   ssd_launch_timing_enable(1) creates the events (SSD_ERR_CUDA on failure),
 *   ssd_launch_timing_enable(0) destroys them.
 *   ssd_launch_timing_read(ms, cap) waits for the last call's events, writes
 *   up to `cap` per-launch durations in milliseconds and returns the number
 *   of launches of that call (-1 if timing is off or no call was recorded).
 *   ssd_launch_timing_name(i) names the kernel of launch i of that call
 *   (static storage; NULL when out of range).
 * Not thread-safe: one host thread should drive a timed sequence of calls.
 */
SSD_API ssd_status_t ssd_launch_timing_enable(int enable);
SSD_API int ssd_launch_timing_read(float *ms, int cap);
SSD_API const char *ssd_launch_timing_name(int i);

#ifdef __cplusplus
}
#endif

#endif /* SSD_H_ */
