/*
 * ssd.h -- C ABI of the B300 (sm_103a) SSD layer library, libssd_b300.so.
 *
 * The library computes the Structured State Space Duality (SSD) layer of
 * Mamba-2, forward only, on one GPU:
 *
 *     h_t = exp(dt_t * A_h) * h_{t-1} + dt_t * x_t B_t^T      (state P x N)
 *     y_t = h_t C_t + D_h * x_t
 *
 * per head h, with A_h one scalar per head and B, C shared by the heads of a
 * group.  Sources: the recurrence "h_t = A_t h_{t-1} + B_t x_t,
 * y_t = C_t^T h_t" ("Mamba-2는 왜 Transformer와 닮았는가", bdev.io, section
 * "문제: 선형 복잡도만으로는 충분하지 않다"); ZOH A-bar = exp(dt A),
 * B-bar ~= dt B and the skip term D x ("20.1 상태 공간 모델 (SSM)",
 * sungeuns.github.io, sec. 1 and the loop of sec. 5); scalar-times-identity
 * A and heads sharing B/C ("Transformers are SSMs Review",
 * dimensionstp.github.io, sec. 3-2 (3) and (5)); the chunked algorithm --
 * intra-chunk quadratic blocks, chunk states, state passing, off-diagonal
 * output -- (same review, sec. 3-2 (4)); varlen packing with the state cut
 * at sequence boundaries (same review, sec. 3-2 (6)).
 *
 * Conventions shared by every entry point
 *  - All tensor pointers are DEVICE pointers owned by the caller.  The
 *    library keeps no pointer after a call returns and allocates no device
 *    or host memory.
 *  - Calls are asynchronous and stream-ordered on `stream` (a cudaStream_t;
 *    NULL = the legacy default stream).  Results are complete when the
 *    stream reaches the point after the call.
 *  - Argument checks run on the host before anything is launched; a failing
 *    check returns SSD_ERR_INVALID or SSD_ERR_UNSUPPORTED and launches
 *    nothing.  A launch failure returns SSD_ERR_CUDA.
 *  - Errors that only the device can see (an invalid cu_seqlens array, a
 *    bounded wait that expired) are written to *dev_status when it is not
 *    NULL: the library clears it at the start of the call and a kernel
 *    stores the SSD_ERR_* code there.  Read it after synchronising.
 *  - Layouts are dense row-major (C order) with the shapes given below.
 *    x, B, C and y must be 16-byte aligned.
 *  - Head h reads group g(h) = floor(h * ngroups / nheads); nheads must be
 *    a multiple of ngroups.
 */
#ifndef SSD_B300_H
#define SSD_B300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    SSD_OK = 0,
    SSD_ERR_INVALID = 1,      /* bad pointer, size or layout */
    SSD_ERR_UNSUPPORTED = 2,  /* valid but outside what the kernels handle */
    SSD_ERR_CUDA = 3,         /* a CUDA runtime call or launch failed */
    SSD_ERR_TIMEOUT = 4       /* device: a bounded inter-block wait expired */
} ssd_status_t;

typedef enum {
    SSD_DT_F32 = 0,   /* x, dt, B, C as float32 */
    SSD_DT_BF16 = 1   /* x, dt, B, C as bfloat16 */
} ssd_dtype_t;

/*
 * ssd_chunk_scan_fwd -- SSD layer forward over whole sequences.
 *
 * Inputs (`in_dtype` elements unless stated):
 *   x   [ntok, nheads, headdim]     ntok = batch * seqlen
 *   dt  [ntok, nheads]              step sizes, already positive
 *   A   [nheads] float32            per-head decay rate (A <= 0 in practice)
 *   B   [ntok, ngroups, dstate]
 *   C   [ntok, ngroups, dstate]
 *   D   [nheads] float32 or NULL    skip weight; NULL means 0
 *   init_states float32 [nseq_or_batch, nheads, headdim, dstate] or NULL
 *               (NULL means a zero state for every sequence)
 *   cu_seqlens  int32 [nseq + 1] DEVICE array or NULL.  NULL: `batch`
 *               independent rows of `seqlen` tokens.  Otherwise `batch`
 *               must be 1 and the nseq sequences are the packed token
 *               ranges [cu_seqlens[s], cu_seqlens[s+1]); cu_seqlens[0] = 0,
 *               non-decreasing, cu_seqlens[nseq] = seqlen.  The state is
 *               reset (or set from init_states[s]) at every sequence start.
 *               A malformed array is detected on the device: nothing is
 *               computed and *dev_status receives SSD_ERR_INVALID.
 * Outputs (float32):
 *   y            [ntok, nheads, headdim]
 *   final_states [nseq_or_batch, nheads, headdim, dstate] or NULL
 * Scratch:
 *   workspace / workspace_bytes: device memory of at least
 *   ssd_chunk_scan_fwd_workspace_size(...) bytes, 256-byte aligned, owned by
 *   the caller; its contents on entry do not matter.  Calls that overlap in
 *   time must not share a workspace.
 * Supported: chunk_size in {64, 128, 256}; headdim in [1, 128] and
 *   dstate in {16, 32, 64, 128, 256} for float32 inputs; for bfloat16
 *   inputs headdim == 64 and dstate == 128 run on the tcgen05 tensor-core
 *   kernel and the other shapes of the float32 list on the CUDA-core
 *   kernels.  The result does not depend on chunk_size beyond rounding: the
 *   chunked algorithm is an exact reordering of the recurrence.
 */
ssd_status_t ssd_chunk_scan_fwd(
    const void *x, const void *dt, const float *A, const void *B, const void *C,
    const float *D, int batch, int seqlen, int nheads, int headdim, int dstate,
    int ngroups, int chunk_size, ssd_dtype_t in_dtype, const float *init_states,
    const int32_t *cu_seqlens, int nseq, float *y, float *final_states,
    void *workspace, size_t workspace_bytes, int32_t *dev_status, void *stream);

/*
 * Fused epilogue options of ssd_chunk_scan_fwd_ex: the steps on either side
 * of the SSD layer in a Mamba block, done inside the forward kernel so that
 * neither the positive dt nor the ungated y makes a round trip through HBM.
 *  - dt_softplus != 0: the layer uses softplus(dt + dt_bias[h]) in place of
 *    dt, where softplus(v) = log(1 + exp(v)); dt_bias [nheads] float32 or
 *    NULL (0).  The step size of the selective SSM is a softplus of a
 *    projection ("20.1 상태 공간 모델 (SSM)", sungeuns.github.io, sec. 2 and
 *    the sec. 5 loop); dt then holds the projection without its bias.
 *  - z != NULL: y is multiplied by silu(z) = z / (1 + exp(-z)) elementwise;
 *    z [ntok, nheads, headdim] in `in_dtype`, 16-byte aligned.  The block's
 *    second branch is a gate multiplied into the SSM output (the Mamba paper
 *    review, feghi.github.io, sec. 5); the pages do not name the gate's
 *    nonlinearity, SiLU is the reading taken here.
 *  - y_bf16 != 0: y is written as bfloat16 (round to nearest even), halving
 *    the largest output stream; `y` then points to bfloat16 storage.
 * Zero-initialised options (or a NULL pointer) select none of them.
 */
typedef struct {
    const float *dt_bias;
    int dt_softplus;
    const void *z;
    int y_bf16;
} ssd_fwd_epilogue_t;

/*
 * ssd_chunk_scan_fwd_ex -- ssd_chunk_scan_fwd with the fused epilogue
 * options above (`epilogue` may be NULL).  Same arguments, layouts and errors;
 * `y` is float32 or, with y_bf16, bfloat16.  Any option set requires the
 * tensor-core configuration (bfloat16 inputs, headdim 64, dstate 128);
 * other shapes return SSD_ERR_UNSUPPORTED and launch nothing.
 */
ssd_status_t ssd_chunk_scan_fwd_ex(
    const void *x, const void *dt, const float *A, const void *B, const void *C,
    const float *D, int batch, int seqlen, int nheads, int headdim, int dstate,
    int ngroups, int chunk_size, ssd_dtype_t in_dtype, const float *init_states,
    const int32_t *cu_seqlens, int nseq, void *y, float *final_states,
    void *workspace, size_t workspace_bytes, int32_t *dev_status, void *stream,
    const ssd_fwd_epilogue_t *epilogue);

/*
 * ssd_chunk_scan_fwd_noalloc -- the same forward for callers that cannot
 * allocate device memory.  The pages have no counterpart: this entry point
 * exists for the deployment side only.  Some callers cannot call cudaMalloc
 * or hand over a workspace: a plugin inside a host framework that owns all
 * device memory and passes in only its inputs and outputs, or a
 * latency-critical loop in which an allocation (which may synchronise the
 * device) is not allowed.  This entry point needs neither.
 *
 * Arguments, layouts and results are those of ssd_chunk_scan_fwd without
 * the workspace pair; the caller still passes every input and output.  It
 * always runs the CUDA-core kernels (fp32 arithmetic), whatever the dtype.
 * Its scratch memory is one fixed 16 MiB array compiled into the library
 * (a file-scope __device__ array): every GPU on which the library is loaded
 * holds those 16 MiB until the process exits.  A problem whose scratch
 * would exceed 16 MiB is rejected with SSD_ERR_UNSUPPORTED before anything
 * is launched; the scratch needed is about 4 * nheads * headdim * dstate
 * bytes per chunk of every sequence.  The first call on a device looks up
 * the array's device address (cudaGetSymbolAddress, with that device
 * current) and caches it.  With lazy module loading (the CUDA default) that
 * first lookup is also when the driver loads the library's device code on
 * that device and reserves the 16 MiB: a one-time step that may
 * synchronise the device.  Make the first call during set-up -- before any
 * stream capture and outside latency-critical loops; from then on the
 * memory stays reserved until the process exits.  The cached address
 * belongs to the device's current context: do not use this entry point
 * across a cudaDeviceReset (or anything else that destroys and recreates
 * the primary context) in the same process.  Every call shares the one
 * array and nothing in it needs to start at zero; calls whose GPU work
 * overlaps in time (other streams, other threads) race on it and must be
 * serialised by the caller.  After that first call no allocation of any
 * kind is made, neither by the library nor by any library it calls.
 */
ssd_status_t ssd_chunk_scan_fwd_noalloc(
    const void *x, const void *dt, const float *A, const void *B, const void *C,
    const float *D, int batch, int seqlen, int nheads, int headdim, int dstate,
    int ngroups, int chunk_size, ssd_dtype_t in_dtype, const float *init_states,
    const int32_t *cu_seqlens, int nseq, float *y, float *final_states,
    int32_t *dev_status, void *stream);

/*
 * Bytes of workspace ssd_chunk_scan_fwd needs for these arguments (0 is a
 * valid answer).  nseq is ignored unless cu_seqlens will be passed
 * (`varlen` != 0).  Returns (size_t)-1 for arguments ssd_chunk_scan_fwd
 * would reject.
 */
size_t ssd_chunk_scan_fwd_workspace_size(int batch, int seqlen, int nheads, int headdim,
                                         int dstate, int ngroups, int chunk_size,
                                         ssd_dtype_t in_dtype, int varlen, int nseq);

/*
 * ssd_state_update -- one decode step for one new token per batch row, in
 * place: the loop body of the recurrence applied to a stored state
 * ("Transformers are SSMs Review", sec. 1-1: constant-size recurrent state
 * for autoregressive inference; "20.1 상태 공간 모델 (SSM)", sec. 5 loop).
 *
 *   state [batch, nheads, headdim, dstate] float32, read and overwritten
 *   x  [batch, nheads, headdim]   dt [batch, nheads]   (in_dtype)
 *   A  [nheads] float32           D [nheads] float32 or NULL
 *   B, C [batch, ngroups, dstate] (in_dtype)
 *   y  [batch, nheads, headdim] float32 output
 * Supported: dstate in {16, 32, 64, 128, 256}, headdim >= 1.  state must be
 * 16-byte aligned.  No workspace.
 */
ssd_status_t ssd_state_update(float *state, const void *x, const void *dt, const float *A,
                              const void *B, const void *C, const float *D, int batch,
                              int nheads, int headdim, int dstate, int ngroups,
                              ssd_dtype_t in_dtype, float *y, void *stream);

/*
 * ssd_chunk_scan_bwd -- backward of ssd_chunk_scan_fwd (batch mode): the
 * gradients of a loss L given dL/dy and dL/dfinal, the reverse-mode
 * derivative of the recurrence above (the state gradient G_t = dL/dh_t runs
 * backwards: G_t = dy_t C_t^T + exp(dt_{t+1} A) G_{t+1}).
 *
 * Inputs: x, dt, A, B, C, D, init_states as for the forward (D and
 *   init_states may be NULL); dy [ntok, nheads, headdim] float32; dfinal
 *   [batch, nheads, headdim, dstate] float32 or NULL (0).
 * Outputs (float32, caller-owned, all overwritten):
 *   dx [ntok, nheads, headdim]; ddt [ntok, nheads]; dA [nheads];
 *   dB, dC [ntok, ngroups, dstate]; dD [nheads] or NULL; dinit [batch,
 *   nheads, headdim, dstate] or NULL.
 * Workspace: ssd_chunk_scan_bwd_workspace_size(...) bytes, 256-byte
 *   aligned, owned by the caller.  With headdim <= 64 and dstate <= 128
 *   (the chunked path, 64-token chunks): the state entering each chunk and
 *   the adjoint leaving it, [chunks][nheads] x headdim x dstate float32
 *   each (on the tensor-core path the same bytes hold each as a bf16
 *   hi/lo pair of [chunks][nheads][dstate][headdim] arrays), and per
 *   (chunk, head) its decay and a 144-float weight row; other
 *   shapes (the step-by-step path): one stored state every 64 steps and the
 *   64 states of one chunk, per (batch row, head).
 * Supported: headdim * dstate <= 16384, either input dtype; no cu_seqlens.
 * Arithmetic: fp32 accumulation.  On the chunked path the products run on
 *   tensor cores with each fp32 operand as a pair of bf16 values (hi =
 *   rn(v), lo = rn(v - hi)).  bf16 inputs with headdim and dstate multiples
 *   of 8: three launches (a weight table, tcgen05 state scans, the tcgen05
 *   gradient kernel); other chunked shapes: five (warp-MMA chunk states,
 *   two state passes, the CUDA-core gradient kernel); the step-by-step
 *   path: one.  dA, ddt, dB, dC and dD are zeroed first (on the tensor-core
 *   path by the weight-table launch, elsewhere by memsets).
 * dev_status: as for the forward (NULL allowed): zeroed by the call on its
 *   stream; a device wait that runs out writes SSD_ERR_TIMEOUT there and the
 *   outputs are undefined.
 */
size_t ssd_chunk_scan_bwd_workspace_size(int batch, int seqlen, int nheads, int headdim,
                                         int dstate, int ngroups, ssd_dtype_t in_dtype);
ssd_status_t ssd_chunk_scan_bwd(const void *x, const void *dt, const float *A, const void *B,
                                const void *C, const float *D, int batch, int seqlen, int nheads,
                                int headdim, int dstate, int ngroups, ssd_dtype_t in_dtype,
                                const float *init_states, const float *dy, const float *dfinal,
                                float *dx, float *ddt, float *dA, float *dB, float *dC, float *dD,
                                float *dinit, void *workspace, size_t workspace_bytes,
                                int32_t *dev_status, void *stream);

/*
 * ssd_chunk_scan_states -- the state at the end of each sequence, without
 * the outputs: the segment-state and state-passing steps of the chunked
 * forward ("Transformers are SSMs Review", dimensionstp.github.io, sec. 3-2
 * (4): chunk states, then the recurrence over chunks; sec. 3-2 (6): only the
 * boundary states cross between pieces of a sequence).
 *   Arguments, layouts and checks as for ssd_chunk_scan_fwd, less C, D and y:
 *   final_states [nseq_or_batch, nheads, headdim, dstate] float32 (required)
 *   receives the state after each sequence from init_states (NULL: zero).
 *   Scratch: workspace of at least ssd_chunk_scan_states_workspace_size(...)
 *   bytes, 256-byte aligned, owned by the caller.
 *   The tensor-core configuration (bfloat16, headdim 64, dstate 128) runs the
 *   segment-state and state-passing kernels only; other shapes run the
 *   CUDA-core forward with y kept in the workspace and dropped.
 *   Returns SSD_OK, SSD_ERR_INVALID, SSD_ERR_UNSUPPORTED or SSD_ERR_CUDA;
 *   errors only the device can see go to *dev_status as for the forward.
 */
size_t ssd_chunk_scan_states_workspace_size(int batch, int seqlen, int nheads, int headdim,
                                            int dstate, int ngroups, int chunk_size,
                                            ssd_dtype_t in_dtype, int varlen, int nseq);
ssd_status_t ssd_chunk_scan_states(
    const void *x, const void *dt, const float *A, const void *B, int batch, int seqlen,
    int nheads, int headdim, int dstate, int ngroups, int chunk_size, ssd_dtype_t in_dtype,
    const float *init_states, const int32_t *cu_seqlens, int nseq, float *final_states,
    void *workspace, size_t workspace_bytes, int32_t *dev_status, void *stream);

/*
 * Context (sequence) parallelism: one sequence cut into R consecutive slices,
 * one per device.  Each device runs ssd_chunk_scan_states on its slice from a
 * zero state and keeps the slice's end state S_r (final_states) and its
 * total log-decay a_r (ssd_segment_decay); the devices exchange these (an
 * all-gather, the caller's collective); ssd_segment_combine composes the
 * slices' affine maps h -> exp(a_r) h + S_r into the state entering each
 * slice; ssd_chunk_scan_fwd from that state gives the exact y and end state
 * of the slice.  The composition rule (a2, b2) o (a1, b1) =
 * (a2 a1, a2 b1 + b2) is that of the Mamba paper review (feghi.github.io,
 * sec. 4); passing states between blocks of the sequence is the SSD
 * review's chunked algorithm (dimensionstp.github.io, sec. 3-2 (4)) at the
 * scale of whole slices.
 *
 * ssd_segment_decay -- decay[b, h] = A[h] * sum_t dt[b, t, h] over the
 *   slice.  dt [batch, seqlen, nheads] (in_dtype), A [nheads] float32,
 *   decay [batch, nheads] float32.  One launch, no workspace.
 */
ssd_status_t ssd_segment_decay(const void *dt, const float *A, int batch, int seqlen, int nheads,
                               ssd_dtype_t in_dtype, float *decay, void *stream);

/*
 * ssd_segment_combine -- the states entering R consecutive slices:
 *   states_in[0] = init_states (NULL: zero), states_in[r + 1] =
 *   exp(decay[r]) * states_in[r] + states[r], elementwise over
 *   [batch, nheads, headdim, dstate].
 *   decay [R, batch, nheads], states [R, batch, nheads, headdim, dstate],
 *   init_states [batch, nheads, headdim, dstate] or NULL, states_in
 *   [R + 1, batch, nheads, headdim, dstate], all float32.  states_in[R] is
 *   the end state of the whole sequence.  One launch, no workspace.
 */
ssd_status_t ssd_segment_combine(const float *decay, const float *states,
                                 const float *init_states, int nsegments, int batch, int nheads,
                                 int headdim, int dstate, float *states_in, void *stream);

/*
 * ssd_selective_scan_fwd -- the Mamba-1 selective scan (S6) forward, with a
 * decay per channel and state: the sequential loop of "20.1 상태 공간 모델
 * (SSM)" (sungeuns.github.io), sec. 5 (Selective SSM forward), with an
 * optional initial state.  Per batch row, channel d and state n:
 *
 *     h_t[d,n] = exp(dt_t[d] * A[d,n]) * h_{t-1}[d,n] + dt_t[d] * B_t[n] * x_t[d]
 *     y_t[d]   = sum_n h_t[d,n] * C_t[n] + D[d] * x_t[d]
 *
 * This is the layer that SSD restricts (A the same scalar for every state
 * of a head); the library offers it so the two can be compared on the same
 * GPU.  Inputs (`in_dtype` unless stated):
 *   x, dt  [batch, seqlen, dmodel]   (dt already positive)
 *   A      [dmodel, dstate] float32
 *   B, C   [batch, seqlen, dstate]   (shared by every channel; 16-byte aligned)
 *   D      [dmodel] float32 or NULL (0)
 *   init_states float32 [batch, dmodel, dstate] or NULL (zero state)
 * Outputs (float32): y [batch, seqlen, dmodel]; final_states
 *   [batch, dmodel, dstate] or NULL.
 * Supported: dstate in {16, 32, 64, 128, 256}, batch <= 65535.  One kernel
 * launch, no workspace; the other conventions are those above.
 */
ssd_status_t ssd_selective_scan_fwd(const void *x, const void *dt, const float *A, const void *B,
                                    const void *C, const float *D, const float *init_states,
                                    int batch, int seqlen, int dmodel, int dstate,
                                    ssd_dtype_t in_dtype, float *y, float *final_states,
                                    void *stream);

/* Short English text for a status code (static storage). */
const char *ssd_status_string(ssd_status_t status);

/* Library version, major * 10000 + minor * 100 + patch. */
int ssd_version(void);

/*
 * Number of CUDA kernels this library has launched in this process so far
 * (all entry points, all devices).  A diagnostic for callers that account
 * for launches; it never resets.
 */
uint64_t ssd_kernel_launches(void);

/*
 * Test hook, not for production use.  Sets, for later calls of
 * ssd_chunk_scan_fwd on the tensor-core path (bf16, headdim 64, dstate 128,
 * no fused-epilogue options), the bound on every device-side wait in
 * nanoseconds (0 restores the default of 2 s) and a work unit that never
 * publishes its segment end state (-1: none).  With a held unit, the unit
 * that waits for it gives up after `wait_ns`, the call records
 * SSD_ERR_TIMEOUT in dev_status, and the kernel returns with its tensor
 * memory freed; the output of that call is undefined.  Work units are
 * numbered sequence by sequence, segment by segment, head by head.  The
 * setting is process-wide and not synchronised with calls in flight.
 */
void ssd_test_set_forward_wait(unsigned long long wait_ns, int hold_unit);

/*
 * Test hook, not for production use.  Sets, for later calls of
 * ssd_chunk_scan_bwd on its tensor-core path (bf16, headdim and dstate
 * multiples of 8, at most 64 and 128), the bound on every mbarrier wait of
 * the state scans and the gradient kernel in polls (0 restores the default,
 * 2^22) and one MMA completion that is never signalled: hold 1, the first
 * dS of gradient block 0; hold 2, the first chunk product of the forward
 * scan of head 0; 0, none.  The waiting threads give up after `polls`, the
 * call records SSD_ERR_TIMEOUT in dev_status, the block stops waiting and
 * frees its tensor memory once its MMAs are done; the gradients of that call
 * are undefined.  Process-wide, not synchronised with calls in flight.
 */
void ssd_test_set_backward_wait(unsigned long long polls, int hold);

#ifdef __cplusplus
}
#endif

#endif /* SSD_B300_H */
