/*
 * ssd.h -- C ABI of libssd.so, the GB300 (sm_103a) Mamba-2 SSD chunked scan.
 *
 * The operation (Mamba-2 state-space duality; the recurrence of the Mamba-3-Lite
 * "SSD Reference" page, section "Math: the recurrence both functions implement",
 * with the dt factor on the input, a D skip, an optional silu(z) gate and
 * initial/final states):
 *
 *   dt_t  = softplus(dt_raw_t + dt_bias_h)                     per token and head
 *   h_t   = exp(dt_t * A_h) * h_{t-1} + dt_t * x_t (outer) B_t    state [P][N] per head
 *   y_t   = (C_t . h_t + D_h * x_t) * silu(z_t)                 (gate only when z is given)
 *
 * Head h reads B/C group g = h / (H / G) (H must be a multiple of G).
 * h_{-1} is the initial state (zero when absent); the final state is h after the
 * last token of each sequence.
 *
 * The scan is evaluated in chunks of `chunk_size` tokens (the chunkwise
 * decomposition of that page's section "ssd_complex_chunkwise -- the production
 * scan": in-chunk cumulative log-decay, intra-chunk segment-sum matrix, per-chunk
 * states, carried chunk states).  The chunk length only changes the association of
 * the arithmetic, never the function, and the library computes with exactly the
 * chunk length the caller passes: 128 on the tensor-core path (one M = 128 tcgen05
 * tile per chunk), 64 on the SIMT path.  Any other value, or a value the chosen path
 * does not compute, returns SSD_ERR_UNSUPPORTED; nothing is re-chunked silently.
 *
 * The chunk grid runs over each batch row's token axis: chunk c holds tokens
 * [c*Q, (c+1)*Q).  With packed sequences (cu_seqlens) chunk boundaries need not meet
 * sequence starts, and a chunk may hold parts (segments) of several sequences; the
 * intra-chunk matrix then couples only tokens of one sequence, the carried state is
 * reset to a sequence's initial state where it starts, mid-chunk or not, and its
 * final state is the state after its last token.  ssd_varlen_metadata returns that
 * grid's metadata.
 *
 * ---------------------------------------------------------------------------
 * Ownership and execution contract (all entry points)
 *   - The caller owns every buffer: inputs, outputs and the workspace.  The
 *     library never allocates, frees or synchronises (except ssd_query_status),
 *     keeps no per-call state outside the workspace, and enqueues all work on
 *     the given stream (a cudaStream_t passed as void*; NULL = legacy stream).
 *   - Pointers in ssd_tensor are DEVICE pointers on the current device.
 *   - Validation runs on the host before any launch; a non-OK return means
 *     nothing was enqueued.  Errors found on the device (bad cu_seqlens
 *     contents, a bounded wait that expired) are written to a status word in the
 *     workspace and read back with ssd_query_status().
 *   - Two calls may share a workspace only if they are ordered on one stream.
 *
 * Tensor conventions (element strides, outermost first, innermost stride 1):
 *   x, z, y, dy, dx, dz : [batch, seqlen, nheads, headdim]        bf16 or f32
 *   B, C, dB, dC        : [batch, seqlen, ngroups, dstate]        same dtype as x
 *   dt, ddt             : [batch, seqlen, nheads]                 f32
 *   A, D, dt_bias, dA, dD, ddt_bias : [nheads], contiguous        f32
 *   initial_states, final_states, dfinal_states, dinitial_states :
 *                         [nstate, nheads, headdim, dstate], contiguous, f32 or
 *                         bf16, each independently (nstate = batch, or nseqs with
 *                         cu_seqlens).  bf16 is a storage dtype only (the state
 *                         cache of a serving stack, whose speed the vLLM pull request
 *                         for the fused Mamba2 SSD kernel reports "depending on state
 *                         dtype", "Purpose"): the scan widens bf16 inputs and carries
 *                         and accumulates every state in f32, then rounds a bf16
 *                         output to nearest even.  The fp32 copies live in the workspace.
 *   cu_seqlens          : int32 [nseqs + 1] device array, batch must be 1;
 *                         cu[0] = 0, non-decreasing, cu[nseqs] = seqlen.
 *                         Sequence s is tokens [cu[s], cu[s+1]) of row 0; its
 *                         scan starts from initial_states[s] and ends in
 *                         final_states[s]; sequences never interact.
 * ---------------------------------------------------------------------------
 */
#ifndef SSD_GB300_H
#define SSD_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define SSD_ABI_VERSION 5

typedef enum {
    SSD_OK = 0,
    SSD_ERR_INVALID_ARGUMENT = 1,   /* bad shape, stride, dtype mix, NULL required pointer, bad cu_seqlens */
    SSD_ERR_UNSUPPORTED = 2,        /* valid but outside the compiled set (headdim/dstate/chunk/algo) */
    SSD_ERR_MISALIGNED = 3,         /* a pointer or stride breaks the 16-byte rule of the TMA path */
    SSD_ERR_WORKSPACE_TOO_SMALL = 4,
    SSD_ERR_CUDA = 5,               /* a CUDA runtime call or a launch failed */
    SSD_ERR_DEVICE_TIMEOUT = 6      /* a bounded inter-CTA wait expired (device-side, via ssd_query_status) */
} ssd_status;

typedef enum { SSD_F32 = 0, SSD_BF16 = 1 } ssd_dtype;

/* Which forward/backward pipeline to run.  AUTO takes the tensor-core path (its single-pass
 * forward) when chunk_size == 128 and the inputs are bf16 with headdim == 64 and dstate 128,
 * 64, 32 or 16 (the compiled tile set is dstate 128; a smaller dstate runs as its
 * zero-extended part -- dstate 64 is the cuDNN frontend Mamba-2 engine's headdim = dstate =
 * 64 shape; tensors that break the
 * 16-byte rule then return SSD_ERR_MISALIGNED), and the SIMT path otherwise (f32 inputs
 * always take SIMT: fp32 inputs are computed in fp32 FMA, never in tf32).  The chunk length
 * is never replaced: the SIMT forward computes chunk_size 32, 64, 128 or 256, the SIMT
 * backward 32 or 64 (its per-chunk Q x Q tiles live in shared memory), the tensor-core path
 * 128; any other combination returns SSD_ERR_UNSUPPORTED.  STAGED forces the SIMT path. */
typedef enum {
    SSD_ALGO_AUTO = 0,
    SSD_ALGO_STAGED = 1,   /* SIMT, one kernel per step: cumsum, chunk_state, state_passing, chunk_scan */
    SSD_ALGO_FUSED = 2,    /* tcgen05/TMA single-pass forward (one persistent kernel); tcgen05 backward */
    SSD_ALGO_SPLIT = 3     /* tcgen05/TMA forward in three launches (chunk states, state passing,
                              outputs; no waits between CTAs); tcgen05 backward whose state
                              recompute (when the forward kept none) uses the first two */
} ssd_algo;

typedef struct {
    void *ptr;          /* device pointer; NULL marks an absent optional tensor */
    int32_t dtype;      /* ssd_dtype */
    int32_t reserved;
    int64_t stride[4];  /* element strides, outermost first; entries past the rank are ignored */
} ssd_tensor;

typedef struct {
    int64_t batch, seqlen, nheads, headdim, ngroups, dstate, chunk_size, nseqs;
    int32_t algo;        /* ssd_algo */
    int32_t seg_chunks;  /* fused path: chunks per work unit, 0 = library choice (for
                            fixed-length batches a number of units per sequence that fills the
                            last round of resident CTAs, units of 4-5 chunks, 3-4 for the
                            backward's recompute), else 1..5 (1..4 for the backward) */
    int32_t bwd_heads;   /* tensor-core backward: heads per work item of the gradient kernel,
                            0 = library choice (whole groups of up to 8 heads, with the pairs of
                            the last partial wave split into halves of a group), else a divisor
                            of nheads/ngroups no larger than 32 (no split) */
    int32_t reserved0;   /* must be 0 */
} ssd_problem;

typedef struct {
    ssd_tensor x, dt, A, B, C, D, z, dt_bias, initial_states;   /* inputs; D, z, dt_bias, initial_states optional */
    ssd_tensor y, final_states;                                 /* outputs; final_states optional */
    const int32_t *cu_seqlens;                                  /* optional device array (see above) */
    void *chunk_states;   /* optional device buffer of ssd_chunk_states_size bytes, 16-byte aligned
                             (tensor-core path only): ssd_fwd writes the carried state entering
                             every chunk into it; ssd_bwd, given the same pointer in its `fwd`
                             arguments, reads them instead of recomputing them */
} ssd_fwd_args;

typedef struct {
    ssd_fwd_args fwd;                 /* the forward's inputs (its y/final_states are ignored) */
    ssd_tensor dy, dfinal_states;     /* upstream gradients; dfinal_states optional (zero) */
    ssd_tensor dx, ddt, dA, dB, dC;   /* required outputs */
    ssd_tensor dD, dz, ddt_bias, dinitial_states;   /* required iff the matching input is given */
} ssd_bwd_args;

/*
 * ssd_fwd_workspace_size / ssd_fwd
 * Forward scan: y and (optionally) final_states from the inputs; with
 * args->chunk_states set, also the carried state entering every chunk (for a
 * later ssd_bwd; see ssd_chunk_states_size).
 * Defined by the recurrence above; steps: chunk cumsum of dt*A, intra-chunk
 * C.B^T under the segment-sum decay mask, chunk states, inter-chunk state
 * passing, chunk output (Mamba-3-Lite "SSD Reference", sections "Chunking and
 * the discretized log-decay", "Intra-chunk outputs and per-chunk states",
 * "Inter-chunk propagation -- the fixed contract", "Readout").
 * Workspace: at least *bytes bytes of device memory, 256-byte aligned, contents
 * need not be initialised; it is clobbered.
 * Returns SSD_OK or the first validation error; nothing is enqueued on error.
 */
ssd_status ssd_fwd_workspace_size(const ssd_problem *prob, const ssd_fwd_args *args, size_t *bytes);
ssd_status ssd_fwd(const ssd_problem *prob, const ssd_fwd_args *args, void *workspace,
                   size_t workspace_bytes, void *stream);

/*
 * ssd_chunk_states_size
 * Size of the chunk-state buffer (ssd_fwd_args.chunk_states) for a problem that
 * takes the tensor-core path: one 16 KB tile per (chunk, head) of the library's
 * 128-token chunk grid (the carried state entering the chunk, bf16 -- the value the
 * scan's readout C . h of that chunk starts from; Mamba-3-Lite "SSD Reference",
 * section "Inter-chunk propagation -- the fixed contract"), for the largest chunk
 * count the problem can have.  The tile layout is internal to the library (it is
 * the operand layout of the backward's tensor-core kernel); its only use is to be
 * handed from ssd_fwd to ssd_bwd of the same problem, inputs and cu_seqlens
 * contents, in stream order.  Returns SSD_ERR_UNSUPPORTED for a problem that takes
 * the SIMT path (which recomputes its states in the backward).
 */
ssd_status ssd_chunk_states_size(const ssd_problem *prob, const ssd_fwd_args *args, size_t *bytes);

/*
 * ssd_bwd_workspace_size / ssd_bwd
 * Gradients of L = sum(dy * y) + sum(dfinal_states * final_states) with respect
 * to x, dt (the raw input, through softplus), A, B, C, and D, z, dt_bias,
 * initial_states when given (Mamba-3-Lite "SSD Reference", section "6. The
 * autograd backward contract": the backward recomputes what the forward did not
 * keep; the stages are those the Helion pull request for the Mamba-2 SSD path times
 * in "Measurements": chunk_scan_bwd_dstates, the reverse state passing,
 * chunk_scan_chunk_state_bwd_dx, chunk_scan_bwd_dC, the dA/dt cumulative-sum
 * gradients).  dB/dC sum over the heads of each group.  All reductions run in a
 * fixed order: results are bitwise reproducible (that page's "Limitations":
 * atomics make its backward nondeterministic; this one uses none).
 * The carried chunk states are recomputed inside (no saved activations are
 * needed) unless args->fwd.chunk_states holds the ones an ssd_fwd call of the same
 * problem and inputs wrote; then the recompute is skipped.
 * Same workspace rules as ssd_fwd.
 */
ssd_status ssd_bwd_workspace_size(const ssd_problem *prob, const ssd_bwd_args *args, size_t *bytes);
ssd_status ssd_bwd(const ssd_problem *prob, const ssd_bwd_args *args, void *workspace,
                   size_t workspace_bytes, void *stream);

/*
 * ssd_query_status
 * Synchronises `stream`, then returns the device-side status word of the most
 * recent ssd_fwd/ssd_bwd call that used `workspace` (SSD_OK,
 * SSD_ERR_INVALID_ARGUMENT for bad cu_seqlens contents, SSD_ERR_DEVICE_TIMEOUT),
 * or SSD_ERR_CUDA if the synchronisation or the read fails.  The status lives in
 * the caller-owned workspace, as the cuDNN frontend's Mamba-2 SSD engine keeps all
 * scratch caller-owned and its calls allocation-free (that pull request's review
 * notes); this is the one call here that synchronises.
 */
ssd_status ssd_query_status(const void *workspace, void *stream);

/*
 * ssd_selftest_bounded_wait
 * Self-test of the device-side failure path (no counterpart on the source pages):
 * enqueues on `stream` one thread block that clears the workspace's status word and
 * then waits for a flag in the workspace header that nothing sets, polling exactly as
 * the kernels' inter-CTA waits do but giving up after `wait_ms` milliseconds (1..2000),
 * when it records SSD_ERR_DEVICE_TIMEOUT as a kernel whose peer never arrives would.
 * Read the result with ssd_query_status; the context stays usable.  The workspace must
 * be device memory of at least 256 bytes (the header); it is scratch for later calls.
 * Returns SSD_ERR_INVALID_ARGUMENT for a NULL or short workspace or a limit out of
 * range, SSD_ERR_CUDA if the launch fails.
 */
ssd_status ssd_selftest_bounded_wait(void *workspace, size_t workspace_bytes, int32_t wait_ms, void *stream);

/*
 * ssd_fwd_noalloc
 * The forward scan (same operation, arguments and results as ssd_fwd) for
 * callers that cannot allocate device memory where they run it: code running
 * while a CUDA graph is captured (allocation is not a capturable operation),
 * serving runtimes that reserve all device memory in their own pools, and
 * real-time loops that must not call the allocator.  There is no counterpart on
 * the source pages: it is a deployment variant of ssd_fwd.
 * The scratch memory is a library-owned static device array of
 * SSD_NOALLOC_SCRATCH_BYTES bytes; a problem whose ssd_fwd workspace would be
 * larger is rejected with SSD_ERR_WORKSPACE_TOO_SMALL before any launch.  The
 * array is loaded on the first call on a device, which also looks up its device
 * address (once per device and context: make that first call before any stream
 * capture); it stays allocated until the process exits.  Nothing is allocated or
 * freed per call.  Errors found on the device are read with
 * ssd_noalloc_query_status.  Device ordinals from 64 up return SSD_ERR_CUDA.
 * All calls share the one array (each call re-initialises the parts that must
 * start at zero), so calls whose work overlaps on the GPU -- on different
 * streams or host threads without ordering -- race and must not be issued.
 */
#define SSD_NOALLOC_SCRATCH_BYTES ((size_t)64 << 20)
ssd_status ssd_fwd_noalloc(const ssd_problem *prob, const ssd_fwd_args *args, void *stream);

/*
 * ssd_noalloc_query_status
 * Synchronises `stream`, then returns the device-side status word that the most
 * recent ssd_fwd_noalloc call on the current device left in the library's scratch
 * array (SSD_OK, SSD_ERR_INVALID_ARGUMENT for bad cu_seqlens contents,
 * SSD_ERR_DEVICE_TIMEOUT), or SSD_ERR_CUDA if the lookup, the synchronisation or the
 * read fails.  The noalloc caller has no workspace to hand to ssd_query_status, so
 * this reader is its only way to see errors found on the device.  No counterpart on
 * the source pages.
 */
ssd_status ssd_noalloc_query_status(void *stream);

/*
 * ssd_varlen_metadata
 * The integer metadata of packed sequences on the chunk grid: for cu_seqlens
 * (int32 [nseqs + 1], device; cu[0] = 0, non-decreasing, cu[nseqs] = seqlen) and
 * chunk length Q = chunk_size (1 .. 65536), with n_chunks = ceil(seqlen / Q):
 *   seq_idx     int32 [seqlen]            the s with cu[s] <= t < cu[s+1], per token t
 *                                         (may be NULL: not written)
 *   chunk_begin int32 [n_chunks + 1]      index of chunk c's first segment; the last
 *                                         entry is the number of segments
 *   segments    int32 [n_chunks + nseqs][3] (seq, first token, end token) of every
 *                                         maximal run of one chunk's tokens (tokens
 *                                         [c*Q, min((c+1)*Q, seqlen))) that belongs to
 *                                         one sequence, chunk by chunk, in token order
 *   status      int32 [1]                 SSD_OK, or SSD_ERR_INVALID_ARGUMENT when the
 *                                         contents of cu_seqlens break the rules above
 *                                         (then nothing else is written)
 * All pointers are device memory owned by the caller; work is enqueued on `stream`.
 * The forward and backward build the same segments internally (one chunk tile per
 * segment).  Definition: the packed (THD) path of the Helion pull request for the
 * Mamba-2 SSD path ("Testing") and the vLLM fused-SSD pull request's cont-batch
 * tests ("Test Plan"), sequences packed on one token axis with the chunk grid over
 * that axis.  Returns SSD_ERR_INVALID_ARGUMENT for NULL required pointers or sizes
 * out of range, SSD_ERR_UNSUPPORTED above 2^24 sequences or 2^30 tokens, SSD_ERR_CUDA
 * if a launch fails.
 */
ssd_status ssd_varlen_metadata(const int32_t *cu_seqlens, int64_t nseqs, int64_t seqlen, int64_t chunk_size,
                               int32_t *seq_idx, int32_t *chunk_begin, int32_t *segments, int32_t *status,
                               void *stream);

/*
 * Gated normalisation over feature groups -- the normalisation that follows the scan in a
 * Mamba-2 block (the gated LayerNorm / RMSNorm whose backward the Helion pull request for the
 * Mamba-2 SSD path times as layer_norm_bwd, "Summary" and "Measurements").  Per row t and
 * group g = features [g * group_size, (g+1) * group_size), with s = silu(z) (s = 1 when z is
 * NULL):
 *
 *   u[t,i]    = y[t,i] * s[t,i]       (default: the gate first)
 *             = y[t,i]                (flags & SSD_NORM_GATE_AFTER)
 *   mu[t,g]   = 0                     (default: RMS normalisation)
 *             = mean_{i in g} u[t,i]  (flags & SSD_NORM_LAYER: LayerNorm, no bias)
 *   rstd[t,g] = 1 / sqrt(mean_{i in g} (u[t,i] - mu[t,g])^2 + eps)
 *   out[t,i]  = (u[t,i] - mu[t,g]) * rstd[t,g] * weight[i]    (times s[t,i] when the gate comes after)
 *
 * Feed it the scan's ungated output (ssd_fwd with z absent) and z; a Mamba-2 block uses
 * group_size = nheads * headdim / ngroups, so a group is the heads of one B/C group.
 * Tensors y, z, out, dout, dy, dz: `rows` rows of `width` contiguous features at an element
 * row stride, all of `dtype` (bf16 or f32), 16-byte aligned with strides a multiple of 8
 * (else SSD_ERR_MISALIGNED).  weight, dweight: f32 [width]; rstd: f32 [rows][width /
 * group_size], written by the forward and read by the backward (which recomputes mu).
 * group_size must divide width (else SSD_ERR_INVALID_ARGUMENT) and be a multiple of 8 no
 * larger than 6144 (else SSD_ERR_UNSUPPORTED); flags other than the two below are
 * SSD_ERR_INVALID_ARGUMENT.  Buffers are the caller's, device memory; work is enqueued on
 * `stream`; the weight gradient is summed in a fixed order (bitwise reproducible).
 */
enum { SSD_NORM_LAYER = 1, SSD_NORM_GATE_AFTER = 2 };
typedef struct {
    int64_t rows, width, group_size;
    float eps;
    int32_t dtype;      /* ssd_dtype of y, z, out, dout, dy, dz */
    int32_t flags;      /* SSD_NORM_LAYER | SSD_NORM_GATE_AFTER, or 0 (gated RMS normalisation) */
} ssd_norm_problem;

ssd_status ssd_gated_norm_fwd(const ssd_norm_problem *prob, const void *y, int64_t y_stride, const void *z,
                              int64_t z_stride, const float *weight, void *out, int64_t out_stride, float *rstd,
                              void *stream);
/* Gradients of sum(dout * out): dy, dz (when z is given) and dweight; `workspace` (at least
 * ssd_gated_norm_bwd_workspace_size bytes, 16-byte aligned) holds the weight gradient's
 * per-row-chunk shares. */
ssd_status ssd_gated_norm_bwd_workspace_size(const ssd_norm_problem *prob, size_t *bytes);
ssd_status ssd_gated_norm_bwd(const ssd_norm_problem *prob, const void *y, int64_t y_stride, const void *z,
                              int64_t z_stride, const float *weight, const float *rstd, const void *dout,
                              int64_t dout_stride, void *dy, int64_t dy_stride, void *dz, int64_t dz_stride,
                              float *dweight, void *workspace, size_t workspace_bytes, void *stream);

/*
 * Causal depthwise convolution over the sequence axis with an optional SiLU -- the step
 * before the scan in a Mamba-2 block, run on the packed xBC = [x | B | C] channels (the
 * Helion pull request for the Mamba-2 SSD path, "Summary": mamba_split_conv1d_scan_combined;
 * "Testing": x, B and C are views of one packed buffer):
 *
 *   pre[t,c] = bias[c] + sum_{k<width} weight[c][k] * u[t - (width-1) + k][c]
 *   out[t,c] = silu(pre[t,c])   (activation 1)   or   pre[t,c]   (activation 0)
 *
 * with u := 0 before the start of t's sequence (a batch row, or with cu_seqlens -- int32
 * [nseqs + 1], device, batch 1 -- a packed sequence): a window never reaches into another
 * sequence.  The scan then reads x, B and C as strided views of out (ssd_tensor strides), so
 * the split costs no copy.  Token tensors u, out, dout, du: [batch][seqlen][channels], channels
 * contiguous, at element strides (per batch row, per token), of `dtype` (bf16 or f32),
 * 16-byte aligned with strides a multiple of 8 (else SSD_ERR_MISALIGNED); weight, dweight: f32
 * [channels][width]; bias, dbias: f32 [channels] (optional).  width 1..8 and channels a
 * multiple of 8 (else SSD_ERR_UNSUPPORTED).  cu_seqlens contents are not validated here
 * (ssd_varlen_metadata reports bad ones); bad ones give unspecified values, yet every access
 * stays inside the tensors described above.  The backward gives du, dweight and dbias (sums over
 * tokens in a fixed order: bitwise reproducible) and needs `workspace` of
 * ssd_conv1d_bwd_workspace_size bytes, 16-byte aligned.
 */
typedef struct {
    int64_t batch, seqlen, channels, width, nseqs;   /* nseqs: packed sequences (cu_seqlens), else 0 */
    int32_t dtype, activation;                       /* ssd_dtype; 0 none, 1 silu */
    int32_t reserved, pad;                           /* reserved must be 0 */
} ssd_conv_problem;

ssd_status ssd_conv1d_fwd(const ssd_conv_problem *prob, const void *u, int64_t u_batch_stride,
                          int64_t u_token_stride, const float *weight, const float *bias,
                          const int32_t *cu_seqlens, void *out, int64_t out_batch_stride,
                          int64_t out_token_stride, void *stream);
ssd_status ssd_conv1d_bwd_workspace_size(const ssd_conv_problem *prob, size_t *bytes);
ssd_status ssd_conv1d_bwd(const ssd_conv_problem *prob, const void *u, int64_t u_batch_stride,
                          int64_t u_token_stride, const float *weight, const float *bias,
                          const int32_t *cu_seqlens, const void *dout, int64_t dout_batch_stride,
                          int64_t dout_token_stride, void *du, int64_t du_batch_stride, int64_t du_token_stride,
                          float *dweight, float *dbias, void *workspace, size_t workspace_bytes, void *stream);

/* Human-readable name of a status code (static string, never NULL). */
const char *ssd_status_string(ssd_status status);

/* SSD_ABI_VERSION of the built library. */
int32_t ssd_abi_version(void);

/* ------------------------------------------------------------------------------------------
 * Complex-A SSD scan, forward (the Mamba-3-Lite variant: Mamba-3-Lite "SSD Reference --
 * complex scan API & kernel contract", sections "Math: the recurrence both functions
 * implement", "ssd_naive_complex", "ssd_complex_chunkwise" and its shape table).
 *
 * Per batch row b and head h, with abar_t = exp(softplus(dt[b,t,h]) * A[h]) (A complex, dt
 * real, no bias) and a complex state h_t [headdim][dstate]:
 *
 *   h_t = abar_t h_{t-1} + x_t (outer) B_t,   y_t[d] = sum_n C_t[n] h_t[d][n]
 *
 * from h_{-1} = initial_states[b,h] (zero when NULL).  No dt factor on the input and no
 * conjugation (C and B enter bilinearly).  y_real = Re y, y_imag = Im y (optional: NULL skips
 * it), final_states = h_{T-1} (optional).  One exact function: the chunking (chunk_size
 * positions per tile) changes only rounding order.
 *
 * Layouts (all contiguous, element offsets; complex = interleaved (re, im) fp32 pairs, the
 * layout of a complex64 tensor): x [batch][seqlen][nheads][headdim] complex; B, C
 * [batch][seqlen][nheads][dstate] complex (one projection per head); dt [batch][seqlen]
 * [nheads] f32; A [nheads] complex; initial/final_states [batch][nheads][headdim][dstate]
 * complex; y_real, y_imag [batch][seqlen][nheads][headdim] f32.  x, B, C, y_*, the states
 * and the workspace 16-byte aligned (else SSD_ERR_MISALIGNED).
 *
 * Compiled set: headdim = dstate = chunk_size = 64 (the 434M Mamba-3-Lite configuration of
 * the page), else SSD_ERR_UNSUPPORTED.  The contractions run on the tensor cores in tf32
 * (10-bit mantissa operands, fp32 accumulation), the decays, the carried state and the
 * outputs in fp32.  `workspace` (>= ssd_complex_fwd_workspace_size bytes, caller-owned)
 * holds the status header that ssd_query_status reads; stream-ordered, no allocation.
 */
typedef struct {
    int64_t batch, seqlen, nheads, headdim, dstate, chunk_size;
} ssd_complex_problem;

ssd_status ssd_complex_fwd_workspace_size(const ssd_complex_problem *prob, size_t *bytes);
ssd_status ssd_complex_fwd(const ssd_complex_problem *prob, const void *x, const float *dt, const void *A,
                           const void *B, const void *C, const void *initial_states, float *y_real,
                           float *y_imag, void *final_states, void *workspace, size_t workspace_bytes,
                           void *stream);

/*
 * ssd_fwd_debug_layout
 * Byte offsets, inside an ssd_fwd workspace, of the intermediates the STAGED
 * forward leaves behind after it completes (for stage-by-stage checks):
 *   meta_counts : int32[4]  {n_chunks, n_units, n_seqs, status}
 *   chunk_info  : 16-byte records {int32 seq, int32 batch row, int32 first token t0 of
 *                 the physical chunk in the row, int16 end - t0, int16 first - t0}: one
 *                 chunk tile per segment of a physical chunk; tile rows [first - t0,
 *                 end - t0) are the sequence's
 *   dt          : f32[n_chunks][nheads][qi]   softplus(dt_raw + dt_bias), 0 past the chunk's length
 *   cs          : f32[n_chunks][nheads][qi]   inclusive in-chunk cumulative sum of dt*A
 *   states      : f32[n_chunks][nheads][headdim][dstate]  carry-in state of each chunk
 *   units       : 32-byte records (fused path) {int32 seq, batch row, t0 of its first
 *                 tile, end of the sequence's rows from t0 (capped at its tiles), tile
 *                 count, index of the sequence's previous unit or -1, unit index j within
 *                 the sequence; int16 1 if last unit of its sequence, int16 first row of
 *                 its first tile}; units are grouped in blocks of 4 and listed by (block,
 *                 sequence, j)
 * where qi is the chunk length (chunk_size) written to *qi.  Tiles are listed sequence
 * by sequence, in order (the same order as chunk by chunk).  Offsets of -1 mean "not
 * produced by algo".
 */
typedef struct {
    int64_t meta_counts, chunk_info, dt, cs, states, units;
    int64_t qi;
} ssd_debug_layout;
ssd_status ssd_fwd_debug_layout(const ssd_problem *prob, const ssd_fwd_args *args, ssd_debug_layout *out);

#ifdef __cplusplus
}
#endif
#endif /* SSD_GB300_H */
