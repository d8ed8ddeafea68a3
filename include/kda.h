/*
 * kda.h — C ABI of the Kimi Delta Attention (KDA) gated delta-rule scan for
 * NVIDIA GB300 (sm_103a). Library: libkda.so.
 *
 * The operation, per sequence and head, with state S in R^{d_k x d_v}
 * (row c = key channel c), per-token log-decay g_t (a_t = exp(g_t) in (0,1]^{d_k}),
 * write strength beta_t and query scale s:
 *
 *     S~_t = Diag(a_t) S_{t-1}
 *     S_t  = S~_t + beta_t k_t (v_t - S~_t^T k_t)^T
 *     o_t  = S_t^T (s q_t)
 *
 * ("Understanding Kimi Delta Attention", box "KDA: Retain, predict, correct";
 *  the query scale as in "Demystifying Kimi Delta Attention", opening KDA
 *  equations.)
 *
 * Conventions shared by every entry point:
 *  - All tensor pointers are DEVICE pointers owned by the caller; the library
 *    keeps no reference after the call returns. Scratch memory is passed in
 *    explicitly (kda_chunk_fwd's workspace); the library itself allocates no
 *    device memory.
 *  - Every call is asynchronous on `stream` (0 = legacy default stream); there
 *    is no implicit synchronisation. Results are valid once the stream
 *    reaches the call.
 *  - Layouts are dense row-major with the last dimension contiguous:
 *      q, k, g    [tokens][H][d_k]     v, out [tokens][H][d_v]
 *      beta       [tokens][H]
 *      states     [num_seqs][H][d_k][d_v]  (fp32; row c = key channel c)
 *    where `tokens` is B*T for fixed-length batches (sequence b occupies
 *    tokens [b*T, (b+1)*T)) and cu_seqlens[num_seqs] for packed sequences.
 *  - q, k, v and out share one storage dtype (kda_dtype); g, beta and the
 *    states are always fp32. Arithmetic is fp32 (bf16 tensor-core operands
 *    with fp32 accumulation on the bf16 prefill path).
 *  - Supported sizes: d_k == d_v, and d_k in {64, 128}. Other sizes return
 *    KDA_ERR_UNSUPPORTED.
 *  - Tensor pointers must be 16-byte aligned, except beta and cu_seqlens
 *    (4-byte aligned).
 *  - Errors are returned as kda_status; nothing is thrown and nothing is
 *    printed. Argument checks happen on the host before any CUDA call; a
 *    launch failure returns KDA_ERR_CUDA (the CUDA error is left for the
 *    caller's cudaGetLastError()/cudaPeekAtLastError() to inspect).
 *  - Inputs are expected to satisfy g <= 0 (finite), beta in [0, 1]. Every
 *    decay a = exp(g) in (0, 1] is handled exactly, however steep (the bf16
 *    prefill takes a slower exact form for any 64-token chunk in which some
 *    key channel decays by more than 64 nats within 16 tokens). Values
 *    outside these ranges are not checked on the device.
 */
#ifndef KDA_H_
#define KDA_H_

#include <stddef.h>
#include <stdint.h>

#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    KDA_OK = 0,
    KDA_ERR_INVALID_ARGUMENT = 1, /* NULL required pointer, bad size or alignment */
    KDA_ERR_UNSUPPORTED = 2,      /* valid request this build does not implement */
    KDA_ERR_WORKSPACE = 3,        /* workspace NULL or smaller than required */
    KDA_ERR_CUDA = 4,             /* a CUDA runtime call or kernel launch failed */
    KDA_ERR_TIMEOUT = 5           /* a bounded device-side wait gave up */
} kda_status;

typedef enum {
    KDA_DTYPE_F32 = 0, /* q, k, v, out are fp32 */
    KDA_DTYPE_BF16 = 1 /* q, k, v, out are bf16 */
} kda_dtype;

/*
 * The decay family, i.e. the layout of g (the pages trace it as DeltaNet ->
 * Gated DeltaNet -> KDA: "Kimi Delta Attention: How It Works, Step by Step",
 * section 6; "Kimi Delta Attention: a half-life per channel", "Promote the
 * scalar to a diagonal"). A scalar decay is the per-channel one with every
 * channel equal; no decay is a = 1.
 */
typedef enum {
    KDA_DECAY_CHANNEL = 0, /* g [tokens][H][dk]: one decay per key channel (KDA) */
    KDA_DECAY_SCALAR = 1,  /* g [tokens][H]: one decay per token and head (Gated DeltaNet) */
    KDA_DECAY_NONE = 2     /* a_t = 1; g is not read and may be NULL (DeltaNet) */
} kda_decay;

/*
 * How the values in g become the log-decay log a_t ("Kimi Delta Attention: a
 * half-life per channel": a_t = sigmoid(x_t W_a); "Understanding Kimi Delta
 * Attention", closing remarks: a negative log-decay bounded below through a
 * sigmoid).
 */
typedef enum {
    KDA_GATE_LOG = 0,        /* g holds log a_t itself (<= 0) */
    KDA_GATE_LOGSIGMOID = 1, /* g holds logits z: a_t = sigmoid(z), log a_t = -log(1 + e^-z) */
    KDA_GATE_BOUNDED = 2     /* g holds logits z: log a_t = gate_lower * sigmoid(z) */
} kda_gate;

/*
 * Options of kda_chunk_fwd_opt and kda_decode_step_opt. A NULL pointer means
 * {KDA_DECAY_CHANNEL, KDA_GATE_LOG, 0, 0, 0, 0}, the behaviour of kda_chunk_fwd
 * and kda_decode_step.
 *  decay       layout of g (above)
 *  gate        meaning of g's values (above); ignored with KDA_DECAY_NONE
 *  gate_lower  KDA_GATE_BOUNDED only: the lower bound of log a_t, finite and
 *              in [-10, 0) (log a_t then lies in (gate_lower, 0))
 *  l2norm_qk   nonzero: q and k are L2-normalised per token and head inside
 *              the kernel, x / sqrt(sum_c x_c^2 + 1e-6), before anything else
 *              uses them ("Kimi Delta Attention: How It Works, Step by Step",
 *              section 16: the key and query are normalised); the query
 *              scale still applies after it
 *  segments    prefill only, tensor-core path (bf16, d = 128) with fixed-length
 *              batches (no cu_seqlens): how the state crosses the chunks.
 *              1: one serial chain per (sequence, head). k >= 2: each sequence
 *              is cut into up to k segments of whole chunks; every segment
 *              but the last first computes its affine map S_out = M S_in + E
 *              from the same recurrence (M from identity columns with v = 0,
 *              E from a zero state), the maps are composed in order, and the
 *              segments then rerun from their true entering states, all in
 *              parallel ("Understanding Kimi Delta Attention": composing the
 *              affine transitions; a chunk-level parallel prefix). k is
 *              clamped so that (sequences x H x k) <= 32 and k <= chunks.
 *              0 (the default): segments only when few (sequence, head)
 *              chains leave most of the GPU idle and T >= 2048, else 1.
 *              Results equal the serial chain's up to fp32 rounding. Must be
 *              >= 0; ignored by the decode step and the fp32 SIMT path.
 *  fused       prefill only, tensor-core path: 0 (the default) lets the call
 *              run phase 1 and the state pass as ONE cooperative launch when
 *              that is expected to be faster: a serial chain (segments
 *              resolves to 1), fixed-length batches or a single packed
 *              sequence, and few enough (sequence, head) chains that the
 *              state pass (two CTAs per chain) leaves SMs to phase 1, which
 *              hands each chunk over through a ready flag in the workspace.
 *              1: the fused launch whenever those conditions (all but the
 *              expected speed) hold. -1: always the two launches. Results
 *              equal the two launches' up to fp32 rounding. Other values are
 *              rejected.
 */
typedef struct {
    kda_decay decay;
    kda_gate gate;
    float gate_lower;
    int l2norm_qk;
    int segments;
    int fused;
} kda_options;

/* Human-readable name of a status code (static storage; never NULL). */
const char *kda_status_string(kda_status status);

/*
 * Bytes of device workspace kda_chunk_fwd needs for these sizes.
 * B, T: batch and per-sequence length when cu_seqlens is NULL; with packed
 * sequences pass B = 1, T = total tokens (= cu_seqlens[num_seqs]) and
 * num_seqs = number of sequences. The bound holds for every split of T into
 * num_seqs sequences. Returns 0 for invalid or unsupported sizes (and for
 * T == 0 with no sequence to carry).
 */
size_t kda_chunk_fwd_workspace_size(int B, int T, int H, int dk, int dv, int num_seqs,
                                    kda_dtype dtype);

/*
 * Chunkwise-parallel prefill ("Understanding Kimi Delta Attention", sections
 * "The triangular system", "Putting the chunks together" and Figure 04):
 * each chunk of up to 64 tokens forms its cumulative log-decay, the
 * correction matrix A, T = (I - A)^{-1} by a triangular solve, and the WY/UT
 * factors; the state then crosses chunk boundaries one chunk at a time, and
 * every token's output is read from the state entering its chunk plus the
 * chunk's own corrections.
 *
 *  q, k       [tokens][H][dk], dtype      query (unscaled) and key
 *  v          [tokens][H][dv], dtype      value
 *  g          [tokens][H][dk], fp32       per-token log-decay log a_t (<= 0)
 *  beta       [tokens][H], fp32           write strength
 *  scale      query scale (normally dk^-1/2), applied to q only
 *  init_state [num_seqs][H][dk][dv] fp32, or NULL for zero initial states
 *  cu_seqlens int32 [num_seqs + 1] device array, or NULL. When given: B must
 *             be 1, T = cu_seqlens[num_seqs], values non-decreasing from 0.
 *             The contents are not read on the host; the first kernel checks
 *             them (see the status word below).
 *  out        [tokens][H][dv], dtype      token outputs o_t (written)
 *  final_state[num_seqs][H][dk][dv] fp32 (written), or NULL. May alias
 *             init_state exactly (in-place state carry).
 *  B, T, H, dk, dv, num_seqs: sizes; without cu_seqlens num_seqs must be B.
 *  workspace  device scratch of at least kda_chunk_fwd_workspace_size(...)
 *             bytes, 256-byte aligned; contents on entry are ignored and on
 *             return are unspecified. Must not alias any other argument.
 *  stream     CUDA stream for all work.
 *
 * A zero-length sequence writes its initial state (or zeros) to final_state.
 *
 * Device-side status: the call's kernels write an int status word at the
 * start of the workspace, to be read once the stream has completed the call.
 * KDA_OK: the call completed. KDA_ERR_INVALID_ARGUMENT: cu_seqlens failed its
 * check (cu_seqlens[0] != 0, a decrease, or cu_seqlens[num_seqs] != T); the
 * call then computed nothing and left out and final_state unwritten.
 * KDA_ERR_TIMEOUT: a bounded wait inside a kernel gave up (the results are
 * not valid; the context stays usable).
 */
kda_status kda_chunk_fwd(const void *q, const void *k, const void *v, const float *g,
                         const float *beta, float scale, const float *init_state,
                         const int32_t *cu_seqlens, void *out, float *final_state, int B, int T,
                         int H, int dk, int dv, int num_seqs, kda_dtype dtype, void *workspace,
                         size_t workspace_bytes, cudaStream_t stream);

/*
 * kda_chunk_fwd with phase markers for timing: identical arguments, results
 * and errors, plus `events`, an array of 4 caller-created CUDA events (any
 * entry may be NULL) recorded on `stream` at the start of the call (0), after
 * the chunk table is built (1), after the intra-chunk phase (2) and after the
 * inter-chunk state pass (3). Pass events created without
 * cudaEventDisableTiming to read phase durations with cudaEventElapsedTime.
 */
kda_status kda_chunk_fwd_timed(const void *q, const void *k, const void *v, const float *g,
                               const float *beta, float scale, const float *init_state,
                               const int32_t *cu_seqlens, void *out, float *final_state, int B,
                               int T, int H, int dk, int dv, int num_seqs, kda_dtype dtype,
                               void *workspace, size_t workspace_bytes, cudaStream_t stream,
                               cudaEvent_t *events);

/*
 * kda_chunk_fwd with options (decay family, gate transform, in-kernel q/k
 * normalisation; see kda_options) and optional phase events (as in
 * kda_chunk_fwd_timed; `events` may be NULL). With KDA_DECAY_SCALAR, g is
 * [tokens][H] fp32 and 4-byte aligned; with KDA_DECAY_NONE it is not read.
 * The workspace is the same as kda_chunk_fwd's. Invalid option values return
 * KDA_ERR_INVALID_ARGUMENT before any CUDA call.
 */
kda_status kda_chunk_fwd_opt(const void *q, const void *k, const void *v, const float *g,
                             const float *beta, float scale, const float *init_state,
                             const int32_t *cu_seqlens, void *out, float *final_state, int B,
                             int T, int H, int dk, int dv, int num_seqs, kda_dtype dtype,
                             const kda_options *options, void *workspace, size_t workspace_bytes,
                             cudaStream_t stream, cudaEvent_t *events);

/*
 * Bytes of device workspace kda_chunk_fwd_host needs: two windows of
 * `window_tokens` tokens (inputs, outputs and up to 16 sequence states in and
 * out each) and the prefill's own workspace for one window. window_tokens must
 * be a positive multiple of 64; options as in kda_chunk_fwd_opt (NULL: the
 * defaults; only the decay family changes the size). Returns 0 for invalid or
 * unsupported sizes.
 */
size_t kda_chunk_fwd_host_workspace_size(int H, int dk, int dv, kda_dtype dtype,
                                         const kda_options *options, int window_tokens);

/*
 * The chunkwise prefill with every tensor in HOST memory (the end-to-end form
 * of kda_chunk_fwd_opt): q, k, v, g, beta, init_state (nullable), out and
 * final_state (nullable) have kda_chunk_fwd's layouts but are host pointers,
 * pinned for the copies to overlap (pageable memory works, serialised).
 * cu_seqlens, when given, is a HOST int32 array of num_seqs + 1 offsets (B must
 * be 1), checked here: rising from 0 to T, else KDA_ERR_INVALID_ARGUMENT.
 *
 * The sequences are cut into windows of at most `window_tokens` tokens and 16
 * sequence pieces, each cut falling on a multiple of 64 tokens from its
 * sequence's start, so that every chunk is the one the single device call
 * forms; the fp32 state of a cut sequence crosses windows on the device. Each
 * window is one kda_chunk_fwd_opt call (serial state pass) on `stream`, while
 * two copy streams created for the call move the next window's inputs in and
 * the previous window's outputs and finished sequences' final states out. The
 * results are bit-identical to kda_chunk_fwd_opt with options->segments = 1 on
 * the same data, and valid once `stream` reaches the end of the call; the host
 * inputs must stay unchanged until then.
 *
 * workspace: device memory of kda_chunk_fwd_host_workspace_size(...) bytes,
 * 256-byte aligned. The call allocates no device memory; it creates two streams
 * and a few events and releases them before returning (their work completes
 * asynchronously). Errors as kda_chunk_fwd; a zero-length sequence's final
 * state (its initial state, or zeros) is written on the host during the call.
 */
kda_status kda_chunk_fwd_host(const void *q, const void *k, const void *v, const float *g,
                              const float *beta, float scale, const float *init_state,
                              const int32_t *cu_seqlens, void *out, float *final_state, int B,
                              int T, int H, int dk, int dv, int num_seqs, kda_dtype dtype,
                              const kda_options *options, int window_tokens, void *workspace,
                              size_t workspace_bytes, cudaStream_t stream);

/*
 * kda_chunk_fwd_opt whose outputs leave through the output gate and RMS
 * normalisation of the module around the scan ("Understanding Kimi Delta
 * Attention", closing remarks: output gating and RMS normalisation):
 *
 *     out_t = w o (o_t / sqrt(mean_c o_t,c^2 + eps)) o sigmoid(z_t)
 *
 * per token and head over the dv channels, o_t the scan's output. Same
 * arguments as kda_chunk_fwd_opt plus
 *  z       [tokens][H][dv], dtype: gate logits (16-byte aligned; not read when
 *          there are no tokens)
 *  weight  [dv] fp32 per-channel scale shared by the heads, or NULL (ones)
 *  eps     finite, > 0 (1e-6 is customary)
 * On the tensor-core path (bf16, d = 128) the state crosses chunks in one
 * serial chain (options->segments is ignored). Where the fused single launch
 * applies (see kda_options.fused) the call runs it with plain outputs and
 * then the gate as a pass over them (kda_output_gate_rmsnorm in place);
 * otherwise the gate is applied inside the state pass, from the fp32 outputs,
 * before the single write of `out`: the four CTAs that hold a head's 128
 * output columns form a thread-block cluster and exchange per-row sums of
 * squares through distributed shared memory. On the fp32 path the gate is a
 * pass over the written outputs. The ungated outputs are not kept.
 * Workspace and errors as kda_chunk_fwd; eps, z and weight are checked first.
 */
kda_status kda_chunk_fwd_gated(const void *q, const void *k, const void *v, const float *g,
                               const float *beta, float scale, const float *init_state,
                               const int32_t *cu_seqlens, const void *z, const float *weight,
                               float eps, void *out, float *final_state, int B, int T, int H,
                               int dk, int dv, int num_seqs, kda_dtype dtype,
                               const kda_options *options, void *workspace, size_t workspace_bytes,
                               cudaStream_t stream, cudaEvent_t *events);

/*
 * Capacity, in bytes, of the scratch array kda_chunk_fwd_noalloc uses: 64 MiB.
 * A problem fits when kda_chunk_fwd_workspace_size(...) for its sizes is at
 * most this value.
 */
#define KDA_NOALLOC_SCRATCH_BYTES (64u << 20)

/*
 * The chunkwise prefill for callers that cannot allocate device memory: code
 * that may not call cudaMalloc (for instance a host callback or stream-ordered
 * work where allocation is forbidden, a process whose allocator must not be
 * re-entered, or an embedding that owns all memory statically). The paper has
 * no counterpart; it is a deployment convenience.
 *
 * Same arguments, results and errors as kda_chunk_fwd, without `workspace`:
 * the scratch is a 256-byte aligned file-scope device array of
 * KDA_NOALLOC_SCRATCH_BYTES inside libkda.so, which every GPU that loads the
 * library holds until the process exits. This call allocates nothing (no
 * cudaMalloc, cudaFree or allocating library routine).
 *  - The arguments are checked first, exactly as kda_chunk_fwd checks them
 *    (same codes, same order); then sizes whose kda_chunk_fwd_workspace_size
 *    exceeds KDA_NOALLOC_SCRATCH_BYTES are rejected with KDA_ERR_WORKSPACE.
 *    Both happen before any CUDA call.
 *  - Every call looks up the array's device address in the current context
 *    with cudaGetSymbolAddress (with the target device current), so a context
 *    created later on the same device, for instance after cudaDeviceReset,
 *    gets its own array. The first call in a context also loads the
 *    library's device code there: make it before any stream capture begins.
 *  - Every call, on every stream, shares the one array and it keeps the last
 *    call's contents. Nothing in it needs to start at zero (each call rebuilds
 *    everything it reads), but calls whose work overlaps on the GPU race on it:
 *    order them on one stream or synchronise between them.
 *  - The device-side status word of kda_chunk_fwd (bad cu_seqlens, a bounded
 *    wait that gave up) lives at the start of the array; read it with
 *    kda_chunk_fwd_noalloc_status.
 */
kda_status kda_chunk_fwd_noalloc(const void *q, const void *k, const void *v, const float *g,
                                 const float *beta, float scale, const float *init_state,
                                 const int32_t *cu_seqlens, void *out, float *final_state, int B,
                                 int T, int H, int dk, int dv, int num_seqs, kda_dtype dtype,
                                 cudaStream_t stream);

/*
 * The device-side status word of the last kda_chunk_fwd_noalloc call on this
 * device (see kda_chunk_fwd's "Device-side status"): KDA_OK, or
 * KDA_ERR_INVALID_ARGUMENT when cu_seqlens failed its check (nothing was
 * computed or written), or KDA_ERR_TIMEOUT. The paper has no counterpart.
 *  status  host int (pageable or pinned) that receives the word.
 *  stream  the stream of that call: one 4-byte device-to-host copy is queued
 *          on it, so the word is that call's once the stream has reached the
 *          copy (after cudaStreamSynchronize(stream), or at return when
 *          `status` is pageable memory).
 * Allocates nothing. Returns KDA_ERR_INVALID_ARGUMENT for a NULL status and
 * KDA_ERR_CUDA if the copy cannot be queued.
 */
kda_status kda_chunk_fwd_noalloc_status(int *status, cudaStream_t stream);

/*
 * One recurrent decode step for N independent sequences ("Kimi Delta
 * Attention: How It Works, Step by Step", section 11; the update of
 * "Understanding Kimi Delta Attention", box "KDA: Retain, predict, correct"),
 * fused into one pass over the state: with a = exp(g),
 *     vhat = (a o k)^T S,  e = beta (v - vhat),
 *     o    = (a o (s q))^T S + (s q^T k) e,   S <- Diag(a) S + k e^T.
 *
 *  q, k   [N][H][dk], dtype;  v, out [N][H][dv], dtype
 *  g      [N][H][dk] fp32;    beta [N][H] fp32
 *  state  [N][H][dk][dv] fp32, read and updated in place
 *  No workspace is needed.
 */
kda_status kda_decode_step(const void *q, const void *k, const void *v, const float *g,
                           const float *beta, float scale, float *state, void *out, int N, int H,
                           int dk, int dv, kda_dtype dtype, cudaStream_t stream);

/*
 * kda_decode_step with options (see kda_options). With KDA_DECAY_SCALAR, g is
 * [N][H] fp32 and 4-byte aligned; with KDA_DECAY_NONE it is not read.
 */
kda_status kda_decode_step_opt(const void *q, const void *k, const void *v, const float *g,
                               const float *beta, float scale, float *state, void *out, int N,
                               int H, int dk, int dv, kda_dtype dtype, const kda_options *options,
                               cudaStream_t stream);

/*
 * Bytes of device workspace kda_decode_host needs for N sequences (two steps'
 * inputs and outputs). Returns 0 for invalid or unsupported sizes.
 */
size_t kda_decode_host_workspace_size(int N, int H, int dk, int dv, kda_dtype dtype,
                                      const kda_options *options);

/*
 * `steps` successive decode steps (kda_decode_step_opt) with the per-step
 * tensors in HOST memory: q, k [steps][N][H][dk], v [steps][N][H][dv], g
 * [steps][N][H][dk] (or [steps][N][H] with KDA_DECAY_SCALAR; unused with
 * KDA_DECAY_NONE), beta [steps][N][H], out [steps][N][H][dv] (written), all
 * host pointers (pinned for overlap). `state` [N][H][dk][dv] fp32 is DEVICE
 * memory, updated in place by every step. Step t + 1's inputs are copied in
 * and step t - 1's outputs copied out on two copy streams created for the call
 * while step t runs on `stream`; results are bit-identical to the device
 * steps and valid once `stream` reaches the end of the call.
 * workspace: device memory of kda_decode_host_workspace_size(...) bytes,
 * 256-byte aligned; nothing is allocated on the device.
 */
kda_status kda_decode_host(const void *q, const void *k, const void *v, const float *g,
                           const float *beta, float scale, float *state, void *out, int steps,
                           int N, int H, int dk, int dv, kda_dtype dtype,
                           const kda_options *options, void *workspace, size_t workspace_bytes,
                           cudaStream_t stream);

/*
 * Output gate and RMS normalisation of the attention outputs, per token and
 * head ("Understanding Kimi Delta Attention", closing remarks: the module
 * applies output gating and RMS normalisation to the heads' outputs):
 *
 *     out_t = w o (o_t / sqrt(mean_c o_t,c^2 + eps)) o sigmoid(z_t)
 *
 * (o = elementwise product; the normalisation runs over the d_v channels of
 * one head).
 *  o, z, out  [tokens][H][dv], dtype (z: gate logits); out may alias o
 *  weight     [dv] fp32 per-channel scale shared by the heads, or NULL (ones)
 *  eps        finite, > 0 (1e-6 is customary)
 *  tokens >= 0, H > 0, dv in {64, 128}. o, z, out 16-byte aligned; weight
 *  4-byte aligned. Asynchronous on `stream`; no workspace.
 */
kda_status kda_output_gate_rmsnorm(const void *o, const void *z, const float *weight, float eps,
                                   void *out, long long tokens, int H, int dv, kda_dtype dtype,
                                   cudaStream_t stream);

/*
 * Diagnostic of the failure detection (no counterpart on the pages): launches
 * one CTA that waits, with the kernels' bounded mbarrier wait limited to
 * `limit` polls (1 .. 4194304), on a barrier nothing ever completes; when the
 * wait gives up it writes KDA_ERR_TIMEOUT into *status (a device int), as the
 * prefill kernels write their workspace status word, and returns. Nothing
 * faults or hangs, and the context stays usable. status must be 4-byte
 * aligned device memory.
 */
kda_status kda_selftest_wait_timeout(int *status, unsigned int limit, cudaStream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* KDA_H_ */
