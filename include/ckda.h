/*
 * ckda.h -- C ABI of libckda, a GB300 (sm_103a) implementation of the
 * Complex KDA (CKDA) recurrence.
 *
 * The operation (one head of one sequence, state H in R^{dk x dv}, rows are
 * key channels):
 *
 *     H_t = (I - beta_t k_t k_t^T) Diag(alpha_t) H_{t-1} + beta_t k_t v_t^T
 *     o_t = H_t^T (scale * q_t)
 *
 * defined in "Complex KDA: Understanding and Enhancing the Expressivity of
 * Kimi Delta Attention", Sec. 2 Eq. (1) and App. B.2 Eq. (9), with the
 * ranges alpha_t in [-1, 1]^dk, beta_t in [0, 2] of Sec. 3 ("CKDA"), unit
 * keys ||k_t|| = 1, and the readout of the updated state shown on the
 * paper-discussion slides ("CKDA keeps the original gate--delta--readout
 * structure").  The pages use no query scale: scale = 1 reproduces them.
 *
 * Conventions shared by every call:
 *   - All tensor arguments are DEVICE pointers to contiguous row-major
 *     arrays owned by the caller.  The library never allocates, frees or
 *     synchronises device memory on these paths; every call is asynchronous
 *     on `stream` (a cudaStream_t passed as void*, NULL = legacy default).
 *   - Argument errors are detected on the host before anything is launched
 *     and returned synchronously (CKDA_ERR_INVALID_ARG / _UNSUPPORTED).
 *     A failed launch returns CKDA_ERR_CUDA.
 *   - Device-side conditions (a bounded wait that ran out, a result that is
 *     not finite) are written to a status word in the caller's
 *     workspace and read back with ckda_fwd_status().
 *   - k is NOT normalised by the library: ||k_t|| = 1 is the caller's
 *     precondition, as on the pages.  The library accepts any finite k.
 *   - The compute calls (ckda_fwd, ckda_fwd_raw, the split forwards,
 *     ckda_decode_step(_raw), ckda_prep(_bwd), ckda_bwd) enqueue only kernels
 *     and asynchronous memsets on `stream`, so they may be captured into a
 *     CUDA graph and replayed; the tensor maps and launch arguments are fixed
 *     at capture.  ckda_fwd_status and ckda_fwd_host synchronise and may not
 *     be captured; ckda_fwd_noalloc only after its first call in the context.
 */
#ifndef CKDA_H
#define CKDA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    CKDA_F32 = 0,   /* IEEE fp32 inputs and outputs */
    CKDA_BF16 = 1   /* bfloat16 inputs and outputs; the state is always fp32 */
} ckda_dtype;

typedef enum {
    CKDA_OK = 0,
    CKDA_ERR_INVALID_ARG = 1,  /* null pointer, bad size, bad cu_seqlens shape */
    CKDA_ERR_UNSUPPORTED = 2,  /* valid arguments outside what is implemented */
    CKDA_ERR_CUDA = 3,         /* a CUDA runtime call or launch failed */
    CKDA_ERR_TIMEOUT = 4,      /* device: a bounded wait ran out (see ckda_fwd_status) */
    CKDA_ERR_WORKSPACE = 5,    /* workspace missing or smaller than required */
    CKDA_ERR_RANGE = 6         /* device: a non-finite o or final state -- a result outside
                                  fp32 / the I/O dtype, non-finite inputs, or (tensor-core
                                  path) a query or key too large for its fp16 operand; v
                                  and h0 of any finite size are scaled into range */
} ckda_status;

/* Version of this ABI: major * 10000 + minor * 100 + patch. */
int ckda_version(void);

/* Human-readable name of a status code (static storage; never NULL). */
const char *ckda_status_string(ckda_status s);

/*
 * Workspace bytes ckda_fwd needs.  num_seqs is the number of packed
 * sequences (cu_seqlens != NULL) or 0 for the dense layout.  The workspace
 * holds the device status word and, for packed input, the longest-first
 * work order of the sequences.  It is scratch: its contents on entry do not
 * matter (each ckda_fwd first clears the status word on its stream) and
 * calls that share one workspace must be stream-ordered.
 */
size_t ckda_fwd_workspace_bytes(int num_seqs, int H);

/*
 * Forward over a batch: computes o for every token and the final state of
 * every (sequence, head).
 *
 * Layouts (io = io_dtype element type):
 *   q, k, alpha : io   [B, H, T, dk]
 *   v, o        : io   [B, H, T, dv]
 *   beta        : io   [B, H, T]
 *   h0, hT      : fp32 [N, H, dk, dv], N = B (dense) or num_seqs (packed)
 *   cu_seqlens  : int32 [num_seqs + 1] device array, or NULL.  When given,
 *                 B must be 1 and the sequences are packed along T:
 *                 sequence n owns tokens [cu_seqlens[n], cu_seqlens[n+1]).
 *                 The offsets must be non-decreasing with cu_seqlens[0] = 0
 *                 and cu_seqlens[num_seqs] = T; they are read on the device
 *                 and not validated there.
 *   h0 == NULL  : zero initial state.   hT == NULL : final state not stored.
 *   hT may alias h0 (each (sequence, head) reads its slice before writing).
 *   o must not alias any input.
 *
 * Paths: io_dtype = CKDA_BF16 with dv = 128 and dk = 128 or 64 runs the
 * chunkwise tensor-core kernel (chunk_size 0 or 64); dk = 64 is the reduced
 * key dimension of a state-reduced head ("On State Reduction in Linear
 * Attention"), run with the key channels padded to 128 inside the kernel
 * (zero keys and queries, unit gates), which leaves the result unchanged.
 * Every other supported shape
 * (dk, dv <= 128) runs the token-serial CUDA-core kernel, which has no
 * chunks (chunk_size 0, 16, 32 or 64 accepted and ignored; results never
 * depend on it).  scale multiplies q.
 *
 * workspace / workspace_bytes: device scratch of at least
 * ckda_fwd_workspace_bytes(cu_seqlens ? num_seqs : 0, H) bytes, 256-byte
 * aligned.
 *
 * Returns CKDA_OK once the work is enqueued on `stream`.
 */
ckda_status ckda_fwd(const void *q, const void *k, const void *v,
                     const void *alpha, const void *beta, const float *h0,
                     void *o, float *hT, const int32_t *cu_seqlens, int num_seqs,
                     int B, int H, int T, int dk, int dv, ckda_dtype io_dtype,
                     float scale, int chunk_size, void *workspace,
                     size_t workspace_bytes, void *stream);

/*
 * ckda_fwd on raw inputs: the input preparation of ckda_prep (unit-norm k,
 * and q if normalize_q; alpha = s [e^-5 + (1 - e^-5) |tanh(a / 2)|];
 * beta = 2 sigma(b)) applied inside the forward kernel as each tile is
 * loaded ("Complex KDA" paper Sec. 6 "Implementation": the signs and the
 * normalisation are fused into the kernels), so the prepared q, k, alpha,
 * beta never pass through HBM.
 *
 *   q_raw, k_raw, a_raw : io [B, H, T, dk]  (the unnormalised q, k and the
 *                                            decay-gate logits)
 *   b_raw               : io [B, H, T]      (the write-strength logits)
 *   v, o, h0, hT, cu_seqlens, num_seqs, scale, workspace: as ckda_fwd.
 *
 * The maps run in fp32 on the loaded bf16 values.  The normalised q and k
 * and alpha then take the forward's own fp16 operand rounding (they are not
 * rounded to bf16 first); beta is rounded to the I/O dtype, exactly as
 * ckda_prep hands it to ckda_fwd.  scale multiplies q after its normalisation.  Tensor-core
 * shapes only (bf16, dv = 128, dk = 128 or 64): others return
 * CKDA_ERR_UNSUPPORTED (use ckda_prep and ckda_fwd).  norm_eps >= 0.
 */
ckda_status ckda_fwd_raw(const void *q_raw, const void *k_raw, const void *v,
                         const void *a_raw, const void *b_raw, const float *h0,
                         void *o, float *hT, const int32_t *cu_seqlens, int num_seqs,
                         int B, int H, int T, int dk, int dv, ckda_dtype io_dtype,
                         float scale, int normalize_q, float norm_eps, void *workspace,
                         size_t workspace_bytes, void *stream);

/*
 * ckda_fwd for callers that cannot allocate device memory.  The paper has no
 * counterpart; this is a deployment variant of ckda_fwd.
 *
 * Same arguments and results as ckda_fwd, minus the workspace.  It is meant
 * for callers that may not call cudaMalloc.  One example is a host
 * application that splits its device memory once at start-up and forbids
 * later allocation.  Another is a plugin whose host owns the only allocator.
 * The scratch ckda_fwd would take from a workspace lives instead in a fixed
 * array in this library's device memory: 256 KiB + 256 B on every GPU that
 * loads the library, held until the process exits.  Nothing is allocated or
 * freed per call.
 *
 *   - Packed input is limited to num_seqs <= 65536; more returns
 *     CKDA_ERR_UNSUPPORTED before anything is launched.
 *   - The first call in a CUDA context looks up the array's device address
 *     in that context (the device's primary context for runtime callers; a
 *     plugin host's own driver-API context if that is the current one).  The
 *     address is cached per context id and never reused in another context,
 *     so a cudaDeviceReset or a different current context gets its own
 *     set-up.  Make the first call in a context before any stream capture.
 *   - Every call shares the one array.  Calls whose GPU work overlaps (on
 *     different streams, or from several threads at once) race on it and
 *     must be serialised by the caller.  Each call clears the status word it
 *     uses and rewrites the work order it reads.
 *   - Device-side conditions (timeout, range) are recorded in the shared
 *     array and are not reported; use ckda_fwd to observe them.
 */
ckda_status ckda_fwd_noalloc(const void *q, const void *k, const void *v,
                             const void *alpha, const void *beta, const float *h0,
                             void *o, float *hT, const int32_t *cu_seqlens, int num_seqs,
                             int B, int H, int T, int dk, int dv, ckda_dtype io_dtype,
                             float scale, int chunk_size, void *stream);

/*
 * Forward over HOST buffers: the operation of ckda_fwd for the dense layout,
 * with every tensor argument in host memory (page-locked memory gives full
 * copy bandwidth; pageable memory works, slower).  Same layouts and dtypes
 * as ckda_fwd: q, k, alpha [B, H, T, dk]; v, o [B, H, T, dv]; beta
 * [B, H, T]; h0, hT fp32 [B, H, dk, dv] (h0 == NULL: zero state; hT == NULL:
 * not stored).  Packed sequences are not accepted here.
 *
 * The token axis is processed in slices of `slice_tokens` tokens (a multiple
 * of 64; 0 picks about T / 4, at least 512): the copy of slice s to the device
 * overlaps the computation of slice s - 1 and the copy of slice s - 2's o
 * back, on two internal streams and the caller's `stream`.  Each
 * (sequence, head) carries its fp32 state between slices in device memory,
 * and slices end on chunk boundaries, so o and hT equal those of one
 * ckda_fwd over the whole sequence.
 *
 * dev_scratch / dev_scratch_bytes: caller-owned device memory of at least
 * ckda_fwd_host_scratch_bytes(...) bytes, 256-byte aligned; it holds the
 * device copies of two slices, the carried state and a status word (read it
 * with ckda_fwd_status(dev_scratch, stream)).  Calls that share a scratch
 * must be ordered on their streams.
 *
 * Returns CKDA_OK once the work is enqueued on `stream`; o and hT in host
 * memory are complete when `stream` is.  The internal streams are shared by
 * the calls of a process on one device (enqueueing is serialised).
 */
size_t ckda_fwd_host_scratch_bytes(int B, int H, int T, int dk, int dv, ckda_dtype io_dtype,
                                   int slice_tokens);
ckda_status ckda_fwd_host(const void *q, const void *k, const void *v,
                          const void *alpha, const void *beta, const float *h0,
                          void *o, float *hT, int B, int H, int T, int dk, int dv,
                          ckda_dtype io_dtype, float scale, int slice_tokens,
                          void *dev_scratch, size_t dev_scratch_bytes, void *stream);

/*
 * Sequence-split forward: the result of ckda_fwd (dense layout) for batches
 * with fewer (sequence, head) pairs than the GPU has SMs, and long sequences.
 *
 * The recurrence is affine in the state: over a run of tokens the final state
 * is P H_in + F, with P the product of the steps' transitions (dk x dk) and F
 * the final state from H_in = 0 (Eq. (1) of "Complex KDA: Understanding and
 * Enhancing the Expressivity of Kimi Delta Attention", applied step after
 * step).  Like the chunked form ("Kimi Delta Attention: a bounded case study",
 * "Chunkwise execution"), splitting a sequence this way changes the cost and
 * not the result.  Each sequence is cut into `segments` runs of whole 64-token
 * chunks.  Pass 1 computes, in parallel:
 *   - segment 0 from h0, including its o;
 *   - for each middle segment, F, and P (as the final state from [I | 0] with
 *     v = 0).
 * A scan then gives the state entering each segment.  Pass 2 runs segments
 * 1..S-1 from those states and writes their o and the final state.
 *
 * Arguments, layouts and results are those of ckda_fwd with cu_seqlens = NULL
 * and chunk_size = 0.  hT may alias h0.
 *   segments : 0 picks the count for the current device (see
 *              ckda_fwd_split_segments); 1 runs ckda_fwd unchanged; S >= 2
 *              cuts each sequence into ceil(chunks / ceil(chunks / S)) <= S
 *              segments.
 * The split runs on the tensor-core shapes (io_dtype = CKDA_BF16, dv = 128,
 * dk = 128 or 64).  With segments >= 2, other shapes return
 * CKDA_ERR_UNSUPPORTED; with segments = 0 they run as ckda_fwd.
 *
 * workspace: device scratch of at least
 * ckda_fwd_split_workspace_bytes(B, H, T, dk, dv, io_dtype, segments) bytes,
 * 256-byte aligned.  It holds the status word (read it with ckda_fwd_status)
 * and, with S >= 2, B * H * S fp32 [dk, 128] states, and as many transitions
 * and zero-start states when S >= 3.  The call is asynchronous on `stream`:
 * two launches of the forward kernel and one of the scan.
 *
 * Every segment's state passes through fp32, and each P carries the same
 * tensor-core rounding as the state of one ckda_fwd.  The results therefore
 * match ckda_fwd within the forward's tolerance, not bit for bit.
 */
/*
 * The segment count ckda_fwd_split picks for segments = 0: the count, at most
 * 16 and at most one per chunk, that minimises a model of the run time.  The
 * model counts chunk steps: whole waves of CTAs over num_sms SMs for both
 * passes, plus small terms for the state I/O and the scan.  A count must beat
 * one plain pass by 10%; otherwise the answer is 1.  num_sms = 0 reads the
 * current device.  Shapes off the tensor-core path, and bad sizes, give 1.
 * Host-only; it enqueues nothing.
 */
int ckda_fwd_split_segments(int B, int H, int T, int dk, int dv, ckda_dtype io_dtype,
                            int num_sms);
size_t ckda_fwd_split_workspace_bytes(int B, int H, int T, int dk, int dv, ckda_dtype io_dtype,
                                      int segments);
ckda_status ckda_fwd_split(const void *q, const void *k, const void *v,
                           const void *alpha, const void *beta, const float *h0,
                           void *o, float *hT, int B, int H, int T, int dk, int dv,
                           ckda_dtype io_dtype, float scale, int segments,
                           void *workspace, size_t workspace_bytes, void *stream);

/*
 * The sequence split for packed input: ckda_fwd with cu_seqlens (same
 * layouts: q, k, alpha [1, H, T, dk], v, o [1, H, T, dv], beta [1, H, T],
 * h0, hT fp32 [num_seqs, H, dk, dv], cu_seqlens device int32 [num_seqs + 1],
 * monotone from 0 to T), where every sequence longer than seg_len tokens is
 * cut into ceil(L / seg_len) segments that run in parallel, chained by the
 * scan of ckda_fwd_split; shorter sequences run whole in the first pass.
 * Sequences are planned longest first on the device, so the host needs no
 * lengths and nothing is synchronised.  Each launch covers an upper bound on
 * the plan's work; CTAs beyond it return at once.
 *
 * seg_len: a positive multiple of 64, or 0 for ckda_fwd_split_varlen_seg_len's
 * choice (the average work per SM; 0 from that function means the shape does
 * not take the tensor-core path).  Bf16 with dv = 128 and dk = 128 or 64 only
 * (CKDA_ERR_UNSUPPORTED otherwise).  The workspace (256-byte aligned) holds
 * the status word, the order, the plan and three state tiles per segment
 * slot: ckda_fwd_split_varlen_workspace_bytes.  Results equal ckda_fwd's up
 * to rounding.  Returns once the five launches are enqueued on `stream`;
 * device conditions are read with ckda_fwd_status.
 */
int ckda_fwd_split_varlen_seg_len(int num_seqs, int H, int T, int dk, int dv,
                                  ckda_dtype io_dtype, int num_sms);
size_t ckda_fwd_split_varlen_workspace_bytes(int num_seqs, int H, int T, int dk, int seg_len);
ckda_status ckda_fwd_split_varlen(const void *q, const void *k, const void *v,
                                  const void *alpha, const void *beta, const float *h0,
                                  void *o, float *hT, const int32_t *cu_seqlens, int num_seqs,
                                  int H, int T, int dk, int dv, ckda_dtype io_dtype, float scale,
                                  int seg_len, void *workspace, size_t workspace_bytes,
                                  void *stream);

/*
 * Reads (and clears) the device status word of a workspace: waits for
 * `stream`, then returns CKDA_OK, CKDA_ERR_TIMEOUT or CKDA_ERR_RANGE for the
 * most recent ckda_fwd (or self-test) enqueued with that workspace.
 * Returns CKDA_ERR_CUDA if the copy or the stream failed.
 */
ckda_status ckda_fwd_status(void *workspace, void *stream);

/*
 * One decode step: applies one token to a resident state, in place.
 * The update is the recurrence above with T = 1, computed as in "Kimi Delta
 * Attention: a bounded case study" (worked case A/B: per-channel decay,
 * read, correct) followed by the readout of the updated state.
 *
 *   q, k, alpha : io   [B, H, dk]
 *   v, o        : io   [B, H, dv]
 *   beta        : io   [B, H]
 *   state       : fp32 [B, H, dk, dv], read and overwritten.
 *
 * dk = dv = 128 runs the vectorised bandwidth kernel; other dk, dv <= 128
 * run the column-per-thread kernel.  Returns CKDA_OK once enqueued.
 */
ckda_status ckda_decode_step(const void *q, const void *k, const void *v,
                             const void *alpha, const void *beta, float *state,
                             void *o, int B, int H, int dk, int dv,
                             ckda_dtype io_dtype, float scale, void *stream);

/*
 * One decode step on raw inputs, with the input preparation of ckda_prep
 * fused in: the step first forms k = k_raw / sqrt(|k_raw|^2 + norm_eps), q
 * likewise when normalize_q (else q = q_raw), alpha = s [e^-5 + (1 - e^-5)
 * |tanh(a_raw / 2)|] with s = +1 for tanh >= 0 else -1, and beta =
 * 2 sigma(b_raw) ("Complex KDA" discussion slides, backup frame "practical
 * gates differ from exact theoretical endpoints"; paper Sec. 2 for the unit
 * keys), in fp32, then applies ckda_decode_step's update and readout.  The
 * prepared values are not written out.
 *
 *   q_raw, k_raw, a_raw : io   [B, H, dk]      v, o : io [B, H, dv]
 *   b_raw               : io   [B, H]          state : fp32 [B, H, dk, dv]
 *
 * dk = dv = 128 only (CKDA_ERR_UNSUPPORTED otherwise; ckda_prep followed by
 * ckda_decode_step covers the other shapes); state 16-byte aligned.  The step
 * is bound by HBM like the plain one: the token inputs are 1 KB against the
 * state's 128 KB per (batch, head).  Argument errors return synchronously;
 * otherwise CKDA_OK once enqueued on `stream`.
 */
ckda_status ckda_decode_step_raw(const void *q_raw, const void *k_raw, const void *v,
                                 const void *a_raw, const void *b_raw, float *state, void *o,
                                 int B, int H, int dk, int dv, ckda_dtype io_dtype,
                                 float scale, int normalize_q, float norm_eps, void *stream);

/*
 * Backward of ckda_fwd: gradients of L = sum_t <o_t, do_t> + <hT, dhT> with
 * respect to q, k, v, alpha, beta and h0, by reverse-mode differentiation of
 * the recurrence ("Complex KDA: Understanding and Enhancing the Expressivity
 * of Kimi Delta Attention", Sec. 2 Eq. (1) and App. B.2 Eq. (9); the paper's
 * Fig. 5 times forward and backward together).  Per token, with
 * G = Diag(alpha) S, p = G^T k, u = beta (v - p), S' = G + k u^T and
 * D = dL/dS' (from dhT):
 *   D += (scale q) do^T;  du = D^T k;  dv = beta du;  dbeta = <du, v - p>;
 *   dp = -beta du;  dk = D u + G dp;  dalpha_i = sum_j (D + k dp^T)_ij S_ij;
 *   D <- Diag(alpha)(D + k dp^T);  dq = scale S' do;  dh0 = the final D.
 *
 *   q, k, alpha, d_q, d_k, d_alpha : io [B, H, T, dk]
 *   v, d_o, d_v                    : io [B, H, T, dv]
 *   beta, d_beta                   : io [B, H, T]
 *   h0, d_hT, d_h0                 : fp32 [N, H, dk, dv]  (N as in ckda_fwd)
 *   cu_seqlens / num_seqs          : as in ckda_fwd (packed sequences, B = 1)
 *
 * h0 == NULL: zero initial state.  d_hT == NULL: no gradient on the final
 * state.  d_h0 == NULL: not stored.  Gradient buffers must not alias inputs.
 * Any dk, dv <= 128 and either I/O dtype; arithmetic is fp32, token by token
 * on CUDA cores.  Each (sequence, head) runs as one thread-block cluster of
 * ceil(dv / 32) CTAs, each holding 32 columns of the state in registers;
 * sums over columns are reduced in a fixed order, so results are
 * deterministic.  Pass 1 reruns the forward and keeps the state before every
 * 64th token in `workspace`.  Pass 2 takes the 64-token chunks in reverse:
 * it reruns a chunk from its checkpoint, keeping the state before every 2nd
 * token, and walks the chunk backward 2 tokens at a time.
 *
 * workspace: device memory of at least ckda_bwd_workspace_bytes(num_seqs, B,
 * H, T, dk, dv) bytes (num_seqs = 0 for dense input), 16-byte aligned, owned
 * by the caller; its contents are scratch.  It holds state slices of 16 KiB
 * (one CTA's 32 columns).  There are ceil(dv / 32) of them per checkpoint:
 * ceil(T/64) checkpoints per dense (batch, head), ceil(T/64) + num_seqs per
 * head when packed.  Each CTA also has 32 slices for the chunk being walked.
 * Argument errors return synchronously with nothing launched; otherwise
 * CKDA_OK once enqueued on `stream`.  The library allocates nothing.
 */
size_t ckda_bwd_workspace_bytes(int num_seqs, int B, int H, int T, int dk, int dv);
ckda_status ckda_bwd(const void *q, const void *k, const void *v, const void *alpha,
                     const void *beta, const float *h0, const void *d_o, const float *d_hT,
                     void *d_q, void *d_k, void *d_v, void *d_alpha, void *d_beta,
                     float *d_h0, const int32_t *cu_seqlens, int num_seqs, int B, int H,
                     int T, int dk, int dv, ckda_dtype io_dtype, float scale,
                     void *workspace, size_t workspace_bytes, void *stream);

/*
 * Input preparation, fused into one pass over HBM: the gate
 * parameterisation of "Complex KDA" (discussion slides, backup frame
 * "practical gates differ from exact theoretical endpoints"; paper App.
 * E-G.1) and the unit-norm keys the recurrence assumes (paper Sec. 2), per
 * token row of dk channels:
 *
 *   r = tanh(a / 2),  s = +1 if r >= 0 else -1,
 *   alpha = s [e^-5 + (1 - e^-5) |r|],       beta = 2 sigma(b) = 2 / (1 + e^-b),
 *   k = k_raw / sqrt(sum_i k_raw_i^2 + norm_eps),
 *   q = q_raw / sqrt(sum_i q_raw_i^2 + norm_eps) if normalize_q, else q_raw.
 *
 * The paper's implementation fuses the gate's sign handling into the key
 * normalisation the same way (Sec. 6 "Implementation").  Its outputs are
 * ckda_fwd's and ckda_decode_step's q, k, alpha, beta.
 *
 *   q_raw, k_raw, a_raw : io [rows, dk]   (rows = B*H*T, or B*H for decode)
 *   b_raw               : io [rows]
 *   q, k, alpha         : io [rows, dk]    beta : io [rows]
 *
 * q_raw and q are both NULL (no query) or both set.  Each output may alias
 * its own input (in place); outputs must not alias other inputs.  Arithmetic
 * is fp32 with one rounding to io_dtype.  norm_eps >= 0; with norm_eps = 0 an
 * all-zero row gives NaN, with norm_eps > 0 it stays zero.  dk <= 128.
 * Argument errors return synchronously with nothing launched (rows = 0
 * launches nothing and returns CKDA_OK); otherwise returns CKDA_OK once
 * enqueued on `stream`.  The library allocates nothing.
 */
ckda_status ckda_prep(const void *q_raw, const void *k_raw, const void *a_raw,
                      const void *b_raw, void *q, void *k, void *alpha, void *beta,
                      long long rows, int dk, ckda_dtype io_dtype, int normalize_q,
                      float norm_eps, void *stream);

/*
 * Backward of ckda_prep: from the gradients of a loss with respect to its
 * outputs (d_q, d_k, d_alpha, d_beta), the gradients with respect to its raw
 * inputs (d_q_raw, d_k_raw, d_a_raw, d_b_raw), per token row:
 *
 *   k = k_raw / n, n = sqrt(sum_i k_raw_i^2 + norm_eps):
 *       d_k_raw = (d_k - k (k . d_k)) / n           (q likewise if normalize_q,
 *                                                     else d_q_raw = d_q)
 *   d_a_raw = d_alpha * (1 - e^-5) (1 - r^2) / 2 with r = tanh(a_raw / 2),
 *             and 0 where a_raw = 0
 *   d_b_raw = d_beta * 2 sigma(b_raw) (1 - sigma(b_raw))
 *
 * The gate's sign s is piecewise constant and carries no gradient; |r| takes
 * the subgradient 0 at r = 0 (where alpha jumps between -e^-5 and +e^-5).
 *
 *   q_raw, k_raw, a_raw, d_q, d_k, d_alpha, d_q_raw, d_k_raw, d_a_raw : io [rows, dk]
 *   b_raw, d_beta, d_b_raw                                           : io [rows]
 *
 * q_raw, d_q and d_q_raw are all NULL (no query) or all set; normalize_q and
 * norm_eps must be those of the forward call.  Each output may alias its own
 * gradient input or its own raw input (in place).  Arithmetic is fp32 with
 * one rounding to io_dtype.  dk <= 128.  Argument errors return
 * synchronously with nothing launched (rows = 0 launches nothing and returns
 * CKDA_OK); otherwise returns CKDA_OK once enqueued on `stream`.  The library
 * allocates nothing.
 */
ckda_status ckda_prep_bwd(const void *q_raw, const void *k_raw, const void *a_raw,
                          const void *b_raw, const void *d_q, const void *d_k,
                          const void *d_alpha, const void *d_beta, void *d_q_raw,
                          void *d_k_raw, void *d_a_raw, void *d_b_raw, long long rows, int dk,
                          ckda_dtype io_dtype, int normalize_q, float norm_eps, void *stream);

/*
 * Self-test of the bounded-wait path: launches one block that waits on a
 * barrier nothing will complete, with a limit of `spin_limit` polls (each
 * sleeping up to about a microsecond, the whole wait at most about a second),
 * after which it records CKDA_ERR_TIMEOUT in the workspace's status word and
 * returns.  It never hangs and never faults.  Read the result with
 * ckda_fwd_status().
 */
ckda_status ckda_selftest_timeout(void *workspace, size_t workspace_bytes,
                                  unsigned int spin_limit, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* CKDA_H */
