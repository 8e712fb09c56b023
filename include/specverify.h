/*
 * specverify.h -- C ABI of libspecverify, the GB300 (sm_103a) verify-and-accept
 * hot path of multi-token-prediction (MTP) speculative decoding.
 *
 * One speculative cycle, as the pages describe it ("MTPLX 2.24x faster TPS",
 * section "Layer 2: Speculative cycle (the hot loop)"): the drafter proposes K
 * tokens; the target model verifies all of them in one batched forward over
 * M = K+1 rows (the last committed token plus the K drafts -- "MTP in
 * llama.cpp", section "How speculative decoding works"); a probability-ratio
 * test accepts a prefix; a rejection emits one replacement from the residual
 * (p - q)+; a full acceptance emits a bonus token; the GatedDeltaNet state is
 * committed by replaying the innovation tape over the accepted prefix.
 *
 * This library provides the data-parallel steps of that cycle:
 *   qmv_smallm        the target's 4-bit small-M quantised mat-vec (M = 1..16)
 *   qmv_plan_*        an ordered list of those mat-vecs in one persistent launch
 *   spec_accept       fp32 acceptance, residual resampling and bonus token
 *   gdn_tape_capture  GatedDeltaNet recurrence over the verify tokens, with a
 *                     (gate, innovation, key) tape per token and head
 *   gdn_tape_replay   rebuild the recurrent state over an accepted prefix
 *   conv_window_*     short convolution windows: outputs, commit of a prefix
 *   qmv_identity_probe  start-up check: block verify rows == single-row calls
 *   qmv_requantize    a bf16 weight matrix -> the 4-bit layout above (the
 *                     drafter's own 4-bit LM head)
 *   qmv_wide          the same product for wide blocks (M = 17..128, e.g. the
 *                     verify blocks of 32 sequences against one LM head) on
 *                     the tcgen05 tensor cores
 *
 * Conventions (all entry points):
 *  - Every tensor argument is a DEVICE pointer owned by the caller, to
 *    contiguous row-major memory.  The library allocates no device memory and
 *    keeps no pointer after a call returns, except a qmv plan (below), which
 *    holds the pointers it was created with.
 *  - Calls are asynchronous on `stream` (NULL = the legacy default stream) and
 *    never synchronise with the host -- except qmv_plan_create and the
 *    start-up probe qmv_identity_probe, which say so.
 *  - Arguments are validated on the host before any launch.  A nonzero status
 *    means nothing was launched (SV_ERR_CUDA: the launch itself failed), except
 *    for qmv_identity_probe, a sequence of launches that stops at the first
 *    failing one.
 *    sv_last_error() returns a thread-local message for the last failure.
 *  - Data-dependent problems found on the device (a draft token out of range,
 *    a NaN logit, ...) never trap: they are reported in per-sequence flag
 *    words and the result stays well defined (see spec_accept).
 *  - No C++ exception crosses this boundary.
 */
#ifndef SPECVERIFY_H
#define SPECVERIFY_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define SV_ABI_VERSION 2

/* A CUDA stream (cudaStream_t); NULL selects the legacy default stream. */
typedef struct CUstream_st *sv_stream_t;

typedef enum {
    SV_OK = 0,
    SV_ERR_INVALID_ARG = 1, /* a pointer, size, alignment or value is invalid     */
    SV_ERR_UNSUPPORTED = 2, /* valid request outside what the kernels implement   */
    SV_ERR_CUDA = 3,        /* a CUDA runtime call or kernel launch failed        */
    SV_ERR_DEVICE_FLAG = 4  /* sv_device_status: a kernel hit a bounded-wait limit */
} sv_status;

typedef enum { SV_F32 = 0, SV_BF16 = 1 } sv_dtype;

/* Per-sequence error flag bits written by spec_accept (err_flags) and
 * gdn_tape_replay. */
#define SV_FLAG_DRAFT_OUT_OF_RANGE 1 /* draft token not in [0, V): rejected          */
#define SV_FLAG_DRAFT_ZERO_Q 2       /* q(d) == 0, the draft could not have been drawn */
#define SV_FLAG_NONFINITE_LOGIT 4    /* a NaN or +inf logit in a row that was used   */
#define SV_FLAG_EMPTY_DIST 8         /* nothing to sample from: token -1 emitted     */
#define SV_FLAG_REPLAY_RANGE 16      /* gdn_tape_replay: record count clamped to [0,T] */

int sv_abi_version(void);
const char *sv_status_string(int status);
/* Message describing the most recent failure on the calling thread ("" if none). */
const char *sv_last_error(void);

/* Programmatic dependent launch (PDL) for qmv_smallm, qmv_plan_run,
 * qmv_wide and qmv_requantize, process-wide, default 0.
 * When enabled, such a kernel may start while the kernel enqueued before it
 * on the same stream is still running.  Before that kernel has finished the
 * products read only w_packed, scales and biases; x is read, and y (or the
 * top-64 lists) written, after it has finished; qmv_requantize reads nothing
 * before it has finished.  Enable it only when no kernel enqueued right
 * before a product writes its weights (a qmv_requantize of those weights
 * directly followed by the product needs PDL off for that launch, or any
 * other kernel in between).  (The GatedDeltaNet kernels always start in
 * stream order but let the kernel after them start early.) */
void sv_set_pdl(int enable);
int sv_get_pdl(void);

/* Reads and clears the device-side error word (synchronises the current
 * device).  Returns SV_OK, or SV_ERR_DEVICE_FLAG if some kernel gave up on a
 * bounded wait since the last call (it then returned without a result). */
sv_status sv_device_status(void);

/* ------------------------------------------------------------------------ */
/* qmv_smallm: Y[M,N] = X[M,K] . W^T with 4-bit affine group-64 weights.     */
/* ------------------------------------------------------------------------ */
/* Source: "MTPLX 2.24x faster TPS", section "Layer 0: MLX Runtime" -- the
 * verify forward multiplies M = 3..6 rows (one per drafted position) by the
 * 4-bit weights, a shape stock large-M kernels handle badly; "MTPLX | Apple
 * Silicon..." (ai-navigate-news), "what I had to solve" item 3 -- MLP
 * projections took 51 % of verify time before the small-M kernel.
 *
 *   W[n,i] = scales[n, i/64] * q[n,i] + biases[n, i/64]
 *   q[n,i] = (w_packed[n*(K/8) + i/8] >> (4*(i%8))) & 15     (LSB-first)
 *   y[m*N + n] = sum_i x[m*K + i] * W[n,i]      (fp32 accumulation)
 *
 * w_packed  uint32 [N][K/8];  scales, biases: bf16 bit patterns [N][K/64];
 * x         [M][K], fp32 (SV_F32) or bf16 (SV_BF16);   y: fp32 [M][N].
 * Requires 1 <= M <= 16 (M == 0 or N == 0: no-op), K > 0, K % 64 == 0,
 * group_size == 64, bits == 4; w_packed, scales, biases and x 16-byte
 * aligned; y 4-byte aligned and not overlapping any input.  Each output is a
 * fixed-order sum (deterministic run to run) whose order does not depend on
 * M: row m of an M-row call equals the same row computed alone, bit for
 * bit.  M = 9..16 (a DFlash-width block, "MTPLX 2.24x faster TPS", section
 * "Layer 0: MLX Runtime") uses two 8-row MMA tiles per weight fragment and
 * one CTA per SM.  Accuracy: fp32 accumulation
 * of exact products; fp32 x is split into two bf16 terms (|x - hi - lo| <=
 * 2^-16 |x|). */
sv_status qmv_smallm(const uint32_t *w_packed, const uint16_t *scales, const uint16_t *biases,
                     const void *x, sv_dtype x_dtype, float *y, int M, int N, int K,
                     int group_size, int bits, sv_stream_t stream);

/* qmv plan: an ordered list of qmv_smallm problems run by one launch.
 * Sources: "MTPLX 2.24x faster TPS", section "Layer 0: MLX Runtime" (the
 * verify forward streams every 4-bit projection of the target model for M =
 * K+1 rows) and "MTP in llama.cpp", section "Theoretical maximum tg t/s" (a
 * decode step is bounded by streaming the active weights once at memory
 * bandwidth).  A verify forward is hundreds of projections; as separate
 * launches each pays a launch and the latency of its first weight stage, so
 * the weight stream stalls at every boundary.  A plan runs the whole list in
 * one persistent launch whose weight stream never stops: problem i reads its
 * activations x only after every earlier problem has written y when
 * `after` is set (x is an earlier output), and at once otherwise.
 *
 * Each problem: Y[M][N] (fp32) = X[M][K] . W^T with W as in qmv_smallm
 * (w_packed uint32 [N][K/8], scales and biases bf16 [N][K/64], group 64,
 * 4 bits); K % 512 == 0; pointers 16-byte aligned (y 4-byte); y may not
 * overlap the problem's inputs, and a problem may read an earlier output
 * only if `after` is set on it or on a problem between them.  M (1..8) and
 * the activation dtype are shared by all problems.  Results equal
 * qmv_smallm's up to fp32 summation order and are deterministic run to run.
 *
 * qmv_plan_device_bytes: device bytes the plan needs (0 on invalid input;
 * see sv_last_error).  qmv_plan_create: validates, encodes the tensor maps
 * and copies them, with zeroed counters, into `device_buffer` (caller-owned,
 * 256-byte aligned, at least qmv_plan_device_bytes; synchronous; the device
 * current at creation runs the plan); *plan_out is a host object freed by
 * qmv_plan_destroy.  The buffer and every problem's tensors must stay valid
 * while the plan is used.  qmv_plan_run: one launch on `stream` of exactly
 * as many CTAs as fit on the device at once (capturable in a CUDA graph);
 * runs of one plan must not overlap in time.  Its CTAs wait on one another
 * (phase counts, split tiles) and it is not a cooperative launch, so every
 * CTA must become resident: on one device, run plans one at a time (not
 * concurrently on several streams) and beside no other kernel whose CTAs
 * wait for one another -- or use qmv_plan_run_cooperative.  Otherwise two
 * such grids can each hold the SMs the other needs; the plan's waits then
 * give up after ~1 s, set the device error word and leave invalid results
 * (no hang).
 * With sv_set_pdl(1) the launch may start while the preceding kernel runs:
 * weights are streamed at once, while x, y and the plan's counters are
 * touched only after that kernel has finished.
 * A phase wait that exceeds ~1 s sets a device error word
 * (sv_device_status) and the launch finishes with invalid results; the
 * plan's counters are then undefined: create it again. */
typedef struct {
    const uint32_t *w_packed;
    const uint16_t *scales;
    const uint16_t *biases;
    const void *x;  /* [M][K] of the plan's dtype */
    float *y;       /* [M][N]; NULL when topk is set */
    int N, K;
    int after;      /* 1: x is written by an earlier problem of the list */
    /* NULL, or the per-row top-64 epilogue (at most one problem per plan):
     * instead of y, each of the plan's G CTAs writes, for every output row
     * m, the 64 largest (logit, index) pairs among the columns it computed
     * as descending 64-bit keys (the ordered float bits of the logit, then
     * the inverted index; 0 = empty), followed by one flag word per (CTA, m)
     * that is nonzero when a NaN or +inf logit was met.  Layout:
     * uint64 [G][M][64] then uint32 [G][M]; qmv_plan_topk_bytes gives its
     * size.  spec_accept_lists reads it ("MTP in llama.cpp", one evaluation
     * boundary per cycle; the logits never travel through memory). */
    uint64_t *topk;
} sv_qmv_problem;

typedef struct sv_qmv_plan sv_qmv_plan;

size_t qmv_plan_device_bytes(const sv_qmv_problem *problems, int n_problems, int M,
                             sv_dtype x_dtype);
sv_status qmv_plan_create(const sv_qmv_problem *problems, int n_problems, int M,
                          sv_dtype x_dtype, void *device_buffer, size_t device_bytes,
                          sv_qmv_plan **plan_out);
sv_status qmv_plan_run(const sv_qmv_plan *plan, sv_stream_t stream);
/* qmv_plan_run as a cooperative launch: the device guarantees that all of
 * the plan's CTAs are resident together, so the plan may run beside other
 * grids whose CTAs wait on one another (or another plan on another stream)
 * without its waits timing out.  No programmatic early start (sv_set_pdl is
 * ignored); measured about 1.5 us slower per launch than qmv_plan_run.
 * Same results, same errors. */
sv_status qmv_plan_run_cooperative(const sv_qmv_plan *plan, sv_stream_t stream);
void qmv_plan_destroy(sv_qmv_plan *plan);
/* CTAs of the plan's launch (the co-resident count), 0 for NULL. */
int qmv_plan_grid(const sv_qmv_plan *plan);
/* Bytes of a top-64 epilogue buffer for plans of M rows and this dtype on the
 * current device (G x M x (64 x 8 + 4)); 0 on invalid input. */
size_t qmv_plan_topk_bytes(int M, sv_dtype x_dtype);

/* ------------------------------------------------------------------------ */
/* qmv_identity_probe: start-up check that block verification is exact.      */
/* ------------------------------------------------------------------------ */
/* Source: "MTP와 DFlash" (mlxcel manual), section "MTP 정확성 검사": when a
 * worker starts, three independent synthetic inputs go through a verify block
 * and through the equivalent single-token steps; block verification is used
 * only if both agree byte for byte, and the verdict is kept per (model,
 * block width).
 *
 * For the given weights (layout of qmv_smallm), three synthetic activation
 * blocks x_s [M][K] (values in [-2, 2) from a hash of the element index,
 * fp32 or bf16 per x_dtype) are generated on the device; each is multiplied
 * with qmv_smallm as one M-row block and as M one-row calls, and the fp32
 * outputs are compared as bit patterns.  *mismatches = the number of outputs
 * (over the three blocks) whose bits differ; 0 means block verification of
 * this projection at width M is exact.  Keeping the verdict per (weights, M)
 * is the caller's part.
 *
 * Requires 1 <= M <= 16, N >= 1, K >= 64, K % 64 == 0; w_packed, scales and
 * biases as qmv_smallm requires.  scratch: caller-owned device memory,
 * 256-byte aligned, at least qmv_identity_probe_bytes(M, N, K, x_dtype)
 * bytes (0 on invalid input), not overlapping the weights; its contents are
 * overwritten.  Runs on `stream` and waits for it (synchronous: call it at
 * start-up, outside stream capture).  On error *mismatches is -1 (or left
 * unchanged when the arguments are rejected before any work). */
size_t qmv_identity_probe_bytes(int M, int N, int K, sv_dtype x_dtype);
sv_status qmv_identity_probe(const uint32_t *w_packed, const uint16_t *scales,
                             const uint16_t *biases, sv_dtype x_dtype, int M, int N, int K,
                             void *scratch, size_t scratch_bytes, int *mismatches,
                             sv_stream_t stream);

/* ------------------------------------------------------------------------ */
/* qmv_wide: y[M][N] = x[M][K] . W^T for wide blocks, tcgen05 tensor cores.  */
/* ------------------------------------------------------------------------ */
/* Sources: "MTP in llama.cpp", section "Theoretical maximum tg t/s" (the
 * verify step streams the quantised weights once, whatever the number of
 * rows) and "MTPLX 2.24x faster TPS", section "Layer 0: MLX Runtime" (the
 * verify block goes through every 4-bit projection, the LM head included).
 * When the verify blocks of many sequences share one weight matrix (32
 * sequences x (K+1) = 128 rows against the LM head) the product is a dense
 * contraction of about 64 flops per weight byte.
 *
 * Same operation, weight format (w_packed, scales, biases) and output layout
 * as qmv_smallm, for bf16 activations x [M][K]:
 *   y[m][n] = sum_i x[m][i] * (s[n][i/64] * q[n][i] + b[n][i/64])  (fp32).
 * Computed as two bf16 products against the exact split s*q = hi + lo plus
 * sum_g b[n][g] * X[m][g] (X = the group sums of x, fp32, split into two bf16
 * parts), all accumulated in fp32 on the tensor cores: the result is exact
 * up to fp32 rounding of the sums and the 2^-17 relative split of X.
 *
 * Requires 0 <= M <= 128, N >= 0, K % 512 == 0; w_packed, scales, biases and
 * x 16-byte aligned, y 4-byte aligned; y must not overlap any input.
 * workspace: caller-owned device memory, 256-byte aligned, at least
 * qmv_wide_workspace_bytes(M, K) bytes (0 on invalid input), not overlapping
 * the inputs or y; it is overwritten (the split group sums of x).  Two
 * launches on `stream` (the group sums, then the product); M = 0 or N = 0
 * launches nothing.  A kernel wait that gives up (only if the device
 * misbehaves) sets a word read by sv_device_status. */
/* ------------------------------------------------------------------------ */
/* qmv_requantize: bf16 weights -> the 4-bit affine group-64 layout.         */
/* ------------------------------------------------------------------------ */
/* Source: "MTPLX 2.24x faster TPS", section "Layer 0: MLX Runtime": the
 * target keeps its LM head at model precision while a separate 4-bit LM head,
 * built in memory, serves the drafter only (draft time down, target accuracy
 * unchanged).  The drafter's logits are then qmv_smallm(w_packed, scales,
 * biases, x) at M = 1.
 *
 * w_bf16 [N][K] bf16 (finite values), row-major, 16-byte aligned.  Writes
 * w_packed [N][K/8] (4-byte aligned), scales and biases [N][K/64] bf16
 * (2-byte aligned), the layout of qmv_smallm.  Per group of 64 inputs of a
 * row, every step one IEEE fp32 operation:
 *   lo = min w, hi = max w (a zero extreme taken as +0),
 *   s = rn_bf16((hi - lo) / 15), b = lo,
 *   q = 0 if s == 0, else clamp(rint((w - b) / s), 0, 15)   (ties to even).
 * Requires N >= 0, K % 64 == 0; no two buffers may overlap.  One launch on
 * `stream` (PDL-capable); N = 0 launches nothing. */
sv_status qmv_requantize(const uint16_t *w_bf16, uint32_t *w_packed, uint16_t *scales,
                         uint16_t *biases, int N, int K, sv_stream_t stream);

size_t qmv_wide_workspace_bytes(int M, int K);
sv_status qmv_wide(const uint32_t *w_packed, const uint16_t *scales, const uint16_t *biases,
                   const uint16_t *x, float *y, int M, int N, int K, void *workspace,
                   size_t workspace_bytes, sv_stream_t stream);

/* ------------------------------------------------------------------------ */
/* spec_accept: probability-ratio verification of K drafts per sequence.     */
/* ------------------------------------------------------------------------ */
/* Sources: "MTPLX 2.24x faster TPS", sections "Layer 2: Speculative cycle"
 * (fp32 Leviathan-Chen acceptance per position, (p - q)+ residual on
 * rejection, bonus token on full acceptance) and "QWEN 3.6 27B @ 63 TPS"
 * (temperature 0.6, top_p 0.95, top_k 20); "MTP in llama.cpp", section
 * "lossless" (temperature 0: accept until the first mismatch with the
 * target's argmax, plus one extra target token).
 *
 * Distribution of a logits row z (target p_k, draft q_k):
 *   z' = z / temperature -> keep the top_k largest (equal values: lower id)
 *   -> softmax over the kept set -> keep the shortest descending prefix whose
 *   cumulative probability >= top_p (at least one) -> renormalise.
 * For k = 1..K: accept d_k iff u_accept[k] < p_k(d_k) / q_k(d_k).  At the
 * first rejection emit the smallest token id x whose cumulative sum of
 * R = max(0, p_k - q_k) (in ascending id order) exceeds u_sample * sum(R)
 * (R = p_k if sum(R) == 0), and stop.  If all K are accepted, emit a bonus
 * token from p_{K+1} the same way.  temperature == 0: greedy (p_k is the
 * argmax one-hot, lowest id on ties; draft_logits is not read, may be NULL).
 *
 * target_logits fp32 [B][K+1][V]; draft_logits fp32 [B][K][V];
 * draft_tokens int32 [B][K]; u_accept fp32 [B][K]; u_sample fp32 [B] (uniforms
 * in [0,1), supplied by the caller).  Outputs: out_tokens int32 [B][K+1]
 * (accepted drafts, then the emitted token, then -1 padding), n_accepted
 * int32 [B] in [0,K], err_flags int32 [B] (SV_FLAG_*; may be NULL).
 * Device-side data errors: a draft outside [0,V) or with q(d) == 0 is
 * rejected; NaN and +inf logits are never kept (-inf is a mask); a
 * distribution with no finite logit is empty and emits -1.
 * Requires B >= 0 (0: no-op), B*(2K+1) <= 65535, 1 <= K <= 8,
 * 1 <= V <= 1048576, all pointers 4-byte aligned (16-byte aligned logits with
 * V % 4 == 0 are streamed through shared memory by bulk copies, and the
 * call is then two kernel launches on `stream`: the chunk selection and a
 * finish per sequence); temperature finite and >= 0; if
 * temperature > 0 then 1 <= top_k <= 64 and 0 < top_p <= 1.  No output may
 * overlap an input or another output.
 * workspace: device memory of spec_accept_workspace_bytes(B, K, V) bytes,
 * 16-byte aligned, with no required contents: every call first clears the
 * counter words it needs (a memset on `stream`), so one workspace serves
 * calls of any shape it is large enough for.  Calls that run concurrently
 * must use different workspaces. */
typedef struct {
    float temperature; /* 0 => greedy */
    int top_k;         /* 1..64 (ignored when temperature == 0) */
    float top_p;       /* (0, 1]; 1 disables */
} sv_sampling;

size_t spec_accept_workspace_bytes(int B, int K, int V);

sv_status spec_accept(const float *target_logits, const float *draft_logits,
                      const int32_t *draft_tokens, const float *u_accept, const float *u_sample,
                      int B, int K, int V, sv_sampling sampling, int32_t *out_tokens,
                      int32_t *n_accepted, int32_t *err_flags, void *workspace,
                      size_t workspace_bytes, sv_stream_t stream);

/* spec_accept_lists: the same acceptance with the target rows given as the
 * per-CTA top-64 lists of a fused LM head (the top-k epilogue of a qmv plan
 * problem, sv_qmv_problem.topk) instead of logits: "MTP in llama.cpp", one
 * evaluation boundary per cycle; the target logits never travel through
 * memory.  target_lists holds B blocks of spec_accept_lists_block_bytes(G, K)
 * bytes, 16-byte aligned; block b is the plan's buffer for sequence b (G
 * CTAs, K+1 rows): uint64 keys [G][K+1][64] (descending, 0 = empty) then
 * uint32 flags [G][K+1] (nonzero: a NaN or +inf logit was met).  Each list
 * holds the 64 largest keys among the columns its CTA computed, so for
 * top_k <= 64 (and greedy) the filtered target distribution is exactly the
 * one spec_accept forms from the full logits; the result is identical to
 * spec_accept on the logits the plan would have written.  Requires
 * 1 <= G <= 2048.  The workspace is spec_accept's, sized by
 * spec_accept_lists_workspace_bytes (equal to spec_accept_workspace_bytes
 * when G <= 32 ceil(V / 16384), e.g. the 151936-token LM head on one GB300);
 * everything else as spec_accept. */
size_t spec_accept_lists_workspace_bytes(int B, int K, int V, int G);
size_t spec_accept_lists_block_bytes(int G, int K);
sv_status spec_accept_lists(const uint64_t *target_lists, int G, const float *draft_logits,
                            const int32_t *draft_tokens, const float *u_accept,
                            const float *u_sample, int B, int K, int V, sv_sampling sampling,
                            int32_t *out_tokens, int32_t *n_accepted, int32_t *err_flags,
                            void *workspace, size_t workspace_bytes, sv_stream_t stream);

/* spec_accept_noalloc: spec_accept on a scratch area that the library holds
 * as a fixed-size device global (spec_accept_noalloc_scratch_bytes() bytes,
 * 2 MiB: e.g. B <= 32 at K = 3, V = 151936).  The pages have no counterpart;
 * this exists for callers that cannot allocate device memory: a plain C
 * host loop that links only this library and has no device allocator of its
 * own, or a decode loop that must not call cudaMalloc / cudaFree per step
 * (cudaFree synchronises the device).
 * Arguments, outputs, flags and results are those of spec_accept without the
 * workspace pair; like every spec_accept call it clears the counter words
 * it needs on `stream` before its kernels, whatever shape the previous call
 * on the scratch had.
 * Errors: SV_ERR_UNSUPPORTED when spec_accept_workspace_bytes(B, K, V)
 * exceeds the scratch size (nothing is launched; use spec_accept with a
 * caller workspace); SV_ERR_CUDA when the scratch address cannot be looked
 * up; otherwise spec_accept's.
 * There is one scratch per device, so calls that overlap in time (different
 * streams or host threads on one device) race on it and must be serialised
 * by the caller.  The first call on each device looks the scratch address up
 * (with that device current); make it before any stream capture begins. */
size_t spec_accept_noalloc_scratch_bytes(void);

sv_status spec_accept_noalloc(const float *target_logits, const float *draft_logits,
                              const int32_t *draft_tokens, const float *u_accept,
                              const float *u_sample, int B, int K, int V, sv_sampling sampling,
                              int32_t *out_tokens, int32_t *n_accepted, int32_t *err_flags,
                              sv_stream_t stream);

/* ------------------------------------------------------------------------ */
/* GatedDeltaNet innovation tape.                                            */
/* ------------------------------------------------------------------------ */
/* Sources: "MTPLX 2.24x faster TPS", section "Layer 0: MLX Runtime"
 * (innovation-tape GDN capture: KB-scale (token, gate, state-delta) tuples;
 * a rejection replays the tape instead of restoring a state snapshot, bit
 * exact); "MTP와 DFlash" (mlxcel manual), section "Qwen3.8-Flash-Next
 * (qwen4_exp) MTP" (rollback replays the GatedDeltaNet recurrence over the
 * accepted tokens).  The update is the gated delta rule, per (b, h) with
 * S in R^{dv x dk}, in this order (fp32):
 *     S' = alpha_t * S;   u = S' k_t;   e_t = beta_t * (v_t - u);
 *     S_t = S' + e_t k_t^T;   o_t = S_t q_t.
 * The state update rounds alpha_t * S, then adds e_t[i] * k_t[j] with one
 * fused multiply-add per element (capture and replay alike).
 * Tape record (b,t,h) = (alpha_t, e_t, k_t).  Tape layout, fp32, in one
 * buffer of gdn_tape_bytes(B,T,H,dk,dv) bytes: B blocks of
 * F = T*H*(dv+dk) + 4*ceil(T*H/4) floats, block b at float offset b*F holding
 *     e     [T][H][dv]  at float 0
 *     k     [T][H][dk]  at float T*H*dv
 *     alpha [T][H]      at float T*H*(dv+dk)   (padded to a multiple of 4)
 * so the tapes of consecutive batches, stacked, form the tape of the
 * concatenated batch (one replay launch can commit several layers).
 * Replaying records t = 0..L-1 applies S[i][j] <- alpha_t*S[i][j] + e_t[i]*k_t[j]
 * (a rounded multiply, then one fused multiply-add: the same roundings as the
 * capture), so the state after replaying L records equals, bit for bit, the
 * capture's state after its first L tokens.
 * Shapes: state [B][H][dv][dk]; q, k [B][T][H][dk]; v [B][T][H][dv];
 * alpha, beta [B][T][H]; out [B][T][H][dv].
 * Requires B >= 0 (0: no-op), 1 <= T <= 16, H >= 1, dk and dv in [4, 128]
 * and multiples of 4, all pointers 16-byte aligned, outputs not
 * overlapping inputs. */
size_t gdn_tape_bytes(int B, int T, int H, int dk, int dv);

/* Runs the recurrence over T tokens from the snapshot state0 (read only) and
 * writes the tape; when not NULL, out receives the outputs o_t and state_out
 * [B][H][dv][dk] the state after all T tokens. */
sv_status gdn_tape_capture(const float *state0, const float *q, const float *k, const float *v,
                           const float *alpha, const float *beta, int B, int T, int H, int dk,
                           int dv, float *out, float *tape, float *state_out, sv_stream_t stream);

/* Applies, in place, the first L_b = n_replay[b % n_replay_count] +
 * n_replay_bias tape records of every head of state row-block b to state
 * (L_b clamped to [0,T]; a clamp sets SV_FLAG_REPLAY_RANGE in err_flags[b]
 * when err_flags != NULL).  n_replay_count in [1, B]: pass B for one count per
 * sequence, or the number of sequences when state and tape stack several
 * layers' [B_seq] blocks ([layers][B_seq][...]) that share one accepted
 * length per sequence.  n_replay is read on the device, so spec_accept's
 * n_accepted can feed it directly (bias 1 when the tape's first record is the
 * last committed token).  Blocks with L_b == 0 are not touched. */
sv_status gdn_tape_replay(float *state, const float *tape, const int32_t *n_replay,
                          int n_replay_count, int n_replay_bias, int B, int T, int H, int dk,
                          int dv, int32_t *err_flags, sv_stream_t stream);

/* ------------------------------------------------------------------------ */
/* Short causal convolution windows of a GatedDeltaNet layer.                */
/* ------------------------------------------------------------------------ */
/* Source: "MTP와 DFlash" (mlxcel manual), section "Qwen3.8-Flash-Next
 * (qwen4_exp) MTP": the rollback replays the GatedDeltaNet recurrence and two
 * convolution windows over the accepted tokens; the batched DFlash paragraph
 * of the same page: linear-attention layers replay the convolution and
 * recurrent state over each row's accepted prefix.  The pages give no
 * formula; implemented is the depthwise causal convolution of width W whose
 * state is the W-1 most recent inputs of each channel:
 *   h(tau) = x[tau][c] for tau >= 0, window[W-1+tau][c] for -(W-1) <= tau < 0
 *   y[t][c] = sum_{j=0}^{W-1} weight[j][c] * h(t - (W-1) + j)   (fp32, j ascending)
 * Layouts (fp32, time-major): window [B][W-1][C], x and y [B][T][C], weight
 * [W][C].  Requires B >= 0 (0: no-op), 1 <= T <= 64, C >= 1, 2 <= W <= 8,
 * 4-byte aligned pointers, no output overlapping an input.
 *
 * conv_window_capture: y for the T verify tokens; the committed window is
 * read only (a rejection needs nothing restored).
 * conv_window_replay: commit: window <- the last W-1 entries of (window,
 * x[0..L_b)) with L_b = n_replay[b % n_replay_count] + n_replay_bias clamped
 * to [0, T] (a clamp sets SV_FLAG_REPLAY_RANGE in err_flags[b] if given);
 * L_b = 0 leaves the window unchanged.  An exact copy: bit for bit.  The
 * verify inputs x are the tape of the convolution.  n_replay is read on the
 * device (spec_accept's n_accepted, bias 1 when the last committed token is
 * among the verify rows). */
sv_status conv_window_capture(const float *window, const float *x, const float *weight, int B,
                              int T, int C, int W, float *y, sv_stream_t stream);
sv_status conv_window_replay(float *window, const float *x, const int32_t *n_replay,
                             int n_replay_count, int n_replay_bias, int B, int T, int C, int W,
                             int32_t *err_flags, sv_stream_t stream);

#ifdef __cplusplus
}
#endif
#endif /* SPECVERIFY_H */
