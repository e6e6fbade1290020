/*
 * spec_verify.h -- C ABI of the GB300 (sm_103a) verify-and-sample step of
 * speculative decoding.
 *
 * One call to spec_verify_run performs, for B independent sequences, the
 * target-side tail of one speculative round:
 *
 *   1. LM-head contraction: logits L[b, i, v] = sum_k hidden[b, i, k] * W_lm[v, k]
 *      for the K+1 verified positions i = 0..K of every sequence.
 *      ("What Actually Happens During Speculative Decoding in LLMs", the
 *      memory-bound section: the verify pass multiplies a [positions x d]
 *      block against weights that are read from memory once.)
 *   2. Temperature softmax: p_{i+1} = softmax(L[b, i, :] / T) and
 *      q_{i+1} = softmax(q_logits[b, i, :] / T), the same T for both.
 *      ("Speculative Decoding: Two Models, One Voice", "The rule that makes
 *      it exact", third remark; "Speculative Decoding: The Algebra and the
 *      Proof", "Where it breaks".)
 *   3. Left-to-right accept test: draft token x_{i+1} survives iff
 *      u[b, i] < p_{i+1}(x) / q_{i+1}(x) (strict; if q(x) == 0 it survives
 *      iff p(x) > 0).  The round stops at the first rejection.
 *      ("Speculative Decoding: Two Models, One Voice", "The idea", step 3;
 *      "Speculative Decoding" (library wiki), "One speculation round".)
 *   4. Final draw with the last uniform u[b, K]: at a rejection at position
 *      j, from norm(max(0, p_j - q_j)) (from p_j if that residual is empty);
 *      if all K survive, the bonus token from p_{K+1}.  Every draw is an
 *      inverse CDF in token-id order: the smallest v with u * S < C_v.
 *      ("Speculative Decoding: Guess Several Tokens, Check Them in One
 *      Pass", Step 3; "What Actually Happens ...", speculative_sample_step.)
 *   5. T == 0 is greedy verification: accept while x_{i+1} equals the
 *      argmax of L[b, i, :] (ties to the smallest id), emit that argmax at
 *      the first mismatch, or the argmax of L[b, K, :] as the bonus.
 *      ("Speculative Decoding: Guess Several Tokens, Check Them in One
 *      Pass", Step 2, verify_greedy; "Two Models, One Voice", first remark.)
 *
 * Conventions for every function:
 *   - Return value: 0 (SV_OK) or a negative SV_ERR_* code.  No function
 *     throws, aborts or prints.
 *   - Pointers named "device" must be device memory (or managed memory)
 *     visible to the handle's device; they are owned by the caller and are
 *     never freed or retained by the library beyond the call.
 *   - All tensors are dense, row-major, and 16-byte aligned.
 *   - Host-detectable errors (bad arguments, alignment, shapes) return
 *     before anything is launched.  Errors found on the device (draft token
 *     out of range, non-finite logits, a bounded wait that ran out) are
 *     written to a device status word; read them with spec_verify_status.
 */
#ifndef SPEC_VERIFY_H
#define SPEC_VERIFY_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Status codes. */
#define SV_OK 0
#define SV_ERR_ARG (-1)       /* null pointer, bad size, bad temperature     */
#define SV_ERR_ALIGN (-2)     /* pointer not 16-byte aligned                 */
#define SV_ERR_SHAPE (-3)     /* V, d, B, K outside the supported limits     */
#define SV_ERR_CUDA (-4)      /* a CUDA runtime/driver call failed           */
#define SV_ERR_ARCH (-5)      /* device is not compute capability 10.3       */
#define SV_ERR_TIMEOUT (-6)   /* a bounded device-side wait ran out          */
#define SV_ERR_TOKEN (-7)     /* a draft token was outside [0, V)            */
#define SV_ERR_NONFINITE (-8) /* logits or draft logits were NaN/inf         */

/* Element type of hidden and W_lm. */
#define SV_BF16 0 /* production path: TMA + tcgen05 tensor-core contraction   */
#define SV_FP32 1 /* reference-precision path for small vocabularies          */
#define SV_FP8 2  /* FP8 E4M3 hidden and W_lm with fp32 row scales: run
                   * through spec_verify_run_fp8                             */

/* Limits checked at create time. */
#define SV_MAX_K 64      /* draft tokens (tree nodes) per sequence           */
#define SV_MAX_B 4096    /* sequences per call                               */
#define SV_MAX_ROWS_BF16 384 /* B * (K+1) for the bf16 path                  */

typedef struct spec_verify spec_verify_t; /* opaque handle */

typedef struct {
  int64_t V;      /* vocabulary size, >= 1                                   */
  int64_t d;      /* hidden size; bf16: multiple of 8, fp32: multiple of 4   */
  int32_t B;      /* sequences per call, 1..SV_MAX_B                         */
  int32_t K;      /* draft tokens per sequence, 0..SV_MAX_K                  */
  int32_t dtype;  /* SV_BF16, SV_FP32 or SV_FP8                              */
  void *stream;   /* cudaStream_t the calls are enqueued on (NULL = legacy)  */
} sv_config_t;

/* Creates a handle for one problem shape on the current CUDA device and
 * allocates its device workspace (logits scratch, softmax partials,
 * per-sequence state, status word, staging buffers for
 * spec_verify_run_host).  *out receives the handle.
 * Errors: SV_ERR_ARG (null pointer, bad dtype), SV_ERR_SHAPE (limits
 * above), SV_ERR_ARCH (not compute capability 10.3), SV_ERR_CUDA
 * (allocation failed).  On error *out is set to NULL. */
int spec_verify_create(const sv_config_t *cfg, spec_verify_t **out);

/* Enqueues one verify-and-sample step (steps 1-5 above) on the handle's
 * stream and returns without synchronising.  Outputs are valid once the
 * stream has reached this point.  The call allocates nothing and does not
 * synchronise the host, so it can be captured in a CUDA graph.
 *   hidden         device, [B, K+1, d] of dtype; row i of sequence b is the
 *                  final hidden state that scores draft position i+1 (row K
 *                  scores the bonus position K+1)
 *   W_lm           device, [V, d] of dtype (the LM-head matrix, read once)
 *   draft_tokens   device, int32 [B, K], each in [0, V); may be NULL if K == 0
 *   q_logits       device, fp32 [B, K, V] draft logits; not read if T == 0.
 *                  NULL: the drafts came without a distribution (prompt
 *                  lookup, a supplied prediction), so q is the point mass at
 *                  each proposed token ("Speculative Decoding: The Algebra
 *                  and the Proof", "Where it breaks": q is the distribution
 *                  that actually generated the proposal).  The accept test
 *                  becomes u < p(x), the residual is p without x, and a draft
 *                  may end early: the first -1 in draft_tokens[b] ends it
 *                  (later entries must be -1 too) and, if every proposed
 *                  token survives, the bonus comes from target row K_b, the
 *                  draft's length.  Applies at T == 0 as well (greedy).
 *   uniforms       device, fp32 [B, K+1] in [0, 1): u[b, i] for the accept
 *                  test of position i+1, u[b, K] for the final draw;
 *                  unused if T == 0
 *   temperature    T > 0 samples; T == 0 selects greedy verification
 *   out_tokens     device, int32 [B, K+1]: the accepted prefix, then the
 *                  resampled or bonus token, then -1
 *   out_n_accepted device, int32 [B]: accepted draft tokens (the round
 *                  emitted n + 1 tokens); -1 for a sequence with an invalid
 *                  draft token or non-finite logits
 * The outputs depend on the inputs only: repeated calls on the same inputs
 * give the same tokens bit for bit (every sum has a fixed order; a tile
 * split between two CTAs is always finished by the same one).
 * Errors (returned): SV_ERR_ARG (null handle/pointer, T < 0 or not finite),
 * SV_ERR_ALIGN, SV_ERR_CUDA (launch failed).
 * Errors (device status word): SV_ERR_TOKEN, SV_ERR_NONFINITE,
 * SV_ERR_TIMEOUT. */
int spec_verify_run(spec_verify_t *h, const void *hidden, const void *W_lm,
                    const int32_t *draft_tokens, const float *q_logits,
                    const float *uniforms, float temperature,
                    int32_t *out_tokens, int32_t *out_n_accepted);

/* The same step end to end from HOST buffers: copies hidden, draft_tokens,
 * q_logits and uniforms (host; pinned memory recommended) into the handle's
 * staging buffers, runs the step, copies out_tokens and out_n_accepted back
 * to the host buffers, and synchronises the stream before returning.  W_lm
 * stays a DEVICE pointer (model weights are resident).  Argument meaning
 * and errors as spec_verify_run; the device status word is also checked
 * and returned. */
int spec_verify_run_host(spec_verify_t *h, const void *hidden_host,
                         const void *W_lm, const int32_t *draft_tokens_host,
                         const float *q_logits_host, const float *uniforms_host,
                         float temperature, int32_t *out_tokens_host,
                         int32_t *out_n_accepted_host);

/* End-to-end rounds from HOST buffers, double-buffered, for a caller with
 * independent rounds to verify back to back (two groups of sequences that
 * alternate, or replicas of a benchmark); a decode loop whose next round
 * needs this round's tokens gains nothing over spec_verify_run_host.
 * spec_verify_submit_host enqueues a round in slot 0 or 1 and returns
 * without waiting: its inputs are copied into the slot's own device buffers
 * on a host-to-device stream (so the copies overlap the kernels of the
 * other slot's round), the step runs on the handle's stream after them, and
 * out_tokens / out_n_accepted and the status word are copied back on a
 * device-to-host stream.  spec_verify_wait_host(h, slot) waits for that
 * round and returns its status (SV_OK, or the device status word, which it
 * then clears).  The host buffers of a submitted round must stay valid, and
 * its outputs unread, until the wait returns; a slot must be waited for
 * before it is submitted again.  The first submit allocates the two slots'
 * buffers, streams and events (later calls allocate nothing).  Arguments
 * and errors as spec_verify_run_host, and SV_ERR_ARG for a slot other than
 * 0 or 1, a busy slot (submit) or an idle one (wait). */
int spec_verify_submit_host(spec_verify_t *h, int slot, const void *hidden_host,
                            const void *W_lm, const int32_t *draft_tokens_host,
                            const float *q_logits_host, const float *uniforms_host,
                            float temperature, int32_t *out_tokens_host,
                            int32_t *out_n_accepted_host);
int spec_verify_wait_host(spec_verify_t *h, int slot);

/* Synchronises the handle's stream, then returns and clears the device
 * status word (SV_OK if no device-side error occurred since the last call),
 * or SV_ERR_CUDA if synchronisation failed. */
int spec_verify_status(spec_verify_t *h);

/* Replaces the stream that later calls are enqueued on. */
int spec_verify_set_stream(spec_verify_t *h, void *stream);

/* Copies the last run's fp32 logits [B*(K+1), V] (row b*(K+1)+i) to dst
 * (host or device, B*(K+1)*V floats).  Synchronises.  For tests. */
int spec_verify_debug_logits(spec_verify_t *h, float *dst);

/* Copies the last run's log-sum-exp normalisers (fp64) to dst (host or
 * device): B*(K+1) values of logits/T, then B*K values of q_logits/T.
 * Synchronises.  For tests; meaningful only when T > 0. */
int spec_verify_debug_lse(spec_verify_t *h, double *dst);

/* Upper bound, in nanoseconds, of every device-side wait (default 1e9).
 * A wait that runs out sets SV_ERR_TIMEOUT and the kernel returns early
 * after draining its own copies in flight.  0 makes the first wait that is
 * not already satisfied give up at once (used to test that path). */
int spec_verify_set_wait_limit(spec_verify_t *h, uint64_t limit_ns);

/* For tests of the timeout path: while enabled (enable != 0), every run's
 * decision/selection kernel first waits for a device flag that nothing
 * sets.  The wait gives up after the handle's wait limit
 * (spec_verify_set_wait_limit), the run reports SV_ERR_TIMEOUT through the
 * status word, and sequence 0 of that run is withdrawn (out_tokens and
 * out_n_accepted -1) when T > 0; the other sequences are verified as usual.
 * Nothing faults or hangs.  Returns SV_OK or SV_ERR_ARG (null handle). */
int spec_verify_debug_stall(spec_verify_t *h, int enable);

/* Kernel timing for the benchmark: while enabled, each run records CUDA
 * events on the handle's stream around the LM-head contraction kernel.
 * spec_verify_timing_read synchronises and returns the summed duration in
 * milliseconds and the number of timed launches since enabling. */
int spec_verify_timing(spec_verify_t *h, int enable);
int spec_verify_timing_read(spec_verify_t *h, double *total_ms,
                            int64_t *launches);

/* Number of kernel launches one spec_verify_run enqueues for temperature
 * T: the LM-head contraction and one fused decision / residual / selection
 * launch (2 for every T). */
int spec_verify_launches_per_run(spec_verify_t *h, float temperature);

/* Launch plan of the tensor-core contraction for a configuration: which
 * accumulation mode runs and how shared memory and tensor memory are laid
 * out.  Host arithmetic only (no CUDA call, no GPU needed); num_sms and
 * smem_optin describe the GPU (152 SMs and 232448 bytes of opt-in shared
 * memory per block on GB300).  For tests and for callers that want to know
 * what a shape will run.  Returns SV_OK, SV_ERR_ARG (null pointer, num_sms
 * < 1, dtype not SV_BF16 or SV_FP8) or SV_ERR_SHAPE (the shape create would
 * reject, or no plan with at least two stages fits smem_optin). */
typedef struct {
  int32_t npad;          /* columns one CTA multiplies (rows padded to 16)       */
  int32_t drain_cols;    /* drain mode: TMEM slot width (16, 32, 64); 0: direct  */
  int32_t half;          /* 1: the two CTAs of a pair split the columns          */
  int32_t kblock_elems;  /* elements of one 128-byte k block (64 bf16, 128 fp8)  */
  int32_t kblocks;       /* k blocks per row: ceil(d / kblock_elems)             */
  int32_t chunks;        /* k blocks per pipeline stage                          */
  int32_t stages;        /* pipeline stages in shared memory                     */
  int32_t stage_bytes;   /* bytes of one stage (multiple of 1024)                */
  int32_t smem_bytes;    /* dynamic shared memory per CTA                        */
  int32_t grid;          /* CTAs (persistent, at most one per SM)                */
  int32_t tmem_cols;     /* TMEM columns allocated per CTA                       */
  int32_t tmem_buffers;  /* direct mode: tiles held in TMEM at once (1 or 2)     */
  int32_t tmem_slots;    /* drain: ring slots; direct: accumulators per tile     */
} sv_plan_t;

int spec_verify_plan(const sv_config_t *cfg, int32_t num_sms, int32_t smem_optin,
                     sv_plan_t *out);

/* Static description of an error code. */
const char *spec_verify_strerror(int code);

/* Frees the handle and its workspace.  NULL is ignored. */
void spec_verify_destroy(spec_verify_t *h);

/* The same step as spec_verify_run for callers that cannot allocate device
 * memory when they call in -- a serving runtime that plans every device
 * buffer in advance and forbids cudaMalloc at run time (it can synchronise
 * the device and fragment a caching allocator), or a plugin host that only
 * passes input and output pointers.  No handle is needed and nothing is
 * allocated: the scratch lives in one fixed device array of 32 MiB inside
 * the library, which every GPU that loads the library holds until the
 * process exits.  (The pages describe no such mode; this is a property of
 * the library, not of the method.)
 *   cfg            shape, dtype (SV_BF16 or SV_FP32) and stream, as for
 *                  spec_verify_create
 *   other arguments as for spec_verify_run
 * The first call on a device looks up that device's copy of the array
 * (cudaGetSymbolAddress); make it before any stream capture.  Every call
 * reuses the same array and clears the counters it needs at its start, so
 * calls that may overlap on the GPU (different streams, or different host
 * threads on the same device) race and must be serialised by the caller.
 * The scratch of a call is about 4*R*V bytes of logits (R = B*(K+1)),
 * 8*(R + B*K)*ceil(V/32) of softmax partials, 1 KiB per column and
 * contraction CTA of stream-K split tiles (up to 152 CTAs, columns = R
 * rounded up to 16), 16*(R + B*K) per CTA of row statistics and small
 * tables: 5.1 MiB for V = 128256, d = 4096, B = 1, K = 4; 15.7 MiB for
 * d = 8192, B = 4, K = 4; 29.1 MiB for d = 4096, B = 8, K = 4.  B = 8,
 * K = 7 at V = 128256 (44.8 MiB) does not fit.
 * Errors (returned): as spec_verify_run, SV_ERR_SHAPE if the scratch for
 * this shape exceeds the array, SV_ERR_ARG if cfg->dtype is not SV_BF16
 * or SV_FP32.  Errors found on the device are not reported through a
 * status word: the affected sequences get out_n_accepted = -1 and
 * out_tokens = -1. */
int spec_verify_run_noalloc(const sv_config_t *cfg, const void *hidden, const void *W_lm,
                            const int32_t *draft_tokens, const float *q_logits,
                            const float *uniforms, float temperature, int32_t *out_tokens,
                            int32_t *out_n_accepted);

/* The step with truncated sampling: as spec_verify_run, with the target
 * distributions warped by (target_top_k, target_top_p) and the draft
 * distributions by (draft_top_k, draft_top_p) before the rule
 * ("Speculative Decoding: Two Models, One Voice", three remarks: warping by
 * temperature, top-k and top-p before forming p and q keeps the rule exact
 * for the warped target; "Speculative Decoding: The Algebra and the Proof",
 * "Where it breaks": p is the requested distribution after temperature and
 * truncation, q the distribution that generated the proposal, and the two
 * may use different settings).  Order: logits / T, then top-k, then top-p
 * on the renormalised top-k distribution.  Both cuts are by value, ties
 * kept: top-k keeps every token whose logit is at least the k-th largest
 * (top_k = 0 or >= V: no cut), top-p every token whose logit is at least
 * that of the first token, in descending order, at which the cumulative
 * probability reaches top_p (top_p = 1: no cut).  Membership is decided on
 * the fp32 logits the step computes; the cumulative masses that place a
 * top-p cut are summed in a fixed order (per-bin masses in fixed point
 * where a whole row is histogrammed), so repeated calls give the same
 * outputs bit for bit, as for spec_verify_run.  At T == 0 (greedy) the cuts change
 * nothing; with q_logits == NULL the draft settings are unused.  One more
 * launch (the cut of every truncated row) runs between the contraction and
 * the decision kernel.
 * Errors: as spec_verify_run, and SV_ERR_ARG for top_k < 0 or top_p outside
 * (0, 1]. */
int spec_verify_run_truncated(spec_verify_t *h, const void *hidden, const void *W_lm,
                              const int32_t *draft_tokens, const float *q_logits,
                              const float *uniforms, float temperature, int32_t target_top_k,
                              float target_top_p, int32_t draft_top_k, float draft_top_p,
                              int32_t *out_tokens, int32_t *out_n_accepted);

/* The step with an FP8 LM head, on a handle created with dtype SV_FP8
 * ("Speculative Decoding: The Algebra and the Proof", "Where it breaks":
 * native FP8 doubles both the arithmetic intensity and the peak, and halves
 * the bytes of the weight stream).  Values are FP8 E4M3 (sign, 4-bit
 * exponent of bias 7, 3-bit mantissa; largest finite 448) with one fp32
 * scale per hidden row and per vocabulary row:
 *   hidden8        device, E4M3 bytes [B, K+1, d] (d a multiple of 16)
 *   hidden_scale   device, fp32 [B, K+1]
 *   W8             device, E4M3 bytes [V, d]
 *   w_scale        device, fp32 [V]
 * The logit of row r and token v is hidden_scale[r] * w_scale[v] *
 * sum_k hidden8[r][k] * W8[v][k]; the contraction runs on the FP8 tensor
 * cores (tcgen05 kind::f8f6f4) with fp32 accumulation, and everything after
 * it is the same step on those logits.  Other arguments, outputs and errors
 * as spec_verify_run; SV_ERR_ARG if the handle is not SV_FP8 or a scale
 * pointer is NULL.  (spec_verify_run, spec_verify_run_host and the variants
 * return SV_ERR_ARG on an SV_FP8 handle: they carry no scales.) */
int spec_verify_run_fp8(spec_verify_t *h, const void *hidden8, const float *hidden_scale,
                        const void *W8, const float *w_scale, const int32_t *draft_tokens,
                        const float *q_logits, const float *uniforms, float temperature,
                        int32_t *out_tokens, int32_t *out_n_accepted);

/* Greedy tree verification ("Speculative Decoding: Guess Several Tokens,
 * Check Them in One Pass", "Tree attention": several draft branches verified
 * in one pass, the longest matching path accepted).  The handle's K is the
 * number of tree nodes N; hidden is [B, N+1, d] with row 0 scoring the
 * continuation of the last committed token (the root) and row 1 + j that of
 * node j (the tree-attention forward pass produces exactly these rows).
 *   tree_tokens    device, int32 [B, N]: node j's token, in [0, V)
 *   tree_parents   device, int32 [B, N]: node j's parent in [-1, j) (-1: the
 *                  root), so parents come before their children
 * A node matches when its parent matches (the root always does) and its
 * token is the argmax of its parent's row (ties to the smallest id).  The
 * round emits the tokens on the path to the deepest matched node (the
 * smallest index among equally deep ones), then the argmax of that node's
 * row; with no match, the argmax of row 0.  (The tie rule is this library's
 * reading.)
 *   out_tokens     device, int32 [B, N+1]: the path's tokens, the final
 *                  argmax, then -1
 *   out_nodes      device, int32 [B, N] or NULL: the path's node indices
 *                  (root first; for KV rollback), then -1
 *   out_n          device, int32 [B]: the path length; -1 for a sequence
 *                  with an invalid token or parent (status SV_ERR_TOKEN) or
 *                  non-finite logits
 * Errors: as spec_verify_run. */
int spec_verify_tree_greedy(spec_verify_t *h, const void *hidden, const void *W_lm,
                            const int32_t *tree_tokens, const int32_t *tree_parents,
                            int32_t *out_tokens, int32_t *out_nodes, int32_t *out_n);

/* ---------------------------------------------------------------------------
 * Prompt-lookup drafting ("Speculative Decoding: Guess Several Tokens, Check
 * Them in One Pass", "Drafts without a model"; "Speculative Decoding: Two
 * Models, One Voice", "No model at all"): propose the tokens that followed
 * an earlier occurrence of the last few context tokens.  For each sequence
 * b with context tokens[b * ld .. b * ld + lengths[b] - 1]:
 *   for n = n_max down to n_min, the pattern is the last n tokens; an
 *   occurrence starts at j with j + n <= lengths[b] - 1 (at least one token
 *   follows it) and equals the pattern token for token.  The first n with
 *   an occurrence wins, and of its occurrences the latest (largest j).
 * (Longest n first and the latest occurrence are this library's reading;
 * the pages leave both open.)
 *   tokens         device, int32 [B, ld] row-major contexts
 *   lengths        device, int32 [B]; a length outside [0, ld] counts as 0
 *   K              draft slots, 1..SV_MAX_K
 *   n_min, n_max   1 <= n_min <= n_max <= SV_NGRAM_MAX
 *   out_draft      device, int32 [B, K]: the up to K tokens following the
 *                  chosen occurrence, then -1 (ready for spec_verify_run
 *                  with q_logits == NULL)
 *   out_len        device, int32 [B]: the draft's length, 0 if no n matched
 *   stream         cudaStream_t (NULL: the default stream)
 * Asynchronous; allocates nothing; graph-capturable.  All pointers 4-byte
 * aligned.  Errors (returned): SV_ERR_ARG (null pointer, B < 1, ld < 1, K or
 * the n bounds out of range), SV_ERR_ALIGN, SV_ERR_ARCH (not compute
 * capability 10.3), SV_ERR_CUDA (launch failed). */
#define SV_NGRAM_MAX 16
int spec_ngram_draft(const int32_t *tokens, int64_t ld, const int32_t *lengths, int32_t B,
                     int32_t K, int32_t n_min, int32_t n_max, int32_t *out_draft,
                     int32_t *out_len, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* SPEC_VERIFY_H */
