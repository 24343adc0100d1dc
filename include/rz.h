/*
 * rz.h -- C ABI of the batch-invariant logprob + REINFORCE Zero loss library
 * for one NVIDIA GB300 (sm_103a).
 *
 * What it computes (sources are web pages on REINFORCE Zero, cited by title
 * and section):
 *   [RZ-page]  "REINFORCE Zero: Kernel Alignment Unlocks Stable Asynchronous
 *              RL with Importance Sampling", project page, section 02 "The
 *              mechanism", block "A minimal REINFORCE objective":
 *                L = -(1/B) sum_i (1/T_i) sum_t A_i pi(a_it|h_it)/mu_i(a_it|h_it),
 *              T_i = valid action tokens of response i, mu = the behaviour
 *              probability recorded at sampling time, gradient through the
 *              numerator pi only.
 *   [vLLM-zh]  "Zero Mismatch, Simple Async RL: REINFORCE Zero, DeepSeek-V4.1
 *              and Kimi K3.1" (todayforai rendering): section 3 (D3 = mean
 *              over all tokens of w - 1 - log w), section 4 items 1-3
 *              (aligned logprobs, unclipped token-level ratio, advantage =
 *              reward minus group mean), section 5 ("diff 0": bitwise-equal
 *              logprob of every sampled token in rollout and trainer).
 *
 * Conventions shared by every entry point:
 *   - Array arguments are DEVICE pointers owned by the caller; the library
 *     never frees or keeps them.  Scalars are written to device pointers.
 *   - The library allocates no device memory.  Scratch space is the caller's
 *     `ws` buffer of at least rz_workspace_size(...) bytes (256-byte aligned).
 *     One exception: rz_token_logprob_noalloc uses a 32 MiB array built into
 *     the library, which every GPU that loads the library holds for the life
 *     of the process (whether or not that entry point is called).
 *   - Calls are asynchronous on `stream` (NULL = legacy default stream) and
 *     never synchronise the host.  A return of RZ_OK means the work was
 *     enqueued; faults found on the device are reported through `err_flag`.
 *   - Layouts are row-major and contiguous.  bf16 arrays are raw 16-bit
 *     bfloat16 values (rz_bf16).  H, W, dH and logits must be 16-byte
 *     aligned; d must be a multiple of 8 (16-byte rows for the tensor-memory
 *     copy engine).
 *   - Sizes: 0 <= T < 2^31, 1 <= V <= 2^24, 8 <= d <= 65536, B >= 0.
 *   - Return value: RZ_OK or an RZ_ERR_* code; nothing is enqueued when an
 *     argument check fails.  RZ_ERR_CUDA (a launch or driver call failed)
 *     can come after some of the call's launches were enqueued: the
 *     outputs are then undefined.  rz_status_string() gives the text.
 *   - err_flag (nullable, device int32): device-side problems are OR-ed
 *     into it (RZ_DEVERR_*).  The caller zeroes it before the call and reads
 *     it afterwards.  No kernel ever traps.
 *   - Batch invariance: the logprob of a row depends only on that row's
 *     hidden state, its token and W -- never on T, on the other rows or on
 *     the row's position -- because the GEMM tile (128x256x64), the K order
 *     and the vocab split (a function of V only) are fixed.
 */
#ifndef RZ_H_
#define RZ_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define RZ_API __attribute__((visibility("default")))
#else
#define RZ_API
#endif

typedef uint16_t rz_bf16;                 /* raw bfloat16 bits */
typedef struct CUstream_st* rz_stream_t;  /* == cudaStream_t */

/* Return codes. */
#define RZ_OK               0
#define RZ_ERR_INVALID_ARG  1  /* null pointer, bad size, B % G != 0, ... */
#define RZ_ERR_UNSUPPORTED  2  /* alignment, d % 8, no sm_103a device */
#define RZ_ERR_WORKSPACE    3  /* ws == NULL or ws_bytes too small */
#define RZ_ERR_CUDA         4  /* a CUDA runtime/driver call failed */
#define RZ_ERR_TOO_LARGE    5  /* exceeds the built-in scratch of rz_token_logprob_noalloc */

/* Bits OR-ed into *err_flag by device code. */
#define RZ_DEVERR_TOKEN_RANGE  1  /* a token id outside [0, V) */
#define RZ_DEVERR_CU_SEQLENS   2  /* cu_seqlens not 0 = cu[0] <= ... <= cu[B] = T */
#define RZ_DEVERR_TIMEOUT      4  /* a pipeline wait gave up (kernel returned early) */
#define RZ_DEVERR_RANGE        8  /* a reference log-sum-exp too far from the row's (rz_loss_fwd_bwd_ref) */

/* Operation ids for rz_workspace_size(). */
#define RZ_OP_TOKEN_LOGPROB   0
#define RZ_OP_LOSS_FWD_BWD    1
#define RZ_OP_LOGITS_LOSS     2
#define RZ_OP_IS_LOSS         3
#define RZ_OP_SAMPLE          4
#define RZ_OP_SC_LOSS_FWD_BWD 5
#define RZ_OP_LOSS_FWD_BWD_REF 6  /* rz_loss_fwd_bwd_ref, and rz_loss_fwd_bwd_shard with ref_lse */

/*
 * Bytes of scratch the operation needs for these sizes (0 if none).  Pure
 * host function; arguments an operation does not use are ignored.  For
 * RZ_OP_TOKEN_LOGPROB and RZ_OP_SAMPLE with at most 64 rows (a decode-sized
 * batch; logits scratch at most 256 MB) the size includes the batch's fp32
 * logits, [T, V rounded up to 64]: with it the call spreads the LM-head GEMM
 * over every SM and folds the stored logits with the fused pass's own
 * operations.  Those two kernels are launched with programmatic stream
 * serialization: each may begin its set-up while the kernel ahead of it in
 * the stream finishes, and waits for that kernel before any memory access,
 * so stream order is kept.  A
 * workspace sized for any larger T serves a smaller batch too (without the
 * logits scratch the call keeps the fused pass); the results are the same
 * bits either way.
 */
RZ_API size_t rz_workspace_size(int op, int64_t T, int32_t d, int32_t V, int32_t B);

/* Static text for a return code (never NULL). */
RZ_API const char* rz_status_string(int status);

/*
 * Rollout side: record log mu of every sampled token [vLLM-zh s.4 item 2;
 * RZ-page s.02 "recorded behavior probability"].
 *   H       [T, d] bf16   hidden state that predicts token t
 *   W       [V, d] bf16   LM-head weight (the rollout's weights)
 *   tokens  [T] int32     sampled token ids
 *   logprob_out [T] fp32  log pi(a_t|h_t) = z_{t,a_t} - logsumexp_v z_tv,
 *                         z = H W^T (fp32 accumulation, temperature 1)
 *   lse_out [T] fp32      logsumexp_v z_tv (nullable); the reference that
 *                         rz_loss_fwd_bwd_ref takes for each row
 * Rows whose token is out of range get NaN and set RZ_DEVERR_TOKEN_RANGE.
 * Rows are processed in blocks of 38,912 (one GEMM launch each).  The learner
 * side (rz_loss_fwd_bwd, rz_loss_fwd_bwd_ref) runs this very computation -- the same tiles, K
 * order, vocab splits and log-sum-exp fold, only keeping more of it for its
 * backward pass -- so both sides agree bit for bit at equal weights
 * [vLLM-zh s.5 "diff 0"].
 */
RZ_API int rz_token_logprob(const rz_bf16* H, const rz_bf16* W, const int32_t* tokens,
                     int64_t T, int32_t d, int32_t V,
                     float* logprob_out, float* lse_out,
                     void* ws, size_t ws_bytes, int32_t* err_flag,
                     rz_stream_t stream);

/*
 * Rollout side with the sampling fused in: draws a_t ~ softmax(z_t),
 * z = H W^T at temperature 1, and records log mu(a_t) in the same pass over
 * the logits [vLLM-zh s.4 item 2: the rollout records the logprob of every
 * token it samples; the pages do not say how it samples].
 * Sampling rule (a reading, exact in law): a two-level weighted reservoir
 * over the row's vocabulary in ascending order, q_v = exp(z_tv - max z_t).
 * Inside each vocab split (the log-sum-exp's splits: whole 256-column
 * tiles, a function of V only) the 32-column chunks c come in order; chunk
 * c becomes the split's candidate when U1 R < Q, Q its sum of q and R the
 * running sum including it, and the token inside the chunk is the first
 * column, visited by class (column mod 4) then by column, at which the
 * running sum of q passes U2 Q.  The splits are taken in order the same
 * way with U3 against the running sum of their totals.  Every token is drawn
 * with probability exactly q_v / sum q.  U = ((x >> 9) + 1/2) 2^-23 for a
 * word x of Philox4x32-10 (Salmon et al., SC 2011) under key (seed low,
 * seed high): U1, U2 = words 0, 1 at counter (c, row_id low 32 bits,
 * row_id high 32 bits, 0); U3 = word 0 at counter (split, row_id low,
 * row_id high, 1).  row_ids [T] int64 (nullable: the row index t) makes a
 * row's sample depend only on its own id, hidden state and W -- never on
 * the batch it sits in.
 *   tokens_out [T] int32, logprob_out [T] fp32 (log mu of the sampled
 *   token), lse_out [T] fp32 (nullable).
 * logprob_out is bitwise equal to what rz_token_logprob (and the learner in
 * rz_loss_fwd_bwd) computes for the same H, W and the sampled tokens.
 * Workspace: rz_workspace_size(RZ_OP_SAMPLE, T, d, V, 0).
 */
RZ_API int rz_sample_logprob(const rz_bf16* H, const rz_bf16* W, const int64_t* row_ids,
                             int64_t T, int32_t d, int32_t V, uint64_t seed,
                             int32_t* tokens_out, float* logprob_out, float* lse_out,
                             void* ws, size_t ws_bytes, int32_t* err_flag,
                             rz_stream_t stream);

/*
 * Group-mean advantage [vLLM-zh s.4 item 3]: A_i = r_i - (1/G) sum_{j in g(i)} r_j,
 * groups are contiguous blocks of G responses.  rewards, adv_out: [B] fp32.
 * B % G != 0 -> RZ_ERR_INVALID_ARG.  No workspace.
 */
RZ_API int rz_group_advantage(const float* rewards, int32_t B, int32_t G,
                       float* adv_out, rz_stream_t stream);

/*
 * The importance-sampled loss on given logprobs [RZ-page s.02 objective]:
 *   w_t = exp(logpi_t - logmu_t) (never clipped)
 *   loss = -(1/B) sum_{i: T_i > 0} A_i (1/T_i) sum_{t in i} w_t
 *   d3   = (1/T) sum_t (w_t - 1 - log w_t)           [vLLM-zh s.3]
 *   coef_out[t] = A_i w_t / (B T_i) = -dloss/dlogpi_t (nullable)
 * cu_seqlens [B+1] int64 (response i owns tokens cu[i] .. cu[i+1]-1),
 * adv [B] fp32.  action_mask [T] uint8 (nullable = all tokens are action
 * tokens): "T_i counts valid action tokens" [RZ-page s.02] -- a token with
 * mask 0 (e.g. a tool output inside an agentic response) enters no sum:
 * T_i counts the valid tokens of response i, D3 averages over valid tokens,
 * coef is 0 for it.  Deterministic (fixed-order reductions).  No valid
 * token gives loss = d3 = 0.  Workspace: rz_workspace_size(RZ_OP_IS_LOSS, T,
 * 0, 0, B).
 */
RZ_API int rz_is_loss(const float* logpi, const float* logmu, const int64_t* cu_seqlens,
               const float* adv, const uint8_t* action_mask, int32_t B, int64_t T,
               float* loss_out, float* d3_out, float* coef_out,
               void* ws, size_t ws_bytes, int32_t* err_flag, rz_stream_t stream);

/*
 * D3 diagnostic alone [vLLM-zh s.3]: d3_out = (1/T) sum_t (w_t - 1 - log w_t),
 * w_t = exp(logpi_t - logmu_t); 0 for T = 0.  One fixed-order reduction, no
 * workspace.
 */
RZ_API int rz_d3(const float* logpi, const float* logmu, int64_t T, float* d3_out,
          rz_stream_t stream);

/*
 * Per-update importance-sampling diagnostics over the T sampled tokens
 * (d_t = logpi_t - logmu_t, w_t = e^{d_t}), one fixed-order reduction:
 *   stats_out[0] D3 = mean(w - 1 - log w)     [vLLM-zh s.3]; for tokens drawn
 *                from mu this is also the "k3" estimator of KL(mu || pi)
 *   stats_out[1] k1 = mean(-d), the plain estimator of KL(mu || pi)
 *   stats_out[2] k2 = mean(d^2 / 2)
 *   stats_out[3..6] mean w, max w, min w, max |d|
 * The pages plot a "sampled rollout-to-learner KL" without defining it
 * [RZ-page Figure 1]; k1 and k3 are the two readings offered.  stats_out is
 * 7 device floats; all zero for T = 0.  No workspace.
 */
RZ_API int rz_is_stats(const float* logpi, const float* logmu, int64_t T, float* stats_out,
                       rz_stream_t stream);

/*
 * Peak-to-median ratio max(x)/median(x) of a per-update series held in HOST
 * memory (the pages report it for D3 across updates: 1.50x with aligned
 * kernels vs 442.54x with standard kernels [vLLM-zh s.3 Figure 1]).  The
 * median of an even count is the mean of the two middle values.  Pure host
 * function; n >= 1.
 */
RZ_API int rz_peak_to_median(const float* series, int64_t n, double* ratio_out);

/*
 * Learner side: the fused logprob + REINFORCE Zero loss, forward and backward
 * [RZ-page s.02 objective and "differentiate through the numerator"].
 *   H [T,d] bf16, W [V,d] bf16, tokens [T] int32, logmu [T] fp32 (recorded by
 *   the rollout), cu_seqlens [B+1] int64, adv [B] fp32, action_mask [T] uint8
 *   (nullable; as in rz_is_loss: masked tokens get log pi but no loss and no
 *   gradient -- their dH rows are 0).
 * Outputs: loss_out, d3_out (fp32 scalars), logprob_out [T] fp32 (nullable),
 *   dH [T,d] bf16 = dz W, dW [V,d] fp32 = dz^T H (overwritten, not
 *   accumulated), with dz_tv = A_i w_t/(B T_i) (softmax_v(z_t) - [v = a_t]).
 * log pi is produced by exactly the rollout computation (bitwise equal to
 * rz_token_logprob on the same H, W, tokens).  Rows are processed in chunks
 * of up to 38,912: the forward pass keeps, for the chunk only, its softmax
 * terms exp(z - running max) in fp16 (the [T, V] logits are never stored or
 * recomputed), from which dz is formed in place; dW is reduced over the
 * chunks in a fixed order, so results are run-to-run deterministic.
 * Workspace: rz_workspace_size(RZ_OP_LOSS_FWD_BWD, T, d, V, B).
 */
RZ_API int rz_loss_fwd_bwd(const rz_bf16* H, const rz_bf16* W, const int32_t* tokens,
                    const float* logmu, const int64_t* cu_seqlens, const float* adv,
                    const uint8_t* action_mask,
                    int32_t B, int64_t T, int32_t d, int32_t V,
                    float* loss_out, float* d3_out, float* logprob_out,
                    rz_bf16* dH, float* dW,
                    void* ws, size_t ws_bytes, int32_t* err_flag,
                    rz_stream_t stream);

/*
 * rz_loss_fwd_bwd with the rollout's log-sum-exp of every row as a reference
 * (no counterpart on the pages; the same outputs by another route).
 *   ref_lse [T] fp32: a per-row reference R_t, normally lse_out of the
 *   rz_token_logprob / rz_sample_logprob call that recorded logmu (the
 *   rollout computes it in the same pass).
 * The forward pass keeps the chunk's softmax terms against R_t instead of a
 * running maximum: e'_tv = exp(z_tv - R_t) in bf16, so the backward pass
 * forms dz_tv = sigma_t e'_tv with one factor per row, sigma_t =
 * c_t exp(R_t - lse_t).  dH applies sigma_t to its rows.  dW multiplies e'
 * with the rows of H scaled by sigma_t.  The sampled column's term is set so
 * that its dz is c_t expm1(log pi_t).  This removes the dz pass over the
 * chunk's terms (4 bytes per logit of HBM traffic) and the running maxima.
 * Results equal rz_loss_fwd_bwd's within the rounding of one more bf16 step
 * (H scaled by sigma): log pi, the loss and D3 bit for bit, dH and dW to
 * ~1e-3 relative.
 * Range: needs max_v z_tv - R_t <= 80 and |lse_t - R_t| <= 60 (nats) for
 * every row.  That holds whenever the learner's weights are those of the
 * rollout or a few updates from them; otherwise RZ_DEVERR_RANGE is set and
 * that row's gradients are undefined (use rz_loss_fwd_bwd).
 * Everything else (arguments, layouts, errors, determinism) as
 * rz_loss_fwd_bwd.  Workspace: rz_workspace_size(RZ_OP_LOSS_FWD_BWD_REF, T,
 * d, V, B) (no running maxima; the chunk's rows of H scaled, [rows, d] bf16).
 */
RZ_API int rz_loss_fwd_bwd_ref(const rz_bf16* H, const rz_bf16* W, const int32_t* tokens,
                               const float* logmu, const float* ref_lse,
                               const int64_t* cu_seqlens, const float* adv,
                               const uint8_t* action_mask,
                               int32_t B, int64_t T, int32_t d, int32_t V,
                               float* loss_out, float* d3_out, float* logprob_out,
                               rz_bf16* dH, float* dW,
                               void* ws, size_t ws_bytes, int32_t* err_flag,
                               rz_stream_t stream);

/*
 * One shard of a data-parallel learner step [RZ-page s.04: the method runs on
 * 16 GPUs].  The loss averages tokens within a response and responses within
 * the batch (s.02 objective), so the batch is split over ranks by whole
 * responses: this call gets B of the batch's B_total responses (contiguous;
 * cu_seqlens, adv, tokens, ... are the shard's own) and normalises by B_total:
 *   c_t = A_i w_t / (B_total T_i),
 *   loss_out = -(1/B_total) sum_{i in shard} A_i (1/T_i) sum_t w_t  (the shard's
 *              share: the batch's loss is the sum over shards),
 *   d3_out   = the mean of w - 1 - log w over the shard's valid tokens (the
 *              batch's D3 is the token-weighted mean over shards),
 *   dH       = the shard's rows of the batch's dH, bitwise what one
 *              rz_loss_fwd_bwd call over the whole batch gives for them,
 *   dW       = the shard's partial; the batch's dW is the sum of the partials
 *              over shards (add them in a fixed order, e.g. with
 *              rz_sum_partials, for a result independent of the backend).
 * ref_lse (nullable): as in rz_loss_fwd_bwd_ref (the shard's rows).
 * Everything else (arguments, layouts, errors) as rz_loss_fwd_bwd; workspace
 * RZ_OP_LOSS_FWD_BWD (RZ_OP_LOSS_FWD_BWD_REF with ref_lse) with the shard's
 * B.  B_total = B is rz_loss_fwd_bwd (rz_loss_fwd_bwd_ref).  B_total < B
 * returns RZ_ERR_INVALID_ARG.
 */
RZ_API int rz_loss_fwd_bwd_shard(const rz_bf16* H, const rz_bf16* W, const int32_t* tokens,
                                 const float* logmu, const float* ref_lse,
                                 const int64_t* cu_seqlens, const float* adv,
                                 const uint8_t* action_mask,
                                 int32_t B, int32_t B_total, int64_t T, int32_t d, int32_t V,
                                 float* loss_out, float* d3_out, float* logprob_out,
                                 rz_bf16* dH, float* dW,
                                 void* ws, size_t ws_bytes, int32_t* err_flag,
                                 rz_stream_t stream);

/*
 * The exchange step of the data-parallel learner: the fixed-order sum of n
 * partials.  parts [n_parts, count] fp32 (device, row r = rank r's partial,
 * e.g. gathered by a collective), out [count] fp32 (device; may not overlap
 * parts):  out[i] = ((parts[0][i] + parts[1][i]) + parts[2][i]) + ..., added
 * in row order in fp32, so every rank that sums the same gathered partials
 * gets the same bits, independent of any collective's own reduction order.
 * No workspace.  n_parts >= 1.
 */
RZ_API int rz_sum_partials(const float* parts, int32_t n_parts, int64_t count, float* out,
                           rz_stream_t stream);

/*
 * Comparison estimator: Score Centering (SC), the learner step WITHOUT
 * importance weights ["REINFORCE Zero" project page, "The full IS
 * correction", items 02-03: the update on sampler tokens carries the drift
 * E_q[A] E_q[s]; centring the sampler score keeps g_SC = Cov_q(A, s)].
 * Per-token reading (the page gives only the expectation): each sampled
 * token's score is centred by the batch mean of the per-response averaged
 * scores, with the token weights of the IS loss, i.e.
 *   L_SC = -(1/B) sum_i ((A_i - Abar)/T_i) sum_{t in i} log pi_t,
 *   Abar = mean of A_i over the responses with at least one valid token,
 *   dz_tv = (A_i - Abar)/(B T_i) (softmax_v(z_t) - [v = a_t]).
 * A constant added to every advantage changes nothing; for advantages that
 * already sum to zero it is the IS update at w = 1 (plain REINFORCE).
 * Arguments, layouts, ownership, errors and determinism as rz_loss_fwd_bwd,
 * without log mu and D3.  log pi (logprob_out, nullable) is bitwise the
 * rollout's.  Workspace: rz_workspace_size(RZ_OP_SC_LOSS_FWD_BWD, T, d, V, B)
 * (the same size as RZ_OP_LOSS_FWD_BWD).
 */
RZ_API int rz_sc_loss_fwd_bwd(const rz_bf16* H, const rz_bf16* W, const int32_t* tokens,
                       const int64_t* cu_seqlens, const float* adv,
                       const uint8_t* action_mask,
                       int32_t B, int64_t T, int32_t d, int32_t V,
                       float* loss_out, float* logprob_out,
                       rz_bf16* dH, float* dW,
                       void* ws, size_t ws_bytes, int32_t* err_flag,
                       rz_stream_t stream);

/*
 * Given-logits variant: the same loss on precomputed logits, with the
 * log-softmax, gather, ratio and dlogits done in place.
 *   logits_inout [T, V] bf16: read as logits, overwritten with
 *   dz_tv = A_i w_t/(B T_i) (softmax_v - onehot) in bf16.  V % 8 == 0.
 *   logprob_out [T] fp32 (required), loss_out, d3_out, action_mask as in
 *   rz_is_loss (masked rows are overwritten with zeros).
 * Workspace: rz_workspace_size(RZ_OP_LOGITS_LOSS, T, 0, V, B).
 */
RZ_API int rz_logits_loss_fwd_bwd(rz_bf16* logits_inout, const int32_t* tokens,
                           const float* logmu, const int64_t* cu_seqlens,
                           const float* adv, const uint8_t* action_mask,
                           int32_t B, int64_t T, int32_t V,
                           float* loss_out, float* d3_out, float* logprob_out,
                           void* ws, size_t ws_bytes, int32_t* err_flag,
                           rz_stream_t stream);

/*
 * LM-head logits z = H W^T as fp32 [T, V] (row-major), from the same
 * tensor-core tile, K order and accumulation as the logprob path: every
 * value equals the z the logprob kernels reduce.  No workspace.
 */
RZ_API int rz_lmhead_logits(const rz_bf16* H, const rz_bf16* W, int64_t T, int32_t d,
                     int32_t V, float* logits_out, int32_t* err_flag,
                     rz_stream_t stream);

/*
 * rz_token_logprob without a caller workspace, for callers that cannot
 * allocate device memory: a sampler hook inside an inference engine whose
 * memory pool is reserved up front, a plug-in whose host owns every
 * allocation, or code running between captured graph segments.  The pages
 * have no counterpart for this entry point; it is a deployment convenience.
 *
 * Same arguments and results as rz_token_logprob (bitwise the same output:
 * it runs the same kernels with the same launch shape), minus ws/ws_bytes.
 * Scratch is a fixed array inside the library of rz_noalloc_scratch_bytes()
 * bytes (32 MiB) on every GPU that loads the library, held until the
 * process exits.  It needs T * (8 * S + 4) bytes plus padding, S = the
 * number of vocab splits (at most 64; 60 at V = 151936) -- about 69,000 rows
 * at V = 151936; larger T returns RZ_ERR_TOO_LARGE and enqueues nothing.
 *   - It never calls cudaMalloc/cudaFree or any allocating library routine.
 *   - The first call on a device (with that device current) looks up the
 *     array's device address; make that first call before any stream capture.
 *     The address is then kept for the life of the process: after a
 *     cudaDeviceReset() of a device, do not call this entry point on it again
 *     (the kept address would name memory of the destroyed context).
 *   - All calls on a device share the array, and it keeps the last call's
 *     contents (nothing in it needs zeroing).  Calls that overlap on the GPU
 *     (different streams, or threads without ordering) race on it and give
 *     undefined results: serialise them.
 */
RZ_API int rz_token_logprob_noalloc(const rz_bf16* H, const rz_bf16* W, const int32_t* tokens,
                                    int64_t T, int32_t d, int32_t V,
                                    float* logprob_out, float* lse_out,
                                    int32_t* err_flag, rz_stream_t stream);

/*
 * Failure-detection self-test (no counterpart on the pages): launches one
 * warp that waits, with the library's bounded pipeline wait, on a barrier
 * nothing ever completes.  After limit_us microseconds (1 .. 2,000,000) the
 * wait gives up, RZ_DEVERR_TIMEOUT is OR-ed into *err_flag (device int32,
 * required) and *done_out (device int32, nullable) is set to 2 (1 would mean
 * the barrier completed).  The GPU is neither faulted nor hung, and the
 * context stays usable.
 */
RZ_API int rz_selftest_wait_timeout(int32_t* err_flag, int32_t* done_out, uint32_t limit_us,
                                    rz_stream_t stream);

/*
 * Debug build only (compiled with -DRZ_CHECKS; no counterpart on the pages):
 * the kernels then check their computed indices (task coordinates, split
 * states, running-max and dz offsets, tensor-store coordinates, output
 * tiles) against the sizes of the call; a failed check skips the access,
 * counts itself and records its site (a small integer naming the check).
 * This call waits for the device, writes the number of failed checks since
 * the last read and the site of the first, and clears both.  The normal
 * build returns RZ_ERR_UNSUPPORTED (it has no checks).
 */
RZ_API int rz_debug_check_failures(uint32_t* count_out, int32_t* first_site_out);

/* Size in bytes of the built-in scratch used by rz_token_logprob_noalloc. */
RZ_API size_t rz_noalloc_scratch_bytes(void);

/*
 * Launch-class timing, a measurement aid (no counterpart on the pages).
 * After rz_profile_begin(), every entry point brackets each class of its
 * launches with a pair of CUDA events recorded on the stream it launches
 * on, so one call's device time can be split by kernel without a profiler.
 * rz_profile_end() waits (host-blocking) for the recorded events, writes
 * the milliseconds of each class to ms_out[RZ_PROF_*] and the number of
 * kernels launched in it to launches_out[RZ_PROF_*] (nullable), releases
 * the events and stops recording.  n_classes >= RZ_PROF_CLASSES.
 *   - Off by default: nothing is recorded and nothing is synchronised.
 *   - The events sit between launches on one stream, so the classes add up
 *     to the calls' device time (plus event gaps of a few microseconds).
 *   - Calls on a stream that is being captured into a CUDA graph are not
 *     recorded.  The recording is process-wide (a mutex guards it).
 * Returns RZ_ERR_INVALID_ARG for a null ms_out or a short array, RZ_ERR_CUDA
 * if an event could not be read (the other classes are still filled).
 */
#define RZ_PROF_LOGPROB_GEMM 0  /* rollout logprob GEMM; fused-sampling GEMM */
#define RZ_PROF_KEEP_GEMM    1  /* learner logits + log-sum-exp GEMM keeping the terms */
#define RZ_PROF_MERGE        2  /* split merges: log pi, lse, c_t, sampled token */
#define RZ_PROF_DZ           3  /* dz pass over the kept terms; on the reference route
                                   the scaling of H's rows by sigma_t */
#define RZ_PROF_DH_GEMM      4  /* dH = dz W */
#define RZ_PROF_DW_GEMM      5  /* dW = dz^T H, accumulated over chunks */
#define RZ_PROF_LOGITS_ROWS  6  /* given-logits row kernel */
#define RZ_PROF_SMALL        7  /* advantages, response factors, loss, D3, statistics */
#define RZ_PROF_CLASSES      8
RZ_API int rz_profile_begin(void);
RZ_API int rz_profile_end(float* ms_out, int32_t* launches_out, int32_t n_classes);

#ifdef __cplusplus
}
#endif

#endif /* RZ_H_ */
