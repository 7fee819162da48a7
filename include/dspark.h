/*
 * dspark.h — C ABI of the DSpark draft-head round on one GB300 (sm_103a).
 *
 * One round of DSpark semi-autoregressive speculative decoding after the
 * parallel backbone, for R requests and gamma draft positions:
 *   a1  base logits through the shared, frozen LM head     (dspark_lm_head)
 *   a2  Markov-head bias B(x_{k-1}, .) = W1[x_{k-1}] W2 added to the logits
 *   a3  sampling of x_k (greedy argmax or Gumbel-max)
 *   a4  confidence head c_k = sigmoid(w^T [h_k; W1[x_{k-1}]] / T_k)
 *                                                         (dspark_markov_draft)
 *   a5  prefix survival products a_{r,j} = prod_{i<=j} c_{r,i}
 *   a6  global descending sort of all R*gamma candidates
 *   a7  Theta = tau * SPS(B) search -> per-request verify lengths
 *                                                         (dspark_schedule)
 *   a8  verification of the admitted prefixes against target logits
 *                                                         (dspark_verify)
 *
 * Sources (page title, section):
 *   "DSpark 深度解读" (zhichai.net) §二 设计一 (Markov head, W1: V x r, W2: r x V),
 *   §二 设计二 (confidence head, Sequential Temperature Scaling, hardware-aware
 *   prefix scheduler with Theta = tau * SPS(B)), §三 挑战1/挑战2 (asynchronous
 *   top-K admission, unconstrained search over stepped SPS curves);
 *   "DSpark整体架构" (10100.com) Fig. 1 (anchor -> draft -> schedule -> verify,
 *   corrected token G*) and the two-stage semi-autoregressive description
 *   (anchor is the first prediction position);
 *   DeepSeek-V4-Pro-0813 DSpark article (demingchina.com) config table
 *   (block size 5, Markov rank 512, fp32 confidence).
 *
 * Conventions for every entry point
 *   - All tensor pointers are DEVICE pointers unless stated otherwise, owned by
 *     the caller, row-major and densely packed.  The library allocates nothing
 *     and keeps no state between calls except the sticky device status word.
 *   - "bf16" = IEEE bfloat16 stored as uint16; "f32" = float; tokens are int32.
 *   - Every call is asynchronous on `stream` (a cudaStream_t; NULL = legacy
 *     default stream).  Inputs are never modified.
 *   - Return value: DSPARK_OK, or a host-detected error (bad argument, short
 *     table, short workspace, CUDA launch failure) in which case nothing was
 *     launched.  Problems found on the device (a token id >= V, a length >
 *     gamma, a bounded wait that ran out) set the sticky device status word,
 *     read with dspark_device_status().
 *   - Random draws use Philox4x32-10 keyed by (seed) with counter
 *     (v >> 2, position, request, stream), word v & 3, u = ((w >> 9) + 0.5) 2^-23;
 *     streams: 0 draft Gumbel, 1 accept uniform, 2 residual Gumbel, 3 bonus Gumbel;
 *     residual trial q: 16 + 8q id Gumbel, 20 + 8q block Gumbel, 21 + 8q
 *     super-block Gumbel, 17 + 8q uniform.
 *
 * Departures from the planned boundary (draft / schedule / verify / status):
 *   - W2 enters once, through dspark_pack_w2, as W2t [V, r]; every later call
 *     takes W2t.  Both operands of the bias contraction are then K-major, as the
 *     tensor-core path needs, and no call pays a transpose of r*V*2 bytes.
 *   - The draft writes no draft-logit rows (pd_logits [R, gamma, V]): the loop
 *     keeps the logits on chip.  It returns log p_d(x_k) and lse_k per position,
 *     which is all the acceptance test needs; on the one rejected row of a
 *     request, dspark_verify rebuilds p_d from the draft's own operands
 *     (base_logits, W1, W2t, lse_d).  Writing and re-reading the rows would add
 *     2 * R*gamma*V*2 bytes of traffic per round (662 MB at R=256, gamma=5,
 *     V=129280).
 *   - Theta is returned as f64: it is computed from an exact fixed-point S_K,
 *     and f64 carries that value without a second rounding.
 *   - The status call is dspark_device_status(stream, clear): it reads the one
 *     word every kernel of the library writes, and clearing is the caller's
 *     choice.
 *   - The LM head is also a call of its own (dspark_lm_head), and the base
 *     logits are a caller-owned buffer, because verify reads them again.
 */
#ifndef DSPARK_H
#define DSPARK_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st *dspark_stream_t; /* identical to cudaStream_t */

typedef struct dspark_dims {
  int32_t R;     /* requests in the batch, >= 1                                   */
  int32_t gamma; /* draft positions per request, 1..32                             */
  int32_t V;     /* vocabulary size, multiple of 8                                 */
  int32_t r;     /* Markov rank, multiple of 64                                    */
  int32_t d;     /* backbone hidden size, multiple of 64                           */
} dspark_dims;

enum {
  DSPARK_OK = 0,
  DSPARK_ERR_ARG = 1,        /* null pointer, bad shape or mode                     */
  DSPARK_ERR_SPS_SHORT = 2,  /* SPS table shorter than R * (gamma + 1)              */
  DSPARK_ERR_CUDA = 3,       /* a CUDA call or launch failed                        */
  DSPARK_ERR_WORKSPACE = 4,  /* workspace missing or smaller than required         */
  DSPARK_ERR_TOKEN = 5,      /* device status: token id outside [0, V)              */
  DSPARK_ERR_LENGTH = 6,     /* device status: verify length outside [0, gamma]     */
  DSPARK_ERR_TIMEOUT = 7,    /* device status: a bounded device-side wait ran out   */
  DSPARK_ERR_TOO_LARGE = 8   /* problem exceeds a fixed library limit (static scratch,
                                sampling verify with V > 13107200)                 */
};

enum {
  DSPARK_SCHED_UNCONSTRAINED = 0, /* K = argmax_K Theta(K) over every budget        */
  DSPARK_SCHED_BREAK = 1,         /* admit in sorted order while Theta increases    */
  DSPARK_SCHED_FIXED_K = 2,       /* admit the top min(k_fixed, R*gamma) candidates */
  DSPARK_SCHED_ASYNC = 3          /* dspark_schedule_async only: top-K with K from the
                                     unconstrained search of two rounds earlier      */
};

/* a1 — base draft logits, "DSpark 深度解读" §二 (parallel backbone -> base logits
 * through the LM head shared with, and frozen from, the target).
 *   h           bf16 [R*gamma, d]   backbone hidden states, row m = r*gamma + k-1
 *   W_lm        bf16 [V, d]         LM head (each vocabulary row d-contiguous)
 *   base_logits bf16 [R*gamma, V]   out: l0[m, v] = sum_i h[m, i] W_lm[v, i],
 *                                   fp32 accumulation, rounded to bf16
 * h, W_lm and base_logits must be 16-byte aligned. */
int dspark_lm_head(const dspark_dims *dims, const void *h, const void *W_lm,
                   void *base_logits, dspark_stream_t stream);

/* Layout preparation for the Markov factor W2 (done once per weight load).
 *   W2   bf16 [r, V]   as the pages define it (B = W1[x] W2)
 *   W2t  bf16 [V, r]   out: W2t[v, i] = W2[i, v]  (rank-contiguous rows)
 * Every later call takes W2t (a departure from taking W2 itself: the bias
 * contraction's operands must both be K-major for TMA and tcgen05). */
int dspark_pack_w2(const dspark_dims *dims, const void *W2, void *W2t, dspark_stream_t stream);

/* Workspace bytes dspark_markov_draft / dspark_draft need for `dims`. */
size_t dspark_markov_workspace_bytes(const dspark_dims *dims);

/* a2-a4 — the gamma-step sequential (Markov) head with the confidence head,
 * "DSpark 深度解读" §二 设计一 and 设计二; "DSpark整体架构" stage two.
 * For k = 1..gamma, with x_0 = anchor:
 *   l_k     = l0_k + W1[x_{k-1}] W2                   (f32, never written out)
 *   x_k     = argmax_v l_k[v]                          tau == 0 (ties: lowest v)
 *           = a draw from softmax(l_k / tau)                             tau > 0
 *             by two-level Gumbel-max: the vocabulary is cut into blocks of 64
 *             ids; block b* = argmax_b log sum_{v in b} e^{l_k[v]/tau}
 *             + Gumbel(seed; r, k, b, stream 4), then x_k = argmax over v in b*
 *             of l_k[v]/tau + Gumbel(seed; r, k, v, stream 0); ties to the
 *             lowest id at both levels
 *   c_k     = sigmoid((w_h . h_k + w_e . W1[x_{k-1}]) / T_k),  w_conf = [w_h; w_e]
 *   lse_k   = logsumexp_v(l_k[v] / tau)      (tau > 0 only; 0 when greedy)
 *   logp_k  = l_k[x_k] / tau - lse_k          (tau > 0 only; 0 when greedy)
 *   base_logits bf16 [R*gamma, V]   from dspark_lm_head
 *   h           bf16 [R*gamma, d]
 *   anchor      int32 [R]           anchor token per request (in [0, V))
 *   W1          bf16 [V, r]         Markov embedding table
 *   W2t         bf16 [V, r]         from dspark_pack_w2
 *   w_conf      bf16 [d + r]        confidence head weight
 *   T           f32  [gamma]        per-position STS temperatures (> 0)
 *   tokens      int32 [R, gamma]    out
 *   conf        f32  [R, gamma]     out
 *   logp_d, lse_d f32 [R, gamma]    out, may be NULL (needed by sampling verify);
 *               they replace draft-logit rows as the draft's output for verify:
 *               the logits are never written to memory
 *   workspace   device buffer of dspark_markov_workspace_bytes(dims) bytes,
 *               256-byte aligned; contents on entry are ignored. */
int dspark_markov_draft(const dspark_dims *dims, const void *base_logits, const void *h,
                        const int32_t *anchor, const void *W1, const void *W2t,
                        const void *w_conf, const float *T, float tau, uint64_t seed,
                        int32_t *tokens, float *conf, float *logp_d, float *lse_d,
                        void *workspace, size_t workspace_bytes, dspark_stream_t stream);

/* Workspace bytes dspark_rnn_draft needs for `dims`. */
size_t dspark_rnn_workspace_bytes(const dspark_dims *dims);

/* a2-a4 with the RNN head variant instead of the Markov head, "DSpark整体架构"
 * stage two (the pages describe it in words only: a block-internal recurrent
 * state, gated update over the history, the previous token's embedding and
 * the backbone hidden state).  Read as, with s_0 = 0 and x_0 = anchor:
 *   pre_k = W_rec [s_{k-1}; W1[x_{k-1}]] + W_hid h_k          (2r values)
 *   s_k   = (1 - g) s_{k-1} + g tanh(c), g = sigmoid(pre_k[0:r]), c = pre_k[r:2r]
 *   l_k   = l0_k + bf16(s_k) W2      (s_{k-1} also enters W_rec in bf16)
 * and then exactly as dspark_markov_draft (sampling, confidence head on
 * [h_k; W1[x_{k-1}]], outputs).
 *   W_rec  bf16 [2r, 2r]  columns [state | embedding] of the gate (rows 0..r-1)
 *                         and candidate (rows r..2r-1) pre-activations
 *   W_hid  bf16 [2r, d]   their hidden-state columns
 * Every other argument is dspark_markov_draft's; the workspace is
 * dspark_rnn_workspace_bytes(dims) bytes, 256-byte aligned. */
int dspark_rnn_draft(const dspark_dims *dims, const void *base_logits, const void *h,
                     const int32_t *anchor, const void *W1, const void *W2t, const void *W_rec,
                     const void *W_hid, const void *w_conf, const float *T, float tau,
                     uint64_t seed, int32_t *tokens, float *conf, float *logp_d, float *lse_d,
                     void *workspace, size_t workspace_bytes, dspark_stream_t stream);

/* Fused single-contraction draft step, a measured variant of a1 + a2
 * ("DSpark 深度解读" §二 设计一: the draft logits are the shared LM head's plus
 * the Markov bias).  Per step k one contraction
 *   l_k = [h_k; W1[x_{k-1}]] . [W_lm; W2t]^T    (f32 accumulation, no bf16 base)
 * replaces the round's LM head plus the bias pass: the base logits never reach
 * HBM, but W_lm is streamed gamma times.  Sampling, the confidence head and
 * the outputs are dspark_markov_draft's.
 *   W_cat  bf16 [V, d + r]  row v = [W_lm[v] | W2t[v]], made by dspark_pack_fused
 * The workspace is dspark_fused_workspace_bytes(dims) bytes, 256-byte aligned. */
size_t dspark_fused_workspace_bytes(const dspark_dims *dims);
int dspark_pack_fused(const dspark_dims *dims, const void *W_lm, const void *W2t, void *W_cat,
                      dspark_stream_t stream);
int dspark_fused_draft(const dspark_dims *dims, const void *h, const int32_t *anchor,
                       const void *W_cat, const void *W1, const void *w_conf, const float *T,
                       float tau, uint64_t seed, int32_t *tokens, float *conf, float *logp_d,
                       float *lse_d, void *workspace, size_t workspace_bytes,
                       dspark_stream_t stream);

/* a1-a4 in one call: dspark_lm_head into `base_logits`, then dspark_markov_draft. */
int dspark_draft(const dspark_dims *dims, const void *h, const int32_t *anchor,
                 const void *W_lm, const void *W1, const void *W2t, const void *w_conf,
                 const float *T, float tau, uint64_t seed, void *base_logits,
                 int32_t *tokens, float *conf, float *logp_d, float *lse_d,
                 void *workspace, size_t workspace_bytes, dspark_stream_t stream);

/* a5-a7 — hardware-aware prefix scheduler, "DSpark 深度解读" §二 设计二 and §三.
 *   conf   f32 [R, gamma]    confidences c_{r,j}
 *   sps    f32 [n_sps]       profiled steps/s, sps[B-1] = SPS(B); n_sps >= R*(gamma+1)
 *   mode   DSPARK_SCHED_*;   k_fixed used by FIXED_K only
 *   len    int32 [R]         out: admitted draft length l_r per request
 *   K_out  int32 [1]         out: total admitted candidates K = sum l_r
 *   theta_out f64 [1]        out: Theta(K) = (R + S_K) * SPS(R + K)
 *   a_out  f32 [R, gamma]    out, may be NULL: survival products (f32, left to right)
 *   order_out int32 [R*gamma] out, may be NULL: candidate ids r*gamma + j-1 sorted by
 *                            a descending, ties by id ascending
 * S_K sums the sorted products in 2^-48 units (each rounded to nearest, halves up;
 * exact integer sums); Theta(K) = f64(R + S_K) * (f64(SPS) * 2^-48).  The argmax
 * takes ties to the smallest K; a NaN Theta never wins.  R*gamma <= 16384.
 * theta_out is f64 rather than f32, so the exact fixed-point S_K reaches the
 * caller without a second rounding. */
int dspark_schedule(const float *conf, int32_t R, int32_t gamma, const float *sps,
                    int32_t n_sps, int32_t mode, int32_t k_fixed, int32_t *len,
                    int32_t *K_out, double *theta_out, float *a_out, int32_t *order_out,
                    dspark_stream_t stream);

/* a5-a7, asynchronous form — "DSpark 深度解读" §三 挑战1 (Zero-Overhead
 * Scheduling): round t-2's confidences predict round t's capacity K; round t
 * sorts its own candidates by their actual survival products and admits the
 * top K.  Admission is then fixed before round t's tokens exist, so it stays
 * lossless, and every round launches with the same arguments (CUDA graphs).
 *   k_ring int32 [3] device state, read and written by the call:
 *          {K slot 0, K slot 1, cursor}.  The call admits K_t = k_ring[cursor]
 *          (clamped to [0, R*gamma]), then stores this round's unconstrained
 *          argmax_K Theta(K) in that slot and flips the cursor (0 <-> 1).
 *          Initialise it to {K for round 0, K for round 1, 0}.
 *   K_out  int32 [1]  out: the admitted K_t;  theta_out f64 [1]: Theta(K_t).
 * Every other argument is that of dspark_schedule.  Calls sharing a ring must
 * run in stream order. */
int dspark_schedule_async(const float *conf, int32_t R, int32_t gamma, const float *sps,
                          int32_t n_sps, int32_t *k_ring, int32_t *len, int32_t *K_out,
                          double *theta_out, float *a_out, int32_t *order_out,
                          dspark_stream_t stream);

/* Confidence logits before the temperature, for calibration:
 *   z[r, j] = w_h . h[r, j] + w_e . W1[x_{j-1}]   (x_0 = anchor; w_conf = [w_h; w_e])
 * "DSpark 深度解读" §二 设计二 Confidence Head.  h, anchor, tokens, W1, w_conf as
 * in dspark_markov_draft (tokens: that call's output); z f32 [R, gamma] out. */
int dspark_conf_logits(const dspark_dims *dims, const void *h, const int32_t *anchor,
                       const int32_t *tokens, const void *W1, const void *w_conf, float *z,
                       dspark_stream_t stream);

/* Workspace bytes dspark_sts_fit needs (0 when the sizes are invalid). */
size_t dspark_sts_workspace_bytes(int32_t N, int32_t gamma, int32_t n_grid, int32_t n_bins);

/* Sequential Temperature Scaling, "DSpark 深度解读" §二 设计二 (STS 校准): the
 * per-position temperatures T_j, fitted left to right on N held-out rounds.
 * For j = 1..gamma, every T of T_grid is scored by the expected calibration
 * error of the prefix survival a_j = a_{j-1} * sigmoid(z_j / T) (f32, left to
 * right, T_1..T_{j-1} already fixed) against the label accepted >= j:
 *   ECE = sum over n_bins equal-width bins b of |sum_{n in b}(label_n - a_n)| / N,
 *   bin of a = min(floor(a * n_bins), n_bins - 1) in f32,
 * and the least (the first on ties) is kept.
 *   z        f32 [N, gamma]   logits from dspark_conf_logits
 *   accepted int32 [N]        drafts accepted by dspark_verify with len = gamma
 *   T_grid   f32 [n_grid]     candidate temperatures (> 0; device memory)
 *   n_bins   1..64
 *   T_out    f32 [gamma] out;  ece_out f64 [gamma] out: ECE at the chosen T_j
 *   workspace device buffer of dspark_sts_workspace_bytes(...) bytes, 256-byte
 *            aligned.  A grid value <= 0 sets DSPARK_ERR_ARG in the status word. */
int dspark_sts_fit(const float *z, const int32_t *accepted, int32_t N, int32_t gamma,
                   const float *T_grid, int32_t n_grid, int32_t n_bins, float *T_out,
                   double *ece_out, void *workspace, size_t workspace_bytes,
                   dspark_stream_t stream);

/* Workspace bytes dspark_verify needs for `dims`. */
size_t dspark_verify_workspace_bytes(const dspark_dims *dims);

/* a8 — verification, "DSpark整体架构" Fig. 1 (accept a run, emit a corrected
 * token G*) with the standard speculative-sampling rule:
 *   tau == 0: accept x_j iff x_j == argmax_v t_j[v]; the first mismatch row's
 *             argmax (or row l_r + 1 when all match) is the bonus token.
 *   tau > 0:  accept x_j iff u * p_d(x_j) < p_t(x_j), u = U(seed; r, j, stream 1);
 *             on the first rejection sample norm(max(0, p_t - p_d)) at that row;
 *             when all l_r are accepted sample target row l_r + 1 (streams 3
 *             and 7).  p = softmax(logits / tau).  Each draw is the two-level
 *             Gumbel-max of dspark_markov_draft (entry stream s, block stream
 *             s + 4).  The residual is drawn by rejection from p_t: trial
 *             q = 0, 1, .. proposes y ~ p_t by Gumbel-max in three levels
 *             (super-blocks of 1024 ids on stream 21 + 8q, their 64-id blocks
 *             on 20 + 8q, ids on 16 + 8q) and keeps it iff
 *             u_q < 1 - p_d(y) / p_t(y), u_q = U(stream 17 + 8q);
 *             the first kept proposal is the token.  After 64 unkept trials the
 *             residual is formed over the whole row and drawn on streams 2 and
 *             6; a residual that is empty in floating point is replaced by p_t
 *             itself (streams 2 and 6).
 *             Returns DSPARK_ERR_TOO_LARGE when tau > 0 and V > 13107200.
 *   anchor   int32 [R];  tokens int32 [R, gamma];  len int32 [R] (0..gamma)
 *   base_logits bf16 [R*gamma, V], W1 bf16 [V, r], W2t bf16 [V, r]: the draft's
 *            operands, used to rebuild p_d on the rejected row (tau > 0 only), in
 *            place of draft-logit rows that the draft does not write
 *   lse_d, logp_d f32 [R, gamma] from dspark_markov_draft (tau > 0 only)
 *   target   bf16 [R, gamma + 1, V]  target logits; row j-1 scores position j
 *   accepted int32 [R] out: accepted draft tokens n_r (0..l_r)
 *   bonus    int32 [R] out: corrected / bonus token emitted after them
 *   workspace device buffer of dspark_verify_workspace_bytes(dims) bytes.
 * Pointers only read when tau > 0 may be NULL when tau == 0. */
int dspark_verify(const dspark_dims *dims, const int32_t *anchor, const int32_t *tokens,
                  const int32_t *len, const void *base_logits, const void *W1,
                  const void *W2t, const float *lse_d, const float *logp_d,
                  const void *target, float tau, uint64_t seed, int32_t *accepted,
                  int32_t *bonus, void *workspace, size_t workspace_bytes,
                  dspark_stream_t stream);

/* After a sampling dspark_verify on `stream` (and with its workspace): how many
 * requests were rejected at some position (their corrected token came from the
 * residual) and how many of those kept none of their 64 rejection trials, so
 * that the residual was formed over the whole row (one W2t pass for all of
 * them).  rejected, explicit_rows: host int32 out.  Copies two device counters
 * and synchronises the stream.  Returns DSPARK_ERR_WORKSPACE for a workspace
 * shorter than dspark_verify_workspace_bytes(dims). */
int dspark_verify_residual_rows(const dspark_dims *dims, const void *workspace,
                                size_t workspace_bytes, int32_t *rejected,
                                int32_t *explicit_rows, dspark_stream_t stream);

/* Failure detection self-test (no fault is involved).  Every device-side wait
 * of the library is bounded in time; on expiry the kernel records
 * DSPARK_ERR_TIMEOUT in the device status word and returns, and the context
 * stays usable.  This call runs that path: one CTA waits, with the library's
 * own bounded wait capped at limit_ns (1 ns .. 2 s), on an mbarrier that
 * nothing arrives on.  Afterwards dspark_device_status reports
 * DSPARK_ERR_TIMEOUT.  Returns DSPARK_ERR_ARG for a limit outside that range. */
int dspark_selftest_wait_timeout(uint64_t limit_ns, dspark_stream_t stream);

/* Bytes of scratch the library keeps inside itself for dspark_markov_draft_static. */
#define DSPARK_STATIC_SCRATCH_BYTES ((size_t)16 << 20)

/* dspark_markov_draft without a caller-provided workspace.  No counterpart on
 * the method's pages: it exists for callers that cannot allocate device
 * memory, such as a plugin interface that hands the library only its input
 * and output tensors with no allocator, or a serving loop whose memory planner
 * forbids allocations once it has started.  The scratch lives in one
 * file-scope device array of DSPARK_STATIC_SCRATCH_BYTES (16 MiB) that every
 * GPU loading the library holds until the process exits; this call itself
 * allocates nothing.
 *   Arguments, outputs and results are those of dspark_markov_draft.
 *   Returns DSPARK_ERR_TOO_LARGE (nothing launched) when
 *   dspark_markov_workspace_bytes(dims) > DSPARK_STATIC_SCRATCH_BYTES; the V4
 *   shape (R=256, gamma=5, V=129280, r=512) needs about 8.6 MB.
 *   The first call on a device looks up the array's device address
 *   (cudaGetSymbolAddress) with that device current; make that first call
 *   before any stream capture.  The address is kept until the process exits,
 *   so a device reset (cudaDeviceReset) followed by further calls is not
 *   supported.
 *   Every call shares the one array: calls whose work overlaps on the GPU
 *   (other streams, other host threads) race and must be serialised by the
 *   caller.  Nothing in the array needs to start at zero. */
int dspark_markov_draft_static(const dspark_dims *dims, const void *base_logits, const void *h,
                               const int32_t *anchor, const void *W1, const void *W2t,
                               const void *w_conf, const float *T, float tau, uint64_t seed,
                               int32_t *tokens, float *conf, float *logp_d, float *lse_d,
                               dspark_stream_t stream);

/* Synchronises `stream`, returns the sticky device status word (DSPARK_OK or a
 * DSPARK_ERR_* code) and clears it when clear != 0.  (Planned as
 * dspark_last_device_status(stream); the clear flag lets a caller keep the word
 * across several reads.) */
int dspark_device_status(dspark_stream_t stream, int clear);

/* Human-readable name of a return / status code (static string). */
const char *dspark_error_string(int code);

/* Number of kernels this library has launched in this process. */
uint64_t dspark_launch_count(void);

#ifdef __cplusplus
}
#endif

#endif /* DSPARK_H */
