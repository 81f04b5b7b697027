/*
 * dspark.h — C ABI of the DSpark per-step hot path on one GPU (sm_103a).
 *
 * Three calls make one decode round's data-parallel work:
 *   dspark_draft_sample  Markov-head draft sampler + confidence head
 *   dspark_schedule      Sequential Temperature Scaling + hardware-aware prefix
 *                        scheduler + flattened verify batch with marker tensor
 *   dspark_verify        lossless rejection-sampling verification
 *
 * Sources (page titles; the section on each page is named at each call):
 *   [DSpark]      "DSpark: Confidence-Scheduled Speculative Decoding with
 *                 Semi-Autoregressive Generation" (papercache.org summary)
 *   [MTP Survey]  "大模型推理 MTP 算法 Survey" (backyes.github.io)
 *
 * Conventions shared by every call
 * --------------------------------
 * - Every pointer in an args struct is a DEVICE pointer unless its comment says
 *   "host".  The caller owns every buffer; the library never allocates,
 *   frees or keeps a pointer after the call returns.
 * - Arrays are dense, row-major, with the shapes given in brackets.  Base
 *   pointers of the large arrays (U, W1, W2, h, w, target_logits, pd_rows) must
 *   be 16-byte aligned.
 * - `stream` is a cudaStream_t passed as void* (NULL = legacy default stream).
 *   Calls only enqueue work on it and return; they never synchronise, except
 *   dspark_read_error.
 * - Argument errors return DSPARK_INVALID_ARG / DSPARK_UNSUPPORTED before any
 *   work is enqueued.  A launch failure returns DSPARK_CUDA_ERROR.  Errors
 *   found by a kernel while it runs (a token id outside [0, V), a bounded wait
 *   that gave up) are written to the workspace error word and read back with
 *   dspark_read_error.  Nothing aborts, exits or prints.
 * - Inputs are read-only.  No state survives a call except the workspace error
 *   word.  Random draws use Philox4x32-10 (Salmon et al., SC'11) with
 *   key = (seed mod 2^32, seed >> 32) and counter = (req_id, position, draw, 0),
 *   u = (out0 >> 8) * 2^-24; draw 0 = draft sample, 1 = accept test,
 *   2 = residual, 3 = bonus.  Results therefore depend on (seed, req_id,
 *   position) only, not on a request's slot in the batch.
 * - Temperature T_r per request: T_r > 0 samples from softmax(logits / T_r);
 *   anything else (0, negative, NaN) is greedy: argmax with ties to the lowest
 *   token id.  Logits must be finite.
 */
#ifndef DSPARK_H
#define DSPARK_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define DSPARK_API __attribute__((visibility("default")))
#else
#define DSPARK_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  DSPARK_OK = 0,
  DSPARK_INVALID_ARG = 1,   /* null pointer, bad size, misaligned pointer      */
  DSPARK_UNSUPPORTED = 2,   /* size beyond a limit, unknown dtype, no sm_103a  */
  DSPARK_CUDA_ERROR = 3,    /* a CUDA call or launch failed                     */
  DSPARK_TIMEOUT = 4,       /* a kernel's bounded wait gave up (error word)     */
  DSPARK_BAD_INPUT = 5      /* a kernel met an out-of-range token id (error word) */
} dspark_status;

typedef enum { DSPARK_BF16 = 0, DSPARK_F32 = 1 } dspark_dtype;

typedef enum {
  DSPARK_SCHED_OFF = 0,        /* verify every draft token: l_r = gamma            */
  DSPARK_SCHED_GREEDY = 1,     /* Algorithm 1 with the early stop                  */
  DSPARK_SCHED_ASYNC_TOPK = 2  /* production variant: capacity from earlier
                                  confidences, top-K of the current candidates    */
} dspark_sched_mode;

/* Limits checked by every call. */
#define DSPARK_MAX_GAMMA 32
#define DSPARK_MAX_RANK 1024
#define DSPARK_MAX_SCHED_KEYS 65536 /* B * gamma for dspark_schedule */
#define DSPARK_MAX_VOCAB 2097152    /* V for every call */

/* Problem sizes.  dtype applies to U, W1, W2, h, w and target_logits; every
 * output probability / confidence is fp32. */
typedef struct {
  int32_t B;      /* requests in the batch, >= 0 (0 = nothing to do)        */
  int32_t gamma;  /* draft block size, 1..DSPARK_MAX_GAMMA                   */
  int32_t V;      /* vocabulary size, 1..DSPARK_MAX_VOCAB                    */
  int32_t r;      /* Markov rank, 0..DSPARK_MAX_RANK (0 = no head, DFlash)    */
  int32_t H;      /* backbone hidden size, >= 0                              */
  int32_t dtype;  /* dspark_dtype                                            */
} dspark_dims;

/* ---------------------------------------------------------------------------
 * Workspace
 * ---------------------------------------------------------------------------
 * dspark_workspace_size: bytes of device scratch one set of dims needs for all
 * three calls (they use disjoint regions, so the three calls may share one
 * workspace while they run in order on one stream).  The caller allocates it
 * (any 256-byte-aligned device buffer) and must call dspark_workspace_init
 * once before first use.  Returns DSPARK_INVALID_ARG for a null pointer or
 * invalid dims. */
DSPARK_API dspark_status dspark_workspace_size(const dspark_dims* dims, size_t* bytes);

/* dspark_workspace_init: clears the workspace error word (enqueued on stream). */
DSPARK_API dspark_status dspark_workspace_init(void* workspace, size_t workspace_bytes, void* stream);

/* dspark_read_error: synchronises `stream`, copies the workspace error word to
 * *code_host (0 = none, else a dspark_status value) and *detail_host (the
 * offending value, e.g. the bad token id; may be NULL), then clears the word.
 * Returns DSPARK_CUDA_ERROR if the copy fails. */
DSPARK_API dspark_status dspark_read_error(void* workspace, int32_t* code_host, int32_t* detail_host, void* stream);

/* ---------------------------------------------------------------------------
 * dspark_draft_sample
 * ---------------------------------------------------------------------------
 * [DSpark] 方法细节, "序列阶段的依赖注入" and "马尔可夫头（Markov head）的实现":
 * for k = 1..gamma, left to right,
 *     l_k(v)  = U_k(v) + W1[x_{k-1}] . W2[:, v]          (x_0 = anchor)
 *     p_d^k   = softmax(l_k / T_r)                          (one-hot if greedy)
 *     x_k     = inverse-CDF draw from p_d^k in token-id order, u from draw 0
 *               at position k (greedy: argmax of l_k)
 * [DSpark] 方法细节, "置信度头的设计":
 *     z_k = w_h . h_k + w_e . W1[x_{k-1}],  c_k = sigmoid(z_k),  w = [w_h; w_e].
 * [DSpark] 方法细节, "并行阶段的局限与设计": the anchor is the first predicted
 * position, so U has gamma rows per request.
 * Inputs  U [B, gamma, V], W1 [V, r], W2 [r, V], h [B, gamma, H], w [H + r]
 *         (all dims.dtype); anchor [B] i32 in [0, V); temp [B] f32;
 *         req_id [B] u32; seed.  W1/W2 may be NULL when r = 0; h/w may be
 *         NULL when H + r = 0.
 * Outputs tokens [B, gamma] i32; pd_rows [B, gamma, V] f32 (the exact
 *         probability row each token was drawn from); pd_tok [B, gamma] f32
 *         (= pd_rows at the drawn token, bit for bit); conf_logit and conf
 *         [B, gamma] f32.
 * An anchor outside [0, V) is replaced by 0 and reported as DSPARK_BAD_INPUT
 * through the error word.
 *
 * pd_stat [B, gamma, 2] f32 (optional): each drawn row's max m and sum S of
 * 2^(y - m) (y = l_k log2(e) / T), so that p_d(v) = 2^(y(v) - m) / S can be
 * recomputed (dspark_verify's rejection residual).  pd_rows may be NULL (the
 * p_d-row-free mode): then pd_stat is required, the Markov head only, and
 * the call needs the fused tensor-core path (bf16, r in {64, 128, 192, 256},
 * V and H multiples of 8, sm_103), else DSPARK_UNSUPPORTED; p_d(x_k) still
 * comes back in pd_tok.
 *
 * head = DSPARK_HEAD_RNN ([DSpark] 方法细节, "RNN头的实现", the optional head)
 * replaces the row W1[x_{k-1}] of the bias product by e_k = tanh(W_o z_k),
 * z_k = [s_{k-1}; W1[x_{k-1}]; h_k] in R^{2r+H}, with the recurrent state
 *     s_k = g * s_{k-1} + (1 - g) * tanh(W_c z_k),  g = sigmoid(W_g z_k),  s_0 = 0.
 * W_rnn [3r, 2r + H] (dims.dtype) holds the rows of W_g, then W_c, then W_o.
 * The confidence head is unchanged.  s_k is fp32; e_k enters the bias product
 * in dims.dtype (rounded to nearest from fp32).  bf16 tensor-core shapes run
 * the tensor-core kernels (with p_d rows, the recurrent step inside the fused
 * draft kernel); fp32 and other shapes run the CUDA-core bias product (fp32
 * FMA).  It needs r >= 1; head = DSPARK_HEAD_MARKOV (0) ignores W_rnn. */
typedef enum { DSPARK_HEAD_MARKOV = 0, DSPARK_HEAD_RNN = 1 } dspark_head;

typedef struct {
  dspark_dims dims;
  const void* U;
  const void* W1;
  const void* W2;
  const void* h;
  const void* w;
  const int32_t* anchor;
  const float* temp;
  const uint32_t* req_id;
  uint64_t seed;
  int32_t* tokens;
  float* pd_rows;
  float* pd_tok;
  float* conf_logit;
  float* conf;
  const void* W_rnn;
  int32_t head;
  float* pd_stat;
} dspark_draft_args;

DSPARK_API dspark_status dspark_draft_sample(const dspark_draft_args* args, void* workspace,
                                  size_t workspace_bytes, void* stream);

/* ---------------------------------------------------------------------------
 * dspark_schedule
 * ---------------------------------------------------------------------------
 * [DSpark] 方法细节, "事后校准（Post-hoc Calibration）": per-position temperature
 * scaling of the confidence, read as c'_{r,k} = sigmoid(z_{r,k} / tau_k); this
 * library evaluates the sigmoid in fp64 and rounds it to fp32.
 * [DSpark] 方法细节, "硬件感知前缀调度器" / "贪心求解与因果性保证", Algorithm 1:
 *     a_{r,j} = c'_{r,1} ... c'_{r,j}   (fp32, left to right)
 *     E = {(r, j): a_{r,j} > 0} sorted by a descending (ties: r, then j asc.)
 *     Theta_0 = B SPS[B];  Theta_i = (B + a_(1) + ... + a_(i)) SPS[B + i]  (fp64)
 *     admit while Theta_i > Theta_{i-1}; stop at the first Theta_i <= Theta_{i-1}
 *     l_r = number of admitted (r, .) candidates
 * [DSpark] 补充细节, "高吞吐量与低延迟推理": the kept prefixes are flattened
 * into one batch with a marker tensor.  Layout (this library's reading):
 * request-major, position ascending; row offsets[r] + j holds the anchor for
 * j = 0 and draft token x_j for j = 1..l_r; mark_req/mark_pos give (r, j).
 * Inputs  conf_logit [B, gamma] f32 (z from dspark_draft_sample); sts_temp
 *         [gamma] f32 (> 0); sps [B (1 + gamma) + 1] f64 engine steps/s indexed
 *         by total verify tokens (may be NULL when mode = OFF); anchor [B];
 *         tokens [B, gamma]; mode.
 * Outputs ell [B]; offsets [B + 1]; flat_tok, mark_req, mark_pos
 *         [B (1 + gamma)] (rows past N_v = offsets[B] are set to -1);
 *         n_verify [1] (= N_v); theta_best [1] f64 (Theta of the kept set;
 *         0 when mode = OFF); optional n_verify_host (pinned HOST i32, written
 *         by a stream-ordered copy) and surv [B, gamma] f32 (the a_{r,j}).
 * B * gamma must not exceed DSPARK_MAX_SCHED_KEYS.
 *
 * Mode DSPARK_SCHED_ASYNC_TOPK ([DSpark] 补充细节, "生产环境中的硬件感知前缀
 * 调度器"): the scheduler runs one step behind the draft.  conf_logit_prev
 * [B, gamma] f32 holds the confidence logits of two steps earlier, mapped by the
 * caller onto this batch's requests; their survival products, sorted as above,
 * give the capacity K = the number of admissions of the best prefix of that path
 * (the first maximum of Theta_i over i = 0 .. n_prev: a global search, no early
 * stop).  This step's candidates are sorted as above and the first min(K, n)
 * are admitted; theta_best is Theta of that admission with the current
 * survivals.  K depends only on the earlier step, which is what keeps the
 * search lossless.  Needs sps and conf_logit_prev; supported while the
 * schedule fits one CTA's shared memory (B rounded up to a power of two times
 * gamma rounded up to a power of two at most 8192 slots), else
 * DSPARK_UNSUPPORTED. */
typedef struct {
  int32_t B;
  int32_t gamma;
  int32_t mode;
  const float* conf_logit;
  const float* sts_temp;
  const double* sps;
  const int32_t* anchor;
  const int32_t* tokens;
  int32_t* ell;
  int32_t* offsets;
  int32_t* flat_tok;
  int32_t* mark_req;
  int32_t* mark_pos;
  int32_t* n_verify;
  int32_t* n_verify_host;
  double* theta_best;
  float* surv;
  const float* conf_logit_prev;  /* mode DSPARK_SCHED_ASYNC_TOPK only; may be NULL otherwise */
} dspark_sched_args;

DSPARK_API dspark_status dspark_schedule(const dspark_sched_args* args, void* workspace,
                              size_t workspace_bytes, void* stream);

/* ---------------------------------------------------------------------------
 * dspark_draft_and_schedule
 * ---------------------------------------------------------------------------
 * dspark_draft_sample(draft) followed by dspark_schedule(sched) on the same
 * stream, with the same results bit for bit, in one call that may overlap the
 * two.  The schedule needs only the confidences and the tokens, which are
 * final once the last position is drawn; the draft then still writes that
 * position's p_d rows.  When the draft runs a fused-sweep tensor-core kernel
 * (the 128-row form or the small-batch form) with p_d rows, the scheduler
 * (one CTA, which then also calibrates the keys that dspark_schedule
 * calibrates on many SMs above 2048 candidates) starts by programmatic
 * dependent launch while that sweep runs: on an SM the draft grid leaves
 * idle, or, when the grid fills every SM, on the SM of one draft CTA that
 * leaves the last sweep to the others.  Other shapes (the row-free mode, the two-pass
 * and CUDA-core paths) run the two calls one after the other.
 * Arguments: as for the two calls, one workspace for both (sized for the
 * draft's dims); sched->B and sched->gamma must equal draft->dims, and
 * sched->conf_logit, sched->tokens and sched->anchor must be the draft's
 * conf_logit, tokens and anchor pointers, else DSPARK_INVALID_ARG.  Every
 * argument check of both calls happens before anything is enqueued. */
DSPARK_API dspark_status dspark_draft_and_schedule(const dspark_draft_args* draft, const dspark_sched_args* sched,
                                                   void* workspace, size_t workspace_bytes, void* stream);

/* ---------------------------------------------------------------------------
 * dspark_schedule_noalloc
 * ---------------------------------------------------------------------------
 * The pages have no counterpart to this entry point: it is a library
 * convenience.  It computes exactly what dspark_schedule computes (same kernel,
 * same outputs, bit for bit) without a caller-provided workspace, for callers
 * that cannot allocate device memory.  Two kinds of caller are meant: code
 * embedded in a host process whose device memory is entirely owned by that
 * host's own pool allocator (a plug-in of a serving engine that reserves the
 * HBM for its KV cache up front, so an extension has no allocator and no
 * budget of its own to draw a workspace from), and latency-critical decode
 * loops that must not call cudaMalloc / cudaFree because those calls can
 * synchronise the device and stall the loop.
 *
 * Scratch: a fixed 1 MiB array compiled into the library (4 x 65536 32-bit
 * entries).  Every GPU on which the library's device code is loaded holds its
 * own copy until the process exits.  This call performs no cudaMalloc,
 * cudaFree or other allocating call.
 * Limit: B * gamma <= DSPARK_MAX_SCHED_KEYS (65536); larger batches return
 * DSPARK_UNSUPPORTED before anything is enqueued.  Other argument errors are
 * those of dspark_schedule.
 * Set-up: every call looks up the array's device address in the context that
 * is current (cudaGetSymbolAddress, which allocates nothing), so the address
 * stays right across a device reset or a caller-made driver-API context.  The
 * first call in a context can load the library's device code there: make
 * the first call on each device, with that device current, before any stream
 * capture begins.  A failed lookup or launch returns DSPARK_CUDA_ERROR and is
 * recorded for dspark_last_cuda_error like the other entry points' errors.
 * Sharing: every call on a device uses the same array, which keeps whatever
 * the last call left in it.  The kernel overwrites every entry it reads, so
 * nothing needs clearing between calls, but two calls whose kernels overlap on
 * the same GPU (for instance on two streams without an ordering between them)
 * race on the array and give undefined results: order them on one stream or
 * with events. */
DSPARK_API dspark_status dspark_schedule_noalloc(const dspark_sched_args* args, void* stream);

/* ---------------------------------------------------------------------------
 * dspark_pack_rows
 * ---------------------------------------------------------------------------
 * [DSpark] 补充细节, "高吞吐量与低延迟推理" (flattened prefixes + marker tensor;
 * the SGLang notes pack ragged requests into a compact buffer): gathers the
 * verify batch.  Row i of dst is row (mark_req[i], mark_pos[i]) of src
 * [R, rows_per_request, V] (dtype) for i < *n_rows, where n_rows is a device
 * count (dspark_schedule's n_verify); rows of dst past the count are not
 * written.  src may be device memory or pinned host memory the GPU addresses
 * directly (only the kept rows then cross the host link).  mark_req,
 * mark_pos, n_rows are device arrays ([max_rows] each, one count); dst is
 * [max_rows, V] device memory; max_rows bounds the count (B * (gamma + 1) for
 * a dspark_schedule batch) and sizes the launch.  A marker outside the source
 * skips its row and is reported in the error word of `workspace` (any dspark
 * workspace; NULL: not reported) as DSPARK_BAD_INPUT, detail = the row. */
typedef struct {
  int32_t V;
  int32_t dtype;
  int32_t rows_per_request;
  int32_t max_rows;
  int64_t n_src_rows;
  const void* src;
  const int32_t* mark_req;
  const int32_t* mark_pos;
  const int32_t* n_rows;
  void* dst;
} dspark_pack_args;

DSPARK_API dspark_status dspark_pack_rows(const dspark_pack_args* args, void* workspace, void* stream);

/* ---------------------------------------------------------------------------
 * dspark_verify
 * ---------------------------------------------------------------------------
 * [DSpark] 背景知识与设计原则, "投机解码的延迟建模": x_k is accepted with
 * probability min(1, p_t^k(x_k) / p_d^k(x_k)), left to right; the first
 * rejection discards the rest.  Implemented as u p_d(x_k) < p_t(x_k) with u
 * from draw 1 at position k.
 * [MTP Survey] §2.2 "拒绝采样": at the first rejection a correction is drawn
 * from norm(max(0, p_t^k - p_d^k)) (draw 2 at position k; if that mass is 0 in
 * fp32, from p_t^k); when all l_r tokens are accepted the bonus is drawn from
 * p_t^{l+1} (draw 3 at position l + 1); greedy requests accept iff
 * x_k = argmax p_t^k and emit that argmax as the correction or bonus.
 * p_t^j = softmax(target_logits[offsets[r] + j - 1] / T_r).
 * Inputs  target_logits [>= offsets[B], V] (dims.dtype), the flattened rows of
 *         dspark_schedule's layout; offsets [B + 1]; ell [B]; tokens [B, gamma];
 *         pd_rows [B, gamma, V]; pd_tok [B, gamma]; temp [B]; req_id [B]; seed.
 * Outputs n_accept [B]; out_tok [B, gamma + 1] (the accepted tokens, then the
 *         correction or bonus, then -1); n_out [B] = n_accept + 1.
 * Cap-accept ([MTP Survey] §8, the SGLang notes' third verify mode: the full
 * block is verified, only the scheduled window is committed): when
 * commit_cap [B] (device, 0..gamma) is not NULL, n_out = min(n_accept,
 * commit_cap) + 1 tokens are committed and out_tok holds -1 after them; when
 * n_accept > commit_cap the last committed token is the accepted draft token
 * x_{commit_cap + 1}.  n_accept stays the count the full verification
 * accepted (the observation).  Pass ell = gamma rows per request for the
 * full block.  A window outside 0..gamma is clamped and reported in the
 * workspace error word (DSPARK_BAD_INPUT, detail = request).
 * residual_mode = DSPARK_RESIDUAL_REJECTION samples the residual by rejection
 * from p_t instead (trial t proposes v ~ p_t with draw 2 and Philox counter
 * word 3 = t, and accepts iff u p_t(v) < p_t(v) - p_d(v) with u from draw 4;
 * after DSPARK_RESIDUAL_TRIALS rejected proposals the residual is drawn by
 * inverse CDF with draw 2, trial DSPARK_RESIDUAL_TRIALS).  It reads no p_d
 * row: p_d(v) is recomputed at the proposed tokens of the Markov head from
 * U [B, gamma, V], W1 [V, r], W2 [r, V] (dims.dtype, dims.r >= 1), anchor [B]
 * and pd_stat [B, gamma, 2] (each draft row's max and sum, written by
 * dspark_draft_sample); pd_rows may then be NULL.
 * Only dims.B, gamma, V, dtype (and r in the rejection mode) are read. */
#define DSPARK_RESIDUAL_INVERSE_CDF 0
#define DSPARK_RESIDUAL_REJECTION 1
#define DSPARK_RESIDUAL_TRIALS 256
typedef struct {
  dspark_dims dims;
  const void* target_logits;
  const int32_t* offsets;
  const int32_t* ell;
  const int32_t* tokens;
  const float* pd_rows;
  const float* pd_tok;
  const float* temp;
  const uint32_t* req_id;
  uint64_t seed;
  int32_t* n_accept;
  int32_t* out_tok;
  int32_t* n_out;
  const int32_t* commit_cap;
  int32_t residual_mode;
  const void* U;
  const void* W1;
  const void* W2;
  const int32_t* anchor;
  const float* pd_stat;
} dspark_verify_args;

DSPARK_API dspark_status dspark_verify(const dspark_verify_args* args, void* workspace,
                            size_t workspace_bytes, void* stream);

/* ---------------------------------------------------------------------------
 * dspark_sts_fit
 * ---------------------------------------------------------------------------
 * [DSpark] 方法细节, "事后校准（Post-hoc Calibration）" (also the MTP survey's
 * §4.2.3 on STS): the per-position temperatures of Sequential Temperature
 * Scaling are fitted on held-out draft blocks left to right.  At position k a
 * 1-D grid search over the candidates picks the one whose calibrated
 * cumulative product P_k = c'_1 ... c'_k (c'_i = fp32(sigmoid(z_i / tau_i)),
 * fp32 products as in dspark_schedule) has the smallest expected calibration
 * error, positions before k held at their chosen temperatures.
 *   ECE = (1/N) sum_m |sum_{n in bin m} (y_n - P_k,n)|, with n_bins equal-width
 *   bins on [0, 1] (bin floor(P n_bins), P = 1 in the last) and y_n = 1 when
 *   accept_len[n] >= k.
 * Ties go to the first candidate; N = 0 gives ECE 0 and the first candidate.
 * Inputs  conf_logit [N, gamma] f32 (the confidence head's logits of each
 *         held-out block); accept_len [N] i32 in 0..gamma (draft tokens of the
 *         block accepted by a verification of the full block); grid [n_grid]
 *         f32 candidate temperatures, finite and > 0.
 * Outputs sts_temp [gamma] f32 (the fitted temperatures, ready for
 *         dspark_sched_args.sts_temp); grid_index [gamma] i32 (may be NULL);
 *         ece [gamma, n_grid] f64, the ECE of every candidate at every position.
 * The ECE sums are exact in 2^-40 fixed point: every ECE is within 2^-41 of
 * its exact value for these fp32 products.  accept_len outside 0..gamma or a
 * grid value that is not finite and positive is reported in the workspace
 * error word (DSPARK_BAD_INPUT, detail = the block or candidate index); the
 * outputs are then unspecified.  All pointers are device pointers; every
 * output is written on the stream.  The workspace (size from
 * dspark_sts_fit_workspace_size, 256-byte aligned, header zeroed once by
 * dspark_workspace_init) is separate from the step workspace. */
#define DSPARK_STS_MAX_SAMPLES 8388607 /* N < 2^23: the fixed-point sums fit in 63 bits */
#define DSPARK_STS_MAX_TABLE 16384     /* n_bins * max(n_grid, 128) */

typedef struct {
  int32_t N;
  int32_t gamma;
  int32_t n_grid;
  int32_t n_bins;
  const float* conf_logit;
  const int32_t* accept_len;
  const float* grid;
  float* sts_temp;
  int32_t* grid_index;
  double* ece;
} dspark_sts_fit_args;

DSPARK_API dspark_status dspark_sts_fit_workspace_size(int32_t N, int32_t gamma, int32_t n_grid, int32_t n_bins,
                                                       size_t* bytes);
DSPARK_API dspark_status dspark_sts_fit(const dspark_sts_fit_args* args, void* workspace, size_t workspace_bytes,
                                        void* stream);

/* Number of CUDA kernels this library has enqueued since it was loaded (a
 * host-side counter, incremented at launch time; a captured CUDA graph counts
 * its kernels once, at capture).  For accounting only: no library behaviour
 * depends on it. */
DSPARK_API uint64_t dspark_launch_count(void);

/* The cudaError_t value behind the most recent DSPARK_CUDA_ERROR that a call
 * on the calling thread returned (0 if none has).  Thread-local; no call
 * resets it. */
DSPARK_API int dspark_last_cuda_error(void);

/* Human-readable name of a status code (static string, never NULL). */
DSPARK_API const char* dspark_status_string(dspark_status s);

/* Library build identification (static string). */
DSPARK_API const char* dspark_version(void);

#ifdef __cplusplus
}
#endif

#endif /* DSPARK_H */
