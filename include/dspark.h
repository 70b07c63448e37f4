/*
 * dspark.h -- C ABI of the DSpark draft / schedule / verify / accept-rate path
 * for one NVIDIA GB300 GPU (sm_103a).
 *
 * Six operations, each a hand-written CUDA kernel sequence:
 *   dspark_draft_block      semi-autoregressive draft block, confidence, survival
 *   dspark_schedule_prefix  hardware-aware prefix scheduler (Algorithm 1)
 *   dspark_verify           rejection-sampling verification + residual/bonus token
 *   dspark_accept_rate_tv   c* = 1 - 1/2 ||softmax(d) - softmax(t)||_1 per row
 *   dspark_training_loss    joint CE + L1 + BCE loss per row, and its gradient
 *   dspark_decode_rounds    draft -> schedule -> verify rounds, anchor carried
 * (and _ex variants of the draft and verify calls for the gated / RNN heads)
 *
 * Sources (cited per call): the DeepSpec / DSpark walkthrough at
 * wangjunjian.com ("DSpark" post, sections 2.1, 3.2, 3.3, 7.2, 8.1-8.3) and the
 * Qwen3.8-27B-DSpark model-card explainer at dpshk.com (AcceptRatePredictor,
 * config.json fields).
 *
 * Conventions shared by every call
 *   - Every pointer is a DEVICE pointer owned by the caller, except where a
 *     comment says "host".  The library allocates nothing and frees nothing on
 *     these calls; it caches only device properties and kernel attributes.
 *   - Every call is asynchronous on `stream` (a cudaStream_t; NULL = legacy
 *     default stream).  The return value reports host-side argument checks
 *     and launch errors only.
 *   - Device-side status: the first 16 bytes of `workspace` hold a status
 *     block {uint32 code, uint32 detail, ...}; the call clears it, and a
 *     kernel that meets a device-side error (an out-of-range token id, a
 *     bounded wait that ran out) writes a nonzero dspark_status_t there and
 *     skips the affected work.  Read it after the stream completes, e.g. with
 *     dspark_workspace_status().
 *   - Layouts are row-major with the vocabulary dimension contiguous.  Float
 *     tensors of one call share one dtype (dspark_dtype_t).  bf16 rows need
 *     V % 8 == 0 and f32 rows V % 4 == 0 (16-byte aligned rows); every tensor
 *     base pointer must be 16-byte aligned and workspace 256-byte aligned.
 *   - Positions k are 1-based as on the pages: U[b][k-1] is the base logit
 *     row of draft position k; t_logits[b][k-1] is the target row that
 *     verifies position k, and t_logits[b][gamma] the bonus row.
 *   - Random draws use Philox4x32-10 (Salmon et al., SC'11) keyed by
 *     (seed_lo, seed_hi) with counter (index >> 2, k, b, stream), output word
 *     index & 3.  Streams: 0 draft token (index = vocabulary index), 1 accept
 *     uniform (index 0), 2 the token verification emits (residual, bonus, or
 *     the draw from p_t when a residual has no mass; one per request).
 *   - Sampling from a softmax is Gumbel-max over the whole vocabulary: the
 *     token argmax_v(lw_v - ln(-ln u_v)) with u_v = ((w_v >> 9) + 1/2) 2^-23
 *     from the word of index v, lw the log-weights (logits / T, or ln q of the
 *     residual q); ties go to the lowest index.  This draws token v with
 *     probability exactly softmax(lw)_v.
 */
#ifndef DSPARK_H
#define DSPARK_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define DSPARK_MAX_GAMMA 32

typedef enum {
    DSPARK_OK = 0,
    DSPARK_ERR_INVALID_ARGUMENT = 1,   /* a host-side check failed; nothing was launched */
    DSPARK_ERR_UNSUPPORTED = 2,        /* valid but outside what the kernels handle */
    DSPARK_ERR_WORKSPACE_TOO_SMALL = 3,
    DSPARK_ERR_CUDA = 4,               /* a CUDA runtime call or launch failed */
    DSPARK_ERR_TIMEOUT = 5,            /* device status only: a bounded wait ran out */
    DSPARK_ERR_DEVICE_CHECK = 6        /* device status only: a device-side input check failed */
} dspark_status_t;

typedef enum { DSPARK_F32 = 0, DSPARK_BF16 = 1 } dspark_dtype_t;

typedef struct CUstream_st* dspark_stream_t;   /* same type as cudaStream_t */

/* Human-readable name of a status code (static storage; never NULL). */
const char* dspark_status_string(dspark_status_t s);

/* Synchronises `stream`, then returns the device status code stored at the
 * head of `workspace` by the last call that used it (DSPARK_OK if none).
 * Returns DSPARK_ERR_CUDA if the synchronisation or the copy fails. */
dspark_status_t dspark_workspace_status(const void* workspace, dspark_stream_t stream);

/* Opt-in L2 residency of the Markov weight W2 (read once per draft position).
 * bytes > 0: sets the persisting-L2 limit of the calling thread's current
 * context on the current device to min(bytes, the device's maximum), and from
 * then on every draft launch (dspark_draft_block, its no-allocation twin,
 * dspark_decode_rounds) and the residual launch of dspark_verify carry an
 * access-policy window over W2 that marks its lines persisting, so they stay
 * in L2 from one position and one call to the next instead of being evicted by
 * the streamed U and target rows.  bytes = 0: drops the window from later
 * launches, returns the persisting lines to normal status and puts the
 * limit back to the value it had before the first enabling call.
 * This changes a context-wide setting: L2 set aside for
 * persisting lines is no longer available to other kernels of the process
 * for their normal lines.  Results are bit-identical either way; only the
 * DRAM traffic (and at small batches the time) changes.  Host-side only: not
 * while a stream is being captured.  DSPARK_ERR_CUDA if the limit cannot be
 * set (e.g. no persisting L2 on the device). */
dspark_status_t dspark_set_l2_residency(size_t bytes);

/* ------------------------------------------------------------------------ *
 * Draft block.  DeepSpec walkthrough section 3.2 (stage two): for k = 1..gamma
 *   z_k = U_k + B(x_{k-1}),  B(x_{k-1}, v) = sum_j W2[v][j] * W1[x_{k-1}][j]
 * (VanillaMarkovHead, paper eq. 5, rank r), x_k ~ softmax(z_k / T) -- the
 * `sample_block_tokens` loop, x_0 = anchor.  Section 3.3 confidence head:
 *   c_k = sigmoid(sum_i w[i] h[b][k-1][i] + sum_j w[H+j] W1[x_{k-1}][j] + bias)
 * (model card: one nn.Linear(H + r, 1) returning a logit), and the Algorithm 1
 * survival a_k = a_{k-1} * c_k in float32, a_0 = 1.
 *
 *   U [B][gamma][V], h [B][gamma][H], W1 [V][r], W2 [V][r], w [H + r] in `dt`;
 *   x0 [B] int32 anchors in [0, V).
 *   temperature > 0 samples; temperature == 0 takes argmax z_k (lowest index
 *   on ties) and writes lse_d = logp_d = 0.
 *   Outputs [B][gamma]: x (int32 tokens), lse_d = logsumexp(z_k / T),
 *   logp_d = z_k[x_k] / T - lse_d, c, a (float32).
 *   U, h and x0 may also point to pinned (page-locked, registered) host
 *   memory.  U and h are then copied to the device first, each in one
 *   copy-engine transfer on `stream` (the host link's full rate), into memory
 *   from a pool private to the library; the pool keeps what it allocated (up
 *   to the largest B * gamma * (V + H) elements staged) until the process
 *   exits.  While `stream` is being captured into a graph, or if that memory
 *   cannot be had, the kernels read U and h over the host link instead, each
 *   byte once; they always read x0 that way.
 *   Unregistered host memory returns DSPARK_ERR_INVALID_ARGUMENT.
 * Requires 1 <= B <= 65535, 1 <= gamma <= DSPARK_MAX_GAMMA, r % 8 == 0 and
 * r <= 256.  bf16 inputs with r % 64 == 0 run the bias on tensor cores.
 * An anchor or token id outside [0, V) sets DSPARK_ERR_DEVICE_CHECK in the
 * workspace status and is read as 0.
 * ------------------------------------------------------------------------ */
size_t dspark_draft_block_workspace_size(int B, int gamma, int V, int r);

dspark_status_t dspark_draft_block(int B, int gamma, int V, int H, int r, dspark_dtype_t dt,
                                   const void* U, const void* h, const void* W1, const void* W2,
                                   const void* w, float bias, const int32_t* x0,
                                   float temperature, uint64_t seed,
                                   int32_t* x, float* lse_d, float* logp_d, float* c, float* a,
                                   void* workspace, size_t workspace_bytes, dspark_stream_t stream);

/* ------------------------------------------------------------------------ *
 * dspark_draft_block without a caller workspace.  The paper has no
 * counterpart: this entry point exists for callers that cannot allocate
 * device memory -- hosts that own all GPU memory through their own pool and
 * forbid cudaMalloc or allocating library calls from plug-in code.  Arguments
 * and results are those of dspark_draft_block; the scratch lives in a fixed
 * 4 MiB array inside the library's device image, held by every GPU that loads
 * the library until the process exits.
 *   - Arguments are checked as dspark_draft_block checks them
 *     (DSPARK_ERR_INVALID_ARGUMENT); then calls whose
 *     dspark_draft_block_workspace_size(B, gamma, V, r) exceeds 4 MiB return
 *     DSPARK_ERR_UNSUPPORTED (B * gamma up to about 2100), and so do calls on
 *     a device ordinal of 64 or more.
 *   - All calls share the one array: calls that overlap on the GPU (other
 *     streams, other host threads) race and corrupt each other's results.
 *     Each call clears what must start at zero.
 *   - U, h and x0 in pinned host memory are read by the kernels over the host
 *     link (no staging copy to the device, which would allocate).
 *   - The first call on a device looks up the array's device address with
 *     cudaGetSymbolAddress (with that device current); make that first call
 *     before any stream capture.
 *   - Device-side status (a token id out of range, or a bounded wait that
 *     ran out) is recorded in the internal array, which the caller cannot
 *     read: such a call still returns DSPARK_OK with unfinished outputs.
 *     Validate x0 beforehand; a timeout needs a GPU that stalls for seconds.
 * Allocates nothing: no cudaMalloc, cudaFree or allocating library routine.
 * ------------------------------------------------------------------------ */
dspark_status_t dspark_draft_block_noalloc(int B, int gamma, int V, int H, int r, dspark_dtype_t dt,
                                           const void* U, const void* h, const void* W1, const void* W2,
                                           const void* w, float bias, const int32_t* x0,
                                           float temperature, uint64_t seed,
                                           int32_t* x, float* lse_d, float* logp_d, float* c, float* a,
                                           dspark_stream_t stream);

/* ------------------------------------------------------------------------ *
 * Prefix scheduler, Algorithm 1 (DeepSpec walkthrough section 3.3 flowchart):
 * sort all (b, j) pairs by a[b][j-1] descending (ties: lower b, then lower
 * j), scan them starting from l_b = 0 for all b, and accept a pair while
 *   Theta = (E / N) * sps[N] > Theta_best
 * with N = sum_b (l_b + 1) verified rows (the bonus row included) and
 * E = sum_b (1 + sum_{j <= l_b} a[b][j-1]) expected emitted tokens; stop at the
 * first pair that does not raise Theta.  E is the exact sum of the float32
 * survivals rounded once to double; Theta is one IEEE double division and one
 * multiplication, so the result is bit-reproducible.
 *
 *   a [B][gamma] float32 survivals, each in [0, 1] and non-increasing in j
 *     (as dspark_draft_block writes them);
 *   sps [B*(gamma+1) + 1] double, sps[N] the verification throughput at N rows
 *     (device memory, or pinned host memory read through its mapping);
 *   outputs: ell [B] int32 (l*_b in 0..gamma), n_sched [1] int32 (N),
 *   theta [1] double (Theta_best).
 * Requires B * gamma <= 16384.  A value of a outside [0, 1] sets
 * DSPARK_ERR_DEVICE_CHECK in the workspace status.
 * ------------------------------------------------------------------------ */
size_t dspark_schedule_prefix_workspace_size(int B, int gamma);

dspark_status_t dspark_schedule_prefix(int B, int gamma, const float* a, const double* sps,
                                       int32_t* ell, int32_t* n_sched, double* theta,
                                       void* workspace, size_t workspace_bytes,
                                       dspark_stream_t stream);

/* ------------------------------------------------------------------------ *
 * Verification (DeepSpec walkthrough section 8.2, verify_draft_tokens): for
 * k = 1..ell[b], accept x_k iff u < min(1, p_t(x_k) / p_d(x_k)) with
 *   p_t = softmax(t_logits[b][k-1] / T),  log p_d(x_k) = logp_d[b][k-1],
 *   u = (Philox word >> 8) * 2^-24, stream 1, counter (0, k, b, 1);
 * stop at the first rejection and draw next_token from norm(max(0, p_t - p_d))
 * at that position, where p_d(v) = exp(z_k(v) / T - lse_d[b][k-1]) and z_k is
 * rebuilt from U, W1, W2 and x_{k-1} exactly as the draft built it; if that
 * residual has no mass, draw from p_t.  If all ell[b] are accepted, draw the
 * bonus token from p_t of row ell[b] + 1 (section 2.1: one extra token per
 * round).  temperature == 0: accept iff x_k == argmax t_k, next_token =
 * argmax t at the stop row.
 *
 *   t_logits [B][gamma+1][V], U [B][gamma][V], W1/W2 [V][r] in `dt`.
 *   t_logits, U and x0 may also point to pinned (page-locked, registered)
 *   host memory: the kernels then read only the rows verification needs (the
 *   scheduled prefix and its stop row; U rows of rejected requests) over the
 *   host link.  Unregistered host memory returns DSPARK_ERR_INVALID_ARGUMENT;
 *   x0 [B], x [B][gamma] int32; lse_d, logp_d [B][gamma] float32 (from the
 *   draft); ell [B] int32 in 0..gamma.
 *   Outputs: n_accept [B] int32 in 0..ell[b]; next_token [B] int32.  The
 *   request emits x[b][0 .. n_accept-1] followed by next_token[b].
 * Only target rows 1..ell[b]+1 of each request are read.
 * ------------------------------------------------------------------------ */
size_t dspark_verify_workspace_size(int B, int gamma, int V, int r);

dspark_status_t dspark_verify(int B, int gamma, int V, int r, dspark_dtype_t dt,
                              const void* t_logits, const void* U, const void* W1, const void* W2,
                              const int32_t* x0, const int32_t* x, const float* lse_d,
                              const float* logp_d, const int32_t* ell, float temperature,
                              uint64_t seed, int32_t* n_accept, int32_t* next_token,
                              void* workspace, size_t workspace_bytes, dspark_stream_t stream);

/* ------------------------------------------------------------------------ *
 * Analytic accept rate, paper eq. 8 (DeepSpec walkthrough section 3.3 and the
 * `_compute_accept_rate_3d` snippet): for each row
 *   c_star[row] = 1 - 1/2 sum_v |softmax(d[row])_v - softmax(t[row])_v|
 * over the full vocabulary, no temperature.  Computed as
 * sum_v min(p_d(v), p_t(v)), which is the same quantity.
 *
 *   d, t [rows][V] in `dt`; c_star [rows] float32.  Each row needs at least
 *   one finite logit.  rows == 0 launches nothing.
 * ------------------------------------------------------------------------ */
size_t dspark_accept_rate_tv_workspace_size(int64_t rows, int V);

dspark_status_t dspark_accept_rate_tv(int64_t rows, int V, dspark_dtype_t dt,
                                      const void* d, const void* t, float* c_star,
                                      void* workspace, size_t workspace_bytes,
                                      dspark_stream_t stream);

/* ------------------------------------------------------------------------ *
 * Sequential heads beyond the Markov head (DeepSpec walkthrough section 3.2,
 * the three heads of markov_head.py).  Every head adds a bias
 *   B_k(v) = W2[v] . e_k                  (the output projection of eq. 5)
 * to the parallel logits U_k; the heads differ in the rank-r vector e_k:
 *   DSPARK_HEAD_MARKOV  e_k = W1[x_{k-1}]                      (VanillaMarkovHead, eq. 5)
 *   DSPARK_HEAD_GATED   e_k = sigmoid(Wg . [h_k ; W1[x_{k-1}]]) (*) W1[x_{k-1}]
 *                       (GatedMarkovHead: a hidden-state gate on the Markov row)
 *   DSPARK_HEAD_RNN     s_k = g (*) s_{k-1} + (1 - g) (*) tanh(Wc . z_k),
 *                       g = sigmoid(Wg . z_k), z_k = [s_{k-1} ; W1[x_{k-1}] ; h_k],
 *                       s_0 = 0, e_k = s_k          (RNNHead, GRU-like, eq. 6)
 * with (*) the element-wise product, s_k in R^r, and h_k = h[b][k-1].
 *   Wg: GATED [r][H + r] (columns: h, then W1 row); RNN [r][2r + H] (columns: s,
 *       W1 row, h); Wc: RNN [r][2r + H]; in the call's dtype, rows 16-byte aligned.
 *   E [B][gamma][r] in the call's dtype: the e_k each position used, written by
 *   dspark_draft_block_ex and read by dspark_verify_ex (the residual rebuilds
 *   z_k from it).  e_k is formed in float32 (the RNN state stays float32) and
 *   rounded to the dtype, as W1 rows are, before the projection.
 * The Markov kind ignores Wg, Wc and E.
 * ------------------------------------------------------------------------ */
typedef enum dspark_head_kind {
    DSPARK_HEAD_MARKOV = 0,
    DSPARK_HEAD_GATED = 1,
    DSPARK_HEAD_RNN = 2
} dspark_head_kind_t;

typedef struct dspark_head {
    int kind;        /* dspark_head_kind_t */
    const void* Wg;
    const void* Wc;
    void* E;
} dspark_head_t;

/* dspark_draft_block with a sequential head (NULL: the Markov head).  Gated
 * and RNN heads run one launch per position with a head kernel before each.
 * Requires H > 0 for them.  Workspace: dspark_draft_block_ex_workspace_size. */
size_t dspark_draft_block_ex_workspace_size(int B, int gamma, int V, int r, int kind);

dspark_status_t dspark_draft_block_ex(int B, int gamma, int V, int H, int r, dspark_dtype_t dt,
                                      const void* U, const void* h, const void* W1, const void* W2,
                                      const void* w, float bias, const int32_t* x0,
                                      float temperature, uint64_t seed, const dspark_head_t* head,
                                      int32_t* x, float* lse_d, float* logp_d, float* c, float* a,
                                      void* workspace, size_t workspace_bytes, dspark_stream_t stream);

/* dspark_verify for a draft made with a sequential head: the residual's p_d
 * is rebuilt from head->E (NULL or the Markov kind: from W1[x_{k-1}]).  The
 * workspace is dspark_verify's. */
dspark_status_t dspark_verify_ex(int B, int gamma, int V, int r, dspark_dtype_t dt,
                                 const void* t_logits, const void* U, const void* W1, const void* W2,
                                 const int32_t* x0, const int32_t* x, const float* lse_d,
                                 const float* logp_d, const int32_t* ell, float temperature,
                                 uint64_t seed, const dspark_head_t* head, int32_t* n_accept,
                                 int32_t* next_token, void* workspace, size_t workspace_bytes,
                                 dspark_stream_t stream);

/* ------------------------------------------------------------------------ *
 * Several decoding rounds in a row (DeepSpec walkthrough sections 8.1 / 8.3,
 * `generate_decoding_sample`: propose, verify, emit, continue from the new
 * context), all enqueued on `stream` with no host synchronisation, so that a
 * caller can capture them in one CUDA graph.  Round i (i = 0 .. rounds-1):
 *   1. dspark_draft_block on pool slot p = i mod pool, x0 = anchor, seed + i;
 *   2. dspark_schedule_prefix on its survivals a;
 *   3. dspark_verify of the scheduled prefix against slot p's target rows;
 *   4. emit x[b][0 .. n_accept-1] then next_token[b]; anchor[b] = next_token[b]
 *      (the last token emitted is the next round's anchor).
 * The synthetic slots stand in for the target model's next context; the
 * carried state is the anchor.  Every round keys its draws with seed + i
 * (64-bit wrap-around).
 *
 *   U [pool][B][gamma][V], h [pool][B][gamma][H], t_logits [pool][B][gamma+1][V],
 *   W1/W2 [V][r], w [H + r] in `dt`; sps as for dspark_schedule_prefix.
 *   t_logits may be pinned host memory, as for dspark_verify.
 *   anchor [B] int32: in, the first round's anchors; out, the last emitted tokens.
 *   Outputs: tokens [rounds][B][gamma+1] int32 (emitted tokens, then -1);
 *   n_emitted [rounds][B] int32 (n_accept + 1); stats [rounds][2] double:
 *   E[tau] = sum_b (1 + sum_{j <= l_b} a[b][j-1]) / B, the expected emitted
 *   tokens per request that the scheduler maximises, and the realised
 *   sum_b n_emitted[b] / B.
 *   trace (host pointer, may be NULL; any member may be NULL): per-round copies
 *   of the draft outputs x, lse_d, logp_d, c, a [rounds][B][gamma] and of ell,
 *   n_accept, next_token [rounds][B].
 * Requirements are those of the three calls.  The workspace holds their
 * workspaces and the round's intermediates; a sub-call's device error is copied
 * to this workspace's status with detail 1000 * stage + the sub-call's detail
 * (stage 1 draft, 2 schedule, 3 verify).  rounds == 0 launches nothing.
 * ------------------------------------------------------------------------ */
typedef struct dspark_round_trace {
    int32_t* x;
    float* lse_d;
    float* logp_d;
    float* c;
    float* a;
    int32_t* ell;
    int32_t* n_accept;
    int32_t* next_token;
} dspark_round_trace_t;

size_t dspark_decode_rounds_workspace_size(int B, int gamma, int V, int r);

dspark_status_t dspark_decode_rounds(int rounds, int pool, int B, int gamma, int V, int H, int r,
                                     dspark_dtype_t dt, const void* U, const void* h,
                                     const void* t_logits, const void* W1, const void* W2,
                                     const void* w, float bias, const double* sps, int32_t* anchor,
                                     float temperature, uint64_t seed, int32_t* tokens,
                                     int32_t* n_emitted, double* stats,
                                     const dspark_round_trace_t* trace,
                                     void* workspace, size_t workspace_bytes,
                                     dspark_stream_t stream);

/* ------------------------------------------------------------------------ *
 * Joint training loss of the drafter and its gradient (DeepSpec walkthrough
 * section 7.2, `compute_dspark_loss`; position weights from
 * `_build_loss_weight_mask`).  For each row, with p = softmax over the full
 * vocabulary (no temperature):
 *   ce   = logsumexp(d) - d[target]
 *   c*   = sum_v min(p_d(v), p_t(v))            (= 1 - 1/2 ||p_d - p_t||_1, eq. 8)
 *   bce  = softplus(s) - c* s                    (BCE with logits, target c*)
 *   row  = omega (alpha_ce ce + alpha_l1 (1 - c*) + alpha_conf bce)
 *   loss = sum over rows of row
 * and, with c* held fixed as the BCE's target and sgn_v = sign(p_d(v) - p_t(v)),
 *   grad_d[v]  = omega (alpha_ce (p_d(v) - [v = target])
 *                      + alpha_l1 / 2 p_d(v) (sgn_v - sum_u p_d(u) sgn_u))
 *   grad_conf  = omega alpha_conf (sigmoid(s) - c*).
 * The page's weights are alpha_ce = 0.1, alpha_l1 = 0.9, alpha_conf = 1.0 and
 * the position weight of block position k is exp(-(k - 1) / 4); the caller
 * folds position weights and any normalisation into omega (omega = w_k /
 * sum w gives the weighted mean).
 *
 *   d, t [rows][V] in `dt` (draft and target logits); target [rows] int32 in
 *   [0, V); conf_logit [rows] float32 (the confidence head's logit s); omega
 *   [rows] float32.
 *   row_out [rows][4] float32: (ce, c*, bce, row); loss [1] float32 (summed
 *   in a fixed order: the same inputs give the same bits).
 *   grad_d [rows][V] in `dt`, or NULL to skip it; grad_conf [rows] float32, or
 *   NULL.  Every byte of d and t is read once; grad_d is written from
 *   registers in the same pass.
 *   A target id outside [0, V) sets DSPARK_ERR_DEVICE_CHECK (that row's ce is
 *   then +inf).  rows == 0 writes loss = 0.
 * ------------------------------------------------------------------------ */
size_t dspark_training_loss_workspace_size(int64_t rows, int V);

dspark_status_t dspark_training_loss(int64_t rows, int V, dspark_dtype_t dt,
                                     const void* d, const void* t, const int32_t* target,
                                     const float* conf_logit, const float* omega,
                                     float alpha_ce, float alpha_l1, float alpha_conf,
                                     float* row_out, float* loss, void* grad_d, float* grad_conf,
                                     void* workspace, size_t workspace_bytes,
                                     dspark_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* DSPARK_H */
