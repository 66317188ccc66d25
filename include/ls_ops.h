/*
 * ls_ops.h -- C ABI of the fused non-GEMM Transformer-layer operators for
 * NVIDIA GB300 (sm_103a): bias+dropout+residual, bias+ReLU+dropout,
 * LayerNorm and masked attention softmax, forward and backward.
 *
 * Where the operators come from (page title, section):
 *  - "CMU 11-868 L10: accelerating the Transformer on GPUs (LightSeq)",
 *    technique 1 "kernel fusion" (slide p.12): every non-GEMM step of the
 *    layer is one fused kernel -- bias+dropout+residual, bias+ReLU+dropout,
 *    and the LayerNorm and softmax reduce kernels; technique 2 "rewrite the
 *    formula": LayerNorm statistics with one synchronisation (slide p.21), the
 *    LayerNorm backward as two parallel sums (slide p.22), and the softmax
 *    specialised by row length (slides p.23-26).
 *  - "LightSeq2: Accelerated Training for Transformer-based Models on GPUs",
 *    section 2.1.1 (fused bias+dropout+residual after self-attention) and
 *    section 2.1.2 (the dropout mask saved in the forward pass and reused in
 *    the backward pass).
 *  - "CS336 Lecture 5: GPU", sections 6.1-6.2 (row softmax of the attention
 *    scores, maximum subtracted).
 *
 * Conventions shared by every entry point
 *  - Storage dtype is FP16 (LS_F16) or FP32 (LS_F32); arithmetic is FP32.
 *    Parameters (bias, gamma, beta) and their gradients use the storage dtype;
 *    LayerNorm statistics (mean, rstd) are FP32.
 *  - Activations are row-major [rows, cols]; attention scores are row-major
 *    [batch, heads, q_len, k_len].  cols (k_len) must be a multiple of 8.
 *  - Every pointer is device memory owned by the caller and must be 16-byte
 *    aligned.  The library allocates nothing, never synchronises, and keeps no
 *    state except a per-thread error message.  Work is enqueued on `stream`
 *    (a cudaStream_t; NULL is the legacy default stream) and the call returns
 *    without waiting for it.
 *  - An output may be the very same pointer as an input of the same shape (in
 *    place); any other overlap between an output and another buffer is
 *    rejected with LS_ERR_INVALID_ARGUMENT.
 *  - Argument errors are returned before anything is enqueued.  A launch
 *    failure returns LS_ERR_CUDA; faults during execution surface at the
 *    caller's next synchronisation, as for any CUDA kernel.
 *  - rows == 0 (or batch*heads*q_len == 0) is a no-op returning LS_OK.
 *
 * Dropout
 *  - Drop probability p must satisfy 0 <= p < 1.  Kept values are scaled by
 *    1/(1-p), computed in FP32.
 *  - Element i (flat row-major index) draws the 32-bit word i & 3 of
 *    Philox-4x32-10 (Salmon et al., SC'11) with key = (lo32(seed), hi32(seed))
 *    and counter = (lo32(i>>2), hi32(i>>2), lo32(offset), hi32(offset)); it is
 *    kept iff word >= floor(p * 2^32).  `offset` tells call sites apart.
 *  - mask_bits holds ceil(rows*cols/32) uint32 words: element i is bit
 *    (i & 31) of word (i >> 5); bits past the last element are written as 0.
 *
 * Column reductions (the bias, gamma and beta gradients)
 *  - These are deterministic: per-tile FP32 partial sums go to `workspace`
 *    and are then added in a fixed order.  Results are bitwise reproducible
 *    for a given shape on any GPU.  The workspace is caller-owned device
 *    memory of at least ls_colreduce_workspace_bytes(rows, cols) bytes; its
 *    contents need no initialisation and are scratch after the call.  Two
 *    calls that run concurrently must not share a workspace.
 */
#ifndef LS_OPS_H
#define LS_OPS_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    LS_OK = 0,
    LS_ERR_INVALID_ARGUMENT = 1,   /* NULL required pointer, bad p/eps, negative size, overlap */
    LS_ERR_MISALIGNED = 2,         /* pointer not 16-byte aligned, or cols % 8 != 0 */
    LS_ERR_UNSUPPORTED_SHAPE = 3,  /* LayerNorm cols > 16384, softmax k_len > 2^20, too many elements */
    LS_ERR_WORKSPACE_TOO_SMALL = 4,
    LS_ERR_CUDA = 5                /* a CUDA call or kernel launch failed; see ls_last_error() */
} ls_status;

typedef enum { LS_F32 = 0, LS_F16 = 1 } ls_dtype;

/* Static description of a status code. */
const char* ls_status_string(ls_status status);
/* Message of the last failing call on this host thread ("" if none). */
const char* ls_last_error(void);
/* Library version, major*10000 + minor*100 + patch. */
int ls_version(void);

/* Device-side failure flags raised since the previous call, cleared by this
 * call.  Kernels that stream rows through shared memory with bulk copies wait
 * for each copy with a bounded number of polls; if a wait runs out (a healthy
 * GPU never gets there), the kernel sets LS_DEVERR_WAIT_TIMEOUT, lets its
 * copies in flight land, and stops early: the outputs of that call are
 * incomplete.  Unlike every other entry point this one synchronises: it waits
 * for all work on the current device before reading the flags.  *flags gets
 * the OR of the flags (0 = none). */
#define LS_DEVERR_WAIT_TIMEOUT 1u
ls_status ls_check_device_errors(uint32_t* flags);

/* Self-test of that failure path (no counterpart on the pages): enqueues one
 * warp that waits, with the library's bounded wait, on a barrier that nothing
 * completes; after `polls` polls (1 .. 2^19, each suspending the warp for up
 * to about 2 us) it records LS_DEVERR_WAIT_TIMEOUT and exits.  Nothing hangs
 * and the context stays usable; ls_check_device_errors then reports and
 * clears the flag. */
ls_status ls_selftest_wait_timeout(uint32_t polls, void* stream);

/* Workspace bytes that the backward calls with a column reduction
 * (ls_bias_dropout_residual_bwd, ls_bias_relu_dropout_bwd, ls_layernorm_bwd)
 * need for an activation of shape [rows, cols]; enough for all three. */
size_t ls_colreduce_workspace_bytes(int64_t rows, int64_t cols);

/* Column reductions on a second stream (a scheduling facility; results are
 * bit-identical to the default).  The backward entries with a bias, gamma or
 * beta gradient (ls_bias_dropout_residual_bwd, ls_bias_relu_dropout_bwd,
 * ls_layernorm_bwd, ls_bias_reshape_qkv_bwd) run a main kernel that writes dx
 * and per-tile partial sums into the workspace, then the fixed-order sum of
 * the partials -- the sums over rows that give dbias ("LightSeq2", section
 * 2.1.2) and dgamma, dbeta ("CMU 11-868 L10 (LightSeq)", technique 2, slide
 * p.22).  After
 * ls_set_reduction_stream(rs), calls made from the calling thread launch that
 * reduction on rs, ordered after the main kernel by an event, so that the
 * caller's next kernel on the main stream does not wait for it.  Until
 * ls_join_reductions(stream) has been called and stream reached that point,
 * the gradients (dbias, dgamma, dbeta) are not ready and the workspaces the
 * pending reductions read must not be written by anything but these entries:
 * a later backward call whose workspace overlaps a pending reduction's makes
 * its own stream wait for that reduction first (correct, but no overlap -- give
 * each backward call of a step its own workspace to overlap).  Join before a
 * stream capture ends (the reduction stream joins the capture at the first
 * fork) and before starting one.  rs = NULL restores the default.  The state
 * (rs, 18 CUDA events of the current device, up to 16 pending reductions) is
 * per host thread.  Errors: LS_ERR_INVALID_ARGUMENT if reductions are pending
 * (join first); LS_ERR_CUDA if the events cannot be created.
 * ls_layernorm_bwd_noalloc keeps its reduction on the caller's stream. */
ls_status ls_set_reduction_stream(void* reduce_stream);

/* Makes stream wait for every reduction forked since the last join (no-op if
 * none), then forgets them.  Errors: LS_ERR_CUDA. */
ls_status ls_join_reductions(void* stream);

/* Fused bias + dropout + residual, forward ("CMU 11-868 L10 (LightSeq)",
 * technique 1; "LightSeq2", section 2.1.1):
 *   out[r,c] = residual[r,c] + keep(i) * (x[r,c] + bias[c]) / (1 - p),  i = r*cols + c.
 * x, residual, out: [rows, cols]; bias: [cols]; mask_bits (nullable): keep bits.
 * out may be x or residual (in place). */
ls_status ls_bias_dropout_residual_fwd(ls_dtype dtype, void* out, uint32_t* mask_bits,
                                       const void* x, const void* bias, const void* residual,
                                       int64_t rows, int64_t cols, float p, uint64_t seed,
                                       uint64_t offset, void* stream);

/* Backward of the above ("LightSeq2", section 2.1.2: the saved mask is reused):
 *   dx = keep * dout / (1 - p);  dbias[c] = sum_r dx[r,c];  d residual = dout
 * (not written: the caller uses dout itself).  mask_bits == NULL draws the
 * keep bits again from (seed, offset); otherwise seed and offset are ignored.
 * dbias may be NULL (then no workspace is needed).  dx may be dout. */
ls_status ls_bias_dropout_residual_bwd(ls_dtype dtype, void* dx, void* dbias, const void* dout,
                                       const uint32_t* mask_bits, int64_t rows, int64_t cols,
                                       float p, uint64_t seed, uint64_t offset, void* workspace,
                                       size_t workspace_bytes, void* stream);

/* Fused bias + ReLU + dropout, forward ("CMU 11-868 L10 (LightSeq)", technique 1):
 *   z = x + bias[c];  bit(i) = (z > 0) and keep(i);  out = bit(i) * z / (1 - p).
 * mask_bits is required: it stores bit(i), which is all the backward needs.
 * ReLU(0) = 0 and its slope at 0 is 0.  out may be x. */
ls_status ls_bias_relu_dropout_fwd(ls_dtype dtype, void* out, uint32_t* mask_bits, const void* x,
                                   const void* bias, int64_t rows, int64_t cols, float p,
                                   uint64_t seed, uint64_t offset, void* stream);

/* Backward of the above:  dx = bit * dout / (1 - p);  dbias[c] = sum_r dx[r,c].
 * dbias may be NULL.  dx may be dout. */
ls_status ls_bias_relu_dropout_bwd(ls_dtype dtype, void* dx, void* dbias, const void* dout,
                                   const uint32_t* mask_bits, int64_t rows, int64_t cols, float p,
                                   void* workspace, size_t workspace_bytes, void* stream);

/* LayerNorm forward ("CMU 11-868 L10 (LightSeq)", technique 2, slide p.21): one
 * pass computes sum(x) and sum(x^2) together (one synchronisation), then
 *   mean = mu(x),  var = max(mu(x^2) - mu(x)^2, 0),  rstd = 1/sqrt(var + eps),
 *   y = gamma * (x - mean) * rstd + beta.
 * (The sums are taken about the row's first element, which leaves the
 * identity unchanged and avoids cancellation for rows with a large mean.)
 * x, y: [rows, cols]; gamma, beta: [cols]; mean, rstd: FP32 [rows] (both
 * nullable).  eps >= 0.  cols <= 16384.  y may be x. */
ls_status ls_layernorm_fwd(ls_dtype dtype, void* y, float* mean, float* rstd, const void* x,
                           const void* gamma, const void* beta, int64_t rows, int64_t cols,
                           float eps, void* stream);

/* LayerNorm backward ("CMU 11-868 L10 (LightSeq)", technique 2, slide p.22): per
 * row the two sums A = sum_j g_j and C = sum_j g_j * xhat_j, g = gamma * dy,
 * xhat = (x - mean) * rstd, are computed together (one synchronisation), then
 *   dx = rstd * (g - A/cols - xhat * C/cols),
 *   dgamma[c] = sum_r dy * xhat,  dbeta[c] = sum_r dy.
 * mean and rstd are the forward's saved statistics.  dgamma and dbeta are
 * both given or both NULL (then no workspace is needed).  dx may be dy or x. */
ls_status ls_layernorm_bwd(ls_dtype dtype, void* dx, void* dgamma, void* dbeta, const void* dy,
                           const void* x, const void* gamma, const float* mean, const float* rstd,
                           int64_t rows, int64_t cols, void* workspace, size_t workspace_bytes,
                           void* stream);

/* LayerNorm backward that needs no caller workspace.  The paper has no
 * counterpart of this entry point.  It computes what ls_layernorm_bwd computes
 * (same kernels, same fixed-order reductions, hence the same bits) for callers
 * that cannot allocate device memory and so cannot hand ls_layernorm_bwd the
 * workspace for the gamma/beta partial sums: for example a plugin running
 * inside a host application that owns every device allocation, or a code path
 * where calling cudaMalloc is not allowed (it synchronises the device, and it
 * fails while a CUDA graph is being captured).
 *  - The scratch is an array of LS_NOALLOC_SCRATCH_BYTES (8 MiB) inside the
 *    library's device image; every GPU that loads the library holds it until
 *    the process exits.  The call itself allocates nothing (no cudaMalloc,
 *    cudaFree or allocating library routine).
 *  - Every shape with cols <= 3448 fits; wider rows fit only for fewer rows.
 *    A shape whose partial sums need more scratch is rejected with
 *    LS_ERR_UNSUPPORTED_SHAPE before anything is enqueued.
 *  - Every call looks up the array's device address in the current context
 *    (cudaGetSymbolAddress; a query, not an allocation).  The array exists
 *    once per context that has loaded the library, so the address is never
 *    cached: calls stay correct in a second context on the same device and
 *    after cudaDeviceReset.  The first call in a context also loads the
 *    library's device code there; make that first call outside any stream
 *    capture.
 *  - The fixed-order reduction of the partial sums always runs on `stream`,
 *    also while ls_set_reduction_stream is in effect (the scratch is shared
 *    by every host thread, so a reduction forked onto another stream could
 *    still be reading it when the next call overwrites it).
 *  - All calls share the one array, which keeps the last call's contents.  A
 *    call overwrites every scratch byte it reads, so nothing has to start at
 *    zero.  Calls ordered on one stream, from any host thread, are safe.
 *    Calls that can overlap on the GPU (on different streams, or graphs
 *    replayed concurrently) race on the array and produce wrong dgamma/dbeta.
 * Arguments, layouts, aliasing and errors are otherwise those of
 * ls_layernorm_bwd; with dgamma = dbeta = NULL no scratch is used. */
#define LS_NOALLOC_SCRATCH_BYTES ((size_t)8 << 20)
ls_status ls_layernorm_bwd_noalloc(ls_dtype dtype, void* dx, void* dgamma, void* dbeta,
                                   const void* dy, const void* x, const void* gamma,
                                   const float* mean, const float* rstd, int64_t rows,
                                   int64_t cols, void* stream);

/* Masked attention softmax over the last axis of [batch, heads, q_len, k_len]
 * ("CMU 11-868 L10 (LightSeq)", slides p.23-26; "CS336 Lecture 5: GPU", 6.1-6.2).
 * Entry (b, h, q, j) is valid iff j < clamp(key_len[b], 0, k_len) (key_len is a
 * device int32 [batch] array, or NULL for no padding mask) and, if causal,
 * j <= q + k_len - q_len.  On valid entries y = exp(x - m) / sum(exp(x - m)),
 * m = max of the valid x; masked entries are written as exactly 0 and are
 * not read; a row with no valid key is all zeros.  No 1/sqrt(d) scaling is
 * applied (the score GEMM applies it).  k_len <= 2^20; rows of up to 4096
 * keys (backward: 16384) are held on chip and read once, longer rows are read
 * twice (an online maximum-and-sum pass, then the output pass).  y may be x. */
ls_status ls_softmax_fwd(ls_dtype dtype, void* y, const void* x, int64_t batch, int64_t heads,
                         int64_t q_len, int64_t k_len, const int32_t* key_len, int causal,
                         void* stream);

/* Softmax backward:  dx = y * (dy - sum_valid(y * dy)) on valid entries, 0 on
 * masked ones (which are not read).  Same mask arguments as the forward.
 * dx may be dy. */
ls_status ls_softmax_bwd(ls_dtype dtype, void* dx, const void* y, const void* dy, int64_t batch,
                         int64_t heads, int64_t q_len, int64_t k_len, const int32_t* key_len,
                         int causal, void* stream);

/* Softmax fused with dropout on the attention probabilities ("CMU 11-868 L10
 * (LightSeq)", technique 1: the elementwise step after the softmax reduce
 * kernel joins it).  Same mask arguments and softmax y as ls_softmax_fwd, and
 *   bit(i) = keep(i) on valid entries, 0 on masked ones   (i = flat index of
 *            [batch, heads, q_len, k_len]; keep as for the other dropouts)
 *   y_drop = bit(i) * y / (1 - p)
 * y (needed by the backward), y_drop (fed to the next GEMM) and mask_bits
 * (ceil(n/32) words) are written.  None may overlap x or another output. */
ls_status ls_softmax_dropout_fwd(ls_dtype dtype, void* y, void* y_drop, uint32_t* mask_bits,
                                 const void* x, int64_t batch, int64_t heads, int64_t q_len,
                                 int64_t k_len, const int32_t* key_len, int causal, float p,
                                 uint64_t seed, uint64_t offset, void* stream);

/* Backward of the above: g = bit(i) * dy_drop / (1 - p), then
 *   dx = y * (g - sum_valid(y * g)) on valid entries, 0 on masked ones.
 * dx may be dy_drop. */
ls_status ls_softmax_dropout_bwd(ls_dtype dtype, void* dx, const void* y, const void* dy_drop,
                                 const uint32_t* mask_bits, int64_t batch, int64_t heads,
                                 int64_t q_len, int64_t k_len, const int32_t* key_len, int causal,
                                 float p, void* stream);

/* Embedding layer ("LightSeq2", section 2.1.2).  tokens: int32 [batch*seq]
 * ids (token i = b*seq + l sits at position l); token_table E: [vocab, hidden];
 * pos_table P: [max_positions >= seq, hidden]; y: [batch*seq, hidden]:
 *   y[i] = bit(i*hidden + c) * (scale * E[tokens[i]] + P[l]) / (1 - p)
 * with the keep bits of the other dropouts over the flat index of y, stored
 * in mask_bits (nullable; the backward needs it).  An id outside [0, vocab)
 * gives a zero row.  hidden must be a multiple of 8. */
ls_status ls_embedding_fwd(ls_dtype dtype, void* y, uint32_t* mask_bits, const int32_t* tokens,
                           const void* token_table, const void* pos_table, int64_t batch,
                           int64_t seq, int64_t hidden, int64_t vocab, int64_t max_positions,
                           float scale, float p, uint64_t seed, uint64_t offset, void* stream);

/* Workspace bytes ls_embedding_bwd needs for `tokens` tokens: 0 (the
 * deterministic backward keeps no scratch; the workspace arguments may be
 * NULL and 0). */
size_t ls_embedding_workspace_bytes(int64_t tokens);

/* Backward of the above into the token table's gradient, FP32 [vocab, hidden],
 * ACCUMULATED INTO (zero it first for a fresh gradient):
 *   d_token_table[w] += scale / (1 - p) * sum over tokens i with id w of bit * dy[i]
 * deterministic == 0: the pages' method, float atomic adds (one pass; the
 * order of the additions, so the last bits, vary from run to run; no
 * workspace).  deterministic != 0: the same bits on every run, each table row
 * updated once, in an order fixed by the ids: an id on at most three tokens
 * by the warp of its first token, which adds their rows in token order; an id
 * on four or more one 256-column block at a time, each block by one CTA,
 * whose 16 warps each add the block's rows of one of 16 equal position
 * slices (from the id's first token on) in token order, the slice sums then
 * added in slice order.  No workspace; at most 16384 tokens
 * per call, calls on one stream accumulate in order.  The position table gets
 * no gradient (the pages' formula has none). */
ls_status ls_embedding_bwd(ls_dtype dtype, float* d_token_table, const void* dy,
                           const uint32_t* mask_bits, const int32_t* tokens, int64_t batch,
                           int64_t seq, int64_t hidden, int64_t vocab, float scale, float p,
                           int deterministic, void* workspace, size_t workspace_bytes,
                           void* stream);

/* Cross entropy over vocabulary rows ("CMU 11-868 L10 (LightSeq)", technique 1,
 * slide p.12: one of the custom reduce kernels; its normaliser is the online
 * softmax of "CS336 Lecture 5: GPU", section 6.2, so each row is read once).
 * logits: [rows, vocab] (vocab a multiple of 8; pad the vocabulary), target:
 * int32 [rows] on the device.  Per row, with lse = log sum_j exp(z_j) and label
 * smoothing eps in [0, 1):
 *   loss = (1 - eps) * (lse - z[target]) + eps * (lse - mean_j z_j)
 * loss and lse (nullable; the backward needs it) are FP32 [rows].  A target
 * equal to ignore_index, or outside [0, vocab), gives loss 0. */
ls_status ls_cross_entropy_fwd(ls_dtype dtype, float* loss, float* lse, const void* logits,
                               const int32_t* target, int64_t rows, int64_t vocab,
                               float label_smoothing, int32_t ignore_index, void* stream);

/* Backward of the above, from the forward's lse:
 *   dlogits = dloss[row] * (exp(z - lse) - (1 - eps) * onehot(target) - eps / vocab)
 * dloss: FP32 [rows], or NULL for 1.  Ignored rows get a zero gradient.
 * dlogits may be logits (in place). */
ls_status ls_cross_entropy_bwd(ls_dtype dtype, void* dlogits, const void* logits,
                               const int32_t* target, const float* lse, const float* dloss,
                               int64_t rows, int64_t vocab, float label_smoothing,
                               int32_t ignore_index, void* stream);

/* Bias + reshape of Q, K, V ("CMU 11-868 L10 (LightSeq)", technique 1,
 * slide p.12: one fused elementwise kernel after the QKV projection GEMM).
 * qkv: [batch*seq, 3*H] row-major, H = heads*head_dim, row b*seq + l holding
 * Q, K, V in that order, each split into heads of head_dim; bias: [3*H].
 *   q_k_v[s, b, h, l, j] = qkv[b*seq + l, s*H + h*head_dim + j] + bias[s*H + h*head_dim + j]
 * q_k_v: [3, batch, heads, seq, head_dim] (Q at offset 0, K, V after it).
 * head_dim must be a multiple of 8.  q_k_v may not overlap qkv or bias.  No
 * 1/sqrt(head_dim) scaling (the score GEMM applies it). */
ls_status ls_bias_reshape_qkv_fwd(ls_dtype dtype, void* q_k_v, const void* qkv, const void* bias,
                                  int64_t batch, int64_t seq, int64_t heads, int64_t head_dim,
                                  void* stream);

/* Backward of the above: dqkv[b*seq + l, s*H + h*head_dim + j] = dq_k_v[s, b, h, l, j];
 * dbias[c] = sum over rows of dqkv[., c] (deterministic; workspace of at least
 * ls_colreduce_workspace_bytes(batch*seq, 3*H) bytes when dbias is not NULL).
 * dqkv may not overlap dq_k_v. */
ls_status ls_bias_reshape_qkv_bwd(ls_dtype dtype, void* dqkv, void* dbias, const void* dq_k_v,
                                  int64_t batch, int64_t seq, int64_t heads, int64_t head_dim,
                                  void* workspace, size_t workspace_bytes, void* stream);

/* Fused trainer update over a flat workspace ("CMU 11-868 L10 (LightSeq)",
 * technique 3 "mixed precision", slide p.29; "LightSeq2", section 2.3): the
 * parameters and gradients of a whole model in one contiguous workspace are
 * updated by one launch, read in the storage dtype, converted to FP32 in
 * registers and written back -- no FP32 copy of either is kept.  The rule (the
 * pages say "e.g. Adam") is Adam with bias correction (Kingma & Ba, ICLR 2015)
 * and decoupled weight decay (Loshchilov & Hutter, ICLR 2019), at step t >= 1:
 *   g' = grad * grad_scale                  (grad_scale = 1 / loss scale)
 *   exp_avg'    = beta1 * exp_avg + (1 - beta1) * g'
 *   exp_avg_sq' = beta2 * exp_avg_sq + (1 - beta2) * g'^2
 *   param' = param * (1 - lr * weight_decay)
 *            - lr * (exp_avg' / (1 - beta1^t)) / (sqrt(exp_avg_sq' / (1 - beta2^t)) + eps)
 * param, grad: [n] in the storage dtype; exp_avg, exp_avg_sq: [n] FP32, all
 * updated in place (none may overlap another or grad).  Any n >= 0 (n == 0 is
 * a no-op); 0 <= beta < 1; lr, eps, weight_decay >= 0 and finite; grad_scale
 * finite.  Every pointer 16-byte aligned. */
ls_status ls_adam_update(ls_dtype dtype, void* param, const void* grad, float* exp_avg,
                         float* exp_avg_sq, int64_t n, float lr, float beta1, float beta2,
                         float eps, float weight_decay, int64_t step, float grad_scale,
                         void* stream);

#ifdef __cplusplus
}
#endif
#endif /* LS_OPS_H */
