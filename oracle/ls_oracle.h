/*
 * ls_oracle.h -- FP64 CPU oracle for the fused non-GEMM Transformer-layer
 * operators (bias+dropout+residual, bias+ReLU+dropout, LayerNorm, masked
 * attention softmax; forward and backward).
 *
 * TEST INFRASTRUCTURE ONLY.  This is the plain, slow, obviously correct
 * definition that the CUDA path is checked against.  Only the tests, the
 * smoke check and the benchmark's CPU-baseline leg may call it.  It shares no
 * code, header, table or constant with the CUDA library.
 *
 * Every floating-point input is an FP64 array holding exactly the values the
 * GPU receives (FP16/FP32 storage values widen to FP64 without rounding).
 * Every result is FP64.  Layouts are row-major:
 *   activations  [rows, cols]            (rows = tokens, cols = hidden or FFN)
 *   scores       [batch, heads, q_len, k_len]
 *   dropout mask ceil(rows*cols/32) uint32 words; element i is bit (i & 31)
 *                of word (i >> 5); bits past the last element are 0.
 */
#ifndef LS_ORACLE_H
#define LS_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Philox-4x32 with 10 rounds (Salmon, Moraes, Dror, Shaw, "Parallel Random
 * Numbers: As Easy as 1, 2, 3", SC'11): out = Philox(ctr, key). */
void or_philox4x32_10(const uint32_t ctr[4], const uint32_t key[2], uint32_t out[4]);

/* The 32-bit uniform word that element i of a dropout call (seed, offset)
 * draws: block i>>2 of the counter stream, word i&3 of that block. */
uint32_t or_dropout_word(uint64_t seed, uint64_t offset, uint64_t i);

/* Keep threshold for drop probability p: element kept iff word >= threshold. */
uint32_t or_dropout_threshold(float p);

/* Keep bits of n elements (ceil(n/32) words). */
void or_dropout_keep_bits(int64_t n, float p, uint64_t seed, uint64_t offset, uint32_t* words);

/* bias + dropout + residual:  out = residual + keep * (x + bias[c]) / (1 - p) */
void or_bdr_fwd(int64_t rows, int64_t cols, const double* x, const double* bias,
                const double* residual, float p, uint64_t seed, uint64_t offset,
                double* out, uint32_t* mask_words);
/* dx = keep * dout / (1 - p);  dbias[c] = sum_r dx[r, c].  mask_words may be
 * NULL, in which case the keep bits are drawn again from (seed, offset). */
void or_bdr_bwd(int64_t rows, int64_t cols, const double* dout, const uint32_t* mask_words,
                float p, uint64_t seed, uint64_t offset, double* dx, double* dbias);

/* bias + ReLU + dropout:  z = x + bias[c];  bit = (z > 0) and keep;
 * out = bit * z / (1 - p). */
void or_brd_fwd(int64_t rows, int64_t cols, const double* x, const double* bias,
                float p, uint64_t seed, uint64_t offset, double* out, uint32_t* mask_words);
void or_brd_bwd(int64_t rows, int64_t cols, const double* dout, const uint32_t* mask_words,
                float p, double* dx, double* dbias);

/* LayerNorm over each row (biased variance, eps inside the square root). */
void or_layernorm_fwd(int64_t rows, int64_t cols, const double* x, const double* gamma,
                      const double* beta, double eps, double* y, double* mean, double* rstd);
void or_layernorm_bwd(int64_t rows, int64_t cols, const double* dy, const double* x,
                      const double* gamma, double eps, double* dx, double* dgamma,
                      double* dbeta);

/* Masked softmax along the last axis of [batch, heads, q_len, k_len].
 * key_len may be NULL (no padding mask).  Entry (b, h, q, j) is valid iff
 * j < clamp(key_len[b], 0, k_len) and, when causal, j <= q + k_len - q_len. */
void or_softmax_fwd(int64_t batch, int64_t heads, int64_t q_len, int64_t k_len,
                    const double* x, const int32_t* key_len, int causal, double* y);
void or_softmax_bwd(int64_t batch, int64_t heads, int64_t q_len, int64_t k_len,
                    const double* y, const double* dy, const int32_t* key_len, int causal,
                    double* dx);

/* Softmax (as or_softmax_fwd) with dropout on the probabilities: bit(i) =
 * keep(i) on valid entries and 0 on masked ones (mask_words: ceil(n/32)
 * words), y_drop = bit * y / (1 - p).  The backward takes the bits and the
 * gradient of y_drop: g = bit * dy_drop / (1 - p), dx = y * (g - <y, g>) on
 * valid entries, 0 on masked ones. */
void or_softmax_dropout_fwd(int64_t batch, int64_t heads, int64_t q_len, int64_t k_len,
                            const double* x, const int32_t* key_len, int causal, float p,
                            uint64_t seed, uint64_t offset, double* y, double* y_drop,
                            uint32_t* mask_words);
void or_softmax_dropout_bwd(int64_t batch, int64_t heads, int64_t q_len, int64_t k_len,
                            const double* y, const double* dy_drop, const uint32_t* mask_words,
                            const int32_t* key_len, int causal, float p, double* dx);

/* Embedding layer: y[i] = bit * (s * E[tokens[i]] + P[i % seq]) / (1 - p) for
 * the batch*seq tokens i (y: [batch*seq, H]; keep bits over the flat index of
 * y; ids outside [0, vocab) give zero rows).  The backward adds
 * s * bit * dy / (1 - p) of every token into dE[tokens[i]] (dE: [vocab, H],
 * accumulated into, token order increasing). */
void or_embedding_fwd(int64_t batch, int64_t seq, int64_t H, int64_t vocab,
                      const int32_t* tokens, const double* E, const double* P, double s,
                      float p, uint64_t seed, uint64_t offset, double* y, uint32_t* mask_words);
void or_embedding_bwd(int64_t T, int64_t H, int64_t vocab, const int32_t* tokens,
                      const double* dy, const uint32_t* mask_words, double s, float p,
                      double* dE);

/* Cross entropy over rows of V logits with integer targets and label
 * smoothing eps: loss[t] = (1-eps)(lse - z[y]) + eps(lse - mean(z)), lse =
 * log sum exp(z) (also returned when lse != NULL); the backward gives
 * dz = dloss[t] (softmax(z) - (1-eps) onehot(y) - eps/V) (dloss NULL: 1).
 * Targets equal to ignore_index or outside [0, V) give loss 0 and dz 0. */
void or_cross_entropy_fwd(int64_t rows, int64_t V, const double* logits, const int32_t* target,
                          double eps, int32_t ignore_index, double* loss, double* lse);
void or_cross_entropy_bwd(int64_t rows, int64_t V, const double* logits, const int32_t* target,
                          const double* dloss, double eps, int32_t ignore_index, double* dlogits);

/* Bias + reshape of the fused QKV projection output: qkv [batch*seq, 3*heads*d]
 * (per row: Q, K, V, each heads x d) plus bias [3*heads*d] into
 * out [3, batch, heads, seq, d]:
 *   out[s, b, h, l, j] = qkv[b*seq + l, s*H + h*d + j] + bias[s*H + h*d + j],  H = heads*d.
 * The backward moves dout [3, batch, heads, seq, d] back to dqkv
 * [batch*seq, 3*heads*d] and sums it over rows into dbias [3*heads*d]. */
void or_bias_reshape_qkv_fwd(int64_t batch, int64_t seq, int64_t heads, int64_t d,
                             const double* qkv, const double* bias, double* out);
void or_bias_reshape_qkv_bwd(int64_t batch, int64_t seq, int64_t heads, int64_t d,
                             const double* dout, double* dqkv, double* dbias);

/* Trainer update over a flat parameter workspace of n elements: Adam (Kingma &
 * Ba, ICLR 2015, Algorithm 1) with bias correction at step `step` (>= 1),
 * decoupled weight decay (Loshchilov & Hutter, ICLR 2019) and the gradient
 * multiplied by grad_scale first (1 / loss scale):
 *   g' = g*grad_scale;  m' = b1*m + (1-b1)*g';  v' = b2*v + (1-b2)*g'^2;
 *   p' = p - lr*wd*p - lr * (m'/(1-b1^t)) / (sqrt(v'/(1-b2^t)) + eps).
 * Outputs may alias the inputs. */
void or_adam_update(int64_t n, const double* p, const double* g, const double* m,
                    const double* v, double lr, double beta1, double beta2, double eps,
                    double weight_decay, int64_t step, double grad_scale, double* p_out,
                    double* m_out, double* v_out);

/* OpenMP threads the row loops use, and setting them (n > 0). */
int or_num_threads(void);
void or_set_num_threads(int n);

#ifdef __cplusplus
}
#endif
#endif
