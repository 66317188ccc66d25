/*
 * ls_oracle.c -- FP64 CPU oracle (test infrastructure only; see ls_oracle.h).
 *
 * Each function writes out the plain definition of what the fused operator
 * computes, element by element, in double precision.  Where the fast method
 * reaches the same result by a rewrite (the single-sync LayerNorm statistics,
 * the two-sum LayerNorm backward) this file does NOT follow the rewrite: it
 * computes the textbook two-pass definition, so that the rewrite is checked
 * against the definition rather than against itself.
 *
 * Sources (page title, section):
 *  [L10]  "CMU 11-868 L10: accelerating the Transformer on GPUs (LightSeq)",
 *         section "Technique 1: kernel fusion" (the fused bias+dropout+residual,
 *         bias+ReLU+dropout, LayerNorm and softmax operators, slide p.12) and
 *         section "Technique 2: rewrite the formula" (LayerNorm statistics,
 *         slide p.21; LayerNorm backward, slide p.22; softmax, slides p.23-26).
 *  [LS2]  "LightSeq2: Accelerated Training for Transformer-based Models on GPUs",
 *         section 2.1.1 (Transformer-layer operator taxonomy and the fused
 *         bias+dropout+residual example) and section 2.1.2 (dropout with a
 *         saved mask m reused in the backward pass).
 *  [CS336] "CS336 Lecture 5: GPU", section 6.1 (row softmax of the attention
 *         score matrix) and section 6.2 (the max-subtracted softmax).
 *  Philox-4x32-10: Salmon, Moraes, Dror, Shaw, "Parallel Random Numbers: As
 *         Easy as 1, 2, 3", SC'11 (the pages name no generator).
 *  Bias + reshape of Q, K, V: [L10] section "Technique 1: kernel fusion"
 *         (slide p.12 lists "add bias + reshape Q, K, V" as one fused
 *         elementwise kernel next to the QKV projection GEMM).
 *  Cross entropy: [L10] section "Technique 1: kernel fusion" (slide p.12 names
 *         cross entropy among the custom reduce kernels); its single-pass
 *         normaliser is the online softmax of [CS336] section 6.2 (the pages
 *         give no criterion formula: the oracle writes the textbook one, with
 *         optional label smoothing, Szegedy et al., CVPR 2016).
 *  Embedding: [LS2] section 2.1.2 (token and position embeddings, scaled,
 *         dropped out; the backward adds every position's gradient of a
 *         token into its row of the table).
 *  Trainer update: [L10] section "Technique 3: mixed precision" (slide p.29)
 *         and [LS2] section 2.3 (one update over the FP16 parameter/gradient
 *         workspace, computed in FP32 registers); the update rule is Adam
 *         (Kingma & Ba, ICLR 2015, Algorithm 1) with decoupled weight decay
 *         (Loshchilov & Hutter, ICLR 2019), which the pages name only as
 *         "e.g. Adam".
 */
#include "ls_oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* ------------------------------------------------------------------------- */
/* Philox-4x32-10 (SC'11, section 3.3 "Philox"; constants from its table of   */
/* multipliers and Weyl key increments).                                      */
/* ------------------------------------------------------------------------- */
#define PHILOX_M0 0xD2511F53u
#define PHILOX_M1 0xCD9E8D57u
#define PHILOX_W0 0x9E3779B9u
#define PHILOX_W1 0xBB67AE85u

void or_philox4x32_10(const uint32_t ctr[4], const uint32_t key[2], uint32_t out[4]) {
    uint32_t c0 = ctr[0], c1 = ctr[1], c2 = ctr[2], c3 = ctr[3];
    uint32_t k0 = key[0], k1 = key[1];
    for (int round = 0; round < 10; ++round) {
        if (round > 0) { /* key schedule: add the Weyl constants between rounds */
            k0 += PHILOX_W0;
            k1 += PHILOX_W1;
        }
        uint64_t p0 = (uint64_t)PHILOX_M0 * (uint64_t)c0;
        uint64_t p1 = (uint64_t)PHILOX_M1 * (uint64_t)c2;
        uint32_t n0 = (uint32_t)(p1 >> 32) ^ c1 ^ k0;
        uint32_t n1 = (uint32_t)p1;
        uint32_t n2 = (uint32_t)(p0 >> 32) ^ c3 ^ k1;
        uint32_t n3 = (uint32_t)p0;
        c0 = n0; c1 = n1; c2 = n2; c3 = n3;
    }
    out[0] = c0; out[1] = c1; out[2] = c2; out[3] = c3;
}

/* Reading (the pages name no generator): the key is the 64-bit seed, the
 * counter's low half is the 128-bit block number i>>2 and its high half is the
 * call's 64-bit offset; element i takes 32-bit word i&3 of its block. */
uint32_t or_dropout_word(uint64_t seed, uint64_t offset, uint64_t i) {
    uint64_t block = i >> 2;
    uint32_t ctr[4] = {(uint32_t)block, (uint32_t)(block >> 32), (uint32_t)offset,
                       (uint32_t)(offset >> 32)};
    uint32_t key[2] = {(uint32_t)seed, (uint32_t)(seed >> 32)};
    uint32_t out[4];
    or_philox4x32_10(ctr, key, out);
    return out[i & 3];
}

/* Keep with probability 1 - p: a uniform 32-bit word u keeps the element iff
 * u >= floor(p * 2^32) (clamped to 2^32 - 1).  p is the FP32 value the caller
 * passes; p = 0 keeps everything. */
uint32_t or_dropout_threshold(float p) {
    double t = floor((double)p * 4294967296.0);
    if (t <= 0.0) return 0u;
    if (t >= 4294967295.0) return 4294967295u;
    return (uint32_t)t;
}

static int keep_bit(uint64_t seed, uint64_t offset, uint64_t i, uint32_t thr) {
    return or_dropout_word(seed, offset, i) >= thr;
}

static int64_t mask_word_count(int64_t n) { return (n + 31) / 32; }

static int get_bit(const uint32_t* words, int64_t i) {
    return (int)((words[i >> 5] >> (i & 31)) & 1u);
}

void or_dropout_keep_bits(int64_t n, float p, uint64_t seed, uint64_t offset, uint32_t* words) {
    uint32_t thr = or_dropout_threshold(p);
    memset(words, 0, (size_t)mask_word_count(n) * sizeof(uint32_t));
    for (int64_t i = 0; i < n; ++i)
        if (keep_bit(seed, offset, (uint64_t)i, thr)) words[i >> 5] |= 1u << (i & 31);
}

/* ------------------------------------------------------------------------- */
/* bias + dropout + residual  ([L10] technique 1; [LS2] 2.1.1)                */
/* ------------------------------------------------------------------------- */
void or_bdr_fwd(int64_t rows, int64_t cols, const double* x, const double* bias,
                const double* residual, float p, uint64_t seed, uint64_t offset,
                double* out, uint32_t* mask_words) {
    const uint32_t thr = or_dropout_threshold(p);
    const double scale = 1.0 / (1.0 - (double)p);
    const int64_t n = rows * cols;
    if (mask_words) memset(mask_words, 0, (size_t)mask_word_count(n) * sizeof(uint32_t));
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < rows; ++r) {
        for (int64_t c = 0; c < cols; ++c) {
            int64_t i = r * cols + c;
            int keep = keep_bit(seed, offset, (uint64_t)i, thr);
            double z = x[i] + bias[c];
            out[i] = residual[i] + (keep ? z * scale : 0.0);
        }
    }
    if (mask_words)
        for (int64_t i = 0; i < n; ++i)
            if (keep_bit(seed, offset, (uint64_t)i, thr)) mask_words[i >> 5] |= 1u << (i & 31);
}

/* Shared by both dropout backward passes: dx = bit * dout / (1 - p), and the
 * bias gradient is the column sum of dx (the bias is broadcast over rows). */
static void dropout_bwd_core(int64_t rows, int64_t cols, const double* dout,
                             const uint32_t* mask_words, int regen, uint32_t thr,
                             uint64_t seed, uint64_t offset, float p, double* dx,
                             double* dbias) {
    const double scale = 1.0 / (1.0 - (double)p);
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < rows; ++r) {
        for (int64_t c = 0; c < cols; ++c) {
            int64_t i = r * cols + c;
            int bit = regen ? keep_bit(seed, offset, (uint64_t)i, thr) : get_bit(mask_words, i);
            dx[i] = bit ? dout[i] * scale : 0.0;
        }
    }
    if (dbias) {
        for (int64_t c = 0; c < cols; ++c) {
            double s = 0.0;
            for (int64_t r = 0; r < rows; ++r) s += dx[r * cols + c];
            dbias[c] = s;
        }
    }
}

void or_bdr_bwd(int64_t rows, int64_t cols, const double* dout, const uint32_t* mask_words,
                float p, uint64_t seed, uint64_t offset, double* dx, double* dbias) {
    dropout_bwd_core(rows, cols, dout, mask_words, mask_words == NULL, or_dropout_threshold(p),
                     seed, offset, p, dx, dbias);
}

/* ------------------------------------------------------------------------- */
/* bias + ReLU + dropout  ([L10] technique 1).  ReLU(0) = 0 and its slope at  */
/* 0 is taken as 0, so the saved bit is (z > 0) and keep.                     */
/* ------------------------------------------------------------------------- */
void or_brd_fwd(int64_t rows, int64_t cols, const double* x, const double* bias,
                float p, uint64_t seed, uint64_t offset, double* out, uint32_t* mask_words) {
    const uint32_t thr = or_dropout_threshold(p);
    const double scale = 1.0 / (1.0 - (double)p);
    const int64_t n = rows * cols;
    if (mask_words) memset(mask_words, 0, (size_t)mask_word_count(n) * sizeof(uint32_t));
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < rows; ++r) {
        for (int64_t c = 0; c < cols; ++c) {
            int64_t i = r * cols + c;
            double z = x[i] + bias[c];
            int bit = (z > 0.0) && keep_bit(seed, offset, (uint64_t)i, thr);
            out[i] = bit ? z * scale : 0.0;
        }
    }
    if (mask_words)
        for (int64_t r = 0; r < rows; ++r)
            for (int64_t c = 0; c < cols; ++c) {
                int64_t i = r * cols + c;
                double z = x[i] + bias[c];
                if ((z > 0.0) && keep_bit(seed, offset, (uint64_t)i, thr))
                    mask_words[i >> 5] |= 1u << (i & 31);
            }
}

void or_brd_bwd(int64_t rows, int64_t cols, const double* dout, const uint32_t* mask_words,
                float p, double* dx, double* dbias) {
    dropout_bwd_core(rows, cols, dout, mask_words, 0, 0u, 0u, 0u, p, dx, dbias);
}

/* ------------------------------------------------------------------------- */
/* LayerNorm ([L10] technique 2, slides p.21-22).  Definition, two passes:    */
/*   mu = mean(x);  var = mean((x - mu)^2);  rstd = 1 / sqrt(var + eps)       */
/*   y  = gamma * (x - mu) * rstd + beta                                       */
/* ------------------------------------------------------------------------- */
static void row_stats(const double* xr, int64_t cols, double eps, double* mu_out,
                      double* rstd_out) {
    double s = 0.0;
    for (int64_t c = 0; c < cols; ++c) s += xr[c];
    double mu = s / (double)cols;
    double v = 0.0;
    for (int64_t c = 0; c < cols; ++c) v += (xr[c] - mu) * (xr[c] - mu);
    v /= (double)cols;
    *mu_out = mu;
    *rstd_out = 1.0 / sqrt(v + eps);
}

void or_layernorm_fwd(int64_t rows, int64_t cols, const double* x, const double* gamma,
                      const double* beta, double eps, double* y, double* mean, double* rstd) {
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < rows; ++r) {
        const double* xr = x + r * cols;
        double mu, rs;
        row_stats(xr, cols, eps, &mu, &rs);
        for (int64_t c = 0; c < cols; ++c) y[r * cols + c] = gamma[c] * (xr[c] - mu) * rs + beta[c];
        if (mean) mean[r] = mu;
        if (rstd) rstd[r] = rs;
    }
}

/* Textbook LayerNorm gradient with xhat = (x - mu) * rstd and g = gamma * dy:
 *   dx     = rstd * (g - mean(g) - xhat * mean(g * xhat))
 *   dgamma = sum over rows of dy * xhat,   dbeta = sum over rows of dy.
 * The statistics are recomputed here from x by the definition above. */
void or_layernorm_bwd(int64_t rows, int64_t cols, const double* dy, const double* x,
                      const double* gamma, double eps, double* dx, double* dgamma,
                      double* dbeta) {
    double* xhat = (double*)malloc((size_t)(rows * cols) * sizeof(double));
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < rows; ++r) {
        const double* xr = x + r * cols;
        const double* dyr = dy + r * cols;
        double mu, rs;
        row_stats(xr, cols, eps, &mu, &rs);
        double mean_g = 0.0, mean_gx = 0.0;
        for (int64_t c = 0; c < cols; ++c) {
            double xh = (xr[c] - mu) * rs;
            xhat[r * cols + c] = xh;
            double g = gamma[c] * dyr[c];
            mean_g += g;
            mean_gx += g * xh;
        }
        mean_g /= (double)cols;
        mean_gx /= (double)cols;
        for (int64_t c = 0; c < cols; ++c) {
            double xh = xhat[r * cols + c];
            double g = gamma[c] * dyr[c];
            dx[r * cols + c] = rs * (g - mean_g - xh * mean_gx);
        }
    }
    for (int64_t c = 0; c < cols; ++c) {
        double sg = 0.0, sb = 0.0;
        for (int64_t r = 0; r < rows; ++r) {
            sg += dy[r * cols + c] * xhat[r * cols + c];
            sb += dy[r * cols + c];
        }
        if (dgamma) dgamma[c] = sg;
        if (dbeta) dbeta[c] = sb;
    }
    free(xhat);
}

/* ------------------------------------------------------------------------- */
/* Masked softmax over the key axis ([L10] slides p.23-26; [CS336] 6.1-6.2).  */
/* ------------------------------------------------------------------------- */
static int64_t valid_len(int64_t b, int64_t q, int64_t q_len, int64_t k_len,
                         const int32_t* key_len, int causal) {
    int64_t v = k_len;
    if (key_len) {
        int64_t kl = key_len[b];
        if (kl < 0) kl = 0;
        if (kl < v) v = kl;
    }
    if (causal) {
        int64_t last = q + k_len - q_len; /* last key the query may see */
        if (last + 1 < v) v = last + 1;
    }
    return v < 0 ? 0 : v;
}

void or_softmax_fwd(int64_t batch, int64_t heads, int64_t q_len, int64_t k_len,
                    const double* x, const int32_t* key_len, int causal, double* y) {
    const int64_t nrows = batch * heads * q_len;
#pragma omp parallel for schedule(static)
    for (int64_t row = 0; row < nrows; ++row) {
        int64_t b = row / (heads * q_len);
        int64_t q = row % q_len;
        const double* xr = x + row * k_len;
        double* yr = y + row * k_len;
        int64_t v = valid_len(b, q, q_len, k_len, key_len, causal);
        double m = -INFINITY;
        for (int64_t j = 0; j < v; ++j)
            if (xr[j] > m) m = xr[j];
        double s = 0.0;
        for (int64_t j = 0; j < v; ++j) s += exp(xr[j] - m);
        for (int64_t j = 0; j < k_len; ++j) yr[j] = (j < v) ? exp(xr[j] - m) / s : 0.0;
    }
}

/* dx = y * (dy - <y, dy>) over the valid keys, 0 on masked keys (the
 * Jacobian-vector product of the row softmax). */
void or_softmax_bwd(int64_t batch, int64_t heads, int64_t q_len, int64_t k_len,
                    const double* y, const double* dy, const int32_t* key_len, int causal,
                    double* dx) {
    const int64_t nrows = batch * heads * q_len;
#pragma omp parallel for schedule(static)
    for (int64_t row = 0; row < nrows; ++row) {
        int64_t b = row / (heads * q_len);
        int64_t q = row % q_len;
        const double* yr = y + row * k_len;
        const double* dyr = dy + row * k_len;
        double* dxr = dx + row * k_len;
        int64_t v = valid_len(b, q, q_len, k_len, key_len, causal);
        double dot = 0.0;
        for (int64_t j = 0; j < v; ++j) dot += yr[j] * dyr[j];
        for (int64_t j = 0; j < k_len; ++j) dxr[j] = (j < v) ? yr[j] * (dyr[j] - dot) : 0.0;
    }
}

int or_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

void or_set_num_threads(int n) {
#ifdef _OPENMP
    if (n > 0) omp_set_num_threads(n);
#else
    (void)n;
#endif
}

/* ------------------------------------------------------------------------- */
/* Trainer update ([LS2] 2.3): Adam with bias correction and decoupled weight */
/* decay, by the definitions, one element at a time.                          */
/* ------------------------------------------------------------------------- */
void or_adam_update(int64_t n, const double* p, const double* g, const double* m,
                    const double* v, double lr, double beta1, double beta2, double eps,
                    double weight_decay, int64_t step, double grad_scale, double* p_out,
                    double* m_out, double* v_out) {
    const double bc1 = 1.0 - pow(beta1, (double)step); /* bias corrections */
    const double bc2 = 1.0 - pow(beta2, (double)step);
    for (int64_t i = 0; i < n; ++i) {
        const double gi = g[i] * grad_scale;                  /* unscaled gradient */
        const double mi = beta1 * m[i] + (1.0 - beta1) * gi;  /* first moment */
        const double vi = beta2 * v[i] + (1.0 - beta2) * gi * gi; /* second moment */
        const double m_hat = mi / bc1;
        const double v_hat = vi / bc2;
        const double decayed = p[i] - lr * weight_decay * p[i]; /* decoupled decay */
        p_out[i] = decayed - lr * m_hat / (sqrt(v_hat) + eps);
        m_out[i] = mi;
        v_out[i] = vi;
    }
}

/* ------------------------------------------------------------------------- */
/* Bias + reshape Q, K, V ([L10] technique 1, slide p.12).  The fused QKV     */
/* projection writes one row of 3*H values per token (row = b*seq + l), the   */
/* H = heads*d columns of Q, then of K, then of V, each split into heads of d */
/* columns.  The kernel adds the bias and moves every value to the head-major */
/* layout [3, batch, heads, seq, d] that the attention GEMMs read.            */
/* ------------------------------------------------------------------------- */
static int64_t qkv_out_index(int64_t batch, int64_t seq, int64_t heads, int64_t d, int64_t row,
                             int64_t c) {
    const int64_t H = heads * d;
    const int64_t s = c / H, h = (c % H) / d, j = c % d; /* which of Q/K/V, head, lane */
    const int64_t b = row / seq, l = row % seq;
    return (((s * batch + b) * heads + h) * seq + l) * d + j;
}

void or_bias_reshape_qkv_fwd(int64_t batch, int64_t seq, int64_t heads, int64_t d,
                             const double* qkv, const double* bias, double* out) {
    const int64_t rows = batch * seq, cols = 3 * heads * d;
    for (int64_t r = 0; r < rows; ++r)
        for (int64_t c = 0; c < cols; ++c)
            out[qkv_out_index(batch, seq, heads, d, r, c)] = qkv[r * cols + c] + bias[c];
}

void or_bias_reshape_qkv_bwd(int64_t batch, int64_t seq, int64_t heads, int64_t d,
                             const double* dout, double* dqkv, double* dbias) {
    const int64_t rows = batch * seq, cols = 3 * heads * d;
    for (int64_t c = 0; c < cols; ++c) dbias[c] = 0.0;
    for (int64_t r = 0; r < rows; ++r)
        for (int64_t c = 0; c < cols; ++c) {
            const double g = dout[qkv_out_index(batch, seq, heads, d, r, c)];
            dqkv[r * cols + c] = g;
            dbias[c] += g; /* rows added in order */
        }
}

/* ------------------------------------------------------------------------- */
/* Softmax with dropout on the probabilities ([L10] technique 1: the dropout  */
/* after the attention softmax joins the softmax kernel).  bit = keep on      */
/* valid entries, 0 on masked ones; y_drop = bit * y / (1 - p).               */
/* ------------------------------------------------------------------------- */
void or_softmax_dropout_fwd(int64_t batch, int64_t heads, int64_t q_len, int64_t k_len,
                            const double* x, const int32_t* key_len, int causal, float p,
                            uint64_t seed, uint64_t offset, double* y, double* y_drop,
                            uint32_t* mask_words) {
    or_softmax_fwd(batch, heads, q_len, k_len, x, key_len, causal, y);
    const uint32_t thr = or_dropout_threshold(p);
    const double scale = 1.0 / (1.0 - (double)p);
    const int64_t nrows = batch * heads * q_len;
    memset(mask_words, 0, (size_t)mask_word_count(nrows * k_len) * sizeof(uint32_t));
    for (int64_t row = 0; row < nrows; ++row) {
        const int64_t v = valid_len(row / (heads * q_len), row % q_len, q_len, k_len, key_len,
                                    causal);
        for (int64_t j = 0; j < k_len; ++j) {
            const int64_t i = row * k_len + j;
            const int bit = j < v && keep_bit(seed, offset, (uint64_t)i, thr);
            if (bit) mask_words[i >> 5] |= 1u << (i & 31);
            y_drop[i] = bit ? y[i] * scale : 0.0;
        }
    }
}

/* g = bit * dy_drop / (1 - p);  dx = y * (g - <y, g>) on valid keys, 0 on masked. */
void or_softmax_dropout_bwd(int64_t batch, int64_t heads, int64_t q_len, int64_t k_len,
                            const double* y, const double* dy_drop, const uint32_t* mask_words,
                            const int32_t* key_len, int causal, float p, double* dx) {
    const double scale = 1.0 / (1.0 - (double)p);
    const int64_t nrows = batch * heads * q_len;
    for (int64_t row = 0; row < nrows; ++row) {
        const int64_t v = valid_len(row / (heads * q_len), row % q_len, q_len, k_len, key_len,
                                    causal);
        const double* yr = y + row * k_len;
        double dot = 0.0;
        for (int64_t j = 0; j < v; ++j) {
            const int64_t i = row * k_len + j;
            const double g = get_bit(mask_words, i) ? dy_drop[i] * scale : 0.0;
            dot += yr[j] * g;
        }
        for (int64_t j = 0; j < k_len; ++j) {
            const int64_t i = row * k_len + j;
            const double g = get_bit(mask_words, i) ? dy_drop[i] * scale : 0.0;
            dx[i] = (j < v) ? yr[j] * (g - dot) : 0.0;
        }
    }
}

/* ------------------------------------------------------------------------- */
/* Cross entropy over vocabulary rows ([L10] technique 1, the criterion      */
/* reduce kernel), by the definitions.  Row t with target y:                  */
/*   lse = log sum_j exp(z_j);  p_j = exp(z_j - lse);                         */
/*   loss = (1-eps) (lse - z_y) + eps (lse - mean_j z_j);                     */
/*   dz_j = dloss * (p_j - (1-eps) [j == y] - eps / V).                        */
/* A target equal to ignore_index, or outside [0, V), gives loss 0 and dz 0. */
/* ------------------------------------------------------------------------- */
static double row_lse(const double* z, int64_t V) {
    double m = -INFINITY;
    for (int64_t j = 0; j < V; ++j)
        if (z[j] > m) m = z[j];
    double s = 0.0;
    for (int64_t j = 0; j < V; ++j) s += exp(z[j] - m);
    return m + log(s);
}

static int target_ok(int32_t y, int64_t V, int32_t ignore_index) {
    return y != ignore_index && y >= 0 && (int64_t)y < V;
}

void or_cross_entropy_fwd(int64_t rows, int64_t V, const double* logits, const int32_t* target,
                          double eps, int32_t ignore_index, double* loss, double* lse) {
#pragma omp parallel for schedule(static)
    for (int64_t t = 0; t < rows; ++t) {
        const double* z = logits + t * V;
        const double l = row_lse(z, V);
        if (lse) lse[t] = l;
        if (!target_ok(target[t], V, ignore_index)) {
            loss[t] = 0.0;
            continue;
        }
        double mean = 0.0;
        for (int64_t j = 0; j < V; ++j) mean += z[j];
        mean /= (double)V;
        loss[t] = (1.0 - eps) * (l - z[target[t]]) + eps * (l - mean);
    }
}

void or_cross_entropy_bwd(int64_t rows, int64_t V, const double* logits, const int32_t* target,
                          const double* dloss, double eps, int32_t ignore_index, double* dlogits) {
#pragma omp parallel for schedule(static)
    for (int64_t t = 0; t < rows; ++t) {
        const double* z = logits + t * V;
        double* dz = dlogits + t * V;
        if (!target_ok(target[t], V, ignore_index)) {
            for (int64_t j = 0; j < V; ++j) dz[j] = 0.0;
            continue;
        }
        const double l = row_lse(z, V);
        const double g = dloss ? dloss[t] : 1.0;
        for (int64_t j = 0; j < V; ++j) {
            const double q = (j == target[t] ? 1.0 - eps : 0.0) + eps / (double)V;
            dz[j] = g * (exp(z[j] - l) - q);
        }
    }
}

/* ------------------------------------------------------------------------- */
/* Embedding layer ([LS2] 2.1.2), by the definitions.  Token i = b*seq + l    */
/* with id w = tokens[i] at position l:                                       */
/*   y[i, :] = bit(i*H + c) * (s * E[w, c] + P[l, c]) / (1 - p)               */
/* (keep bits over the flat index of y, as for the other dropouts), and the  */
/* backward adds  s * bit * dy[i, c] / (1 - p)  into dE[w, c] for every i,    */
/* in increasing i.  Token ids outside [0, vocab) give a zero row and no      */
/* gradient.                                                                  */
/* ------------------------------------------------------------------------- */
void or_embedding_fwd(int64_t batch, int64_t seq, int64_t H, int64_t vocab,
                      const int32_t* tokens, const double* E, const double* P, double s,
                      float p, uint64_t seed, uint64_t offset, double* y, uint32_t* mask_words) {
    const uint32_t thr = or_dropout_threshold(p);
    const double scale = 1.0 / (1.0 - (double)p);
    const int64_t T = batch * seq;
    memset(mask_words, 0, (size_t)mask_word_count(T * H) * sizeof(uint32_t));
    for (int64_t i = 0; i < T; ++i) {
        const int64_t l = i % seq, w = tokens[i];
        for (int64_t c = 0; c < H; ++c) {
            const int64_t k = i * H + c;
            const int bit = keep_bit(seed, offset, (uint64_t)k, thr);
            if (bit) mask_words[k >> 5] |= 1u << (k & 31);
            const double v = (w >= 0 && w < vocab) ? s * E[w * H + c] + P[l * H + c] : 0.0;
            y[k] = bit ? v * scale : 0.0;
        }
    }
}

void or_embedding_bwd(int64_t T, int64_t H, int64_t vocab, const int32_t* tokens,
                      const double* dy, const uint32_t* mask_words, double s, float p,
                      double* dE) {
    const double scale = 1.0 / (1.0 - (double)p);
    for (int64_t i = 0; i < T; ++i) {
        const int64_t w = tokens[i];
        if (w < 0 || w >= vocab) continue;
        for (int64_t c = 0; c < H; ++c) {
            const int64_t k = i * H + c;
            if (get_bit(mask_words, k)) dE[w * H + c] += s * dy[k] * scale;
        }
    }
}

