// ls_internal.h -- launchers behind the C ABI.  Arguments reaching these
// functions have been validated by ls_api.cu; each launcher only picks a
// kernel instance and grid for the shape and enqueues it on the stream.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "../../include/ls_ops.h"

namespace ls {

enum class DType { F32 = 0, F16 = 1 };

struct DropoutRng {
    uint32_t thr;       // keep iff Philox word >= thr
    float scale;        // 1 / (1 - p) in FP32
    uint64_t seed;
    uint64_t offset;
};

// Column-reduction plan shared by the launchers and the workspace query.
// Partial sums are FP32 [parts, width]; `parts` depends only on the shape, so
// results are bitwise reproducible on any GPU.
struct ColReducePlan {
    int64_t parts;
    int64_t width;
    size_t bytes() const { return static_cast<size_t>(parts * width) * sizeof(float); }
};
ColReducePlan dropout_bwd_plan(int64_t rows, int64_t cols);
ColReducePlan layernorm_bwd_plan(int64_t rows, int64_t cols, size_t esize);  // esize: 2 or 4

// Sum `parts` FP32 rows of `width` columns in a fixed order; columns
// [0, split) go to out0[0..split) and columns [split, width) to
// out1[0..width-split) (out1 may be null when split == width).
cudaError_t launch_colreduce(DType dt, void* out0, void* out1, int64_t split,
                             const float* partial, int64_t parts, int64_t width, cudaStream_t s);

cudaError_t launch_dropout_fwd(DType dt, bool relu, void* out, uint8_t* mask, const void* x,
                               const void* bias, const void* residual, int64_t rows, int64_t cols,
                               const DropoutRng& rng, cudaStream_t s);
// mask == nullptr: redraw keep bits from rng.  partial == nullptr: no bias gradient.
cudaError_t launch_dropout_bwd(DType dt, void* dx, float* partial, const void* dout,
                               const uint8_t* mask, int64_t rows, int64_t cols,
                               const DropoutRng& rng, cudaStream_t s);

cudaError_t launch_layernorm_fwd(DType dt, void* y, float* mean, float* rstd, const void* x,
                                 const void* gamma, const void* beta, int64_t rows, int64_t cols,
                                 float eps, cudaStream_t s);
cudaError_t launch_layernorm_bwd(DType dt, void* dx, float* partial, const void* dy,
                                 const void* x, const void* gamma, const float* mean,
                                 const float* rstd, int64_t rows, int64_t cols, cudaStream_t s);

struct SoftmaxShape {
    int64_t batch, heads, q_len, k_len;
    const int32_t* key_len;
    int causal;
};
cudaError_t launch_softmax_fwd(DType dt, void* y, const void* x, const SoftmaxShape& sh,
                               cudaStream_t s);
cudaError_t launch_softmax_bwd(DType dt, void* dx, const void* y, const void* dy,
                               const SoftmaxShape& sh, cudaStream_t s);
// Softmax fused with dropout on the probabilities: the forward also writes
// y_drop = bit * y / (1-p) and the bits (keep on valid entries, 0 on masked
// ones); the backward takes the gradient of y_drop and the bits.
cudaError_t launch_softmax_dropout_fwd(DType dt, void* y, void* y_drop, uint8_t* mask,
                                       const void* x, const SoftmaxShape& sh,
                                       const DropoutRng& rng, cudaStream_t s);
cudaError_t launch_softmax_dropout_bwd(DType dt, void* dx, const void* y, const void* dy_drop,
                                       const uint8_t* mask, const SoftmaxShape& sh, float scale,
                                       cudaStream_t s);

constexpr int64_t kMaxRowLen = 16384;          // LayerNorm rows
constexpr int64_t kMaxSoftmaxRowLen = 1 << 20;  // softmax rows (long rows read twice)

// Bias + reshape of Q, K, V: [batch*seq, 3*heads*d] (+ bias) <-> [3, batch,
// heads, seq, d].  The backward writes one FP32 partial row of the bias
// gradient per 128 rows (dropout_bwd_plan(batch*seq, 3*heads*d)) when partial
// is not null.
cudaError_t launch_qkv_fwd(DType dt, void* out, const void* qkv, const void* bias, int64_t batch,
                           int64_t seq, int64_t heads, int64_t d, cudaStream_t s);
cudaError_t launch_qkv_bwd(DType dt, void* dqkv, float* partial, const void* dout, int64_t batch,
                           int64_t seq, int64_t heads, int64_t d, cudaStream_t s);

// Embedding layer: gather + dropout forward; deterministic scatter-add
// backward into an FP32 dE (each id's sum in an order fixed by the ids; every
// CTA of 16 tokens stages and scans all the ids, so the work grows with the
// square of the tokens and the ids must fit in shared memory: at most
// kEmbeddingMaxTokens per call).
constexpr int64_t kEmbeddingMaxTokens = 16384;
cudaError_t launch_embedding_fwd(DType dt, void* y, uint8_t* mask, const int32_t* tokens,
                                 const void* E, const void* P, int64_t batch, int64_t seq,
                                 int64_t H, int64_t vocab, float s, const DropoutRng& rng,
                                 cudaStream_t st);
cudaError_t launch_embedding_bwd(DType dt, float* dE, const void* dy, const uint8_t* mask,
                                 const int32_t* tokens, int64_t T, int64_t H, int64_t vocab,
                                 float coef, cudaStream_t st);
cudaError_t launch_embedding_bwd_atomic(DType dt, float* dE, const void* dy, const uint8_t* mask,
                                        const int32_t* tokens, int64_t T, int64_t H,
                                        int64_t vocab, float coef, cudaStream_t st);

// Cross entropy over rows of `vocab` logits (vocab % 8 == 0), one CTA per row.
cudaError_t launch_cross_entropy_fwd(DType dt, float* loss, float* lse, const void* logits,
                                     const int32_t* target, int64_t rows, int64_t vocab,
                                     float eps, int32_t ignore_index, cudaStream_t s);
cudaError_t launch_cross_entropy_bwd(DType dt, void* dlogits, const void* logits,
                                     const int32_t* target, const float* lse, const float* dloss,
                                     int64_t rows, int64_t vocab, float eps, int32_t ignore_index,
                                     cudaStream_t s);

// Trainer update (Adam with decoupled weight decay) over a flat workspace.
struct AdamHyper {
    float lr, beta1, beta2, eps, weight_decay, grad_scale;
    int64_t step;
};
cudaError_t launch_adam(DType dt, void* param, const void* grad, float* m, float* v, int64_t n,
                        const AdamHyper& h, cudaStream_t s);

// Read and clear the device-side failure flags of one translation unit's
// kernels (synchronous).
cudaError_t softmax_take_device_error(unsigned int* flags);
// One warp waits (polls bounded polls) on a barrier nothing completes and
// records LS_DEVERR_WAIT_TIMEOUT in the softmax unit's failure word.
cudaError_t launch_wait_timeout_selftest(uint32_t polls, cudaStream_t s);
cudaError_t dropout_take_device_error(unsigned int* flags);
cudaError_t layernorm_take_device_error(unsigned int* flags);

// Streaming multiprocessors of the current device (queried once per device).
int sm_count();

// ls_layernorm_bwd with a choice of where the column reduction runs:
// inline_reduction keeps it on `stream` even when a reduction stream is set
// (the allocation-free entry point, whose scratch all host threads share).
ls_status layernorm_bwd_entry(ls_dtype dtype, void* dx, void* dgamma, void* dbeta, const void* dy,
                              const void* x, const void* gamma, const float* mean,
                              const float* rstd, int64_t rows, int64_t cols, void* workspace,
                              size_t workspace_bytes, void* stream, bool inline_reduction);

// Set this host thread's ls_last_error() message (printf-style).
void set_last_error_message(const char* fmt, ...);

}  // namespace ls
