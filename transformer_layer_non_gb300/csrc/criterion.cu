// criterion.cu -- cross entropy over vocabulary rows ("CMU 11-868 L10
// (LightSeq)", technique 1, slide p.12: cross entropy is one of the custom
// reduce kernels), forward and backward.
//
// Forward, one CTA per row: every thread walks its 16-byte vectors of the row
// once and keeps a running maximum m and a running sum l of exp(z - m),
// rescaling l when a vector raises the maximum -- the online softmax of
// "CS336 Lecture 5: GPU", section 6.2 -- plus the plain sum of z (for label
// smoothing) and, in the one thread that meets it, the target's logit.  The
// (m, l) pairs merge across the CTA by the same rule, so the row is read from
// HBM exactly once: lse = m + log l and
//   loss = (1 - eps) (lse - z[y]) + eps (lse - mean(z)).
// Backward, one CTA per row: dz = dloss * (exp(z - lse) - (1 - eps) [j == y]
// - eps / V), from the forward's lse; one read and one write per element.
// A target equal to ignore_index, or outside [0, V), gives loss 0 and a zero
// gradient row.
#include <math.h>

#include "ls_device.cuh"
#include "ls_internal.h"

namespace ls {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kUnroll = 4;  // vectors per thread in flight
constexpr float kLog2e = 1.4426950408889634f;

struct CeArgs {
    int64_t vocab;
    int nvec;  // vocab / 8
    float eps;
    int32_t ignore_index;
};

__device__ __forceinline__ bool target_ok(int32_t y, const CeArgs& a) {
    return y != a.ignore_index && y >= 0 && static_cast<int64_t>(y) < a.vocab;
}

// (m, l) <- the pair for the union of two element sets.
__device__ __forceinline__ void merge(float& m, float& l, float m2, float l2) {
    const float mm = fmaxf(m, m2);
    if (mm == -INFINITY) return;  // both empty
    l = l * exp2_approx((m - mm) * kLog2e) + l2 * exp2_approx((m2 - mm) * kLog2e);
    m = mm;
}

template <typename T>
__global__ void __launch_bounds__(kThreads)
ce_fwd_kernel(float* __restrict__ loss, float* __restrict__ lse_out, const T* __restrict__ logits,
              const int32_t* __restrict__ target, const __grid_constant__ CeArgs a) {
    __shared__ float sm_m[kWarps], sm_l[kWarps], sm_s[kWarps];
    __shared__ float sm_zy;
    pdl_enter();
    const int64_t row = blockIdx.x;
    const T* z = logits + row * a.vocab;
    const int32_t y = target[row];
    const int yv = (y >= 0) ? y / kVec : -1;
    if (threadIdx.x == 0) sm_zy = 0.f;
    float m = -INFINITY, l = 0.f, sz = 0.f, zy = 0.f;
    bool have_zy = false;
    for (int v0 = threadIdx.x; v0 < a.nvec; v0 += kThreads * kUnroll) {
        Raw8<T> r[kUnroll];
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            const int v = v0 + u * kThreads;
            if (v < a.nvec) r[u] = load8<T>(z + static_cast<int64_t>(v) * kVec);
        }
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            const int v = v0 + u * kThreads;
            if (v >= a.nvec) break;
            float f[kVec];
            unpack(r[u], f);
            const float vm = vmax8(r[u]);
            if (vm > m) {  // rescale the running sum to the new maximum
                l *= exp2_approx((m - vm) * kLog2e);
                m = vm;
            }
            const float ml = m == -INFINITY ? 0.f : m * kLog2e;  // all -inf so far: e = 0
#pragma unroll
            for (int j = 0; j < kVec; ++j) {
                l += exp2_approx(fmaf(f[j], kLog2e, -ml));
                sz += f[j];
            }
            if (v == yv) {
                zy = f[y - v * kVec];
                have_zy = true;
            }
        }
    }
    // Merge across the warp, then across warps (fixed order).
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const float m2 = __shfl_xor_sync(0xffffffffu, m, o);
        const float l2 = __shfl_xor_sync(0xffffffffu, l, o);
        merge(m, l, m2, l2);
        sz += __shfl_xor_sync(0xffffffffu, sz, o);
    }
    const int warp = threadIdx.x >> 5;
    __syncthreads();  // sm_zy initialised
    if (have_zy) sm_zy = zy;
    if ((threadIdx.x & 31) == 0) {
        sm_m[warp] = m;
        sm_l[warp] = l;
        sm_s[warp] = sz;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        float M = sm_m[0], Lsum = sm_l[0], S = sm_s[0];
        for (int w = 1; w < kWarps; ++w) {
            merge(M, Lsum, sm_m[w], sm_l[w]);
            S += sm_s[w];
        }
        const float lse = M + logf(Lsum);
        if (lse_out) lse_out[row] = lse;
        loss[row] = target_ok(y, a) ? (1.f - a.eps) * (lse - sm_zy) +
                                          a.eps * (lse - S / static_cast<float>(a.vocab))
                                    : 0.f;
    }
}

template <typename T>
__global__ void __launch_bounds__(kThreads)
ce_bwd_kernel(T* dlogits, const T* logits, const int32_t* __restrict__ target,
              const float* __restrict__ lse, const float* __restrict__ dloss,
              const __grid_constant__ CeArgs a) {
    pdl_enter();
    const int64_t row = blockIdx.x;
    const int32_t y = target[row];
    const bool ok = target_ok(y, a);
    const float g = ok ? (dloss ? dloss[row] : 1.f) : 0.f;
    const float ll = lse[row] * kLog2e;
    const float q0 = a.eps / static_cast<float>(a.vocab);
    const float qy = 1.f - a.eps + q0;
    const T* z = logits + row * a.vocab;
    T* dz = dlogits + row * a.vocab;
    for (int v0 = threadIdx.x; v0 < a.nvec; v0 += kThreads * kUnroll) {
        Raw8<T> r[kUnroll];
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            const int v = v0 + u * kThreads;
            if (v < a.nvec && ok) r[u] = load8<T>(z + static_cast<int64_t>(v) * kVec);
        }
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            const int v = v0 + u * kThreads;
            if (v >= a.nvec) break;
            float o[kVec];
            if (ok) {
                float f[kVec];
                unpack(r[u], f);
#pragma unroll
                for (int j = 0; j < kVec; ++j) {
                    const float q = (v * kVec + j == y) ? qy : q0;
                    o[j] = g * (exp2_approx(fmaf(f[j], kLog2e, -ll)) - q);
                }
            } else {
#pragma unroll
                for (int j = 0; j < kVec; ++j) o[j] = 0.f;
            }
            store8f<T>(dz + static_cast<int64_t>(v) * kVec, o);
        }
    }
}

CeArgs make_args(int64_t vocab, float eps, int32_t ignore_index) {
    CeArgs a;
    a.vocab = vocab;
    a.nvec = static_cast<int>(vocab / kVec);
    a.eps = eps;
    a.ignore_index = ignore_index;
    return a;
}

}  // namespace

cudaError_t launch_cross_entropy_fwd(DType dt, float* loss, float* lse, const void* logits,
                                     const int32_t* target, int64_t rows, int64_t vocab,
                                     float eps, int32_t ignore_index, cudaStream_t s) {
    const CeArgs a = make_args(vocab, eps, ignore_index);
    const dim3 grid(static_cast<unsigned>(rows));
    if (dt == DType::F16)
        return launch_pdl(ce_fwd_kernel<__half>, grid, dim3(kThreads), 0, s, loss, lse,
                          static_cast<const __half*>(logits), target, a);
    return launch_pdl(ce_fwd_kernel<float>, grid, dim3(kThreads), 0, s, loss, lse,
                      static_cast<const float*>(logits), target, a);
}

cudaError_t launch_cross_entropy_bwd(DType dt, void* dlogits, const void* logits,
                                     const int32_t* target, const float* lse, const float* dloss,
                                     int64_t rows, int64_t vocab, float eps, int32_t ignore_index,
                                     cudaStream_t s) {
    const CeArgs a = make_args(vocab, eps, ignore_index);
    const dim3 grid(static_cast<unsigned>(rows));
    if (dt == DType::F16)
        return launch_pdl(ce_bwd_kernel<__half>, grid, dim3(kThreads), 0, s,
                          static_cast<__half*>(dlogits), static_cast<const __half*>(logits),
                          target, lse, dloss, a);
    return launch_pdl(ce_bwd_kernel<float>, grid, dim3(kThreads), 0, s,
                      static_cast<float*>(dlogits), static_cast<const float*>(logits), target, lse,
                      dloss, a);
}

}  // namespace ls
