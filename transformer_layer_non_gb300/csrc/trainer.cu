// trainer.cu -- the fused trainer update ("CMU 11-868 L10 (LightSeq)",
// technique 3 "mixed precision", slide p.29; "LightSeq2", section 2.3).  The
// parameters and gradients of the whole model sit in one flat FP16 workspace,
// so one launch updates all of them: each thread reads FP16 parameters and
// gradients into registers, converts them to FP32, applies the update and
// writes the parameters back in FP16 -- no FP32 copy of either lives in
// memory.  The pages name the rule only as Adam; this is Adam with bias
// correction (Kingma & Ba, ICLR 2015, Algorithm 1) and decoupled weight decay
// (Loshchilov & Hutter, ICLR 2019), the moments kept in FP32.
//
// Layout: a persistent grid (a multiple of the SM count) walks 8-element
// vectors -- one 16-byte load each of parameters and gradients in FP16, two
// each of the FP32 moments -- and a scalar tail covers n % 8.  22 bytes move
// per FP16 element; nothing is re-read.
#include "ls_device.cuh"
#include "ls_internal.h"

namespace ls {
namespace {

constexpr int kThreads = 256;

// Kernel arguments (constant bank).  The bias corrections are folded on the
// host: step_size = lr / (1 - beta1^t), inv_sqrt_bc2 = 1 / sqrt(1 - beta2^t).
struct AdamArgs {
    uint64_t nv;  // whole 8-element vectors
    uint64_t n;   // elements
    float b1, b2, omb1, omb2;
    float step_size, inv_sqrt_bc2, eps;
    float decay;  // 1 - lr * weight_decay
    float grad_scale;
};

// One element, in FP32: g' = g * grad_scale; m' = b1 m + (1 - b1) g';
// v' = b2 v + (1 - b2) g'^2; p' = p (1 - lr wd) - lr m'/(1 - b1^t) /
// (sqrt(v'/(1 - b2^t)) + eps).
__device__ __forceinline__ void adam1(float& p, float g, float& m, float& v, const AdamArgs& a) {
    g *= a.grad_scale;
    m = a.b1 * m + a.omb1 * g;
    v = a.b2 * v + a.omb2 * (g * g);
    const float denom = sqrtf(v) * a.inv_sqrt_bc2 + a.eps;
    p = p * a.decay - a.step_size * m / denom;
}

template <typename T> __device__ __forceinline__ float to_f(T x) { return static_cast<float>(x); }
template <> __device__ __forceinline__ float to_f<__half>(__half x) { return __half2float(x); }
template <typename T> __device__ __forceinline__ T from_f(float x) { return static_cast<T>(x); }
template <> __device__ __forceinline__ __half from_f<__half>(float x) { return __float2half_rn(x); }

template <typename T, typename I>
__global__ void __launch_bounds__(kThreads)
adam_kernel(T* __restrict__ param, const T* __restrict__ grad, float* __restrict__ m,
            float* __restrict__ v, const __grid_constant__ AdamArgs a) {
    pdl_enter();
    const I nv = static_cast<I>(a.nv);
    const I S = static_cast<I>(gridDim.x) * kThreads;
    for (I i = static_cast<I>(blockIdx.x) * kThreads + threadIdx.x; i < nv; i += S) {
        const size_t e = static_cast<size_t>(i) * kVec;
        float pf[kVec], gf[kVec];
        const Raw8<T> pr = load8<T>(param + e);
        const Raw8<T> gr = load8<T>(grad + e);
        float4 m0 = *reinterpret_cast<const float4*>(m + e);
        float4 m1 = *reinterpret_cast<const float4*>(m + e + 4);
        float4 v0 = *reinterpret_cast<const float4*>(v + e);
        float4 v1 = *reinterpret_cast<const float4*>(v + e + 4);
        unpack(pr, pf);
        unpack(gr, gf);
        float mf[kVec] = {m0.x, m0.y, m0.z, m0.w, m1.x, m1.y, m1.z, m1.w};
        float vf[kVec] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
#pragma unroll
        for (int j = 0; j < kVec; ++j) adam1(pf[j], gf[j], mf[j], vf[j], a);
        store8f<T>(param + e, pf);
        *reinterpret_cast<float4*>(m + e) = make_float4(mf[0], mf[1], mf[2], mf[3]);
        *reinterpret_cast<float4*>(m + e + 4) = make_float4(mf[4], mf[5], mf[6], mf[7]);
        *reinterpret_cast<float4*>(v + e) = make_float4(vf[0], vf[1], vf[2], vf[3]);
        *reinterpret_cast<float4*>(v + e + 4) = make_float4(vf[4], vf[5], vf[6], vf[7]);
    }
    // The last n % 8 elements, one per thread of the first CTA.
    const uint64_t j = a.nv * kVec + threadIdx.x;
    if (blockIdx.x == 0 && j < a.n) {
        float pf = to_f(param[j]), mf = m[j], vf = v[j];
        adam1(pf, to_f(grad[j]), mf, vf, a);
        param[j] = from_f<T>(pf);
        m[j] = mf;
        v[j] = vf;
    }
}

template <typename K>
int occupancy(K kernel) {
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kernel, kThreads, 0) != cudaSuccess ||
        n < 1)
        n = 1;
    return n;
}

template <typename T>
cudaError_t adam_impl(void* param, const void* grad, float* m, float* v, const AdamArgs& a,
                      cudaStream_t s) {
    static const int occ = occupancy(adam_kernel<T, uint64_t>);
    const int64_t want = static_cast<int64_t>((a.nv + kThreads - 1) / kThreads);
    const int64_t grid = std::max<int64_t>(1, std::min<int64_t>(want, int64_t{sm_count()} * occ));
    // 32-bit indices while no index the loop forms reaches 2^31.
    const bool narrow = a.nv + static_cast<uint64_t>(grid) * kThreads < (uint64_t{1} << 31);
    auto kern = narrow ? adam_kernel<T, uint32_t> : adam_kernel<T, uint64_t>;
    return launch_pdl(kern, dim3(static_cast<unsigned>(grid)), dim3(kThreads), 0, s,
                      static_cast<T*>(param), static_cast<const T*>(grad), m, v, a);
}

}  // namespace

cudaError_t launch_adam(DType dt, void* param, const void* grad, float* m, float* v, int64_t n,
                        const AdamHyper& h, cudaStream_t s) {
    AdamArgs a;
    a.n = static_cast<uint64_t>(n);
    a.nv = a.n / kVec;
    a.b1 = h.beta1;
    a.b2 = h.beta2;
    a.omb1 = 1.0f - h.beta1;
    a.omb2 = 1.0f - h.beta2;
    const double bc1 = 1.0 - pow(static_cast<double>(h.beta1), static_cast<double>(h.step));
    const double bc2 = 1.0 - pow(static_cast<double>(h.beta2), static_cast<double>(h.step));
    a.step_size = static_cast<float>(static_cast<double>(h.lr) / bc1);
    a.inv_sqrt_bc2 = static_cast<float>(1.0 / sqrt(bc2));
    a.eps = h.eps;
    a.decay = static_cast<float>(1.0 - static_cast<double>(h.lr) * h.weight_decay);
    a.grad_scale = h.grad_scale;
    if (dt == DType::F16) return adam_impl<__half>(param, grad, m, v, a, s);
    return adam_impl<float>(param, grad, m, v, a, s);
}

}  // namespace ls
