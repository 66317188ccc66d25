// layernorm.cu -- LayerNorm forward and backward ("CMU 11-868 L10 (LightSeq)",
// technique 2 "rewrite the formula": slide p.21 computes mu(x) and mu(x^2)
// together so sigma = sqrt(mu(x^2) - mu(x)^2) needs one synchronisation
// instead of two; slide p.22 rewrites the backward as two independent sums
// plus elementwise work; FP32 arithmetic on FP16 storage).
//
// Row mapping.  Rows of up to 2048 elements are held in registers by a group
// of LPR lanes (LPR = 1..32, VPT 8-element vectors per lane); a CTA of 256
// threads holds 256/LPR rows.  Longer rows (up to 16384) use a whole CTA per
// row.  Each lane owns the same columns in every row it visits, so the
// backward's gamma/beta gradient partial sums never leave the SM until the
// CTA has finished its rows.
#include <algorithm>

#include "ls_device.cuh"
#include "ls_internal.h"

namespace ls {
namespace {

constexpr int kThreads = 256;
constexpr int kCtaRowThreshold = 256;  // vectors per row held by one warp at most

// ----------------------------------------------------------------------------
// Forward, group-per-row, persistent.  Row round k gives group slot q of CTA b
// the row k*stride + q*gridDim + b (stride = all groups), so a partial last
// round is spread over every CTA.  Each group keeps two register buffers: the
// next row's loads are in flight while the current row is reduced and stored,
// so a group with two rows waits for DRAM once.  At 3 vectors per lane (FP16)
// and for FP32 rows of 3 or more vectors the second buffer would spill; those
// keep one buffer (at 768 FP16 columns a 4096-row batch is one row per warp).
// Loop conditions are warp-uniform (__any_sync) because the groups of one warp
// reduce with full-warp shuffles.
// ----------------------------------------------------------------------------
template <typename T, int LPR, int VPT>
__device__ __forceinline__ void ln_fwd_load(Raw8<T> (&xr)[VPT], const T* x, int64_t r,
                                            int64_t rows, int cols, int gl) {
    if (r >= rows) return;
    const int nvec = cols / kVec;
#pragma unroll
    for (int k = 0; k < VPT; ++k) {
        const int v = gl + k * LPR;
        if (v < nvec) xr[k] = load8<T>(x + r * cols + v * kVec);
    }
}

// Element 0 of a vector as FP32.
__device__ __forceinline__ float first_elem(const Raw8<__half>& r) {
    return __low2float(*reinterpret_cast<const __half2*>(&r.v.x));
}
__device__ __forceinline__ float first_elem(const Raw8<float>& r) { return r.a.x; }

// Rows that keep two buffers at 4 or more vectors per lane: the output pass
// forms d = x - K again from the raw vector instead of keeping d in registers
// (the same subtract, so the same bits), which keeps the second buffer within
// the register budget.
template <typename T, int VPT>
constexpr bool ln_fwd_double() {
    return VPT <= 2 || (sizeof(T) == 2 && VPT >= 4);
}
template <typename T, int VPT>
constexpr bool ln_fwd_keep_d() {
    return VPT <= 3 || !ln_fwd_double<T, VPT>();
}

// One row of the forward.  The differences d = x - K from the row's first
// element K are formed once (FP16 converts exactly, folded into the subtract)
// and, where the registers allow, kept for both passes; the sums and the
// output use packed FP32 pairs.  Each result is the FP32 operation on the same operands, rounded
// once, as in the plain form.  gamma/beta are read per row, after the row's
// loads: measured on GB300, loading every lane's gamma/beta columns when the
// kernel starts is slower (4.8 against 4.1 us at 4096 x 768), as every warp
// then asks L2 for the same few lines at the same moment.
template <typename T, int LPR, int VPT>
__device__ __forceinline__ void ln_fwd_row(const Raw8<T> (&xr)[VPT], T* y, float* mean,
                                           float* rstd, const T* __restrict__ gamma,
                                           const T* __restrict__ beta, int64_t r, int64_t rows,
                                           int cols, float eps, int gl) {
    const bool row_ok = r < rows;
    const int nvec = cols / kVec;
    // Sums about the row's first element K (held by the group's lane 0):
    // var = mu((x-K)^2) - mu(x-K)^2 is the same identity, without cancellation
    // when |mean| >> std.
    const float K = __shfl_sync(0xffffffffu, first_elem(xr[0]), 0, LPR);
    float d[VPT][kVec];
    float2 sa = make_float2(0.f, 0.f), sb = make_float2(0.f, 0.f);
#pragma unroll
    for (int k = 0; k < VPT; ++k) {
        if (row_ok && gl + k * LPR < nvec) {
            sub8(xr[k], K, d[k]);
#pragma unroll
            for (int j = 0; j < kVec; j += 2) {
                const float2 dj = make_float2(d[k][j], d[k][j + 1]);
                sa = add2(sa, dj);
                sb = fma2(dj, dj, sb);
            }
        }
    }
    float2 s = make_float2(sa.x + sa.y, sb.x + sb.y);
    s = group_sum2<LPR>(s);  // the single synchronisation
    const float inv_n = 1.f / static_cast<float>(cols);
    const float m1 = s.x * inv_n;
    const float var = fmaxf(fmaf(-m1, m1, s.y * inv_n), 0.f);
    const float rs = rsqrtf(var + eps);
    if (!row_ok) return;
    const float2 m2 = make_float2(-m1, -m1), r2 = make_float2(rs, rs);
#pragma unroll
    for (int k = 0; k < VPT; ++k) {
        const int v = gl + k * LPR;
        if (v < nvec) {
            float o[kVec], g[kVec], b[kVec];
            load8f<T>(gamma + v * kVec, g);
            load8f<T>(beta + v * kVec, b);
            if constexpr (!ln_fwd_keep_d<T, VPT>()) sub8(xr[k], K, d[k]);
#pragma unroll
            for (int j = 0; j < kVec; j += 2) {
                float2 t = mul2(add2(make_float2(d[k][j], d[k][j + 1]), m2), r2);
                t = fma2(t, make_float2(g[j], g[j + 1]), make_float2(b[j], b[j + 1]));
                o[j] = t.x;
                o[j + 1] = t.y;
            }
            store8f<T>(y + r * cols + v * kVec, o);
        }
    }
    if (gl == 0) {
        if (mean) mean[r] = K + m1;
        if (rstd) rstd[r] = rs;
    }
}

template <typename T, int LPR, int VPT>
__global__ void __launch_bounds__(kThreads, min_ctas<T>(VPT == 2 ? 3 : (VPT <= 3 ? 4 : (VPT <= 6 ? 3 : 2))))
ln_fwd_group_kernel(T* y, float* __restrict__ mean, float* __restrict__ rstd, const T* x,
                    const T* __restrict__ gamma, const T* __restrict__ beta, int64_t rows,
                    int cols, float eps) {
    constexpr int RPC = kThreads / LPR;
    const int gl = threadIdx.x % LPR;
    const int slot = threadIdx.x / LPR;
    const int64_t stride = static_cast<int64_t>(gridDim.x) * RPC;
    int64_t r = static_cast<int64_t>(slot) * gridDim.x + blockIdx.x;
    // Before the wait: the lines of this group's first row and of
    // gamma/beta, into L2.  (Only the first row: prefetching both rows of a
    // two-buffer group was slower, 7.85 against 7.54 us at 4096 x 2048 and
    // 4.20 against 4.10 at 1024, measured on GB300.)
    {
        const int nvec = cols / kVec;
#pragma unroll
        for (int k = 0; k < VPT; ++k) {
            const int v = gl + k * LPR;
            if (r < rows && v < nvec) prefetch_l2(x + r * cols + v * kVec);
        }
        prefetch_params_l2(gamma, static_cast<size_t>(cols) * sizeof(T));
        prefetch_params_l2(beta, static_cast<size_t>(cols) * sizeof(T));
    }
    pdl_enter();
    Raw8<T> xa[VPT];
    const T* gs = gamma;
    const T* bs = beta;
    ln_fwd_load<T, LPR, VPT>(xa, x, r, rows, cols, gl);
    if constexpr (!ln_fwd_double<T, VPT>()) {
        while (__any_sync(0xffffffffu, r < rows)) {
            ln_fwd_row<T, LPR, VPT>(xa, y, mean, rstd, gs, bs, r, rows, cols, eps, gl);
            r += stride;
            if (!__any_sync(0xffffffffu, r < rows)) break;
            ln_fwd_load<T, LPR, VPT>(xa, x, r, rows, cols, gl);
        }
    } else {
        Raw8<T> xb[VPT];
        while (__any_sync(0xffffffffu, r < rows)) {
            const int64_t r1 = r + stride;
            ln_fwd_load<T, LPR, VPT>(xb, x, r1, rows, cols, gl);
            ln_fwd_row<T, LPR, VPT>(xa, y, mean, rstd, gs, bs, r, rows, cols, eps, gl);
            if (!__any_sync(0xffffffffu, r1 < rows)) break;
            r = r1 + stride;
            ln_fwd_load<T, LPR, VPT>(xa, x, r, rows, cols, gl);
            ln_fwd_row<T, LPR, VPT>(xb, y, mean, rstd, gs, bs, r1, rows, cols, eps, gl);
        }
    }
}

// ----------------------------------------------------------------------------
// Forward, CTA-per-row (rows longer than a warp holds).
// ----------------------------------------------------------------------------
template <typename T, int WARPS, int VPT>
__global__ void __launch_bounds__(WARPS * 32)
ln_fwd_cta_kernel(T* y, float* __restrict__ mean, float* __restrict__ rstd, const T* x,
                  const T* __restrict__ gamma, const T* __restrict__ beta, int cols, float eps) {
    constexpr int NT = WARPS * 32;
    pdl_enter();
    const int64_t r = blockIdx.x;
    const int nvec = cols / kVec;
    const T* xr = x + r * cols;
    const float K = static_cast<float>(xr[0]);
    float f[VPT][kVec];
    float2 s = make_float2(0.f, 0.f);
#pragma unroll
    for (int k = 0; k < VPT; ++k) {
        const int v = threadIdx.x + k * NT;
        if (v < nvec) {
            load8f<T>(xr + v * kVec, f[k]);
#pragma unroll
            for (int j = 0; j < kVec; ++j) {
                const float d = f[k][j] - K;
                s.x += d;
                s.y = fmaf(d, d, s.y);
            }
        }
    }
    s = group_sum2<32>(s);
    __shared__ float2 part[WARPS];
    if ((threadIdx.x & 31) == 0) part[threadIdx.x >> 5] = s;
    __syncthreads();  // the single synchronisation
    s = make_float2(0.f, 0.f);
#pragma unroll
    for (int w = 0; w < WARPS; ++w) {
        s.x += part[w].x;
        s.y += part[w].y;
    }
    const float inv_n = 1.f / static_cast<float>(cols);
    const float m1 = s.x * inv_n;
    const float var = fmaxf(fmaf(-m1, m1, s.y * inv_n), 0.f);
    const float rs = rsqrtf(var + eps);
#pragma unroll
    for (int k = 0; k < VPT; ++k) {
        const int v = threadIdx.x + k * NT;
        if (v < nvec) {
            float g[kVec], b[kVec], o[kVec];
            load8f<T>(gamma + v * kVec, g);
            load8f<T>(beta + v * kVec, b);
#pragma unroll
            for (int j = 0; j < kVec; ++j) o[j] = fmaf((f[k][j] - K - m1) * rs, g[j], b[j]);
            store8f<T>(y + r * cols + v * kVec, o);
        }
    }
    if (threadIdx.x == 0) {
        if (mean) mean[r] = K + m1;
        if (rstd) rstd[r] = rs;
    }
}

// ----------------------------------------------------------------------------
// Backward, group-per-row.  Per row, with g = gamma*dy and xh = (x-mean)*rstd,
// the two sums A = sum g and C = sum g*xh are reduced together; then
//   dx = rstd * (g - A/H - xh * C/H).
// (The pages' second sum is sum gamma*dy*x; taking it about the saved mean and
// scaled by rstd gives C = rstd*(B - mean*A), the same algebra.)
// dgamma/dbeta partial sums accumulate in shared memory per row slot (each
// slot's lanes own disjoint columns), and are summed over the slots in a fixed
// order at the end into partial[blockIdx.x, 0:H] and [blockIdx.x, H:2H].
// ----------------------------------------------------------------------------
template <typename T, int LPR, int VPT>
__global__ void __launch_bounds__(kThreads, min_ctas<T>(VPT <= 2 ? 3 : (VPT <= 5 ? 2 : 1)))
ln_bwd_group_kernel(T* dx, float* __restrict__ partial, const T* dy, const T* x,
                    const T* __restrict__ gamma, const float* __restrict__ mean,
                    const float* __restrict__ rstd, int64_t rows, int cols, int rows_per_cta) {
    constexpr int RPC = kThreads / LPR;  // row slots per CTA
    extern __shared__ __align__(16) float acc[];  // [RPC][2*cols] when partial != nullptr
    pdl_enter();
    const int gl = threadIdx.x % LPR;
    const int slot = threadIdx.x / LPR;
    const int nvec = cols / kVec;
    const float inv_n = 1.f / static_cast<float>(cols);
    float* my_acc = acc + static_cast<size_t>(slot) * 2 * cols;

    if (partial) {
        for (int k = gl; k < 2 * cols; k += LPR) my_acc[k] = 0.f;
    }
    float gm[VPT][kVec];
#pragma unroll
    for (int k = 0; k < VPT; ++k) {
        const int v = gl + k * LPR;
        if (v < nvec) load8f<T>(gamma + v * kVec, gm[k]);
    }

    const int64_t base = static_cast<int64_t>(blockIdx.x) * rows_per_cta;
    const int64_t end = std::min<int64_t>(rows, base + rows_per_cta);
    const int steps = (rows_per_cta + RPC - 1) / RPC;
    for (int st = 0; st < steps; ++st) {
        const int64_t r = base + static_cast<int64_t>(st) * RPC + slot;
        const bool row_ok = r < end;
        Raw8<T> xr[VPT], dr[VPT];
#pragma unroll
        for (int k = 0; k < VPT; ++k) {
            const int v = gl + k * LPR;
            if (row_ok && v < nvec) {
                xr[k] = load8<T>(x + r * cols + v * kVec);
                dr[k] = load8<T>(dy + r * cols + v * kVec);
            }
        }
        const float mu = row_ok ? mean[r] : 0.f;
        const float rs = row_ok ? rstd[r] : 0.f;
        float2 s = make_float2(0.f, 0.f);
#pragma unroll
        for (int k = 0; k < VPT; ++k) {
            if (row_ok && gl + k * LPR < nvec) {
                float xf[kVec], df[kVec];
                unpack(xr[k], xf);
                unpack(dr[k], df);
#pragma unroll
                for (int j = 0; j < kVec; ++j) {
                    const float g = gm[k][j] * df[j];
                    const float xh = (xf[j] - mu) * rs;
                    s.x += g;
                    s.y = fmaf(g, xh, s.y);
                }
            }
        }
        s = group_sum2<LPR>(s);  // the single synchronisation
        const float a_n = s.x * inv_n;
        const float c_n = s.y * inv_n;
        if (!row_ok) continue;
#pragma unroll
        for (int k = 0; k < VPT; ++k) {
            const int v = gl + k * LPR;
            if (v < nvec) {
                float xf[kVec], df[kVec], o[kVec];
                unpack(xr[k], xf);
                unpack(dr[k], df);
                float xh[kVec];
#pragma unroll
                for (int j = 0; j < kVec; ++j) {
                    xh[j] = (xf[j] - mu) * rs;
                    const float g = gm[k][j] * df[j];
                    o[j] = rs * (g - a_n - xh[j] * c_n);
                }
                store8f<T>(dx + r * cols + v * kVec, o);
                if (partial) {
                    float4* pg = reinterpret_cast<float4*>(my_acc + v * kVec);
                    float4* pb = reinterpret_cast<float4*>(my_acc + cols + v * kVec);
                    float4 g0 = pg[0], g1 = pg[1], b0 = pb[0], b1 = pb[1];
                    g0.x = fmaf(df[0], xh[0], g0.x); g0.y = fmaf(df[1], xh[1], g0.y);
                    g0.z = fmaf(df[2], xh[2], g0.z); g0.w = fmaf(df[3], xh[3], g0.w);
                    g1.x = fmaf(df[4], xh[4], g1.x); g1.y = fmaf(df[5], xh[5], g1.y);
                    g1.z = fmaf(df[6], xh[6], g1.z); g1.w = fmaf(df[7], xh[7], g1.w);
                    b0.x += df[0]; b0.y += df[1]; b0.z += df[2]; b0.w += df[3];
                    b1.x += df[4]; b1.y += df[5]; b1.z += df[6]; b1.w += df[7];
                    pg[0] = g0; pg[1] = g1; pb[0] = b0; pb[1] = b1;
                }
            }
        }
    }
    if (partial == nullptr) return;
    __syncthreads();
    for (int k = threadIdx.x; k < 2 * cols; k += kThreads) {
        float t = 0.f;
        for (int q = 0; q < RPC; ++q) t += acc[static_cast<size_t>(q) * 2 * cols + k];
        partial[static_cast<int64_t>(blockIdx.x) * 2 * cols + k] = t;
    }
}

// ----------------------------------------------------------------------------
// Backward, warp per row, rows fed by bulk copies (136 <= H <= 1280 while the
// ring fits in 200 KB).  One 16-warp CTA per SM: CTA b owns rows [b*R,
// (b+1)*R) (R from the shape-only plan, about rows/152); warp w takes rows
// b*R + w + 16k.  Each warp's x and dy rows arrive in a two-stage ring of
// shared memory (cp.async.bulk, bounded mbarrier waits), so both of a warp's
// rows are in flight at once without holding them in registers.  dgamma/dbeta partial
// sums stay in registers (each lane owns the same columns in every row); when
// all rows are done the warps' sums are added in warp order through the
// (now free) stage memory into partial[b, 0:2H].
// ----------------------------------------------------------------------------
constexpr int kLnTmaWarps = 16;
constexpr int kLnTmaStages = 2;
constexpr uint32_t kLnTmaBarBytes = 256;  // 16 warps x 2 stages x 8 bytes
// Shared-memory layout: barriers | gamma (cols, rounded to 128 B) | stages.
__host__ __device__ inline size_t ln_tma_gamma_bytes(int cols, size_t esize) {
    return ((static_cast<size_t>(cols) * esize + 127) / 128) * 128;
}


template <typename T, int VPT>
__global__ void __launch_bounds__(kLnTmaWarps * 32, 1)
ln_bwd_tma_kernel(T* dx, float* __restrict__ partial, const T* dy, const T* x,
                  const T* __restrict__ gamma, const float* __restrict__ mean,
                  const float* __restrict__ rstd, int64_t rows, int cols, int rows_per_cta) {
    extern __shared__ __align__(128) unsigned char smem[];
    constexpr int S = kLnTmaStages;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t row_bytes = static_cast<uint32_t>(cols) * sizeof(T);
    const uint32_t stage_bytes = 2 * row_bytes;
    T* gsm = reinterpret_cast<T*>(smem + kLnTmaBarBytes);
    unsigned char* data = smem + kLnTmaBarBytes + ln_tma_gamma_bytes(cols, sizeof(T));
    WarpRing<S> ring;
    ring.init(reinterpret_cast<uint64_t*>(smem) + warp * S,
              data + static_cast<size_t>(warp) * S * stage_bytes, stage_bytes);
    // The dependent launch (the column reduction, whose CTAs need whole SMs)
    // is released as these CTAs finish rather than at their start, so that
    // its waiting CTAs do not hold SMs that this grid's CTAs still need.
    pdl_wait();
    const int nvec = cols / kVec;
    // gamma's loads go out first (its single vector per thread is in flight
    // while the row copies are issued) and are stored to shared memory after.
    constexpr int kGammaVecs = (5 * 32 + kLnTmaWarps * 32 - 1) / (kLnTmaWarps * 32);
    Raw8<T> graw[kGammaVecs];
#pragma unroll
    for (int q = 0; q < kGammaVecs; ++q) {
        const int v = threadIdx.x + q * kLnTmaWarps * 32;
        if (v < nvec) graw[q] = load8<T>(gamma + v * kVec);
    }
    const float inv_n = 1.f / static_cast<float>(cols);
    const int64_t base = static_cast<int64_t>(blockIdx.x) * rows_per_cta;
    const int64_t end = std::min<int64_t>(rows, base + rows_per_cta);
    float ag[VPT][kVec], ab[VPT][kVec];
#pragma unroll
    for (int k = 0; k < VPT; ++k)
#pragma unroll
        for (int j = 0; j < kVec; ++j) ag[k][j] = ab[k][j] = 0.f;
    uint32_t parity[S] = {0, 0};
    float mu_of[S], rs_of[S];
    // Only the warp's first row is requested now; its second goes out when
    // the first has landed.  (Measured on GB300 at 4096 x 1280: requesting
    // both at once makes every CTA's rows land anywhere in the time DRAM needs
    // for the whole 21 MB, and all reads precede all dx writes; staggered,
    // the first rows land sooner and the second rows' reads overlap the first
    // rows' writes: 10.56 -> 9.97 us, 7.43 -> 7.18 at 4096 x 768.)
    {
        const int64_t r = base + warp;
        if (r < end) {
            ring.issue(0, x + r * cols, row_bytes, dy + r * cols, row_bytes, row_bytes);
            mu_of[0] = mean[r];
            rs_of[0] = rstd[r];
        }
    }
#pragma unroll
    for (int q = 0; q < kGammaVecs; ++q) {
        const int v = threadIdx.x + q * kLnTmaWarps * 32;
        if (v < nvec) store8<T>(gsm + v * kVec, graw[q]);
    }
    bool done = false;  // set when the warp's rows are done (or a wait failed)
    __syncthreads();  // gamma staged
    // Unrolled by the stage count so that the stage index is a constant.
    for (int k0 = 0; !done; k0 += S) {
#pragma unroll
    for (int s = 0; s < S; ++s) {
        const int64_t r = base + warp + static_cast<int64_t>(k0 + s) * kLnTmaWarps;
        if (r >= end) {
            done = true;
            break;
        }
        const bool ok = ring.wait(s, parity[s]);
        if (!__all_sync(0xffffffffu, ok)) {
            ring.drain(parity);
            done = true;
            break;
        }
        parity[s] ^= 1u;
        if (k0 == 0 && s == 0) {
            const int64_t r1 = base + warp + kLnTmaWarps;
            if (r1 < end) {
                ring.issue(1, x + r1 * cols, row_bytes, dy + r1 * cols, row_bytes, row_bytes);
                mu_of[1] = mean[r1];
                rs_of[1] = rstd[r1];
            }
        }
        const float mu = mu_of[s], rs = rs_of[s];
        const T* xs = reinterpret_cast<const T*>(ring.stage(s));
        const T* ds = reinterpret_cast<const T*>(ring.stage(s) + row_bytes);
        // g = gamma*dy and xhat = (x - mu)*rstd, formed once per element with the
        // mixed-precision forms (FP16 operands convert exactly inside them);
        // kept in registers for the second pass when they fit, else re-formed.
        constexpr bool kKeep = VPT <= 3;
        float gk[kKeep ? VPT : 1][kVec], hk[kKeep ? VPT : 1][kVec];
        float2 sa = make_float2(0.f, 0.f), sb = make_float2(0.f, 0.f);
        const float2 rs2 = make_float2(rs, rs);
#pragma unroll
        for (int k2 = 0; k2 < VPT; ++k2) {
            const int v = lane + k2 * 32;
            if (v < nvec) {
                float g[kVec], h[kVec];
                mul8(load8_smem<T>(gsm + v * kVec), load8_smem<T>(ds + v * kVec), g);
                sub8(load8_smem<T>(xs + v * kVec), mu, h);
#pragma unroll
                for (int j = 0; j < kVec; j += 2) {
                    const float2 hj = mul2(make_float2(h[j], h[j + 1]), rs2);
                    const float2 gj = make_float2(g[j], g[j + 1]);
                    sa = add2(sa, gj);
                    sb = fma2(gj, hj, sb);
                    h[j] = hj.x;
                    h[j + 1] = hj.y;
                }
                if (kKeep) {
#pragma unroll
                    for (int j = 0; j < kVec; ++j) {
                        gk[kKeep ? k2 : 0][j] = g[j];
                        hk[kKeep ? k2 : 0][j] = h[j];
                    }
                }
            }
        }
        float2 sum = make_float2(sa.x + sa.y, sb.x + sb.y);
        sum = group_sum2<32>(sum);  // the single synchronisation
        const float2 na = make_float2(-sum.x * inv_n, -sum.x * inv_n);
        const float2 nc = make_float2(-sum.y * inv_n, -sum.y * inv_n);
#pragma unroll
        for (int k2 = 0; k2 < VPT; ++k2) {
            const int v = lane + k2 * 32;
            if (v < nvec) {
                const Raw8<T> dr = load8_smem<T>(ds + v * kVec);
                float g[kVec], h[kVec], df[kVec], o[kVec];
                if (kKeep) {
#pragma unroll
                    for (int j = 0; j < kVec; ++j) {
                        g[j] = gk[kKeep ? k2 : 0][j];
                        h[j] = hk[kKeep ? k2 : 0][j];
                    }
                } else {
                    mul8(load8_smem<T>(gsm + v * kVec), dr, g);
                    sub8(load8_smem<T>(xs + v * kVec), mu, h);
#pragma unroll
                    for (int j = 0; j < kVec; j += 2) {
                        const float2 hj = mul2(make_float2(h[j], h[j + 1]), rs2);
                        h[j] = hj.x;
                        h[j + 1] = hj.y;
                    }
                }
                unpack(dr, df);
#pragma unroll
                for (int j = 0; j < kVec; j += 2) {
                    // dx = rstd * ((g - A/H) - xhat * C/H)
                    const float2 hj = make_float2(h[j], h[j + 1]);
                    const float2 t = fma2(hj, nc, add2(make_float2(g[j], g[j + 1]), na));
                    const float2 oj = mul2(t, rs2);
                    o[j] = oj.x;
                    o[j + 1] = oj.y;
                    const float2 dj = make_float2(df[j], df[j + 1]);
                    const float2 agj = fma2(dj, hj, make_float2(ag[k2][j], ag[k2][j + 1]));
                    const float2 abj = add2(dj, make_float2(ab[k2][j], ab[k2][j + 1]));
                    ag[k2][j] = agj.x;
                    ag[k2][j + 1] = agj.y;
                    ab[k2][j] = abj.x;
                    ab[k2][j + 1] = abj.y;
                }
                store8f<T>(dx + r * cols + v * kVec, o);
            }
        }
        __syncwarp();  // every lane has used its reads of stage s
        const int64_t rn = r + S * kLnTmaWarps;
        if (rn < end) {
            ring.issue(s, x + rn * cols, row_bytes, dy + rn * cols, row_bytes, row_bytes);
            mu_of[s] = mean[rn];
            rs_of[s] = rstd[rn];
        }
    }
    }
    if (partial == nullptr) return;
    // Cross-warp sum of the parameter-gradient partials, in warp order.  Each
    // warp stores its sums in its own stage memory as soon as its rows are
    // done (every copy into it has landed and been read), while other warps
    // still compute: four arrays of half-vectors -- dgamma elements 0..3 and
    // 4..7 of every vector, then dbeta's -- 8*H bytes, which is the warp's
    // stage memory at FP16 (twice that at FP32).  A lane's 16-byte stores are
    // 16 bytes apart, and the summing threads take consecutive vectors of one
    // array, so neither side has bank conflicts (whole 8-float vectors were
    // 32 bytes apart: a two-way conflict on 160 KB at H = 1280).  The
    // association of every sum is unchanged: warps 0..15 in order.
    const int hc = cols / 2;  // floats per half-vector array
    const size_t wstride = static_cast<size_t>(S) * stage_bytes / sizeof(float);
    float* red = reinterpret_cast<float*>(data);  // warp w's arrays at w * wstride
    __syncwarp();
    {
        float* mine = red + static_cast<size_t>(warp) * wstride;
#pragma unroll
        for (int k2 = 0; k2 < VPT; ++k2) {
            const int v = lane + k2 * 32;
            if (v < nvec) {
                *reinterpret_cast<float4*>(mine + 0 * hc + v * 4) =
                    make_float4(ag[k2][0], ag[k2][1], ag[k2][2], ag[k2][3]);
                *reinterpret_cast<float4*>(mine + 1 * hc + v * 4) =
                    make_float4(ag[k2][4], ag[k2][5], ag[k2][6], ag[k2][7]);
                *reinterpret_cast<float4*>(mine + 2 * hc + v * 4) =
                    make_float4(ab[k2][0], ab[k2][1], ab[k2][2], ab[k2][3]);
                *reinterpret_cast<float4*>(mine + 3 * hc + v * 4) =
                    make_float4(ab[k2][4], ab[k2][5], ab[k2][6], ab[k2][7]);
            }
        }
    }
    __syncthreads();
    // Thread q sums vector v of array a (a = q / nvec: dgamma low/high
    // half, dbeta low/high half).
    for (int q = threadIdx.x; q < 4 * nvec; q += kLnTmaWarps * 32) {
        const int a = q / nvec;
        const int v = q - a * nvec;
        const int off = a * hc + v * 4;
        float4 t = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int w = 0; w < kLnTmaWarps; ++w) {
            const float4 p = *reinterpret_cast<const float4*>(red + static_cast<size_t>(w) * wstride + off);
            t.x += p.x;
            t.y += p.y;
            t.z += p.z;
            t.w += p.w;
        }
        *reinterpret_cast<float4*>(partial + static_cast<int64_t>(blockIdx.x) * 2 * cols +
                                   (a >> 1) * cols + v * kVec + (a & 1) * 4) = t;
    }
}

// ----------------------------------------------------------------------------
// Backward, CTA-per-row.  Threads own disjoint columns, so the gradient
// partial sums live in one [2*cols] shared array without conflicts.
// ----------------------------------------------------------------------------
template <typename T, int WARPS, int VPT>
__global__ void __launch_bounds__(WARPS * 32)
ln_bwd_cta_kernel(T* dx, float* __restrict__ partial, const T* dy, const T* x,
                  const T* __restrict__ gamma, const float* __restrict__ mean,
                  const float* __restrict__ rstd, int64_t rows, int cols, int steps) {
    constexpr int NT = WARPS * 32;
    extern __shared__ __align__(16) float acc[];  // [2*cols]
    __shared__ float2 part[WARPS];
    pdl_enter();
    const int nvec = cols / kVec;
    const float inv_n = 1.f / static_cast<float>(cols);
    if (partial)
        for (int k = threadIdx.x; k < 2 * cols; k += NT) acc[k] = 0.f;
    float gm[VPT][kVec];
#pragma unroll
    for (int k = 0; k < VPT; ++k) {
        const int v = threadIdx.x + k * NT;
        if (v < nvec) load8f<T>(gamma + v * kVec, gm[k]);
    }
    for (int st = 0; st < steps; ++st) {
        const int64_t r = static_cast<int64_t>(blockIdx.x) * steps + st;
        if (r >= rows) break;  // uniform across the CTA
        Raw8<T> xr[VPT], dr[VPT];
#pragma unroll
        for (int k = 0; k < VPT; ++k) {
            const int v = threadIdx.x + k * NT;
            if (v < nvec) {
                xr[k] = load8<T>(x + r * cols + v * kVec);
                dr[k] = load8<T>(dy + r * cols + v * kVec);
            }
        }
        const float mu = mean[r];
        const float rs = rstd[r];
        float2 s = make_float2(0.f, 0.f);
#pragma unroll
        for (int k = 0; k < VPT; ++k) {
            if (threadIdx.x + k * NT < nvec) {
                float xf[kVec], df[kVec];
                unpack(xr[k], xf);
                unpack(dr[k], df);
#pragma unroll
                for (int j = 0; j < kVec; ++j) {
                    const float g = gm[k][j] * df[j];
                    s.x += g;
                    s.y = fmaf(g, (xf[j] - mu) * rs, s.y);
                }
            }
        }
        s = group_sum2<32>(s);
        __syncthreads();  // previous row's readers of part[] are done
        if ((threadIdx.x & 31) == 0) part[threadIdx.x >> 5] = s;
        __syncthreads();  // the single synchronisation of this row's sums
        s = make_float2(0.f, 0.f);
#pragma unroll
        for (int w = 0; w < WARPS; ++w) {
            s.x += part[w].x;
            s.y += part[w].y;
        }
        const float a_n = s.x * inv_n;
        const float c_n = s.y * inv_n;
#pragma unroll
        for (int k = 0; k < VPT; ++k) {
            const int v = threadIdx.x + k * NT;
            if (v < nvec) {
                float xf[kVec], df[kVec], o[kVec];
                unpack(xr[k], xf);
                unpack(dr[k], df);
#pragma unroll
                for (int j = 0; j < kVec; ++j) {
                    const float xh = (xf[j] - mu) * rs;
                    o[j] = rs * (gm[k][j] * df[j] - a_n - xh * c_n);
                    if (partial) {
                        acc[v * kVec + j] = fmaf(df[j], xh, acc[v * kVec + j]);
                        acc[cols + v * kVec + j] += df[j];
                    }
                }
                store8f<T>(dx + r * cols + v * kVec, o);
            }
        }
    }
    if (partial == nullptr) return;
    __syncthreads();
    for (int k = threadIdx.x; k < 2 * cols; k += NT)
        partial[static_cast<int64_t>(blockIdx.x) * 2 * cols + k] = acc[k];
}

// ----------------------------------------------------------------------------
// Dispatch.
// ----------------------------------------------------------------------------
int pow2_at_least(int n) {
    int p = 1;
    while (p < n) p <<= 1;
    return p;
}

struct LnPlan {
    bool cta;     // CTA per row
    int lpr;      // group path: lanes per row
    int vpt;      // vectors per lane
    int warps;    // CTA path: warps per row
    int64_t grid;
    int steps;    // backward: rows per CTA (both paths)
};

// Target number of backward CTAs: about two per SM on a 152-SM part.  It is a
// constant, not the device's SM count, so that the partial sums -- and with
// them the bits of dgamma/dbeta -- do not depend on which GPU runs the call.
constexpr int64_t kBwdTargetCtas = 304;
// The bulk-copy backward runs one 16-warp CTA per SM (measured on GB300: faster
// than two 8-warp CTAs per SM, and half the partial rows).
constexpr int64_t kBwdTmaTargetCtas = 152;
constexpr size_t kLnTmaMaxSmem = 200 * 1024;

size_t ln_tma_smem(int64_t cols, size_t esize) {
    // A warp's stage memory (2 stages of x and dy rows, at least 2-byte
    // elements) also holds its 2*cols FP32 sums at the end.
    return kLnTmaBarBytes + ln_tma_gamma_bytes(static_cast<int>(cols), esize) +
           static_cast<size_t>(kLnTmaWarps) * kLnTmaStages * 2 * static_cast<size_t>(cols) * esize;
}

// Whether the backward of rows of `cols` elements of `esize` bytes takes the
// bulk-copy kernel (warp per row, 1..5 vectors per lane, its ring fits).
bool ln_bwd_uses_tma(int64_t cols, size_t esize) {
    const int64_t nvec = cols / kVec;
    return nvec > 16 && nvec <= 5 * 32 && ln_tma_smem(cols, esize) <= kLnTmaMaxSmem;
}

LnPlan plan_for(int64_t rows, int64_t cols, bool bwd, size_t esize) {
    const int nvec = static_cast<int>(cols / kVec);
    LnPlan p{};
    if (nvec <= kCtaRowThreshold) {
        p.cta = false;
        if (nvec <= 32) {
            p.lpr = pow2_at_least(nvec);
            p.vpt = 1;
        } else {
            p.lpr = 32;
            p.vpt = (nvec + 31) / 32;
        }
        const int64_t rpc = kThreads / p.lpr;
        if (bwd) {
            const int64_t target = ln_bwd_uses_tma(cols, esize) ? kBwdTmaTargetCtas
                                                                : kBwdTargetCtas;
            p.steps = static_cast<int>(std::max<int64_t>(1, (rows + target - 1) / target));
            p.grid = (rows + p.steps - 1) / p.steps;
        } else {
            p.steps = 1;
            p.grid = (rows + rpc - 1) / rpc;  // upper bound; the launcher caps it
        }
    } else {
        p.cta = true;
        p.warps = nvec <= 512 ? 4 : 8;
        p.vpt = (nvec + p.warps * 32 - 1) / (p.warps * 32);
        if (bwd) {
            p.steps = static_cast<int>(
                std::max<int64_t>(1, (rows + kBwdTargetCtas - 1) / kBwdTargetCtas));
            p.grid = (rows + p.steps - 1) / p.steps;
        } else {
            p.steps = 1;
            p.grid = rows;
        }
    }
    return p;
}

// Raises the kernel's dynamic shared-memory limit (once per kernel and
// device) when `bytes` needs more than the default 48 KB.
template <typename K>
cudaError_t set_smem(K kernel, size_t bytes, int (&done)[kMaxDevices]) {
    if (bytes <= 48 * 1024) return cudaSuccess;
    return allow_max_dynamic_smem(kernel, done);
}

template <typename K>
int occupancy(K kernel, int threads, size_t smem) {
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kernel, threads, smem) != cudaSuccess ||
        n < 1)
        n = 1;
    return n;
}

template <typename T, int LPR, int VPT>
cudaError_t fwd_group(void* y, float* mean, float* rstd, const void* x, const void* gamma,
                      const void* beta, int64_t rows, int64_t cols, float eps, const LnPlan& p,
                      cudaStream_t s) {
    auto kern = ln_fwd_group_kernel<T, LPR, VPT>;
    static const int occ = occupancy(kern, kThreads, 0);
    const int64_t grid = std::min<int64_t>(p.grid, int64_t{sm_count()} * occ);
    return launch_pdl(kern, dim3(static_cast<unsigned>(grid)), dim3(kThreads), 0, s,
                      static_cast<T*>(y), mean, rstd, static_cast<const T*>(x),
                      static_cast<const T*>(gamma), static_cast<const T*>(beta), rows,
                      static_cast<int>(cols), eps);
}

template <typename T, int WARPS, int VPT>
cudaError_t fwd_cta(void* y, float* mean, float* rstd, const void* x, const void* gamma,
                    const void* beta, int64_t rows, int64_t cols, float eps, const LnPlan& p,
                    cudaStream_t s) {
    return launch_pdl(ln_fwd_cta_kernel<T, WARPS, VPT>, dim3(static_cast<unsigned>(p.grid)),
                      dim3(WARPS * 32), 0, s, static_cast<T*>(y), mean, rstd,
                      static_cast<const T*>(x), static_cast<const T*>(gamma),
                      static_cast<const T*>(beta), static_cast<int>(cols), eps);
}

template <typename T, int LPR, int VPT>
cudaError_t bwd_group(void* dx, float* partial, const void* dy, const void* x, const void* gamma,
                      const float* mean, const float* rstd, int64_t rows, int64_t cols,
                      const LnPlan& p, cudaStream_t s) {
    if constexpr (LPR == 32 && VPT >= 1 && VPT <= 5) {
        if (ln_bwd_uses_tma(cols, sizeof(T))) {
            const size_t smem = ln_tma_smem(cols, sizeof(T));
            auto kern = ln_bwd_tma_kernel<T, VPT>;
            static int done[kMaxDevices] = {};
            cudaError_t e = set_smem(kern, smem, done);
            if (e != cudaSuccess) return e;
            return launch_pdl(kern, dim3(static_cast<unsigned>(p.grid)), dim3(kLnTmaWarps * 32),
                              smem, s, static_cast<T*>(dx), partial, static_cast<const T*>(dy),
                              static_cast<const T*>(x), static_cast<const T*>(gamma), mean, rstd,
                              rows, static_cast<int>(cols), p.steps);
        }
    }
    const size_t smem = partial ? static_cast<size_t>(kThreads / LPR) * 2 * cols * sizeof(float)
                                : 0;
    auto kern = ln_bwd_group_kernel<T, LPR, VPT>;
    static int done[kMaxDevices] = {};
    cudaError_t e = set_smem(kern, smem, done);
    if (e != cudaSuccess) return e;
    return launch_pdl(kern, dim3(static_cast<unsigned>(p.grid)), dim3(kThreads), smem, s,
                      static_cast<T*>(dx), partial, static_cast<const T*>(dy),
                      static_cast<const T*>(x), static_cast<const T*>(gamma), mean, rstd, rows,
                      static_cast<int>(cols), p.steps);
}

template <typename T, int WARPS, int VPT>
cudaError_t bwd_cta(void* dx, float* partial, const void* dy, const void* x, const void* gamma,
                    const float* mean, const float* rstd, int64_t rows, int64_t cols,
                    const LnPlan& p, cudaStream_t s) {
    const size_t smem = partial ? 2 * static_cast<size_t>(cols) * sizeof(float) : 0;
    auto kern = ln_bwd_cta_kernel<T, WARPS, VPT>;
    static int done[kMaxDevices] = {};
    cudaError_t e = set_smem(kern, smem, done);
    if (e != cudaSuccess) return e;
    return launch_pdl(kern, dim3(static_cast<unsigned>(p.grid)), dim3(WARPS * 32), smem, s,
                      static_cast<T*>(dx), partial, static_cast<const T*>(dy),
                      static_cast<const T*>(x), static_cast<const T*>(gamma), mean, rstd, rows,
                      static_cast<int>(cols), p.steps);
}

// Expand a runtime (lpr, vpt) or (warps, vpt) into a template instance.
#define LS_GROUP_CASES(FN, T, ...)                                       \
    if (p.lpr < 32) {                                                    \
        switch (p.lpr) {                                                 \
            case 1: return FN<T, 1, 1>(__VA_ARGS__);                     \
            case 2: return FN<T, 2, 1>(__VA_ARGS__);                     \
            case 4: return FN<T, 4, 1>(__VA_ARGS__);                     \
            case 8: return FN<T, 8, 1>(__VA_ARGS__);                     \
            case 16: return FN<T, 16, 1>(__VA_ARGS__);                   \
        }                                                                \
    } else {                                                             \
        switch (p.vpt) {                                                 \
            case 1: return FN<T, 32, 1>(__VA_ARGS__);                    \
            case 2: return FN<T, 32, 2>(__VA_ARGS__);                    \
            case 3: return FN<T, 32, 3>(__VA_ARGS__);                    \
            case 4: return FN<T, 32, 4>(__VA_ARGS__);                    \
            case 5: return FN<T, 32, 5>(__VA_ARGS__);                    \
            case 6: return FN<T, 32, 6>(__VA_ARGS__);                    \
            case 7: return FN<T, 32, 7>(__VA_ARGS__);                    \
            case 8: return FN<T, 32, 8>(__VA_ARGS__);                    \
        }                                                                \
    }                                                                    \
    return cudaErrorInvalidConfiguration;

#define LS_CTA_CASES(FN, T, ...)                                         \
    if (p.warps == 4) {                                                  \
        switch (p.vpt) {                                                 \
            case 3: return FN<T, 4, 3>(__VA_ARGS__);                     \
            case 4: return FN<T, 4, 4>(__VA_ARGS__);                     \
        }                                                                \
    } else {                                                             \
        switch (p.vpt) {                                                 \
            case 3: return FN<T, 8, 3>(__VA_ARGS__);                     \
            case 4: return FN<T, 8, 4>(__VA_ARGS__);                     \
            case 5: return FN<T, 8, 5>(__VA_ARGS__);                     \
            case 6: return FN<T, 8, 6>(__VA_ARGS__);                     \
            case 7: return FN<T, 8, 7>(__VA_ARGS__);                     \
            case 8: return FN<T, 8, 8>(__VA_ARGS__);                     \
        }                                                                \
    }                                                                    \
    return cudaErrorInvalidConfiguration;

template <typename T>
cudaError_t fwd_dispatch(void* y, float* mean, float* rstd, const void* x, const void* gamma,
                         const void* beta, int64_t rows, int64_t cols, float eps,
                         cudaStream_t s) {
    const LnPlan p = plan_for(rows, cols, false, sizeof(T));
    if (!p.cta) {
        LS_GROUP_CASES(fwd_group, T, y, mean, rstd, x, gamma, beta, rows, cols, eps, p, s)
    } else {
        LS_CTA_CASES(fwd_cta, T, y, mean, rstd, x, gamma, beta, rows, cols, eps, p, s)
    }
}

template <typename T>
cudaError_t bwd_dispatch(void* dx, float* partial, const void* dy, const void* x,
                         const void* gamma, const float* mean, const float* rstd, int64_t rows,
                         int64_t cols, cudaStream_t s) {
    const LnPlan p = plan_for(rows, cols, true, sizeof(T));
    if (!p.cta) {
        LS_GROUP_CASES(bwd_group, T, dx, partial, dy, x, gamma, mean, rstd, rows, cols, p, s)
    } else {
        LS_CTA_CASES(bwd_cta, T, dx, partial, dy, x, gamma, mean, rstd, rows, cols, p, s)
    }
}

}  // namespace

ColReducePlan layernorm_bwd_plan(int64_t rows, int64_t cols, size_t esize) {
    const LnPlan p = plan_for(rows, cols, true, esize);
    return ColReducePlan{p.grid, 2 * cols};
}

cudaError_t layernorm_take_device_error(unsigned int* flags) {
    return take_device_error_word(flags);
}

cudaError_t launch_layernorm_fwd(DType dt, void* y, float* mean, float* rstd, const void* x,
                                 const void* gamma, const void* beta, int64_t rows, int64_t cols,
                                 float eps, cudaStream_t s) {
    if (dt == DType::F16)
        return fwd_dispatch<__half>(y, mean, rstd, x, gamma, beta, rows, cols, eps, s);
    return fwd_dispatch<float>(y, mean, rstd, x, gamma, beta, rows, cols, eps, s);
}

cudaError_t launch_layernorm_bwd(DType dt, void* dx, float* partial, const void* dy,
                                 const void* x, const void* gamma, const float* mean,
                                 const float* rstd, int64_t rows, int64_t cols, cudaStream_t s) {
    if (dt == DType::F16)
        return bwd_dispatch<__half>(dx, partial, dy, x, gamma, mean, rstd, rows, cols, s);
    return bwd_dispatch<float>(dx, partial, dy, x, gamma, mean, rstd, rows, cols, s);
}

}  // namespace ls
