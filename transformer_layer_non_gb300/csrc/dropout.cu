// dropout.cu -- fused bias+dropout+residual and bias+ReLU+dropout, forward and
// backward ("CMU 11-868 L10 (LightSeq)", technique 1, slide p.12: each chain of
// elementwise steps between two GEMMs is one kernel; "LightSeq2", sections
// 2.1.1-2.1.2: the dropout mask is saved in the forward and reused backward).
//
// Layout.  A CTA of 256 threads works on a tile of (256/LANES)*U rows by
// LANES*8 columns.  Lane `l` of a row group owns one 8-element column vector
// (16 bytes in FP16) and keeps it for every row of the tile, so bias values
// are loaded once per thread and bias-gradient partial sums accumulate in
// registers.  All U row loads of a thread are issued before any arithmetic so
// that U (or 2U) independent 16-byte loads per thread are in flight.
//
// Mask.  With cols % 8 == 0 the 8 elements of a vector are one mask byte
// (byte i/8 of the little-endian uint32 word array), so every thread writes or
// reads exactly one byte per vector.
#include "ls_device.cuh"
#include "ls_internal.h"

namespace ls {
namespace {

constexpr int kThreads = 256;

// Forward.  RELU=false: out = residual + keep*(x+bias)*scale, bit = keep.
//           RELU=true:  z = x+bias; bit = (z>0)&keep; out = bit*z*scale.
template <typename T, bool RELU, int LANES, int U>
__global__ void __launch_bounds__(kThreads)
dropout_fwd_kernel(T* out, uint8_t* __restrict__ mask, const T* x, const T* __restrict__ bias,
                   const T* residual, int64_t rows, int cols, uint32_t thr, float scale,
                   PhiloxKey key, uint32_t off_lo, uint32_t off_hi, int mask_tail_bytes) {
    constexpr int RPS = kThreads / LANES;  // rows per step
    const int lane = threadIdx.x % LANES;
    const int slot = threadIdx.x / LANES;
    const int nvec = cols / kVec;
    const int cv = blockIdx.y * LANES + lane;
    const bool col_ok = cv < nvec;
    const int c0 = cv * kVec;
    const int64_t r0 = static_cast<int64_t>(blockIdx.x) * (RPS * U) + slot;

    Raw8<T> xr[U];
    Raw8<T> rr[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
        const int64_t r = r0 + static_cast<int64_t>(u) * RPS;
        if (col_ok && r < rows) {
            const int64_t off = r * cols + c0;
            xr[u] = load8<T>(x + off);
            if (!RELU) rr[u] = load8<T>(residual + off);
        }
    }
    float b[kVec];
    if (col_ok) load8f<T>(bias + c0, b);

#pragma unroll
    for (int u = 0; u < U; ++u) {
        const int64_t r = r0 + static_cast<int64_t>(u) * RPS;
        if (!(col_ok && r < rows)) continue;
        const int64_t i = r * cols + c0;
        const uint32_t keep = keep_bits8(static_cast<uint64_t>(i), thr, key, off_lo, off_hi);
        float xf[kVec], o[kVec];
        unpack(xr[u], xf);
        uint32_t bits = 0;
        if (RELU) {
#pragma unroll
            for (int j = 0; j < kVec; ++j) {
                const float z = xf[j] + b[j];
                const bool on = (z > 0.f) && ((keep >> j) & 1u);
                bits |= on ? (1u << j) : 0u;
                o[j] = on ? z * scale : 0.f;
            }
        } else {
            float rf[kVec];
            unpack(rr[u], rf);
#pragma unroll
            for (int j = 0; j < kVec; ++j) {
                const float z = xf[j] + b[j];
                o[j] = ((keep >> j) & 1u) ? rf[j] + z * scale : rf[j];
            }
            bits = keep;
        }
        store8f<T>(out + i, o);
        if (mask) mask[i >> 3] = static_cast<uint8_t>(bits);
    }
    // Bytes of the last mask word past the last element are defined as 0.
    if (mask && mask_tail_bytes > 0 && blockIdx.x == 0 && blockIdx.y == 0 && threadIdx.x == 0) {
        const int64_t nbytes = rows * cols / 8;
        for (int k = 0; k < mask_tail_bytes; ++k) mask[nbytes + k] = 0;
    }
}

// Backward: dx = bit * dout * scale; the bit comes from the mask, or (REGEN)
// is drawn again from Philox.  With partial != nullptr the column sums of dx
// over the CTA's rows go to partial[blockIdx.x, :].
template <typename T, bool REGEN, int LANES, int U>
__global__ void __launch_bounds__(kThreads)
dropout_bwd_kernel(T* dx, float* __restrict__ partial, const T* dout,
                   const uint8_t* __restrict__ mask, int64_t rows, int cols, uint32_t thr,
                   float scale, PhiloxKey key, uint32_t off_lo, uint32_t off_hi) {
    constexpr int RPS = kThreads / LANES;
    const int lane = threadIdx.x % LANES;
    const int slot = threadIdx.x / LANES;
    const int nvec = cols / kVec;
    const int cv = blockIdx.y * LANES + lane;
    const bool col_ok = cv < nvec;
    const int c0 = cv * kVec;
    const int64_t r0 = static_cast<int64_t>(blockIdx.x) * (RPS * U) + slot;

    Raw8<T> dr[U];
    uint32_t mb[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
        const int64_t r = r0 + static_cast<int64_t>(u) * RPS;
        mb[u] = 0;
        if (col_ok && r < rows) {
            const int64_t off = r * cols + c0;
            dr[u] = load8<T>(dout + off);
            if (!REGEN) mb[u] = mask[off >> 3];
        }
    }
    float acc[kVec];
#pragma unroll
    for (int j = 0; j < kVec; ++j) acc[j] = 0.f;

#pragma unroll
    for (int u = 0; u < U; ++u) {
        const int64_t r = r0 + static_cast<int64_t>(u) * RPS;
        if (!(col_ok && r < rows)) continue;
        const int64_t i = r * cols + c0;
        const uint32_t bits =
            REGEN ? keep_bits8(static_cast<uint64_t>(i), thr, key, off_lo, off_hi) : mb[u];
        float g[kVec];
        unpack(dr[u], g);
#pragma unroll
        for (int j = 0; j < kVec; ++j) {
            g[j] = ((bits >> j) & 1u) ? g[j] * scale : 0.f;
            acc[j] += g[j];
        }
        store8f<T>(dx + i, g);
    }
    if (partial == nullptr) return;

    // Sum the RPS row slots of each column in a fixed order.
    __shared__ __align__(16) float red[RPS][LANES * kVec];
    float4* dst = reinterpret_cast<float4*>(&red[slot][lane * kVec]);
    dst[0] = make_float4(acc[0], acc[1], acc[2], acc[3]);
    dst[1] = make_float4(acc[4], acc[5], acc[6], acc[7]);
    __syncthreads();
    for (int k = threadIdx.x; k < LANES * kVec; k += kThreads) {
        const int col = blockIdx.y * LANES * kVec + k;
        if (col >= cols) continue;
        float s = 0.f;
#pragma unroll 8
        for (int q = 0; q < RPS; ++q) s += red[q][k];
        partial[static_cast<int64_t>(blockIdx.x) * cols + col] = s;
    }
}

// partial [parts, width] FP32 -> out [width] in T, summing rows in a fixed
// order: thread group g takes rows g, g+G, ...; then the G group sums are added
// in group order.
constexpr int kRedCols = 32;
constexpr int kRedGroups = 16;
template <typename T>
__global__ void __launch_bounds__(kRedCols* kRedGroups)
colreduce_kernel(T* __restrict__ out0, T* __restrict__ out1, int64_t split,
                 const float* __restrict__ partial, int64_t parts, int64_t width) {
    const int cx = threadIdx.x % kRedCols;
    const int gy = threadIdx.x / kRedCols;
    const int64_t col = static_cast<int64_t>(blockIdx.x) * kRedCols + cx;
    float s = 0.f;
    if (col < width) {
#pragma unroll 4
        for (int64_t p = gy; p < parts; p += kRedGroups) s += partial[p * width + col];
    }
    __shared__ float sm[kRedGroups][kRedCols + 1];
    sm[gy][cx] = s;
    __syncthreads();
    if (gy == 0 && col < width) {
        float t = 0.f;
#pragma unroll
        for (int g = 0; g < kRedGroups; ++g) t += sm[g][cx];
        if (col < split)
            out0[col] = static_cast<T>(t);
        else
            out1[col - split] = static_cast<T>(t);
    }
}

// Tile shapes.  Forward: 32 lanes x 8 elements = 256 columns per tile, so a
// warp writes one full 32-byte mask sector per row.  Backward: 8 lanes
// (64 columns) per row and 128 rows per tile, so the bias-gradient partial
// sums are few (one row of `cols` floats per 128 input rows).
constexpr int kFwdLanes = 32, kFwdU = 4;
constexpr int kBwdLanes = 8, kBwdU = 4;
constexpr int kBwdRowsPerTile = (kThreads / kBwdLanes) * kBwdU;

PhiloxKey make_key(uint64_t seed) {
    return PhiloxKey{static_cast<uint32_t>(seed), static_cast<uint32_t>(seed >> 32)};
}

template <typename T, bool RELU>
cudaError_t fwd_impl(void* out, uint8_t* mask, const void* x, const void* bias,
                     const void* residual, int64_t rows, int64_t cols, const DropoutRng& rng,
                     cudaStream_t s) {
    constexpr int RPT = (kThreads / kFwdLanes) * kFwdU;
    const int64_t nvec = cols / kVec;
    dim3 grid(static_cast<unsigned>((rows + RPT - 1) / RPT),
              static_cast<unsigned>((nvec + kFwdLanes - 1) / kFwdLanes));
    const int64_t n = rows * cols;
    const int tail = static_cast<int>(((n + 31) / 32) * 4 - n / 8);
    dropout_fwd_kernel<T, RELU, kFwdLanes, kFwdU><<<grid, kThreads, 0, s>>>(
        static_cast<T*>(out), mask, static_cast<const T*>(x), static_cast<const T*>(bias),
        static_cast<const T*>(residual), rows, static_cast<int>(cols), rng.thr, rng.scale,
        make_key(rng.seed), static_cast<uint32_t>(rng.offset),
        static_cast<uint32_t>(rng.offset >> 32), tail);
    return cudaGetLastError();
}

template <typename T>
cudaError_t bwd_impl(void* dx, float* partial, const void* dout, const uint8_t* mask,
                     int64_t rows, int64_t cols, const DropoutRng& rng, cudaStream_t s) {
    const int64_t nvec = cols / kVec;
    dim3 grid(static_cast<unsigned>((rows + kBwdRowsPerTile - 1) / kBwdRowsPerTile),
              static_cast<unsigned>((nvec + kBwdLanes - 1) / kBwdLanes));
    const PhiloxKey key = make_key(rng.seed);
    const uint32_t olo = static_cast<uint32_t>(rng.offset);
    const uint32_t ohi = static_cast<uint32_t>(rng.offset >> 32);
    if (mask)
        dropout_bwd_kernel<T, false, kBwdLanes, kBwdU><<<grid, kThreads, 0, s>>>(
            static_cast<T*>(dx), partial, static_cast<const T*>(dout), mask, rows,
            static_cast<int>(cols), rng.thr, rng.scale, key, olo, ohi);
    else
        dropout_bwd_kernel<T, true, kBwdLanes, kBwdU><<<grid, kThreads, 0, s>>>(
            static_cast<T*>(dx), partial, static_cast<const T*>(dout), nullptr, rows,
            static_cast<int>(cols), rng.thr, rng.scale, key, olo, ohi);
    return cudaGetLastError();
}

}  // namespace

ColReducePlan dropout_bwd_plan(int64_t rows, int64_t cols) {
    return ColReducePlan{(rows + kBwdRowsPerTile - 1) / kBwdRowsPerTile, cols};
}

cudaError_t launch_colreduce(DType dt, void* out0, void* out1, int64_t split,
                             const float* partial, int64_t parts, int64_t width, cudaStream_t s) {
    const unsigned grid = static_cast<unsigned>((width + kRedCols - 1) / kRedCols);
    if (dt == DType::F16)
        colreduce_kernel<__half><<<grid, kRedCols * kRedGroups, 0, s>>>(
            static_cast<__half*>(out0), static_cast<__half*>(out1), split, partial, parts, width);
    else
        colreduce_kernel<float><<<grid, kRedCols * kRedGroups, 0, s>>>(
            static_cast<float*>(out0), static_cast<float*>(out1), split, partial, parts, width);
    return cudaGetLastError();
}

cudaError_t launch_dropout_fwd(DType dt, bool relu, void* out, uint8_t* mask, const void* x,
                               const void* bias, const void* residual, int64_t rows, int64_t cols,
                               const DropoutRng& rng, cudaStream_t s) {
    if (dt == DType::F16)
        return relu ? fwd_impl<__half, true>(out, mask, x, bias, residual, rows, cols, rng, s)
                    : fwd_impl<__half, false>(out, mask, x, bias, residual, rows, cols, rng, s);
    return relu ? fwd_impl<float, true>(out, mask, x, bias, residual, rows, cols, rng, s)
                : fwd_impl<float, false>(out, mask, x, bias, residual, rows, cols, rng, s);
}

cudaError_t launch_dropout_bwd(DType dt, void* dx, float* partial, const void* dout,
                               const uint8_t* mask, int64_t rows, int64_t cols,
                               const DropoutRng& rng, cudaStream_t s) {
    if (dt == DType::F16) return bwd_impl<__half>(dx, partial, dout, mask, rows, cols, rng, s);
    return bwd_impl<float>(dx, partial, dout, mask, rows, cols, rng, s);
}

}  // namespace ls
