// qkv.cu -- bias + reshape of Q, K, V ("CMU 11-868 L10 (LightSeq)", technique 1
// "kernel fusion", slide p.12: adding the bias and reshaping Q, K and V is one
// fused elementwise kernel after the QKV projection GEMM).
//
// The projection writes, per token row (row = b*seq + l), 3*H values: Q, K and
// V, each H = heads*d columns split into heads of d.  The forward adds the bias
// and moves each 8-element vector (d % 8 == 0, so a vector never straddles a
// head) to the head-major [3, batch, heads, seq, d] layout that the attention
// GEMMs read: the reads are contiguous rows, the writes contiguous runs of d
// elements.  The backward gathers the gradient back into rows and sums it
// over rows for the bias gradient, on the 128-row x 64-column tiles of the
// dropout backward (one FP32 partial row per 128 rows, then the fixed-order
// column reduction), so the bias gradient is reproducible bit for bit.
#include "ls_device.cuh"
#include "ls_internal.h"

namespace ls {
namespace {

constexpr int kThreads = 256;

// Index arithmetic of the reshape, on vectors: a column vector cv of a row
// (0 <= cv < 3*H/8) is (s, h, jv) = (which of Q/K/V, head, vector within the
// head); the row is (b, l).
struct QkvShape {
    uint32_t nvr;        // vectors per row = 3*H/8
    uint32_t seq, heads, dv;  // dv = d/8
    uint64_t batch;
    FastDiv by_nvr, by_hv, by_dv, by_seq;  // hv = H/8
};

template <typename I>
__device__ __forceinline__ uint64_t out_vector(uint64_t row, uint32_t cv, const QkvShape& q) {
    uint32_t s, rem, h, jv;
    s = fdiv(cv, q.by_hv);
    rem = cv - s * q.by_hv.d;
    h = fdiv(rem, q.by_dv);
    jv = rem - h * q.dv;
    uint64_t b, l;
    if (sizeof(I) == 4) {
        b = fdiv(static_cast<uint32_t>(row), q.by_seq);
        l = row - b * q.seq;
    } else {
        b = row / q.seq;
        l = row - b * q.seq;
    }
    return (((static_cast<uint64_t>(s) * q.batch + b) * q.heads + h) * q.seq + l) * q.dv + jv;
}

template <typename T, typename I>
__global__ void __launch_bounds__(kThreads)
qkv_fwd_kernel(T* __restrict__ out, const T* __restrict__ qkv, const T* __restrict__ bias,
               uint64_t nv, const __grid_constant__ QkvShape q) {
    pdl_enter();
    const I n = static_cast<I>(nv);
    const I S = static_cast<I>(gridDim.x) * kThreads;
    for (I v = static_cast<I>(blockIdx.x) * kThreads + threadIdx.x; v < n; v += S) {
        uint64_t row;
        uint32_t cv;
        if (sizeof(I) == 4) {
            row = fdiv(static_cast<uint32_t>(v), q.by_nvr);
            cv = static_cast<uint32_t>(v - row * q.nvr);
        } else {
            row = static_cast<uint64_t>(v) / q.nvr;
            cv = static_cast<uint32_t>(static_cast<uint64_t>(v) - row * q.nvr);
        }
        float x[kVec], b[kVec], o[kVec];
        load8f<T>(qkv + static_cast<size_t>(v) * kVec, x);
        load8f<T>(bias + static_cast<size_t>(cv) * kVec, b);
#pragma unroll
        for (int j = 0; j < kVec; ++j) o[j] = x[j] + b[j];
        store8f<T>(out + out_vector<I>(row, cv, q) * kVec, o);
    }
}

// Backward tiles: 128 rows x 64 columns; lane l of an 8-lane group owns one
// column vector, each of the 32 row slots 4 rows per tile.
constexpr int kLanes = 8;
constexpr int kSlots = kThreads / kLanes;   // 32
constexpr int kRowsPerSlot = 4;
constexpr int kTileRows = kSlots * kRowsPerSlot;  // 128
constexpr int kTileCols = kLanes * kVec;          // 64

struct QkvBwdArgs {
    int64_t rows;
    int cols;  // 3*H
    int nbands;
    int64_t ntiles;
};

template <typename T, typename I>
__global__ void __launch_bounds__(kThreads)
qkv_bwd_kernel(T* __restrict__ dqkv, float* __restrict__ partial, const T* __restrict__ dout,
               const __grid_constant__ QkvBwdArgs a, const __grid_constant__ QkvShape q) {
    __shared__ __align__(16) float red[kSlots][kTileCols];
    pdl_enter();
    const int lane = threadIdx.x % kLanes;
    const int slot = threadIdx.x / kLanes;
    for (int64_t tile = blockIdx.x; tile < a.ntiles; tile += gridDim.x) {
        const int64_t chunk = tile / a.nbands;
        const int band = static_cast<int>(tile - chunk * a.nbands);
        const int c0 = (band * kLanes + lane) * kVec;
        const uint32_t cv = static_cast<uint32_t>(c0 / kVec);
        const int64_t r0 = chunk * kTileRows + slot;
        Raw8<T> g[kRowsPerSlot];
#pragma unroll
        for (int u = 0; u < kRowsPerSlot; ++u) {
            const int64_t r = r0 + static_cast<int64_t>(u) * kSlots;
            if (c0 < a.cols && r < a.rows)
                g[u] = load8<T>(dout + out_vector<I>(static_cast<uint64_t>(r), cv, q) * kVec);
        }
        float acc[kVec];
#pragma unroll
        for (int j = 0; j < kVec; ++j) acc[j] = 0.f;
#pragma unroll
        for (int u = 0; u < kRowsPerSlot; ++u) {
            const int64_t r = r0 + static_cast<int64_t>(u) * kSlots;
            if (!(c0 < a.cols && r < a.rows)) continue;
            store8<T>(dqkv + r * a.cols + c0, g[u]);
            float f[kVec];
            unpack(g[u], f);
#pragma unroll
            for (int j = 0; j < kVec; ++j) acc[j] += f[j];
        }
        if (partial == nullptr) continue;
        // The 32 row slots of each column, added in slot order.
        __syncthreads();  // the previous tile's readers of red[] are done
        float4* dst = reinterpret_cast<float4*>(&red[slot][lane * kVec]);
        dst[0] = make_float4(acc[0], acc[1], acc[2], acc[3]);
        dst[1] = make_float4(acc[4], acc[5], acc[6], acc[7]);
        __syncthreads();
        if (threadIdx.x < kTileCols) {
            const int col = band * kTileCols + threadIdx.x;
            if (col < a.cols) {
                float s = 0.f;
#pragma unroll 8
                for (int k = 0; k < kSlots; ++k) s += red[k][threadIdx.x];
                partial[chunk * a.cols + col] = s;
            }
        }
    }
}

QkvShape make_shape(int64_t batch, int64_t seq, int64_t heads, int64_t d) {
    QkvShape q;
    const uint32_t hv = static_cast<uint32_t>(heads * d / kVec);
    q.nvr = 3 * hv;
    q.seq = static_cast<uint32_t>(seq);
    q.heads = static_cast<uint32_t>(heads);
    q.dv = static_cast<uint32_t>(d / kVec);
    q.batch = static_cast<uint64_t>(batch);
    q.by_nvr = make_fastdiv(q.nvr);
    q.by_hv = make_fastdiv(hv);
    q.by_dv = make_fastdiv(q.dv);
    q.by_seq = make_fastdiv(q.seq);
    return q;
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
cudaError_t fwd_impl(void* out, const void* qkv, const void* bias, int64_t batch, int64_t seq,
                     int64_t heads, int64_t d, cudaStream_t s) {
    const QkvShape q = make_shape(batch, seq, heads, d);
    const uint64_t nv = static_cast<uint64_t>(batch * seq) * q.nvr;
    static const int occ = occupancy(qkv_fwd_kernel<T, uint64_t>);
    const int64_t want = static_cast<int64_t>((nv + kThreads - 1) / kThreads);
    const int64_t grid = std::max<int64_t>(1, std::min<int64_t>(want, int64_t{sm_count()} * occ));
    // 32-bit indices (and multiply-shift division) while every index < 2^31.
    const bool narrow = nv + static_cast<uint64_t>(grid) * kThreads < (uint64_t{1} << 31);
    auto kern = narrow ? qkv_fwd_kernel<T, uint32_t> : qkv_fwd_kernel<T, uint64_t>;
    return launch_pdl(kern, dim3(static_cast<unsigned>(grid)), dim3(kThreads), 0, s,
                      static_cast<T*>(out), static_cast<const T*>(qkv),
                      static_cast<const T*>(bias), nv, q);
}

template <typename T>
cudaError_t bwd_impl(void* dqkv, float* partial, const void* dout, int64_t batch, int64_t seq,
                     int64_t heads, int64_t d, cudaStream_t s) {
    const QkvShape q = make_shape(batch, seq, heads, d);
    QkvBwdArgs a;
    a.rows = batch * seq;
    a.cols = static_cast<int>(3 * heads * d);
    a.nbands = (a.cols + kTileCols - 1) / kTileCols;
    a.ntiles = ((a.rows + kTileRows - 1) / kTileRows) * a.nbands;
    static const int occ = occupancy(qkv_bwd_kernel<T, uint64_t>);
    const int64_t grid = std::max<int64_t>(1, std::min<int64_t>(a.ntiles, int64_t{sm_count()} * occ));
    // Multiply-shift division of the row index while rows < 2^31.
    auto kern = a.rows < (int64_t{1} << 31) ? qkv_bwd_kernel<T, uint32_t>
                                             : qkv_bwd_kernel<T, uint64_t>;
    return launch_pdl(kern, dim3(static_cast<unsigned>(grid)), dim3(kThreads), 0, s,
                      static_cast<T*>(dqkv), partial, static_cast<const T*>(dout), a, q);
}

}  // namespace

cudaError_t launch_qkv_fwd(DType dt, void* out, const void* qkv, const void* bias, int64_t batch,
                           int64_t seq, int64_t heads, int64_t d, cudaStream_t s) {
    if (dt == DType::F16) return fwd_impl<__half>(out, qkv, bias, batch, seq, heads, d, s);
    return fwd_impl<float>(out, qkv, bias, batch, seq, heads, d, s);
}

cudaError_t launch_qkv_bwd(DType dt, void* dqkv, float* partial, const void* dout, int64_t batch,
                           int64_t seq, int64_t heads, int64_t d, cudaStream_t s) {
    if (dt == DType::F16) return bwd_impl<__half>(dqkv, partial, dout, batch, seq, heads, d, s);
    return bwd_impl<float>(dqkv, partial, dout, batch, seq, heads, d, s);
}

}  // namespace ls
