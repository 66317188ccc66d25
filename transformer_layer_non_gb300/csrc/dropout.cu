// dropout.cu -- fused bias+dropout+residual and bias+ReLU+dropout, forward and
// backward ("CMU 11-868 L10 (LightSeq)", technique 1, slide p.12: each chain of
// elementwise steps between two GEMMs is one kernel; "LightSeq2", sections
// 2.1.1-2.1.2: the dropout mask is saved in the forward and reused backward).
//
// Forward layout.  The activation is a flat array of 8-element vectors (16
// bytes in FP16); with cols % 8 == 0 a vector never straddles a row and its 8
// keep bits are one mask byte.  A persistent grid (a multiple of the SM count)
// walks the vectors in rounds: in round k, warp w of CTA b takes the 32
// consecutive vectors starting at (k * W + b + w * gridDim) * 32, W = all warps.
// The last, partial round is thus spread over every CTA instead of piling onto
// a few SMs.  A thread handles U rounds at a time: it issues their loads and
// draws their Philox words (two Philox calls per vector) while the loads are in
// flight, then computes in FP32 and stores.  bias+dropout+residual keeps the
// keep bits packed (one byte per vector, five CTAs per SM); bias+ReLU+dropout
// is software-pipelined over two register buffers and selects with predicates
// on the FMA pipes (its Philox work is a large share of its time).
//
// Backward layout.  The bias gradient needs column sums, so the backward works
// on 2-D tiles of 128 rows x 64 columns: lane l of an 8-lane row group owns one
// column vector for all rows of the tile and accumulates its partial sums in
// registers; the 32 row slots are summed in shared memory in a fixed order into
// one FP32 partial row per tile.  A persistent grid walks the tiles.  A second
// kernel adds the partial rows of each column in a fixed order, so the result
// does not depend on the grid or the GPU.
#include "ls_device.cuh"
#include "ls_internal.h"

namespace ls {
namespace {

constexpr int kThreads = 256;

// ---------------------------------------------------------------------------
// Forward.
// ---------------------------------------------------------------------------
// Kernel arguments live in the constant bank, so the Philox round keys,
// computed once on the host, are instruction operands rather than registers.
struct FwdArgs {
    uint64_t nv;        // vectors in the tensor (rows * cols / 8)
    uint32_t nvr;       // vectors per row
    uint32_t step_col;  // (vectors per round) mod nvr
    uint32_t thr;
    float scale;
    PhiloxSchedule ks;
    uint32_t off_lo, off_hi;
    int mask_tail_bytes;
    int prefetch;  // bias+dropout+residual: prefetch the first vector before the wait
};

template <typename T, bool RELU, int U, typename I>
__device__ __forceinline__ void fwd_load(Raw8<T> (&xr)[U], Raw8<T> (&rr)[U], const T* x,
                                         const T* residual, I v, I S, I nv) {
#pragma unroll
    for (int u = 0; u < U; ++u) {
        const I vu = v + u * S;
        if (vu < nv) {
            xr[u] = load8<T>(x + static_cast<size_t>(vu) * kVec);
            if (!RELU) rr[u] = load8<T>(residual + static_cast<size_t>(vu) * kVec);
        }
    }
}

// Keep bits of the U vectors of a chunk (bit j of keep[u] decides element j of
// vector u); called right after the chunk's loads are issued, so the Philox
// arithmetic overlaps their latency.  The bias+dropout+residual forward keeps
// only these 8 bits per vector in registers (its two input streams need the
// occupancy more than fewer integer instructions).
template <int U, typename I>
__device__ __forceinline__ void fwd_keep(uint32_t (&keep)[U], I v, I S, I nv,
                                         const FwdArgs& a, const PhiloxSchedule& ks) {
#pragma unroll
    for (int u = 0; u < U; ++u) {
        const I vu = v + u * S;
        if (sizeof(I) == 4)
            keep[u] = vu < nv ? keep_bits8_blk(static_cast<uint32_t>(vu) * 2u, 0u, a.thr, ks,
                                               a.off_lo, a.off_hi)
                              : 0u;
        else
            keep[u] = vu < nv ? keep_bits8(static_cast<uint64_t>(vu) * kVec, a.thr, ks, a.off_lo,
                                           a.off_hi)
                              : 0u;
    }
}

// bias + dropout + residual on the U vectors of a chunk.
template <typename T, int U, typename I>
__device__ __forceinline__ void bdr_compute(const Raw8<T> (&xr)[U], const Raw8<T> (&rr)[U],
                                            const uint32_t (&kp)[U], T* out, uint8_t* mask,
                                            const T* __restrict__ bias, I v, uint32_t cv, I S,
                                            I nv, const FwdArgs& a) {
#pragma unroll
    for (int u = 0; u < U; ++u) {
        const I vu = v + u * S;
        if (vu >= nv) break;
        float b[kVec], z[kVec], o[kVec], rf[kVec];
        load8f<T>(bias + static_cast<size_t>(cv) * kVec, b);
        add8(xr[u], b, z);  // z = x + bias, exact conversion of x folded in
        unpack(rr[u], rf);
        const uint32_t keep = kp[u];
#pragma unroll
        for (int j = 0; j < kVec; ++j)
            o[j] = ((keep >> j) & 1u) ? rf[j] + z[j] * a.scale : rf[j];
        store8f<T>(out + static_cast<size_t>(vu) * kVec, o);
        if (mask) mask[vu] = static_cast<uint8_t>(keep);
        cv += a.step_col;
        if (cv >= a.nvr) cv -= a.nvr;
    }
}

// Philox words of the U vectors of a chunk (8 per vector: word j decides
// element j); called right after the chunk's loads are issued, so the Philox
// arithmetic overlaps their latency.  With 32-bit indices (the host picks them
// when every vector index and its counter block 2 * vector index fit in 32
// bits) the block's high word is 0.
template <int U, typename I>
__device__ __forceinline__ void fwd_words(uint4 (&wa)[U], uint4 (&wb)[U], I v, I S, I nv,
                                          const FwdArgs& a, const PhiloxSchedule& ks) {
#pragma unroll
    for (int u = 0; u < U; ++u) {
        const I vu = v + u * S;
        if (vu < nv) {
            uint32_t lo, hi;
            if (sizeof(I) == 4) {
                lo = static_cast<uint32_t>(vu) * 2u;
                hi = 0u;
            } else {
                const uint64_t blk = static_cast<uint64_t>(vu) * 2u;
                lo = static_cast<uint32_t>(blk);
                hi = static_cast<uint32_t>(blk >> 32);
            }
            wa[u] = philox4x32_10(make_uint4(lo, hi, a.off_lo, a.off_hi), ks);
            // lo is even, so lo + 1 never carries into hi.
            wb[u] = philox4x32_10(make_uint4(lo + 1u, hi, a.off_lo, a.off_hi), ks);
        }
    }
}

// One element of the bias+ReLU+dropout epilogue, as predicated selects (FSEL
// runs on the FMA pipes; only the two compares use the integer ALU, which the
// Philox rounds already load): with keep = (w >= thr),
//   on = keep && z > 0;  o = on ? zs : 0;  bit = on,
// the bit returned as the float 2^j or 0, to be summed exactly.
__device__ __forceinline__ void brd_elem(uint32_t w, uint32_t thr, float z, float zs, float pow2j,
                                         float& o, float& bit) {
    asm("{\n\t.reg .pred p, q;\n\t"
        "setp.hs.u32 p, %2, %3;\n\t"
        "setp.gt.and.f32 q, %4, 0f00000000, p;\n\t"
        "selp.f32 %0, %5, 0f00000000, q;\n\t"
        "selp.f32 %1, %6, 0f00000000, q;\n\t}"
        : "=f"(o), "=f"(bit)
        : "r"(w), "r"(thr), "f"(z), "f"(zs), "f"(pow2j));
}
// 2^23 plus the sum of the bits' values 2^j (j < 8) is exact in FP32 and its
// low byte is the mask byte: the byte store takes it from the float's bits.
constexpr float kMaskMagic = 8388608.0f;

// Bias of column vector cv in FP32: from the CTA's shared-memory copy when the
// row fits there (SMEMB), else loaded and converted.
template <typename T, bool SMEMB>
__device__ __forceinline__ void bias8(const float* bsm, const T* __restrict__ bias, uint32_t cv,
                                      float (&b)[kVec]) {
    if (SMEMB) {
        const float4 b0 = *reinterpret_cast<const float4*>(bsm + cv * kVec);
        const float4 b1 = *reinterpret_cast<const float4*>(bsm + cv * kVec + 4);
        b[0] = b0.x; b[1] = b0.y; b[2] = b0.z; b[3] = b0.w;
        b[4] = b1.x; b[5] = b1.y; b[6] = b1.z; b[7] = b1.w;
    } else {
        load8f<T>(bias + static_cast<size_t>(cv) * kVec, b);
    }
}

template <typename T, bool SMEMB, int U, typename I>
__device__ __forceinline__ void brd_compute(const Raw8<T> (&xr)[U], const uint4 (&wa)[U],
                                            const uint4 (&wb)[U], T* out,
                                            uint8_t* mask, const float* bsm,
                                            const T* __restrict__ bias, I v, uint32_t cv, I S,
                                            I nv, const FwdArgs& a) {
#pragma unroll
    for (int u = 0; u < U; ++u) {
        const I vu = v + u * S;
        if (vu >= nv) break;
        float b[kVec], z[kVec], o[kVec], bit[kVec];
        bias8<T, SMEMB>(bsm, bias, cv, b);
        add8(xr[u], b, z);  // z = x + bias, exact conversion of x folded in
        const uint32_t w[kVec] = {wa[u].x, wa[u].y, wa[u].z, wa[u].w,
                                  wb[u].x, wb[u].y, wb[u].z, wb[u].w};
#pragma unroll
        for (int j = 0; j < kVec; j += 2) {
            const float2 zs = mul2(make_float2(z[j], z[j + 1]), make_float2(a.scale, a.scale));
            brd_elem(w[j], a.thr, z[j], zs.x, static_cast<float>(1u << j), o[j], bit[j]);
            brd_elem(w[j + 1], a.thr, z[j + 1], zs.y, static_cast<float>(1u << (j + 1)), o[j + 1],
                     bit[j + 1]);
        }
        store8f<T>(out + static_cast<size_t>(vu) * kVec, o);
        if (mask) {
            const float m = ((kMaskMagic + bit[0]) + (bit[1] + bit[2])) +
                            ((bit[3] + bit[4]) + (bit[5] + (bit[6] + bit[7])));
            mask[vu] = static_cast<uint8_t>(__float_as_uint(m));
        }
        cv += a.step_col;
        if (cv >= a.nvr) cv -= a.nvr;
    }
}

// bias + dropout + residual: a chunk's loads are issued, its keep bits drawn
// while they are in flight, then it is computed and stored.  (Measured on
// GB300, two register buffers per thread gain nothing here: five CTAs per SM
// keep enough loads in flight, and the Philox work fits under the two input
// streams' memory time.)
template <typename T, int U, typename I>
__global__ void __launch_bounds__(kThreads, sizeof(T) == 2 ? 5 : 2)
bdr_fwd_kernel(T* out, uint8_t* mask, const T* x, const T* __restrict__ bias, const T* residual,
               const __grid_constant__ FwdArgs a) {
    const PhiloxSchedule& ks = a.ks;
    const I nv = static_cast<I>(a.nv);
    const I S = static_cast<I>(gridDim.x) * kThreads;  // vectors per round
    const I gw = blockIdx.x + static_cast<I>(threadIdx.x >> 5) * gridDim.x;
    I v = gw * 32 + (threadIdx.x & 31);
    // Before the wait, when the launch is about one chunk: the lines of the
    // first vector of x and residual, into L2.  (Measured on GB300 over
    // L2-cold launches: at 4096 x 768, one chunk, 4.71 -> 4.40 us, and 4.48
    // with both vectors; at 4096 x 1280, 1.7 chunks, every prefetch of part of
    // the input was slower, 6.9 -> 7.3-8.4 us, and of all of it no faster.)
    if (a.prefetch && v < nv) {
        prefetch_l2(x + static_cast<size_t>(v) * kVec);
        prefetch_l2(residual + static_cast<size_t>(v) * kVec);
    }
    pdl_enter();
    uint32_t cv = static_cast<uint32_t>(v % a.nvr);
    uint32_t stepU = 0;  // (U rounds) mod nvr, from the per-round step
#pragma unroll
    for (int u = 0; u < U; ++u) {
        stepU += a.step_col;
        if (stepU >= a.nvr) stepU -= a.nvr;
    }
    Raw8<T> xa[U], ra[U];
    uint32_t ka[U];
    while (v < nv) {
        fwd_load<T, false, U>(xa, ra, x, residual, v, S, nv);
        fwd_keep<U>(ka, v, S, nv, a, ks);
        bdr_compute<T, U>(xa, ra, ka, out, mask, bias, v, cv, S, nv, a);
        v += U * S;
        cv += stepU;
        if (cv >= a.nvr) cv -= a.nvr;
    }
    // Bytes of the last mask word past the last element are defined as 0.
    if (mask && a.mask_tail_bytes > 0 && blockIdx.x == 0 && threadIdx.x == 0)
        for (int k = 0; k < a.mask_tail_bytes; ++k) mask[a.nv + k] = 0;
}

// Largest row whose bias the bias+ReLU+dropout forward keeps in shared memory
// as FP32 (32 KB).
constexpr int64_t kFwdSmemBiasMaxCols = 8192;

// bias + ReLU + dropout, software-pipelined over two register buffers: while
// chunk k is computed and stored, chunk k+1's loads are in flight, and its
// Philox words are drawn right after, before it is needed.  The Philox and
// select work of this operator is a large part of its time, so it runs under
// the next chunk's memory latency instead of after it.  Measured on GB300 at
// BERT-base / GPT-2-large FFN widths: 14.1 / 23.0 us against 15.6 / 25.1 us for
// the unpipelined kernel with integer keep masks; two vectors per chunk at
// three CTAs per SM beat one vector at four, and a non-persistent grid (one
// chunk per thread) is slower (15.8 / 24.3 us).
template <typename T, bool SMEMB, int U, typename I>
__global__ void __launch_bounds__(kThreads, sizeof(T) == 2 ? 3 : 2)
brd_fwd_kernel(T* out, uint8_t* mask, const T* x, const T* __restrict__ bias,
               const __grid_constant__ FwdArgs a) {
    extern __shared__ __align__(16) float bsm[];  // [cols] FP32 bias when SMEMB
    const PhiloxSchedule& ks = a.ks;
    const I nv = static_cast<I>(a.nv);
    const I S = static_cast<I>(gridDim.x) * kThreads;  // vectors per round
    const I gw = blockIdx.x + static_cast<I>(threadIdx.x >> 5) * gridDim.x;
    I v = gw * 32 + (threadIdx.x & 31);
    pdl_enter();
    uint32_t cv = static_cast<uint32_t>(v % a.nvr);
    uint32_t stepU = 0;  // (U rounds) mod nvr, from the per-round step
#pragma unroll
    for (int u = 0; u < U; ++u) {
        stepU += a.step_col;
        if (stepU >= a.nvr) stepU -= a.nvr;
    }
    Raw8<T> xa[U], xb[U], unused[U];
    uint4 wa[U], wb[U];
    // The first chunk's loads go out before the bias is staged, so that the
    // bias's first (cold) read overlaps them instead of preceding them.
    if (v < nv) fwd_load<T, true, U>(xa, unused, x, nullptr, v, S, nv);
    if (SMEMB) {
        for (uint32_t c = threadIdx.x; c < a.nvr; c += kThreads) {
            float b[kVec];
            load8f<T>(bias + static_cast<size_t>(c) * kVec, b);
            float4* d = reinterpret_cast<float4*>(bsm + c * kVec);
            d[0] = make_float4(b[0], b[1], b[2], b[3]);
            d[1] = make_float4(b[4], b[5], b[6], b[7]);
        }
    }
    if (v < nv) fwd_words<U>(wa, wb, v, S, nv, a, ks);
    if (SMEMB) __syncthreads();
    while (v < nv) {
        const I v1 = v + U * S;
        fwd_load<T, true, U>(xb, unused, x, nullptr, v1, S, nv);
        brd_compute<T, SMEMB, U>(xa, wa, wb, out, mask, bsm, bias, v, cv, S, nv, a);
        cv += stepU;
        if (cv >= a.nvr) cv -= a.nvr;
        if (v1 >= nv) break;
        fwd_words<U>(wa, wb, v1, S, nv, a, ks);
        const I v2 = v1 + U * S;
        fwd_load<T, true, U>(xa, unused, x, nullptr, v2, S, nv);
        brd_compute<T, SMEMB, U>(xb, wa, wb, out, mask, bsm, bias, v1, cv, S, nv, a);
        cv += stepU;
        if (cv >= a.nvr) cv -= a.nvr;
        if (v2 >= nv) break;
        fwd_words<U>(wa, wb, v2, S, nv, a, ks);
        v = v2;
    }
    // Bytes of the last mask word past the last element are defined as 0.
    if (mask && a.mask_tail_bytes > 0 && blockIdx.x == 0 && threadIdx.x == 0)
        for (int k = 0; k < a.mask_tail_bytes; ++k) mask[a.nv + k] = 0;
}

// ---------------------------------------------------------------------------
// Backward.
// ---------------------------------------------------------------------------
constexpr int kBwdLanes = 8;                         // lanes per row segment (64 columns)
constexpr int kBwdRps = kThreads / kBwdLanes;        // row slots per CTA
constexpr int kBwdU = 4;                             // rows per slot per tile
constexpr int kBwdRowsPerTile = kBwdRps * kBwdU;     // 128
constexpr int kBwdColsPerTile = kBwdLanes * kVec;    // 64

struct BwdArgs {
    int64_t rows;
    int cols;
    int nbands;
    FastDiv by_nbands;  // tile -> (row chunk, column band); tile indices stay below 2^31
    int64_t ntiles;
    int late_trigger;  // CTAs loop over several tiles: release dependents at exit
    uint32_t thr;
    float scale;
    PhiloxSchedule ks;
    uint32_t off_lo, off_hi;
};

// Loads of one tile; with REGEN the keep bits are drawn here, after the loads
// are issued, so the Philox arithmetic overlaps their latency.
template <typename T, bool REGEN>
__device__ __forceinline__ void bwd_load(Raw8<T> (&dr)[kBwdU], uint32_t (&mb)[kBwdU],
                                         const T* dout, const uint8_t* mask, int64_t tile,
                                         const BwdArgs& a, const PhiloxSchedule& ks) {
    const uint32_t chunk32 = fdiv(static_cast<uint32_t>(tile), a.by_nbands);
    const int64_t chunk = chunk32;
    const int band = static_cast<int>(static_cast<uint32_t>(tile) - chunk32 * a.by_nbands.d);
    const int lane = threadIdx.x % kBwdLanes;
    const int c0 = (band * kBwdLanes + lane) * kVec;
    const int64_t r0 = chunk * kBwdRowsPerTile + threadIdx.x / kBwdLanes;
#pragma unroll
    for (int u = 0; u < kBwdU; ++u) {
        const int64_t r = r0 + static_cast<int64_t>(u) * kBwdRps;
        mb[u] = 0;
        if (tile < a.ntiles && c0 < a.cols && r < a.rows) {
            const int64_t off = r * a.cols + c0;
            dr[u] = load8<T>(dout + off);
            if (!REGEN) mb[u] = mask[off >> 3];
        }
    }
    if (REGEN) {
#pragma unroll
        for (int u = 0; u < kBwdU; ++u) {
            const int64_t r = r0 + static_cast<int64_t>(u) * kBwdRps;
            if (tile < a.ntiles && c0 < a.cols && r < a.rows)
                mb[u] = keep_bits8(static_cast<uint64_t>(r * a.cols + c0), a.thr, ks, a.off_lo,
                                   a.off_hi);
        }
    }
}

template <typename T, bool REGEN>
__device__ __forceinline__ void bwd_compute(const Raw8<T> (&dr)[kBwdU],
                                            const uint32_t (&mb)[kBwdU], T* dx, float* partial,
                                            float (*red)[kBwdColsPerTile], int64_t tile,
                                            const BwdArgs& a) {
    const uint32_t chunk32 = fdiv(static_cast<uint32_t>(tile), a.by_nbands);
    const int64_t chunk = chunk32;
    const int band = static_cast<int>(static_cast<uint32_t>(tile) - chunk32 * a.by_nbands.d);
    const int lane = threadIdx.x % kBwdLanes;
    const int slot = threadIdx.x / kBwdLanes;
    const int c0 = (band * kBwdLanes + lane) * kVec;
    const int64_t r0 = chunk * kBwdRowsPerTile + slot;
    float acc[kVec];
#pragma unroll
    for (int j = 0; j < kVec; ++j) acc[j] = 0.f;
#pragma unroll
    for (int u = 0; u < kBwdU; ++u) {
        const int64_t r = r0 + static_cast<int64_t>(u) * kBwdRps;
        if (!(c0 < a.cols && r < a.rows)) continue;
        const int64_t i = r * a.cols + c0;
        const uint32_t bits = mb[u];
        float g[kVec];
        unpack(dr[u], g);
#pragma unroll
        for (int j = 0; j < kVec; ++j) {
            g[j] = ((bits >> j) & 1u) ? g[j] * a.scale : 0.f;
            acc[j] += g[j];
        }
        store8f<T>(dx + i, g);
    }
    if (partial == nullptr) return;
    // Sum the row slots of each column in a fixed order.
    __syncthreads();  // the previous tile's readers of red[] are done
    float4* dst = reinterpret_cast<float4*>(&red[slot][lane * kVec]);
    dst[0] = make_float4(acc[0], acc[1], acc[2], acc[3]);
    dst[1] = make_float4(acc[4], acc[5], acc[6], acc[7]);
    __syncthreads();
    if (threadIdx.x < kBwdColsPerTile) {
        const int col = band * kBwdColsPerTile + threadIdx.x;
        if (col < a.cols) {
            float s = 0.f;
#pragma unroll 8
            for (int q = 0; q < kBwdRps; ++q) s += red[q][threadIdx.x];
            partial[chunk * a.cols + col] = s;
        }
    }
}

template <typename T, bool REGEN>
__global__ void __launch_bounds__(kThreads, sizeof(T) == 2 ? 4 : 2)
dropout_bwd_kernel(T* dx, float* __restrict__ partial, const T* dout,
                   const uint8_t* __restrict__ mask, const __grid_constant__ BwdArgs a) {
    __shared__ __align__(16) float red[kBwdRps][kBwdColsPerTile];
    const PhiloxSchedule& ks = a.ks;
    // Before the wait: the first tile's lines, into L2.  (Only the first:
    // prefetching both tiles a CTA loads at once was slower, 16.13 against
    // 15.88 us at 4096 x 5120, measured on GB300.)
    {
        const int lane = threadIdx.x % kBwdLanes;
        const int64_t tile = blockIdx.x;
        const uint32_t chunk32 = fdiv(static_cast<uint32_t>(tile), a.by_nbands);
        const int64_t chunk = chunk32;
        const int band = static_cast<int>(static_cast<uint32_t>(tile) - chunk32 * a.by_nbands.d);
        const int c0 = (band * kBwdLanes + lane) * kVec;
        const int64_t r0 = chunk * kBwdRowsPerTile + threadIdx.x / kBwdLanes;
#pragma unroll
        for (int u = 0; u < kBwdU; ++u) {
            const int64_t r = r0 + static_cast<int64_t>(u) * kBwdRps;
            if (tile < a.ntiles && c0 < a.cols && r < a.rows) {
                const int64_t off = r * a.cols + c0;
                prefetch_l2(dout + off);
                if (!REGEN && lane == 0) prefetch_l2(mask + (off >> 3));
            }
        }
    }
    // With several tiles per CTA the dependent launch is released as CTAs
    // exit (measured faster); with one tile per CTA at their start.
    pdl_wait();
    if (!a.late_trigger) pdl_trigger();
    int64_t t = blockIdx.x;
    Raw8<T> da[kBwdU], db[kBwdU];
    uint32_t ma[kBwdU], mbb[kBwdU];
    bwd_load<T, REGEN>(da, ma, dout, mask, t, a, ks);
    while (t < a.ntiles) {
        const int64_t t1 = t + gridDim.x;
        bwd_load<T, REGEN>(db, mbb, dout, mask, t1, a, ks);
        bwd_compute<T, REGEN>(da, ma, dx, partial, red, t, a);
        if (t1 >= a.ntiles) break;
        t = t1 + gridDim.x;
        bwd_load<T, REGEN>(da, ma, dout, mask, t, a, ks);
        bwd_compute<T, REGEN>(db, mbb, dx, partial, red, t1, a);
    }
}

// ---------------------------------------------------------------------------
// Fixed-order column reduction: partial [parts, width] FP32 -> out0/out1.
// A CTA covers COLS columns with 32 groups; group g adds rows g, g + 32, ... of
// its column in that order, then the 32 group sums are added in group order.
// The association depends only on (parts, width).  Few partial rows take
// narrow 8-column CTAs (more CTAs, one load each); many take 32 columns per
// CTA (measured on GB300: each faster in its own range).
// ---------------------------------------------------------------------------
constexpr int kRedGroups = 32;
constexpr int64_t kRedNarrowMaxParts = 64;
template <typename T, int COLS>
__global__ void __launch_bounds__(COLS* kRedGroups)
colreduce_kernel(T* __restrict__ out0, T* __restrict__ out1, int64_t split,
                 const float* __restrict__ partial, int64_t parts, int64_t width) {
    __shared__ float sm[kRedGroups][COLS + 1];
    pdl_enter();
    const int cx = threadIdx.x % COLS;
    const int gy = threadIdx.x / COLS;
    const int64_t col = static_cast<int64_t>(blockIdx.x) * COLS + cx;
    float s = 0.f;
    if (col < width) {
#pragma unroll 4
        for (int64_t p = gy; p < parts; p += kRedGroups) s += partial[p * width + col];
    }
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

PhiloxKey make_key(uint64_t seed) {
    return PhiloxKey{static_cast<uint32_t>(seed), static_cast<uint32_t>(seed >> 32)};
}

template <typename K>
int occupancy(K kernel, int threads, size_t smem) {
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kernel, threads, smem) != cudaSuccess ||
        n < 1)
        n = 1;
    return n;
}

constexpr int kFwdU = 2;
// bias + ReLU + dropout: vectors per thread per chunk (two chunks in flight).
constexpr int kBrdU = 2;

FwdArgs fwd_args(int64_t rows, int64_t cols, const DropoutRng& rng, int64_t grid) {
    FwdArgs a;
    a.nv = static_cast<uint64_t>(rows) * static_cast<uint64_t>(cols) / kVec;
    a.nvr = static_cast<uint32_t>(cols / kVec);
    a.step_col = static_cast<uint32_t>((static_cast<uint64_t>(grid) * kThreads) % a.nvr);
    a.thr = rng.thr;
    a.scale = rng.scale;
    a.ks = philox_schedule(make_key(rng.seed));
    a.off_lo = static_cast<uint32_t>(rng.offset);
    a.off_hi = static_cast<uint32_t>(rng.offset >> 32);
    a.mask_tail_bytes = static_cast<int>(((a.nv + 3) / 4) * 4 - a.nv);
    a.prefetch = 0;
    return a;
}

// 32-bit indices when no index the loop forms (up to nv + (U+2) rounds) and no
// counter block (2 * index) reaches 2^32.
bool narrow_index(uint64_t nv, int64_t grid) {
    return nv + static_cast<uint64_t>(kFwdU + 2) * static_cast<uint64_t>(grid) * kThreads <
           (uint64_t{1} << 31);
}

template <typename T>
cudaError_t bdr_fwd_impl(void* out, uint8_t* mask, const void* x, const void* bias,
                         const void* residual, int64_t rows, int64_t cols, const DropoutRng& rng,
                         cudaStream_t s) {
    static const int occ = occupancy(bdr_fwd_kernel<T, kFwdU, uint64_t>, kThreads, 0);
    const uint64_t nv = static_cast<uint64_t>(rows) * static_cast<uint64_t>(cols) / kVec;
    const int64_t want = static_cast<int64_t>((nv + kThreads * kFwdU - 1) / (kThreads * kFwdU));
    const int64_t grid = std::max<int64_t>(1, std::min<int64_t>(want, int64_t{sm_count()} * occ));
    FwdArgs a = fwd_args(rows, cols, rng, grid);
    const uint64_t chunk = static_cast<uint64_t>(grid) * kThreads * kFwdU;
    a.prefetch = nv <= chunk + chunk / 16 ? 1 : 0;
    auto kern = narrow_index(a.nv, grid) ? bdr_fwd_kernel<T, kFwdU, uint32_t>
                                         : bdr_fwd_kernel<T, kFwdU, uint64_t>;
    return launch_pdl(kern, dim3(static_cast<unsigned>(grid)), dim3(kThreads), 0, s,
                      static_cast<T*>(out), mask, static_cast<const T*>(x),
                      static_cast<const T*>(bias), static_cast<const T*>(residual), a);
}

template <typename T>
cudaError_t brd_fwd_impl(void* out, uint8_t* mask, const void* x, const void* bias, int64_t rows,
                         int64_t cols, const DropoutRng& rng, cudaStream_t s) {
    const bool smemb = cols <= kFwdSmemBiasMaxCols;
    const size_t smem = smemb ? static_cast<size_t>(cols) * sizeof(float) : 0;
    static const int occ = occupancy(brd_fwd_kernel<T, false, kBrdU, uint64_t>, kThreads, 0);
    static const int occ_s = occupancy(brd_fwd_kernel<T, true, kBrdU, uint64_t>, kThreads,
                                       kFwdSmemBiasMaxCols * sizeof(float));
    const uint64_t nv = static_cast<uint64_t>(rows) * static_cast<uint64_t>(cols) / kVec;
    const int64_t want = static_cast<int64_t>((nv + kThreads * kBrdU - 1) / (kThreads * kBrdU));
    const int64_t grid = std::max<int64_t>(
        1, std::min<int64_t>(want, int64_t{sm_count()} * (smemb ? occ_s : occ)));
    const FwdArgs a = fwd_args(rows, cols, rng, grid);
    const bool narrow = narrow_index(a.nv, grid);
    auto kern = smemb ? (narrow ? brd_fwd_kernel<T, true, kBrdU, uint32_t>
                                : brd_fwd_kernel<T, true, kBrdU, uint64_t>)
                      : (narrow ? brd_fwd_kernel<T, false, kBrdU, uint32_t>
                                : brd_fwd_kernel<T, false, kBrdU, uint64_t>);
    return launch_pdl(kern, dim3(static_cast<unsigned>(grid)), dim3(kThreads), smem, s,
                      static_cast<T*>(out), mask, static_cast<const T*>(x),
                      static_cast<const T*>(bias), a);
}

template <typename T>
cudaError_t bwd_impl(void* dx, float* partial, const void* dout, const uint8_t* mask,
                     int64_t rows, int64_t cols, const DropoutRng& rng, cudaStream_t s) {
    BwdArgs a;
    a.rows = rows;
    a.cols = static_cast<int>(cols);
    a.nbands = static_cast<int>((cols + kBwdColsPerTile - 1) / kBwdColsPerTile);
    a.by_nbands = make_fastdiv(static_cast<uint32_t>(a.nbands));
    a.ntiles = ((rows + kBwdRowsPerTile - 1) / kBwdRowsPerTile) * a.nbands;
    a.thr = rng.thr;
    a.scale = rng.scale;
    a.ks = philox_schedule(make_key(rng.seed));
    a.off_lo = static_cast<uint32_t>(rng.offset);
    a.off_hi = static_cast<uint32_t>(rng.offset >> 32);
    auto kern = mask ? dropout_bwd_kernel<T, false> : dropout_bwd_kernel<T, true>;
    static const int occ_mask = occupancy(dropout_bwd_kernel<T, false>, kThreads, 0);
    static const int occ_regen = occupancy(dropout_bwd_kernel<T, true>, kThreads, 0);
    const int occ = mask ? occ_mask : occ_regen;
    const int64_t grid = std::min<int64_t>(a.ntiles, int64_t{sm_count()} * occ);
    // Every tile index the kernel forms (up to ntiles + 2 * grid) is divided
    // with the 31-bit FastDiv: 2^31 tiles would be 2^44 elements.
    if (a.ntiles + 2 * grid >= (int64_t{1} << 31)) return cudaErrorInvalidValue;
    a.late_trigger = a.ntiles > grid ? 1 : 0;
    return launch_pdl(kern, dim3(static_cast<unsigned>(grid)), dim3(kThreads), 0, s,
                      static_cast<T*>(dx), partial, static_cast<const T*>(dout), mask, a);
}

}  // namespace

cudaError_t dropout_take_device_error(unsigned int* flags) {
    return take_device_error_word(flags);
}

ColReducePlan dropout_bwd_plan(int64_t rows, int64_t cols) {
    return ColReducePlan{(rows + kBwdRowsPerTile - 1) / kBwdRowsPerTile, cols};
}

template <typename T, int COLS>
cudaError_t colreduce_impl(void* out0, void* out1, int64_t split, const float* partial,
                           int64_t parts, int64_t width, cudaStream_t s) {
    const dim3 grid(static_cast<unsigned>((width + COLS - 1) / COLS));
    return launch_pdl(colreduce_kernel<T, COLS>, grid, dim3(COLS * kRedGroups), 0, s,
                      static_cast<T*>(out0), static_cast<T*>(out1), split, partial, parts, width);
}

cudaError_t launch_colreduce(DType dt, void* out0, void* out1, int64_t split,
                             const float* partial, int64_t parts, int64_t width, cudaStream_t s) {
    const bool narrow = parts <= kRedNarrowMaxParts;
    if (dt == DType::F16)
        return narrow ? colreduce_impl<__half, 8>(out0, out1, split, partial, parts, width, s)
                      : colreduce_impl<__half, 32>(out0, out1, split, partial, parts, width, s);
    return narrow ? colreduce_impl<float, 8>(out0, out1, split, partial, parts, width, s)
                  : colreduce_impl<float, 32>(out0, out1, split, partial, parts, width, s);
}

cudaError_t launch_dropout_fwd(DType dt, bool relu, void* out, uint8_t* mask, const void* x,
                               const void* bias, const void* residual, int64_t rows, int64_t cols,
                               const DropoutRng& rng, cudaStream_t s) {
    if (dt == DType::F16)
        return relu ? brd_fwd_impl<__half>(out, mask, x, bias, rows, cols, rng, s)
                    : bdr_fwd_impl<__half>(out, mask, x, bias, residual, rows, cols, rng, s);
    return relu ? brd_fwd_impl<float>(out, mask, x, bias, rows, cols, rng, s)
                : bdr_fwd_impl<float>(out, mask, x, bias, residual, rows, cols, rng, s);
}

cudaError_t launch_dropout_bwd(DType dt, void* dx, float* partial, const void* dout,
                               const uint8_t* mask, int64_t rows, int64_t cols,
                               const DropoutRng& rng, cudaStream_t s) {
    if (dt == DType::F16) return bwd_impl<__half>(dx, partial, dout, mask, rows, cols, rng, s);
    return bwd_impl<float>(dx, partial, dout, mask, rows, cols, rng, s);
}

}  // namespace ls
