// softmax.cu -- masked attention softmax, forward and backward, specialised by
// row length ("CMU 11-868 L10 (LightSeq)", slides p.23-26: the two dependent
// reductions of the softmax -- row maximum, then sum of exponentials -- are
// kept, and instead the number of lanes per row and elements per lane are
// fixed at compile time for each row length and the right instance is picked
// at call time; "CS336 Lecture 5: GPU", section 6.2: subtract the row maximum
// before exponentiating).
//
// Row-length classes (k_len = 8 * nvec):
//   nvec <= 32        LPR = next power of two >= nvec lanes per row, one
//                     16-byte vector per lane; 256/LPR rows per 256-thread CTA
//                     (k_len 16 -> 2 lanes/row, 128 rows per CTA).
//   32 < nvec <= 128  a warp per row, VPT = 2..4 vectors per lane.
//   nvec > 128        a CTA per row (4 or 8 warps), partial results of the two
//                     reductions through shared memory.
//   nvec > 2048       a CTA per row that reads the row twice: an online
//   (fwd: > 512)      (maximum, sum) pass, then the output pass.
// Masked keys are never loaded: a lane loads a vector only if it holds at
// least one valid key; masked outputs are written as exact zeros.
#include <math.h>

#include <algorithm>

#include "ls_device.cuh"
#include "ls_internal.h"

namespace ls {
namespace {

constexpr int kThreads = 256;
constexpr float kLog2e = 1.4426950408889634f;

struct RowMask {
    const int32_t* key_len;  // [batch] or nullptr
    FastDiv heads_q;         // row / (heads * q_len) = batch index
    FastDiv q_len;           // row % q_len = query index
    int shift;               // k_len - q_len (causal diagonal offset)
    int causal;
};

// Number of leading valid keys of a row (0..k_len).
// Rows number fewer than 2^31 (checked on the host), so the batch and query
// indices come from multiply-shift division.
__device__ __forceinline__ int valid_len(int64_t row, int k_len, const RowMask& m) {
    int v = k_len;
    const uint32_t r32 = static_cast<uint32_t>(row);
    if (m.key_len) {
        const int kl = m.key_len[fdiv(r32, m.heads_q)];
        v = min(v, max(kl, 0));
    }
    if (m.causal) {
        const int q = static_cast<int>(fmod_(r32, m.q_len));
        v = min(v, max(q + m.shift + 1, 0));
    }
    return v;
}

// ----------------------------------------------------------------------------
// Group-per-row kernels, persistent.  Row round k gives group slot q of CTA b
// the row k*stride + q*gridDim + b, so the partial last round is spread over
// every CTA.  For rows of up to 2 vectors per lane, two register buffers per
// group: the next row's loads are in flight while the current row is reduced
// and stored (wider rows keep one buffer and rely on occupancy).  Loop
// conditions are warp-uniform because the groups of a warp reduce with
// full-warp shuffles.
// ----------------------------------------------------------------------------
template <typename T, int LPR, int VPT>
struct RowBuf {
    Raw8<T> a[VPT];  // x (forward) or y (backward)
    Raw8<T> b[VPT];  // dy (backward only)
    uint32_t mb[VPT];  // dropout bits of each vector (fused dropout backward only)
    int vlen;
};

// Dropout on the probabilities, fused into the softmax ("CMU 11-868 L10
// (LightSeq)", technique 1: the elementwise step after a reduce kernel joins
// it).  Forward: y_drop = bit * y * scale, with bit = keep on valid entries
// and 0 on masked ones, one mask byte per 8-element vector (bit j = element
// 8v + j); backward: the mask is read.  Unused by the plain softmax.
struct DropArgs {
    void* y_drop;
    uint8_t* mask;
    uint32_t thr;
    float scale;
    PhiloxSchedule ks;
    uint32_t off_lo, off_hi;
    uint64_t tail_at;  // forward: the bytes [tail_at, tail_at + tail) of the last
    int tail;          // mask word lie past the last element and are written as 0
};

// The forward's one-thread duty: zero the mask bytes past the last element.
__device__ __forceinline__ void drop_tail(const DropArgs& d) {
    if (blockIdx.x == 0 && threadIdx.x == 0)
        for (int k = 0; k < d.tail; ++k) d.mask[d.tail_at + k] = 0;
}

// Valid length of a row, 0 past the last row.  With per-batch key lengths it
// costs a dependent load, so the kernels fetch it one row ahead of the row's
// data loads.
__device__ __forceinline__ int row_vlen(int64_t row, int64_t nrows, int k_len, const RowMask& mk) {
    return row < nrows ? valid_len(row, k_len, mk) : 0;
}

template <typename T, int LPR, int VPT, bool BWD, bool DROP>
__device__ __forceinline__ void sm_load(RowBuf<T, LPR, VPT>& buf, const T* p, const T* q,
                                        int64_t row, int vlen, int k_len, int gl,
                                        const DropArgs& d) {
    buf.vlen = vlen;
    const int64_t base = row * k_len;
#pragma unroll
    for (int k = 0; k < VPT; ++k) {
        const int v = gl + k * LPR;
        if (v * kVec < buf.vlen) {
            buf.a[k] = load8<T>(p + base + v * kVec);
            if (BWD) buf.b[k] = load8<T>(q + base + v * kVec);
            if (BWD && DROP) buf.mb[k] = d.mask[(base >> 3) + v];
        }
    }
}

// Fused dropout epilogue of one output vector v of a row (forward): the keep
// bits of its valid elements, the dropped probabilities and the mask byte.
template <typename T>
__device__ __forceinline__ void drop_store(const float (&o)[kVec], int64_t base, int v, int vlen,
                                           const DropArgs& d) {
    const int cnt = min(max(vlen - v * kVec, 0), kVec);
    uint32_t bits = 0;
    if (cnt > 0)
        bits = keep_bits8(static_cast<uint64_t>(base + v * kVec), d.thr, d.ks, d.off_lo,
                          d.off_hi) &
               ((1u << cnt) - 1u);
    float od[kVec];
#pragma unroll
    for (int j = 0; j < kVec; ++j) od[j] = ((bits >> j) & 1u) ? o[j] * d.scale : 0.f;
    store8f<T>(static_cast<T*>(d.y_drop) + base + v * kVec, od);
    d.mask[(base >> 3) + v] = static_cast<uint8_t>(bits);
}

// The forward row is branch-free across the valid/masked boundary: element j
// of vector v is valid iff j < cnt(v) = clamp(vlen - 8v, 0, 8); invalid
// elements are replaced by selects (vectors that were not loaded hold
// arbitrary bits, which a select discards).  Divergent branches at the
// boundary would run the full, partial and empty paths one after another.
template <typename T, int LPR, int VPT, bool DROP>
__device__ __forceinline__ void sm_fwd_row(const RowBuf<T, LPR, VPT>& buf, T* y, int64_t row,
                                           int64_t nrows, int k_len, int gl, const DropArgs& d) {
    const int nvec = k_len / kVec;
    const int vlen = buf.vlen;
    float f[VPT][kVec];
    float m = -INFINITY;
#pragma unroll
    for (int k = 0; k < VPT; ++k) {
        const int v = gl + k * LPR;
        const int cnt = min(max(vlen - v * kVec, 0), kVec);
        unpack(buf.a[k], f[k]);
        if (LPR == 32 && (k + 1) * LPR * kVec <= vlen) {
            // the warp's k-th slot lies wholly in the valid prefix (the same
            // test in every lane): packed maximum, no per-element selects
            m = fmaxf(m, vmax8(buf.a[k]));
            continue;
        }
#pragma unroll
        for (int j = 0; j < kVec; ++j) {
            f[k][j] = j < cnt ? f[k][j] : -INFINITY;
            m = fmaxf(m, f[k][j]);
        }
    }
    m = group_max<LPR>(m);
    const float ml = m == -INFINITY ? 0.f : m * kLog2e;  // empty row: every e is 0
    float2 acc = make_float2(0.f, 0.f);
#pragma unroll
    for (int k = 0; k < VPT; ++k)
#pragma unroll
        for (int j = 0; j < kVec; j += 2) {  // two at a time; -inf -> 0
            float2 t = fma2(make_float2(f[k][j], f[k][j + 1]), make_float2(kLog2e, kLog2e),
                            make_float2(-ml, -ml));
            t.x = exp2_approx(t.x);
            t.y = exp2_approx(t.y);
            f[k][j] = t.x;
            f[k][j + 1] = t.y;
            acc = add2(acc, t);
        }
    float s = group_sum<LPR>(acc.x + acc.y);
    if (row >= nrows) return;
    const float inv = s > 0.f ? __fdividef(1.f, s) : 0.f;
    const int64_t base = row * k_len;
#pragma unroll
    for (int k = 0; k < VPT; ++k) {
        const int v = gl + k * LPR;
        if (v < nvec) {
            float o[kVec];
#pragma unroll
            for (int j = 0; j < kVec; j += 2) {  // masked: 0 * inv = +0
                const float2 t = mul2(make_float2(f[k][j], f[k][j + 1]), make_float2(inv, inv));
                o[j] = t.x;
                o[j + 1] = t.y;
            }
            store8f<T>(y + base + v * kVec, o);
            if (DROP) drop_store<T>(o, base, v, vlen, d);
        }
    }
}

// The backward branches (branch-free needs more registers and measured
// slower).  A vector wholly inside the valid prefix takes the unpredicated
// path, with the FP16 conversions folded into mixed-precision instructions.
// With a warp per row the branch is taken per slot of 32 vectors (the warp's
// k-th vectors) rather than per lane, so it is warp-uniform: a slot that
// straddles the end of the valid prefix runs only the predicated path instead
// of the full, predicated and empty paths one after another.
template <typename T, int LPR, int VPT, bool DROP>
__device__ __forceinline__ void sm_bwd_row(const RowBuf<T, LPR, VPT>& buf, T* dx, int64_t row,
                                           int64_t nrows, int k_len, int gl, const DropArgs& d) {
    const int nvec = k_len / kVec;
    const int vlen = buf.vlen;
    if (DROP) {
        // g = bit * dy_drop * scale, then the softmax backward of g.
        float dot = 0.f;
#pragma unroll
        for (int k = 0; k < VPT; ++k) {
            const int v = gl + k * LPR;
            if (v * kVec < vlen) {
                float yf[kVec], df[kVec];
                unpack(buf.a[k], yf);
                unpack(buf.b[k], df);
#pragma unroll
                for (int j = 0; j < kVec; ++j) {
                    const bool on = v * kVec + j < vlen && ((buf.mb[k] >> j) & 1u);
                    dot = fmaf(yf[j], on ? df[j] * d.scale : 0.f, dot);
                }
            }
        }
        dot = group_sum<LPR>(dot);
        if (row >= nrows) return;
        const int64_t base = row * k_len;
#pragma unroll
        for (int k = 0; k < VPT; ++k) {
            const int v = gl + k * LPR;
            if (v < nvec) {
                float o[kVec];
                if (v * kVec < vlen) {
                    float yf[kVec], df[kVec];
                    unpack(buf.a[k], yf);
                    unpack(buf.b[k], df);
#pragma unroll
                    for (int j = 0; j < kVec; ++j) {
                        const bool valid = v * kVec + j < vlen;
                        const float g = valid && ((buf.mb[k] >> j) & 1u) ? df[j] * d.scale : 0.f;
                        o[j] = valid ? yf[j] * (g - dot) : 0.f;
                    }
                } else {
#pragma unroll
                    for (int j = 0; j < kVec; ++j) o[j] = 0.f;
                }
                store8f<T>(dx + base + v * kVec, o);
            }
        }
        return;
    }
    // full(k): vector gl + k*LPR lies wholly in the valid prefix; any(k): it
    // holds a valid element.  Warp-uniform (whole slot) for a warp per row.
    constexpr bool kSlot = LPR == 32;
    auto full = [&](int k) {
        return ((kSlot ? k * LPR + LPR : gl + k * LPR + 1) * kVec) <= vlen;
    };
    auto any = [&](int k) { return ((kSlot ? k * LPR : gl + k * LPR) * kVec) < vlen; };
    float dot = 0.f;
#pragma unroll
    for (int k = 0; k < VPT; ++k) {
        const int v = gl + k * LPR;
        if (full(k)) {
            dot = dot8_acc(buf.a[k], buf.b[k], dot);
        } else if (any(k)) {
            float yf[kVec], df[kVec];
            unpack(buf.a[k], yf);
            unpack(buf.b[k], df);
#pragma unroll
            for (int j = 0; j < kVec; ++j)
                dot = v * kVec + j < vlen ? fmaf(yf[j], df[j], dot) : dot;  // unloaded: discarded
        }
    }
    dot = group_sum<LPR>(dot);
    if (row >= nrows) return;
    const int64_t base = row * k_len;
#pragma unroll
    for (int k = 0; k < VPT; ++k) {
        const int v = gl + k * LPR;
        if (v < nvec) {
            float o[kVec];
            if (full(k)) {
                float yf[kVec];
                unpack(buf.a[k], yf);
                sub8(buf.b[k], dot, o);
#pragma unroll
                for (int j = 0; j < kVec; j += 2) {
                    const float2 t = mul2(make_float2(o[j], o[j + 1]),
                                          make_float2(yf[j], yf[j + 1]));
                    o[j] = t.x;
                    o[j + 1] = t.y;
                }
            } else if (any(k)) {
                float yf[kVec], df[kVec];
                unpack(buf.a[k], yf);
                unpack(buf.b[k], df);
#pragma unroll
                for (int j = 0; j < kVec; ++j)
                    o[j] = (v * kVec + j < vlen) ? yf[j] * (df[j] - dot) : 0.f;
            } else {
#pragma unroll
                for (int j = 0; j < kVec; ++j) o[j] = 0.f;
            }
            store8f<T>(dx + base + v * kVec, o);
        }
    }
}

// BWD = false: out = y, p = x.   BWD = true: out = dx, p = y, q = dy.
// DROP: dropout on the probabilities fused in (forward writes d.y_drop and
// d.mask; backward reads d.mask and q = dy_drop).
template <typename T, int LPR, int VPT, bool BWD, bool DROP>
__global__ void __launch_bounds__(kThreads, min_ctas<T>((VPT == 1 || (BWD && VPT == 2))
                                                           ? 4
                                                           : (DROP && !BWD && VPT > 2 &&
                                                                      sizeof(T) == 2
                                                                  ? 2
                                                                  : 3)))
softmax_group_kernel(T* out, const T* p, const T* q, int64_t nrows, int k_len, RowMask mk,
                     const __grid_constant__ DropArgs d) {
    constexpr int RPC = kThreads / LPR;
    const int gl = threadIdx.x % LPR;
    const int slot = threadIdx.x / LPR;
    const int64_t stride = static_cast<int64_t>(gridDim.x) * RPC;
    int64_t r = static_cast<int64_t>(slot) * gridDim.x + blockIdx.x;
    // Before the wait, when every row (or pair of rows) has its own key
    // length: the L2 lines of the key lengths of this group's first two rows
    // (a row's data loads need its valid length first, so without this the
    // first row pays two DRAM round trips; measured on GB300 on 2^22 elements
    // with a key length per row: 2-5% at 32..1024 keys).  With one key length
    // per batch entry every warp would prefetch the same line -- L2 requests
    // queue at one slice, where plain loads mostly hit in L1 (BERT-base:
    // softmax forward 17.1 -> 21.5 us) -- so none is prefetched then.  The
    // rows themselves are not prefetched: their valid length is not known.
    if (mk.key_len && mk.heads_q.d <= 2 && gl == 0) {
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int64_t rr = r + h * stride;
            if (rr < nrows) prefetch_l2(mk.key_len + fdiv(static_cast<uint32_t>(rr), mk.heads_q));
        }
    }
    pdl_enter();
    if (DROP && !BWD) drop_tail(d);
    RowBuf<T, LPR, VPT> ba, bb;
    // Wide rows keep one buffer (a second would cost occupancy) -- except in
    // the FP16 softmax + dropout forward, whose per-row Philox draws and
    // three stores otherwise stand between one row's loads and the next's:
    // with two buffers at two CTAs per SM, 92.1 -> 85.5 us at 4 x 20 x 1024^2
    // causal, 52.6 -> 49.3 at 768 keys (measured on GB300).
    if (VPT > 2 && !(DROP && !BWD && sizeof(T) == 2)) {
        int vl = row_vlen(r, nrows, k_len, mk);
        for (; __any_sync(0xffffffffu, r < nrows); r += stride) {
            const int vln = row_vlen(r + stride, nrows, k_len, mk);
            sm_load<T, LPR, VPT, BWD, DROP>(ba, p, q, r, vl, k_len, gl, d);
            if (BWD)
                sm_bwd_row<T, LPR, VPT, DROP>(ba, out, r, nrows, k_len, gl, d);
            else
                sm_fwd_row<T, LPR, VPT, DROP>(ba, out, r, nrows, k_len, gl, d);
            vl = vln;
        }
        return;
    }
    sm_load<T, LPR, VPT, BWD, DROP>(ba, p, q, r, row_vlen(r, nrows, k_len, mk), k_len, gl, d);
    int vl_next = row_vlen(r + stride, nrows, k_len, mk);  // the row bb takes next
    while (__any_sync(0xffffffffu, r < nrows)) {
        const int64_t r1 = r + stride;
        sm_load<T, LPR, VPT, BWD, DROP>(bb, p, q, r1, vl_next, k_len, gl, d);
        vl_next = row_vlen(r1 + stride, nrows, k_len, mk);
        if (BWD)
            sm_bwd_row<T, LPR, VPT, DROP>(ba, out, r, nrows, k_len, gl, d);
        else
            sm_fwd_row<T, LPR, VPT, DROP>(ba, out, r, nrows, k_len, gl, d);
        if (!__any_sync(0xffffffffu, r1 < nrows)) break;
        r = r1 + stride;
        sm_load<T, LPR, VPT, BWD, DROP>(ba, p, q, r, vl_next, k_len, gl, d);
        vl_next = row_vlen(r + stride, nrows, k_len, mk);
        if (BWD)
            sm_bwd_row<T, LPR, VPT, DROP>(bb, out, r1, nrows, k_len, gl, d);
        else
            sm_fwd_row<T, LPR, VPT, DROP>(bb, out, r1, nrows, k_len, gl, d);
    }
}

// ----------------------------------------------------------------------------
// Warp-per-row kernels fed by bulk copies (k_len 256..1024).  Each warp owns an
// S-stage ring of row buffers in shared memory; lane 0 copies the valid prefix
// of the warp's next rows (x, or y and dy) with cp.async.bulk while the warp
// computes the current row from shared memory, so S rows per warp are in
// flight independently of registers.  Measured on GB300: two stages of four
// warps per CTA serve the forward best (more stages cost warps per SM, and the
// per-row work then limits); the backward, which reads twice the bytes per
// row, is faster from registers (softmax_group_kernel), so only the forward
// dispatches here.  Rows are interleaved over warps of all
// CTAs (row = warp_slot + k * all_warps).  A wait that runs out of time flags
// the failure, lets the warp's copies land and ends the warp.
// ----------------------------------------------------------------------------
constexpr int kTmaWarps = 4;
constexpr int kTmaStages = 2;
constexpr int kTmaMaxLen = 1024;  // longest row of the warp-per-row path

__host__ __device__ constexpr uint32_t tma_bar_bytes() {
    return ((kTmaWarps * kTmaStages * 8 + 127) / 128) * 128;
}

template <typename T, int VPT, bool BWD>
__global__ void __launch_bounds__(kTmaWarps * 32)
softmax_tma_kernel(T* out, const T* p, const T* q, int64_t nrows, int k_len, RowMask mk) {
    extern __shared__ __align__(128) unsigned char smem[];
    constexpr int S = kTmaStages;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t row_bytes = static_cast<uint32_t>(k_len) * sizeof(T);
    const uint32_t stage_bytes = BWD ? 2 * row_bytes : row_bytes;
    WarpRing<S> ring;
    ring.init(reinterpret_cast<uint64_t*>(smem) + warp * S,
              smem + tma_bar_bytes() + static_cast<size_t>(warp) * S * stage_bytes, stage_bytes);
    const int nvec = k_len / kVec;
    const int64_t W = static_cast<int64_t>(gridDim.x) * kTmaWarps;
    const int64_t first = static_cast<int64_t>(blockIdx.x) + static_cast<int64_t>(warp) * gridDim.x;
    // Before the wait: the L2 lines of the key lengths of the warp's first S
    // rows, when each row (or pair) has its own (as in softmax_group_kernel).
    if (mk.key_len && mk.heads_q.d <= 2 && lane < S) {
        const int64_t rr = first + lane * W;
        if (rr < nrows) prefetch_l2(mk.key_len + fdiv(static_cast<uint32_t>(rr), mk.heads_q));
    }
    pdl_enter();
    uint32_t parity[S];
    int vlen_of[S];
#pragma unroll
    for (int s = 0; s < S; ++s) {
        parity[s] = 0;
        vlen_of[s] = 0;
        const int64_t r = first + s * W;
        if (r < nrows) {
            const int vl = valid_len(r, k_len, mk);
            vlen_of[s] = vl;
            const uint32_t n = static_cast<uint32_t>((vl + kVec - 1) / kVec) * kVec * sizeof(T);
            ring.issue(s, p + r * k_len, n, BWD ? q + r * k_len : nullptr, BWD ? n : 0, row_bytes);
        }
    }
    // Unrolled by the stage count so that the stage index is a constant.
    for (int64_t k0 = 0;; k0 += S) {
#pragma unroll
    for (int s = 0; s < S; ++s) {
        const int64_t r = first + (k0 + s) * W;
        if (r >= nrows) return;
        const bool ok = ring.wait(s, parity[s]);
        if (!__all_sync(0xffffffffu, ok)) {  // the warp leaves together
            ring.drain(parity);
            return;
        }
        parity[s] ^= 1u;
        const int vlen = vlen_of[s];
        const T* xs = reinterpret_cast<const T*>(ring.stage(s));
        const int64_t base = r * k_len;
        // No divergent branch over the valid/masked boundary: element j of
        // vector v is valid iff j < cnt(v) = clamp(vlen - 8v, 0, 8).  A slot
        // of 32 vectors (one per lane) is wholly valid, straddles vlen, or lies
        // past it -- the same case in every lane.  Wholly valid slots take the
        // packed maximum; in the straddling slot invalid elements become -inf
        // before the maximum, so their exponentials are exactly 0 with no
        // further test; slots past vlen are stored as zeros.
        float f[VPT][kVec];
        float m = -INFINITY;
#pragma unroll
        for (int k2 = 0; k2 < VPT; ++k2) {
            const int v = lane + k2 * 32;
            if (vlen >= (k2 + 1) * 32 * kVec) {
                // every vector of the slot is valid (same test in every lane)
                const Raw8<T> raw = load8_smem<T>(xs + v * kVec);
                m = fmaxf(m, vmax8(raw));
                unpack(raw, f[k2]);
            } else if (vlen > k2 * 32 * kVec) {
                const int cnt = min(max(vlen - v * kVec, 0), kVec);
                unpack(load8_smem<T>(xs + v * kVec), f[k2]);
#pragma unroll
                for (int j = 0; j < kVec; ++j) {
                    f[k2][j] = j < cnt ? f[k2][j] : -INFINITY;
                    m = fmaxf(m, f[k2][j]);
                }
            }
        }
        m = group_max<32>(m);
        const float ml = m == -INFINITY ? 0.f : m * kLog2e;  // empty row: all e = 0
        // Exponentials and their sum two lanes at a time (packed FP32): the
        // even and odd elements keep separate partial sums, added at the end.
        float2 acc = make_float2(0.f, 0.f);
#pragma unroll
        for (int k2 = 0; k2 < VPT; ++k2) {
            if (vlen > k2 * 32 * kVec) {
#pragma unroll
                for (int j = 0; j < kVec; j += 2) {
                    float2 t = fma2(make_float2(f[k2][j], f[k2][j + 1]),
                                    make_float2(kLog2e, kLog2e), make_float2(-ml, -ml));
                    t.x = exp2_approx(t.x);
                    t.y = exp2_approx(t.y);
                    f[k2][j] = t.x;
                    f[k2][j + 1] = t.y;
                    acc = add2(acc, t);
                }
            }
        }
        float sum = group_sum<32>(acc.x + acc.y);
        const float inv = sum > 0.f ? __fdividef(1.f, sum) : 0.f;
#pragma unroll
        for (int k2 = 0; k2 < VPT; ++k2) {
            const int v = lane + k2 * 32;
            if (v >= nvec) continue;
            T* dst = out + base + v * kVec;
            if (vlen > k2 * 32 * kVec) {
                float o[kVec];
#pragma unroll
                for (int j = 0; j < kVec; j += 2) {
                    const float2 t = mul2(make_float2(f[k2][j], f[k2][j + 1]),
                                          make_float2(inv, inv));
                    o[j] = t.x;
                    o[j + 1] = t.y;
                }
                store8f<T>(dst, o);
            } else {
                store8<T>(dst, zero8<T>());
            }
        }
        __syncwarp();  // every lane has used its reads of stage s
        const int64_t rn = r + S * W;
        if (rn < nrows) {
            const int vl = valid_len(rn, k_len, mk);
            vlen_of[s] = vl;
            const uint32_t n = static_cast<uint32_t>((vl + kVec - 1) / kVec) * kVec * sizeof(T);
            ring.issue(s, p + rn * k_len, n, BWD ? q + rn * k_len : nullptr, BWD ? n : 0,
                       row_bytes);
        }
    }
    }
}

// ----------------------------------------------------------------------------
// CTA-per-row kernels (k_len > 1024).
// ----------------------------------------------------------------------------
template <int WARPS>
__device__ __forceinline__ float cta_max(float v, float* red) {
    v = group_max<32>(v);
    __syncthreads();
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
    __syncthreads();
    float r = red[0];
#pragma unroll
    for (int w = 1; w < WARPS; ++w) r = fmaxf(r, red[w]);
    return r;
}
template <int WARPS>
__device__ __forceinline__ float cta_sum(float v, float* red) {
    v = group_sum<32>(v);
    __syncthreads();
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
    __syncthreads();
    float r = 0.f;
#pragma unroll
    for (int w = 0; w < WARPS; ++w) r += red[w];
    return r;
}

template <typename T, int WARPS, int VPT, bool DROP>
__global__ void __launch_bounds__(WARPS * 32)
softmax_fwd_cta_kernel(T* y, const T* x, int k_len, RowMask mk,
                       const __grid_constant__ DropArgs d) {
    constexpr int NT = WARPS * 32;
    __shared__ float red[WARPS];
    pdl_enter();
    if (DROP) drop_tail(d);
    const int64_t row = blockIdx.x;
    const int vlen = valid_len(row, k_len, mk);
    const int nvec = k_len / kVec;
    const int64_t base = row * k_len;
    float f[VPT][kVec];
    float m = -INFINITY;
#pragma unroll
    for (int k = 0; k < VPT; ++k) {
        const int v = threadIdx.x + k * NT;
        if (v * kVec < vlen) {
            load8f<T>(x + base + v * kVec, f[k]);
            if ((v + 1) * kVec <= vlen) {  // a whole vector: no per-element tests
#pragma unroll
                for (int j = 0; j < kVec; ++j) m = fmaxf(m, f[k][j]);
            } else {
#pragma unroll
                for (int j = 0; j < kVec; ++j)
                    if (v * kVec + j < vlen) m = fmaxf(m, f[k][j]);
            }
        }
    }
    m = cta_max<WARPS>(m, red);
    const float ml = m == -INFINITY ? 0.f : m * kLog2e;  // no valid or all -inf: e = 0
    float s = 0.f;
#pragma unroll
    for (int k = 0; k < VPT; ++k) {
        const int v = threadIdx.x + k * NT;
        if ((v + 1) * kVec <= vlen) {  // exponentials two at a time
            float2 acc = make_float2(0.f, 0.f);
#pragma unroll
            for (int j = 0; j < kVec; j += 2) {
                float2 t = fma2(make_float2(f[k][j], f[k][j + 1]), make_float2(kLog2e, kLog2e),
                                make_float2(-ml, -ml));
                t.x = exp2_approx(t.x);
                t.y = exp2_approx(t.y);
                f[k][j] = t.x;
                f[k][j + 1] = t.y;
                acc = add2(acc, t);
            }
            s += acc.x + acc.y;
        } else {
#pragma unroll
            for (int j = 0; j < kVec; ++j) {
                const bool on = v * kVec + j < vlen;
                const float e = on ? exp2_approx(fmaf(f[k][j], kLog2e, -ml)) : 0.f;
                f[k][j] = e;
                s += e;
            }
        }
    }
    s = cta_sum<WARPS>(s, red);
    const float inv = s > 0.f ? 1.f / s : 0.f;
#pragma unroll
    for (int k = 0; k < VPT; ++k) {
        const int v = threadIdx.x + k * NT;
        if (v < nvec) {
            float o[kVec];
#pragma unroll
            for (int j = 0; j < kVec; j += 2) {
                const float2 t = mul2(make_float2(f[k][j], f[k][j + 1]), make_float2(inv, inv));
                o[j] = t.x;
                o[j + 1] = t.y;
            }
            store8f<T>(y + base + v * kVec, o);
            if (DROP) drop_store<T>(o, base, v, vlen, d);
        }
    }
}

template <typename T, int WARPS, int VPT, bool DROP>
__global__ void __launch_bounds__(WARPS * 32)
softmax_bwd_cta_kernel(T* dx, const T* y, const T* dy, int k_len, RowMask mk,
                       const __grid_constant__ DropArgs d) {
    constexpr int NT = WARPS * 32;
    __shared__ float red[WARPS];
    pdl_enter();
    const int64_t row = blockIdx.x;
    const int vlen = valid_len(row, k_len, mk);
    const int nvec = k_len / kVec;
    const int64_t base = row * k_len;
    Raw8<T> yr[VPT], dr[VPT];
    uint32_t mb[VPT];
#pragma unroll
    for (int k = 0; k < VPT; ++k) {
        const int v = threadIdx.x + k * NT;
        mb[k] = 0;
        if (v * kVec < vlen) {
            yr[k] = load8<T>(y + base + v * kVec);
            dr[k] = load8<T>(dy + base + v * kVec);
            if (DROP) mb[k] = d.mask[(base >> 3) + v];
        }
    }
    // With fused dropout the incoming gradient is g = bit * dy_drop * scale.
    auto grad = [&](int k, const float (&df)[kVec], int j) {
        return DROP ? (((mb[k] >> j) & 1u) ? df[j] * d.scale : 0.f) : df[j];
    };
    float dot = 0.f;
#pragma unroll
    for (int k = 0; k < VPT; ++k) {
        const int v = threadIdx.x + k * NT;
        if (!DROP && (v + 1) * kVec <= vlen) {  // a whole vector: no per-element tests
            dot = dot8_acc(yr[k], dr[k], dot);
        } else if (v * kVec < vlen) {
            float yf[kVec], df[kVec];
            unpack(yr[k], yf);
            unpack(dr[k], df);
#pragma unroll
            for (int j = 0; j < kVec; ++j)
                if (v * kVec + j < vlen) dot = fmaf(yf[j], grad(k, df, j), dot);
        }
    }
    dot = cta_sum<WARPS>(dot, red);
#pragma unroll
    for (int k = 0; k < VPT; ++k) {
        const int v = threadIdx.x + k * NT;
        if (v < nvec) {
            float o[kVec];
            if (!DROP && (v + 1) * kVec <= vlen) {  // (dy - dot) * y, two at a time
                float yf[kVec];
                unpack(yr[k], yf);
                sub8(dr[k], dot, o);
#pragma unroll
                for (int j = 0; j < kVec; j += 2) {
                    const float2 t = mul2(make_float2(o[j], o[j + 1]),
                                          make_float2(yf[j], yf[j + 1]));
                    o[j] = t.x;
                    o[j + 1] = t.y;
                }
            } else if (v * kVec < vlen) {
                float yf[kVec], df[kVec];
                unpack(yr[k], yf);
                unpack(dr[k], df);
#pragma unroll
                for (int j = 0; j < kVec; ++j)
                    o[j] = (v * kVec + j < vlen) ? yf[j] * (grad(k, df, j) - dot) : 0.f;
            } else {
#pragma unroll
                for (int j = 0; j < kVec; ++j) o[j] = 0.f;
            }
            store8f<T>(dx + base + v * kVec, o);
        }
    }
}

// ----------------------------------------------------------------------------
// Long rows (forward: k_len > 4096, backward: k_len > 16384): a CTA per row
// streams the valid prefix twice.  Forward: the first pass keeps each thread's running
// maximum and its rescaled running sum of exponentials -- the online softmax
// normaliser of "CS336 Lecture 5: GPU", section 6.2 -- and the CTA merges the
// pairs by the same rule; the second pass writes y (and the dropout
// epilogue).  Backward: the first pass sums y*g, the second writes dx.  The
// row's second read comes from L2 (a row is at most 2 MB).
// ----------------------------------------------------------------------------
// CTA sizes: the forward takes 256 threads for rows of up to 32768 keys (four
// rows in flight per SM hide its two phases better: 0.76 against 0.52 of the
// copy bandwidth at 16384 keys) and 512 for longer rows; the backward 512.
constexpr int kStreamThreads = 512;
constexpr int kStreamThreadsShort = 256;
constexpr int64_t kStreamShortMaxLen = 32768;
// Vectors per thread in flight: 64 bytes of either storage type.
template <typename T>
constexpr int stream_unroll() { return sizeof(T) == 2 ? 4 : 2; }

__device__ __forceinline__ void online_merge(float& m, float& l, float m2, float l2) {
    const float mm = fmaxf(m, m2);
    if (mm == -INFINITY) return;  // both empty
    l = l * exp2_approx((m - mm) * kLog2e) + l2 * exp2_approx((m2 - mm) * kLog2e);
    m = mm;
}

// Loads the vectors v0 + u * THREADS (u < U) of a row that hold at least one
// of its vlen valid elements.
template <typename T, int U, int THREADS>
__device__ __forceinline__ void stream_load(Raw8<T> (&r)[U], const T* row_ptr, int v0,
                                            int vlen) {
#pragma unroll
    for (int u = 0; u < U; ++u) {
        const int v = v0 + u * THREADS;
        if (v * kVec < vlen) r[u] = load8<T>(row_ptr + v * kVec);
    }
}

template <typename T, bool DROP, int THREADS>
__global__ void __launch_bounds__(THREADS, 2)
softmax_fwd_stream_kernel(T* y, const T* x, int k_len, RowMask mk,
                          const __grid_constant__ DropArgs d) {
    constexpr int U = stream_unroll<T>();
    constexpr int kWarps = THREADS / 32;
    __shared__ float sm_m[kWarps], sm_l[kWarps];
    pdl_enter();
    if (DROP) drop_tail(d);
    const int64_t row = blockIdx.x;
    const int vlen = valid_len(row, k_len, mk);
    const int nvec = k_len / kVec;
    const int64_t base = row * k_len;
    float m = -INFINITY, l = 0.f;
    for (int v0 = threadIdx.x; v0 * kVec < vlen; v0 += THREADS * U) {
        Raw8<T> r[U];
        stream_load<T, U, THREADS>(r, x + base, v0, vlen);
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int v = v0 + u * THREADS;
            const int cnt = min(vlen - v * kVec, kVec);
            if (cnt <= 0) break;
            float f[kVec];
            unpack(r[u], f);
            if (cnt == kVec) {
                // a whole vector (every one but the row's last): packed maximum,
                // exponentials two at a time
                const float vm = vmax8(r[u]);
                if (vm > m) {  // rescale the running sum to the new maximum
                    l *= exp2_approx((m - vm) * kLog2e);
                    m = vm;
                }
                const float ml = m == -INFINITY ? 0.f : m * kLog2e;  // all -inf so far: e = 0
                float2 acc = make_float2(0.f, 0.f);
#pragma unroll
                for (int j = 0; j < kVec; j += 2) {
                    float2 t = fma2(make_float2(f[j], f[j + 1]), make_float2(kLog2e, kLog2e),
                                    make_float2(-ml, -ml));
                    t.x = exp2_approx(t.x);
                    t.y = exp2_approx(t.y);
                    acc = add2(acc, t);
                }
                l += acc.x + acc.y;
                continue;
            }
            float vm = -INFINITY;
#pragma unroll
            for (int j = 0; j < kVec; ++j) vm = fmaxf(vm, j < cnt ? f[j] : -INFINITY);
            if (vm > m) {  // rescale the running sum to the new maximum
                l *= exp2_approx((m - vm) * kLog2e);
                m = vm;
            }
            const float ml = m == -INFINITY ? 0.f : m * kLog2e;  // all -inf so far: e = 0
#pragma unroll
            for (int j = 0; j < kVec; ++j)
                l += j < cnt ? exp2_approx(fmaf(f[j], kLog2e, -ml)) : 0.f;
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
        online_merge(m, l, __shfl_xor_sync(0xffffffffu, m, o), __shfl_xor_sync(0xffffffffu, l, o));
    if ((threadIdx.x & 31) == 0) {
        sm_m[threadIdx.x >> 5] = m;
        sm_l[threadIdx.x >> 5] = l;
    }
    __syncthreads();
    float M = sm_m[0], L = sm_l[0];
    for (int w = 1; w < kWarps; ++w) online_merge(M, L, sm_m[w], sm_l[w]);
    const float ml = M == -INFINITY ? 0.f : M * kLog2e;
    const float inv = L > 0.f ? __fdividef(1.f, L) : 0.f;
    for (int v0 = threadIdx.x; v0 < nvec; v0 += THREADS * U) {
        Raw8<T> r[U];
        stream_load<T, U, THREADS>(r, x + base, v0, vlen);
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int v = v0 + u * THREADS;
            if (v >= nvec) break;
            const int cnt = min(max(vlen - v * kVec, 0), kVec);
            float o[kVec];
            if (cnt == kVec) {
                float f[kVec];
                unpack(r[u], f);
#pragma unroll
                for (int j = 0; j < kVec; j += 2) {
                    float2 t = fma2(make_float2(f[j], f[j + 1]), make_float2(kLog2e, kLog2e),
                                    make_float2(-ml, -ml));
                    t.x = exp2_approx(t.x);
                    t.y = exp2_approx(t.y);
                    t = mul2(t, make_float2(inv, inv));
                    o[j] = t.x;
                    o[j + 1] = t.y;
                }
            } else if (cnt > 0) {
                float f[kVec];
                unpack(r[u], f);
#pragma unroll
                for (int j = 0; j < kVec; ++j)
                    o[j] = j < cnt ? exp2_approx(fmaf(f[j], kLog2e, -ml)) * inv : 0.f;
            } else {
#pragma unroll
                for (int j = 0; j < kVec; ++j) o[j] = 0.f;
            }
            store8f<T>(y + base + v * kVec, o);
            if (DROP) drop_store<T>(o, base, v, vlen, d);
        }
    }
}

template <typename T, bool DROP>
__global__ void __launch_bounds__(kStreamThreads, 2)
softmax_bwd_stream_kernel(T* dx, const T* y, const T* dy, int k_len, RowMask mk,
                          const __grid_constant__ DropArgs d) {
    constexpr int U = stream_unroll<T>();
    constexpr int kWarps = kStreamThreads / 32;
    __shared__ float red[kWarps];
    pdl_enter();
    const int64_t row = blockIdx.x;
    const int vlen = valid_len(row, k_len, mk);
    const int nvec = k_len / kVec;
    const int64_t base = row * k_len;
    // g = dy, or bit * dy_drop * scale with the fused dropout
    auto grads = [&](const Raw8<T>& r, uint32_t bits, float (&g)[kVec]) {
        unpack(r, g);
        if (DROP) {
#pragma unroll
            for (int j = 0; j < kVec; ++j) g[j] = ((bits >> j) & 1u) ? g[j] * d.scale : 0.f;
        }
    };
    auto load_bits = [&](uint32_t (&mb)[U], int v0) {
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int v = v0 + u * kStreamThreads;
            mb[u] = (DROP && v * kVec < vlen) ? d.mask[(base >> 3) + v] : 0u;
        }
    };
    float dot = 0.f;
    for (int v0 = threadIdx.x; v0 * kVec < vlen; v0 += kStreamThreads * U) {
        Raw8<T> ry[U], rg[U];
        uint32_t mb[U];
        stream_load<T, U, kStreamThreads>(ry, y + base, v0, vlen);
        stream_load<T, U, kStreamThreads>(rg, dy + base, v0, vlen);
        load_bits(mb, v0);
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int v = v0 + u * kStreamThreads;
            const int cnt = min(vlen - v * kVec, kVec);
            if (cnt <= 0) break;
            if (!DROP && cnt == kVec) {  // a whole vector: no per-element tests
                dot = dot8_acc(ry[u], rg[u], dot);
                continue;
            }
            float yf[kVec], g[kVec];
            unpack(ry[u], yf);
            grads(rg[u], mb[u], g);
#pragma unroll
            for (int j = 0; j < kVec; ++j)
                if (j < cnt) dot = fmaf(yf[j], g[j], dot);
        }
    }
    dot = cta_sum<kWarps>(dot, red);
    for (int v0 = threadIdx.x; v0 < nvec; v0 += kStreamThreads * U) {
        Raw8<T> ry[U], rg[U];
        uint32_t mb[U];
        stream_load<T, U, kStreamThreads>(ry, y + base, v0, vlen);
        stream_load<T, U, kStreamThreads>(rg, dy + base, v0, vlen);
        load_bits(mb, v0);
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int v = v0 + u * kStreamThreads;
            if (v >= nvec) break;
            const int cnt = min(max(vlen - v * kVec, 0), kVec);
            float o[kVec];
            if (!DROP && cnt == kVec) {  // a whole vector: (dy - dot) * y, two at a time
                float yf[kVec];
                unpack(ry[u], yf);
                sub8(rg[u], dot, o);
#pragma unroll
                for (int j = 0; j < kVec; j += 2) {
                    const float2 t = mul2(make_float2(o[j], o[j + 1]),
                                          make_float2(yf[j], yf[j + 1]));
                    o[j] = t.x;
                    o[j + 1] = t.y;
                }
            } else if (cnt > 0) {
                float yf[kVec], g[kVec];
                unpack(ry[u], yf);
                grads(rg[u], mb[u], g);
#pragma unroll
                for (int j = 0; j < kVec; ++j) o[j] = j < cnt ? yf[j] * (g[j] - dot) : 0.f;
            } else {
#pragma unroll
                for (int j = 0; j < kVec; ++j) o[j] = 0.f;
            }
            store8f<T>(dx + base + v * kVec, o);
        }
    }
}

// ----------------------------------------------------------------------------
// Dispatch by row length.
// ----------------------------------------------------------------------------
struct SmPlan {
    bool cta, stream;
    int lpr, vpt, warps;
    int64_t grid;
};

// Longest rows held in registers: 8 warps x 8 vectors x 8 elements for the
// backward.  The forward streams from 4104 keys on: measured on 2^26 FP16
// elements, the CTA-per-row forward reaches 0.72 / 0.68 of the copy bandwidth
// at 2048 / 4096 keys (the two-pass kernel 0.29 / 0.46) but 0.65 / 0.52 at
// 8192 / 12288 keys (two-pass, 256 threads: 0.69 / 0.75); at 8 vectors per
// lane it needs 128 registers.
constexpr int64_t kMaxRegisterRowLen = 16384;
constexpr int64_t kMaxRegisterRowLenFwd = 4096;

SmPlan plan_for(int64_t nrows, int64_t k_len, bool fwd) {
    const int nvec = static_cast<int>(k_len / kVec);
    SmPlan p{};
    if (nvec <= 128) {
        p.cta = false;
        if (nvec <= 32) {
            p.lpr = 1;
            while (p.lpr < nvec) p.lpr <<= 1;
            p.vpt = 1;
        } else {
            p.lpr = 32;
            p.vpt = (nvec + 31) / 32;
        }
        const int64_t rpc = kThreads / p.lpr;
        p.grid = (nrows + rpc - 1) / rpc;
    } else if (k_len <= (fwd ? kMaxRegisterRowLenFwd : kMaxRegisterRowLen)) {
        p.cta = true;
        p.warps = nvec <= 512 ? 4 : 8;
        p.vpt = (nvec + p.warps * 32 - 1) / (p.warps * 32);
        p.grid = nrows;
    } else {
        p.stream = true;
        p.grid = nrows;
    }
    return p;
}

RowMask make_mask(const SoftmaxShape& sh) {
    RowMask m;
    m.key_len = sh.key_len;
    m.heads_q = make_fastdiv(static_cast<uint32_t>(std::max<int64_t>(1, sh.heads * sh.q_len)));
    m.q_len = make_fastdiv(static_cast<uint32_t>(std::max<int64_t>(1, sh.q_len)));
    m.shift = static_cast<int>(sh.k_len - sh.q_len);
    m.causal = sh.causal;
    return m;
}

template <typename K>
int occupancy(K kernel, int threads, size_t smem) {
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kernel, threads, smem) != cudaSuccess ||
        n < 1)
        n = 1;
    return n;
}

template <typename T, int LPR, int VPT, bool BWD, bool DROP>
cudaError_t group_launch(T* out, const T* p, const T* q, int64_t nrows, int k_len,
                         const RowMask& m, const DropArgs& d, const SmPlan& pl, cudaStream_t s) {
    auto kern = softmax_group_kernel<T, LPR, VPT, BWD, DROP>;
    static const int occ = occupancy(kern, kThreads, 0);
    const int64_t grid = std::min<int64_t>(pl.grid, int64_t{sm_count()} * occ);
    return launch_pdl(kern, dim3(static_cast<unsigned>(grid)), dim3(kThreads), 0, s, out, p, q,
                      nrows, k_len, m, d);
}
template <typename T, int VPT, bool BWD>
cudaError_t tma_launch(T* out, const T* p, const T* q, int64_t nrows, int k_len,
                       const RowMask& m, cudaStream_t s) {
    auto kern = softmax_tma_kernel<T, VPT, BWD>;
    const size_t stage = static_cast<size_t>(k_len) * sizeof(T) * (BWD ? 2 : 1);
    const size_t smem = tma_bar_bytes() + static_cast<size_t>(kTmaWarps) * kTmaStages * stage;
    if (smem > 48 * 1024) {
        static int done[kMaxDevices] = {};
        const cudaError_t e = allow_max_dynamic_smem(kern, done);
        if (e != cudaSuccess) return e;
    }
    // Resident CTAs for this row length, queried once per length (k_len <= 1024
    // on this path: 128 lengths) rather than on every launch.
    static int occ_by_len[kTmaMaxLen / kVec + 1] = {};
    const int li = k_len / kVec;
    int occ = li <= kTmaMaxLen / kVec ? __atomic_load_n(&occ_by_len[li], __ATOMIC_RELAXED) : 0;
    if (occ == 0) {
        occ = occupancy(kern, kTmaWarps * 32, smem);
        if (li <= kTmaMaxLen / kVec) __atomic_store_n(&occ_by_len[li], occ, __ATOMIC_RELAXED);
    }
    const int64_t need = (nrows + kTmaWarps - 1) / kTmaWarps;
    const int64_t grid = std::max<int64_t>(1, std::min<int64_t>(need, int64_t{sm_count()} * occ));
    return launch_pdl(kern, dim3(static_cast<unsigned>(grid)), dim3(kTmaWarps * 32), smem, s, out,
                      p, q, nrows, k_len, m);
}

// The plain forward of warp-per-row lengths takes the bulk-copy kernel; the
// fused-dropout forward stays on the register kernel.
template <typename T, bool DROP, int LPR, int VPT>
cudaError_t fwd_group(void* y, const void* x, int64_t nrows, int k_len, const RowMask& m,
                      const DropArgs& d, const SmPlan& p, cudaStream_t s) {
    if constexpr (LPR == 32 && !DROP)
        return tma_launch<T, VPT, false>(static_cast<T*>(y), static_cast<const T*>(x),
                                         static_cast<const T*>(nullptr), nrows, k_len, m, s);
    else
        return group_launch<T, LPR, VPT, false, DROP>(static_cast<T*>(y), static_cast<const T*>(x),
                                                      static_cast<const T*>(nullptr), nrows,
                                                      k_len, m, d, p, s);
}
template <typename T, bool DROP, int LPR, int VPT>
cudaError_t bwd_group(void* dx, const void* y, const void* dy, int64_t nrows, int k_len,
                      const RowMask& m, const DropArgs& d, const SmPlan& p, cudaStream_t s) {
    return group_launch<T, LPR, VPT, true, DROP>(static_cast<T*>(dx), static_cast<const T*>(y),
                                                 static_cast<const T*>(dy), nrows, k_len, m, d,
                                                 p, s);
}
template <typename T, bool DROP, int WARPS, int VPT>
cudaError_t fwd_cta(void* y, const void* x, int64_t nrows, int k_len, const RowMask& m,
                    const DropArgs& d, const SmPlan& p, cudaStream_t s) {
    return launch_pdl(softmax_fwd_cta_kernel<T, WARPS, VPT, DROP>,
                      dim3(static_cast<unsigned>(p.grid)), dim3(WARPS * 32), 0, s,
                      static_cast<T*>(y), static_cast<const T*>(x), k_len, m, d);
}
template <typename T, bool DROP, int WARPS, int VPT>
cudaError_t bwd_cta(void* dx, const void* y, const void* dy, int64_t nrows, int k_len,
                    const RowMask& m, const DropArgs& d, const SmPlan& p, cudaStream_t s) {
    return launch_pdl(softmax_bwd_cta_kernel<T, WARPS, VPT, DROP>,
                      dim3(static_cast<unsigned>(p.grid)), dim3(WARPS * 32), 0, s,
                      static_cast<T*>(dx), static_cast<const T*>(y), static_cast<const T*>(dy),
                      k_len, m, d);
}

#define LS_SM_T_DROP T, DROP
#define LS_SM_GROUP_CASES(FN, T, ...)                                    \
    switch (p.lpr) {                                                     \
        case 1: return FN<T, 1, 1>(__VA_ARGS__);                         \
        case 2: return FN<T, 2, 1>(__VA_ARGS__);                         \
        case 4: return FN<T, 4, 1>(__VA_ARGS__);                         \
        case 8: return FN<T, 8, 1>(__VA_ARGS__);                         \
        case 16: return FN<T, 16, 1>(__VA_ARGS__);                       \
        case 32:                                                         \
            switch (p.vpt) {                                             \
                case 1: return FN<T, 32, 1>(__VA_ARGS__);                \
                case 2: return FN<T, 32, 2>(__VA_ARGS__);                \
                case 3: return FN<T, 32, 3>(__VA_ARGS__);                \
                case 4: return FN<T, 32, 4>(__VA_ARGS__);                \
            }                                                            \
    }                                                                    \
    return cudaErrorInvalidConfiguration;

#define LS_SM_CTA_CASES(FN, T, ...)                                      \
    if (p.warps == 4) {                                                  \
        switch (p.vpt) {                                                 \
            case 2: return FN<T, 4, 2>(__VA_ARGS__);                     \
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

template <typename T, bool DROP>
cudaError_t fwd_dispatch(void* y, const void* x, const SoftmaxShape& sh, const DropArgs& d,
                         cudaStream_t s) {
    const int64_t nrows = sh.batch * sh.heads * sh.q_len;
    const int k_len = static_cast<int>(sh.k_len);
    const SmPlan p = plan_for(nrows, sh.k_len, true);
    const RowMask m = make_mask(sh);
    if (p.stream)
        return sh.k_len <= kStreamShortMaxLen
                   ? launch_pdl(softmax_fwd_stream_kernel<T, DROP, kStreamThreadsShort>,
                                dim3(static_cast<unsigned>(p.grid)), dim3(kStreamThreadsShort), 0,
                                s, static_cast<T*>(y), static_cast<const T*>(x), k_len, m, d)
                   : launch_pdl(softmax_fwd_stream_kernel<T, DROP, kStreamThreads>,
                                dim3(static_cast<unsigned>(p.grid)), dim3(kStreamThreads), 0, s,
                                static_cast<T*>(y), static_cast<const T*>(x), k_len, m, d);
    if (!p.cta) {
        LS_SM_GROUP_CASES(fwd_group, LS_SM_T_DROP, y, x, nrows, k_len, m, d, p, s)
    } else {
        LS_SM_CTA_CASES(fwd_cta, LS_SM_T_DROP, y, x, nrows, k_len, m, d, p, s)
    }
}

template <typename T, bool DROP>
cudaError_t bwd_dispatch(void* dx, const void* y, const void* dy, const SoftmaxShape& sh,
                         const DropArgs& d, cudaStream_t s) {
    const int64_t nrows = sh.batch * sh.heads * sh.q_len;
    const int k_len = static_cast<int>(sh.k_len);
    const SmPlan p = plan_for(nrows, sh.k_len, false);
    const RowMask m = make_mask(sh);
    if (p.stream)
        return launch_pdl(softmax_bwd_stream_kernel<T, DROP>, dim3(static_cast<unsigned>(p.grid)),
                          dim3(kStreamThreads), 0, s, static_cast<T*>(dx),
                          static_cast<const T*>(y), static_cast<const T*>(dy), k_len, m, d);
    if (!p.cta) {
        LS_SM_GROUP_CASES(bwd_group, LS_SM_T_DROP, dx, y, dy, nrows, k_len, m, d, p, s)
    } else {
        LS_SM_CTA_CASES(bwd_cta, LS_SM_T_DROP, dx, y, dy, nrows, k_len, m, d, p, s)
    }
}

DropArgs no_drop() {
    DropArgs d{};
    return d;
}

DropArgs make_drop(void* y_drop, uint8_t* mask, const DropoutRng& rng, uint64_t n) {
    DropArgs d{};
    d.tail_at = n / 8;  // n is a multiple of 8
    d.tail = static_cast<int>(((n + 31) / 32) * 4 - n / 8);
    d.y_drop = y_drop;
    d.mask = mask;
    d.thr = rng.thr;
    d.scale = rng.scale;
    d.ks = philox_schedule(PhiloxKey{static_cast<uint32_t>(rng.seed),
                                     static_cast<uint32_t>(rng.seed >> 32)});
    d.off_lo = static_cast<uint32_t>(rng.offset);
    d.off_hi = static_cast<uint32_t>(rng.offset >> 32);
    return d;
}

// Self-test of the bounded-wait failure path: one warp waits on a barrier
// that expects one arrival nobody makes.  After `polls` bounded polls it
// records the timeout in this unit's failure word and returns, as the
// bulk-copy rings do when a copy never lands.
__global__ void __launch_bounds__(32) wait_timeout_selftest_kernel(uint32_t polls) {
    __shared__ __align__(8) uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        mbar_init_fence();
    }
    __syncwarp();
    bool done = false;
    for (uint32_t i = 0; i < polls && !done; ++i) done = mbar_try_wait(&bar, 0);
    if (!done && threadIdx.x == 0) flag_device_error(kDevErrWaitTimeout);
}

}  // namespace

cudaError_t launch_wait_timeout_selftest(uint32_t polls, cudaStream_t s) {
    wait_timeout_selftest_kernel<<<1, 32, 0, s>>>(polls);
    return cudaGetLastError();
}

cudaError_t softmax_take_device_error(unsigned int* flags) {
    return take_device_error_word(flags);
}

cudaError_t launch_softmax_fwd(DType dt, void* y, const void* x, const SoftmaxShape& sh,
                               cudaStream_t s) {
    if (dt == DType::F16) return fwd_dispatch<__half, false>(y, x, sh, no_drop(), s);
    return fwd_dispatch<float, false>(y, x, sh, no_drop(), s);
}

cudaError_t launch_softmax_bwd(DType dt, void* dx, const void* y, const void* dy,
                               const SoftmaxShape& sh, cudaStream_t s) {
    if (dt == DType::F16) return bwd_dispatch<__half, false>(dx, y, dy, sh, no_drop(), s);
    return bwd_dispatch<float, false>(dx, y, dy, sh, no_drop(), s);
}

cudaError_t launch_softmax_dropout_fwd(DType dt, void* y, void* y_drop, uint8_t* mask,
                                       const void* x, const SoftmaxShape& sh,
                                       const DropoutRng& rng, cudaStream_t s) {
    const DropArgs d = make_drop(y_drop, mask, rng,
                                 static_cast<uint64_t>(sh.batch * sh.heads * sh.q_len * sh.k_len));
    if (dt == DType::F16) return fwd_dispatch<__half, true>(y, x, sh, d, s);
    return fwd_dispatch<float, true>(y, x, sh, d, s);
}

cudaError_t launch_softmax_dropout_bwd(DType dt, void* dx, const void* y, const void* dy_drop,
                                       const uint8_t* mask, const SoftmaxShape& sh, float scale,
                                       cudaStream_t s) {
    DropArgs d{};
    d.mask = const_cast<uint8_t*>(mask);  // read only in the backward
    d.scale = scale;
    if (dt == DType::F16) return bwd_dispatch<__half, true>(dx, y, dy_drop, sh, d, s);
    return bwd_dispatch<float, true>(dx, y, dy_drop, sh, d, s);
}

}  // namespace ls
