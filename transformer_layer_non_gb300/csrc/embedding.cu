// embedding.cu -- the embedding layer ("LightSeq2", section 2.1.2), forward
// and backward.
//
// Forward: token i = b*seq + l with id w gives the row
//   y[i] = bit * (s * E[w] + P[l]) / (1 - p),
// the keep bits drawn over the flat index of y exactly as for the other
// dropouts.  A persistent grid walks 16-byte vectors of y: each gathers one
// vector of E's row w and of P's row l, draws its 8 keep bits and writes one
// mask byte.
//
// Backward: dE[w] += s / (1 - p) * sum over the tokens i with id w of
// bit * dy[i].  The pages add the rows with atomicAdd, whose order (and so
// whose rounding) changes from run to run; that is one mode here (vector
// float atomics, one pass).  The other mode is deterministic: each row of dE
// is updated once, by one warp or one CTA, with the id's rows added in an
// order fixed by the ids alone (emb_det_kernel), so no atomics.
#include "ls_device.cuh"
#include "ls_internal.h"

namespace ls {
namespace {

constexpr int kThreads = 256;

struct EmbFwdArgs {
    uint64_t nv;       // vectors of y
    uint32_t nvr;      // vectors per row (H / 8)
    uint32_t seq;
    int64_t vocab;
    float s;           // embedding scale
    uint32_t thr;
    float scale;       // 1 / (1 - p)
    PhiloxSchedule ks;
    uint32_t off_lo, off_hi;
    FastDiv by_nvr, by_seq;
    int mask_tail;     // mask bytes past the last element (written as 0)
};

template <typename T, typename I>
__global__ void __launch_bounds__(kThreads)
emb_fwd_kernel(T* __restrict__ y, uint8_t* __restrict__ mask, const int32_t* __restrict__ tokens,
               const T* __restrict__ E, const T* __restrict__ P,
               const __grid_constant__ EmbFwdArgs a) {
    pdl_enter();
    const I n = static_cast<I>(a.nv);
    const I S = static_cast<I>(gridDim.x) * kThreads;
    for (I v = static_cast<I>(blockIdx.x) * kThreads + threadIdx.x; v < n; v += S) {
        uint64_t i, l;
        uint32_t cv;
        if (sizeof(I) == 4) {
            i = fdiv(static_cast<uint32_t>(v), a.by_nvr);
            cv = static_cast<uint32_t>(v - i * a.nvr);
            l = fmod_(static_cast<uint32_t>(i), a.by_seq);
        } else {
            i = static_cast<uint64_t>(v) / a.nvr;
            cv = static_cast<uint32_t>(static_cast<uint64_t>(v) - i * a.nvr);
            l = i % a.seq;
        }
        const int32_t w = tokens[i];
        float o[kVec];
        const uint32_t bits = keep_bits8(static_cast<uint64_t>(v) * kVec, a.thr, a.ks, a.off_lo,
                                         a.off_hi);
        if (w >= 0 && static_cast<int64_t>(w) < a.vocab) {
            float e[kVec], p[kVec];
            load8f<T>(E + static_cast<size_t>(w) * a.nvr * kVec + cv * kVec, e);
            load8f<T>(P + static_cast<size_t>(l) * a.nvr * kVec + cv * kVec, p);
#pragma unroll
            for (int j = 0; j < kVec; ++j)
                o[j] = ((bits >> j) & 1u) ? fmaf(a.s, e[j], p[j]) * a.scale : 0.f;
        } else {
#pragma unroll
            for (int j = 0; j < kVec; ++j) o[j] = 0.f;
        }
        store8f<T>(y + static_cast<size_t>(v) * kVec, o);
        if (mask) mask[v] = static_cast<uint8_t>(bits);
    }
    if (mask && blockIdx.x == 0 && threadIdx.x == 0)
        for (int k = 0; k < a.mask_tail; ++k) mask[a.nv + k] = 0;
}

// --- backward ------------------------------------------------------------
struct EmbBwdArgs {
    int T;
    int nvr;     // H / 8
    int64_t H;
    int64_t vocab;
    float coef;  // s / (1 - p)
};

// Rows in flight per warp in the shared sum of a frequent id (32 registers).
template <typename T> constexpr int heavy_batch() { return sizeof(T) == 2 ? 8 : 4; }

// Ids as the deterministic backward keeps them in shared memory: 16 bits when
// every valid id lies below the 0xFFFF sentinel, else 32.  A lane compares
// IdScan<ID>::kPerLane consecutive ids (one 16-byte shared load), a warp
// kStep per step.
template <typename ID> struct IdScan {
    static constexpr int kPerLane = 16 / static_cast<int>(sizeof(ID));
    static constexpr int kStep = 32 * kPerLane;
    static constexpr uint32_t kNone = sizeof(ID) == 2 ? 0xFFFFu : 0xFFFFFFFFu;
    // Bit k set iff ids[base + kPerLane*lane + k] == w (w < kNone).
    static __device__ __forceinline__ uint32_t lane_bits(const ID* ids, int base, int lane,
                                                         uint32_t w) {
        const uint4 q = *reinterpret_cast<const uint4*>(ids + base + kPerLane * lane);
        if constexpr (sizeof(ID) == 2) {
            const uint32_t wp = w | (w << 16);
            const uint32_t m0 = __vcmpeq2(q.x, wp), m1 = __vcmpeq2(q.y, wp);
            const uint32_t m2 = __vcmpeq2(q.z, wp), m3 = __vcmpeq2(q.w, wp);
            return (m0 & 1u) | ((m0 >> 15) & 2u) | ((m1 & 1u) << 2) | ((m1 >> 13) & 8u) |
                   ((m2 & 1u) << 4) | ((m2 >> 11) & 32u) | ((m3 & 1u) << 6) | ((m3 >> 9) & 128u);
        } else {
            return static_cast<uint32_t>(q.x == w) | (static_cast<uint32_t>(q.y == w) << 1) |
                   (static_cast<uint32_t>(q.z == w) << 2) | (static_cast<uint32_t>(q.w == w) << 3);
        }
    }
    static __device__ __forceinline__ uint32_t of(int32_t t, int64_t vocab) {
        return t >= 0 && static_cast<int64_t>(t) < vocab ? static_cast<uint32_t>(t) : kNone;
    }
};

// Bits k of a lane's run of n ids starting at position p0 whose position lies
// in [lo, hi).
__device__ __forceinline__ uint32_t range_bits(int p0, int n, int lo, int hi) {
    const int a = min(max(lo - p0, 0), n), b = min(max(hi - p0, 0), n);
    return ((1u << b) - 1u) & ~((1u << a) - 1u);
}

// Warps (tokens) per CTA of the deterministic backward, and the CTAs per SM
// its registers are sized for: two at 64 registers for FP16 rows (32 warps
// per SM, so a 4096-token batch is one wave), one at 128 for FP32 rows.
constexpr int kDetWarps = 16;
template <typename T> constexpr int det_min_ctas() { return sizeof(T) == 4 ? 1 : 2; }

// Ids on at least this many tokens are summed by a whole CTA.
constexpr int kFrequent = 4;

// Deterministic backward: dE[w] += coef * sum over the tokens i with id w of
// bit * dy[i], each row of dE written by one warp or CTA, in an order fixed
// by the ids alone, so the bits are the same on every run (no atomics).
//
// One warp per token, W tokens per CTA; each warp's gradient row and mask
// bytes are asked of L2 before the dependency wait.  Each CTA copies all T
// ids into shared memory (padded with a sentinel to whole scan steps) and
// passes over them once, counting for each of its tokens j with id w the
// tokens with id w before j (r) and after it, so n = all of them:
//   - n <= 3: the first of them (r = 0) adds its own row and the later ones,
//     in token order: dE[w] += coef * (((0 + bit*dy[j]) + bit*dy[i1]) + ...);
//   - n >= 4 ("frequent"): each 32-vector column block b of the row is an
//     independent sum, handed to the CTA of the id's token of rank
//     (h + b) mod n, h a hash of w.  After the light sums, the CTA takes its
//     blocks one by one: the positions [f, T) (f: the id's first token) cut
//     into W equal slices, warp s sums, in increasing index, the rows of
//     slice s with id w (heavy_batch rows in flight) into S_s, and
//     dE[w][block] += coef * (((0 + S_0) + S_1) + ... + S_{W-1}) through
//     shared memory.
// The tokens of an id are spread over the batch, so the hash spreads the
// frequent ids' blocks over the CTAs (their first tokens all lie early in the
// batch), and an id's blocks over as many CTAs as it has blocks.
// Light sums take NB column vectors per lane per pass.
template <typename T, typename ID, int NB>
__global__ void __launch_bounds__(32 * kDetWarps, det_min_ctas<T>())
emb_det_kernel(float* __restrict__ dE, const T* __restrict__ dy,
               const uint8_t* __restrict__ mask, const int32_t* __restrict__ tokens,
               const __grid_constant__ EmbBwdArgs a) {
    using S = IdScan<ID>;
    constexpr int W = kDetWarps;
    constexpr int P = S::kPerLane;
    constexpr int STEP = S::kStep;
    constexpr int B = heavy_batch<T>();
    extern __shared__ __align__(16) unsigned char det_smem[];
    ID* ids = reinterpret_cast<ID*>(det_smem);  // [Tp]
    __shared__ int s_first[W];  // first token of the frequent id warp t hands over, or -1
    __shared__ int s_blk[W], s_cnt[W];  // its first column block and its token count
    __shared__ uint32_t s_tab[256];  // bit t: token t's id has these low 8 bits
    __shared__ uint32_t s_wid[W];
    // Per counting warp c and token t: earlier / later tokens with t's id, the
    // first earlier one, and the first two later ones it met.
    __shared__ int s_rank[W][W], s_low[W][W], s_nlater[W][W], s_next[W][W][2];
    __shared__ __align__(16) float s_part[W][32][kVec];
    __shared__ uint16_t s_list[W][STEP];

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int ntok = a.T, nvr = a.nvr;
    const int Tp = (ntok + STEP - 1) / STEP * STEP;
    const int j = blockIdx.x * W + warp;
    const bool have = j < ntok;
    const int64_t rowv = static_cast<int64_t>(j) * nvr;  // first vector of row j

    // Before the dependency wait: this warp's gradient row and mask bytes, and
    // one line of the ids per CTA (the CTAs together cover them), into L2.
    if (have) {
        const char* row = reinterpret_cast<const char*>(dy + rowv * kVec);
        const int bytes = nvr * kVec * static_cast<int>(sizeof(T));
        for (int c = lane * 128; c < bytes; c += 32 * 128) prefetch_l2(row + c);
        if (lane == 31) prefetch_l2(row + bytes - 1);
        if (lane == 0) prefetch_l2(mask + rowv);
        if (lane == 1) prefetch_l2(mask + rowv + nvr - 1);
    }
    if (threadIdx.x == 0) {
        const int lines = (ntok + 31) / 32;
        prefetch_l2(tokens + static_cast<int64_t>(blockIdx.x % lines) * 32);
    }
    pdl_enter();

    for (int k = threadIdx.x; k < 256; k += 32 * W) s_tab[k] = 0u;
    if (lane < W) {
        s_rank[warp][lane] = s_nlater[warp][lane] = 0;
        s_low[warp][lane] = ntok;
    }
    // All ids into shared memory, four per 16-byte load where aligned.
    int k0 = 0;
    if ((reinterpret_cast<uintptr_t>(tokens) & 15u) == 0) {
        const int n4 = ntok >> 2;
        const int4* t4 = reinterpret_cast<const int4*>(tokens);
#pragma unroll 2
        for (int k = threadIdx.x; k < n4; k += 32 * W) {
            const int4 t = t4[k];
            const uint32_t x = S::of(t.x, a.vocab), y = S::of(t.y, a.vocab);
            const uint32_t z = S::of(t.z, a.vocab), u = S::of(t.w, a.vocab);
            if constexpr (sizeof(ID) == 2)
                *reinterpret_cast<uint2*>(ids + 4 * k) = make_uint2(x | (y << 16), z | (u << 16));
            else
                *reinterpret_cast<uint4*>(ids + 4 * k) = make_uint4(x, y, z, u);
        }
        k0 = 4 * n4;
    }
#pragma unroll 4
    for (int k = k0 + threadIdx.x; k < Tp; k += 32 * W)
        ids[k] = static_cast<ID>(k < ntok ? S::of(tokens[k], a.vocab) : S::kNone);
    __syncthreads();

    const uint32_t w = have ? static_cast<uint32_t>(ids[j]) : S::kNone;
    const bool valid = w != S::kNone;
    if (valid) {  // the dE row into L2 (harmless if this token is not the one to update it)
        const float* row = dE + static_cast<int64_t>(w) * a.H;
        for (int c = lane * 32; c < nvr * kVec; c += 32 * 32) prefetch_l2(row + c);
        if (lane == 31) prefetch_l2(row + nvr * kVec - 1);
    }
    // One pass of the CTA over all ids finds the tokens with the CTA's W ids:
    // s_tab[x & 255] has bit t set if token t's id has those low bits, so an
    // id is compared in full only on a hit.  For token t it counts the earlier
    // tokens with its id (s_rank) and the first of them (s_low), and the later
    // ones (s_nlater), keeping the first two it meets (s_next).  Each warp
    // counts into its own row of these arrays -- a frequent id's hundreds of
    // matches would otherwise queue on one shared-memory word -- and the rows
    // are combined after the pass (sums and minima: the order does not matter).
    if (lane == 0) {
        s_wid[warp] = w;
        if (valid) atomicOr(&s_tab[w & 255u], 1u << warp);
    }
    __syncthreads();
    for (int k = P * threadIdx.x; k < Tp; k += P * 32 * W) {
        const uint4 q = *reinterpret_cast<const uint4*>(ids + k);
        uint32_t x[P];
        if constexpr (sizeof(ID) == 2) {
            x[0] = q.x & 0xFFFFu; x[1] = q.x >> 16; x[2] = q.y & 0xFFFFu; x[3] = q.y >> 16;
            x[4] = q.z & 0xFFFFu; x[5] = q.z >> 16; x[6] = q.w & 0xFFFFu; x[7] = q.w >> 16;
        } else {
            x[0] = q.x; x[1] = q.y; x[2] = q.z; x[3] = q.w;
        }
#pragma unroll
        for (int i = 0; i < P; ++i) {
            if (x[i] == S::kNone) continue;
            for (uint32_t m = s_tab[x[i] & 255u]; m; m &= m - 1) {
                const int t = __ffs(m) - 1;
                if (s_wid[t] != x[i]) continue;
                const int pos = k + i, jt = blockIdx.x * W + t;
                if (pos < jt) {
                    atomicAdd(&s_rank[warp][t], 1);
                    atomicMin(&s_low[warp][t], pos);
                } else if (pos > jt) {
                    const int slot = atomicAdd(&s_nlater[warp][t], 1);
                    if (slot < 2) s_next[warp][t][slot] = pos;
                }
            }
        }
    }
    __syncthreads();
    // Token `warp`'s counts: lane c reads counting warp c's row.  p1 < p2 are
    // the two smallest later positions (all of them when there are at most two).
    const int cr = lane < W ? s_rank[lane][warp] : 0;
    const int cl = lane < W ? s_nlater[lane][warp] : 0;
    const int r = __reduce_add_sync(0xffffffffu, cr);
    const int later = __reduce_add_sync(0xffffffffu, cl);
    const int first = r > 0 ? __reduce_min_sync(0xffffffffu, lane < W ? s_low[lane][warp] : ntok)
                            : j;
    const int e0 = cl >= 1 ? s_next[lane][warp][0] : ntok;
    const int e1 = cl >= 2 ? s_next[lane][warp][1] : ntok;
    const int p1 = __reduce_min_sync(0xffffffffu, min(e0, e1));
    const int p2 = __reduce_min_sync(0xffffffffu, min(e0, e1) == p1 ? max(e0, e1) : min(e0, e1));
    const int n = r + 1 + later;
    const bool frequent = valid && n >= kFrequent;
    const int ncb = (nvr + 31) / 32;  // 32-vector column blocks of a row
    if (lane == 0) {
        // Column block b of a frequent id goes to its token of rank (h + b) mod n,
        // h a hash of the id: this token takes blocks b0, b0 + n, ...
        const int h = static_cast<int>(__umulhi(w * 2654435761u, static_cast<uint32_t>(n)));
        const int b0 = r >= h ? r - h : r - h + n;
        s_first[warp] = frequent && b0 < ncb ? first : -1;
        s_blk[warp] = b0;
        s_cnt[warp] = n;
    }

    if (valid && !frequent && r == 0) {
        const int64_t row1 = static_cast<int64_t>(p1) * nvr, row2 = static_cast<int64_t>(p2) * nvr;
        for (int cb = 0; cb < nvr; cb += 32 * NB) {
            Raw8<T> g0[NB];  // the own row's block (in L2 since before the dependency wait)
            uint32_t b0[NB];
#pragma unroll
            for (int b = 0; b < NB; ++b) {
                const int cv = cb + b * 32 + lane;
                b0[b] = 0u;
                if (cv < nvr) {
                    g0[b] = load8<T>(dy + (rowv + cv) * kVec);
                    b0[b] = mask[rowv + cv];
                }
            }
#pragma unroll
            for (int b = 0; b < NB; ++b) {
                const int cv = cb + b * 32 + lane;
                if (cv >= nvr) continue;
                float acc[kVec], f[kVec];
                unpack(g0[b], f);
#pragma unroll
                for (int q = 0; q < kVec; ++q) {
                    acc[q] = 0.f;
                    if ((b0[b] >> q) & 1u) acc[q] += f[q];
                }
                for (int m = 0; m < later; ++m) {  // at most 2, in token order
                    const int64_t iv = (m == 0 ? row1 : row2) + cv;
                    unpack(load8<T>(dy + iv * kVec), f);
                    const uint32_t bits = mask[iv];
#pragma unroll
                    for (int q = 0; q < kVec; ++q)
                        if ((bits >> q) & 1u) acc[q] += f[q];
                }
                float* dst = dE + static_cast<int64_t>(w) * a.H + static_cast<int64_t>(cv) * kVec;
                float4 d0 = *reinterpret_cast<const float4*>(dst);
                float4 d1 = *reinterpret_cast<const float4*>(dst + 4);
                d0.x = fmaf(a.coef, acc[0], d0.x); d0.y = fmaf(a.coef, acc[1], d0.y);
                d0.z = fmaf(a.coef, acc[2], d0.z); d0.w = fmaf(a.coef, acc[3], d0.w);
                d1.x = fmaf(a.coef, acc[4], d1.x); d1.y = fmaf(a.coef, acc[5], d1.y);
                d1.z = fmaf(a.coef, acc[6], d1.z); d1.w = fmaf(a.coef, acc[7], d1.w);
                *reinterpret_cast<float4*>(dst) = d0;
                *reinterpret_cast<float4*>(dst + 4) = d1;
            }
        }
    }

    // The column blocks of frequent ids handed to this CTA, one after another,
    // by all its warps: warp s sums slice s of the positions [f, T).
    __syncthreads();
    for (int t = 0; t < W; ++t) {
        const int f = s_first[t];  // the same in every thread of the CTA
        if (f < 0) continue;
        const uint32_t wt = ids[blockIdx.x * W + t];
        const int per = (ntok - f + W - 1) / W;
        const int lo = min(ntok, f + warp * per), hi = min(ntok, lo + per);
        for (int cb = s_blk[t]; cb < ncb; cb += s_cnt[t]) {
            const int cv = cb * 32 + lane;
            float acc[kVec];
#pragma unroll
            for (int q = 0; q < kVec; ++q) acc[q] = 0.f;
            for (int base = lo - lo % STEP; base < hi; base += STEP) {
                // This step's matches, in increasing position, listed in s_list.
                const uint32_t m =
                    S::lane_bits(ids, base, lane, wt) & range_bits(base + P * lane, P, lo, hi);
                const uint32_t c = __popc(m);
                uint32_t incl = c;
#pragma unroll
                for (int d = 1; d < 32; d <<= 1) {
                    const uint32_t o = __shfl_up_sync(0xffffffffu, incl, d);
                    if (lane >= d) incl += o;
                }
                const int total = static_cast<int>(__shfl_sync(0xffffffffu, incl, 31));
                int slot = static_cast<int>(incl - c);
                for (uint32_t rb = m; rb; rb &= rb - 1)
                    s_list[warp][slot++] = static_cast<uint16_t>(P * lane + __ffs(rb) - 1);
                __syncwarp();
                for (int q0 = 0; q0 < total; q0 += B) {
                    Raw8<T> g[B];
                    uint32_t bits[B];
#pragma unroll
                    for (int u = 0; u < B; ++u) {
                        bits[u] = 0u;
                        if (q0 + u < total && cv < nvr) {
                            const int64_t iv =
                                static_cast<int64_t>(base + s_list[warp][q0 + u]) * nvr + cv;
                            g[u] = load8<T>(dy + iv * kVec);
                            bits[u] = mask[iv];
                        }
                    }
#pragma unroll
                    for (int u = 0; u < B; ++u) {
                        if (q0 + u >= total || cv >= nvr) continue;
                        float fv[kVec];
                        unpack(g[u], fv);
#pragma unroll
                        for (int q = 0; q < kVec; ++q)
                            if ((bits[u] >> q) & 1u) acc[q] += fv[q];
                    }
                }
                __syncwarp();
            }
            float4* pp = reinterpret_cast<float4*>(s_part[warp][lane]);
            pp[0] = make_float4(acc[0], acc[1], acc[2], acc[3]);
            pp[1] = make_float4(acc[4], acc[5], acc[6], acc[7]);
            __syncthreads();
            if (threadIdx.x < 32 * kVec) {
                const int v = threadIdx.x / kVec, e = threadIdx.x % kVec;
                const int vv = cb * 32 + v;
                if (vv < nvr) {
                    float sum = 0.f;
#pragma unroll
                    for (int s2 = 0; s2 < W; ++s2) sum += s_part[s2][v][e];
                    float* d = dE + static_cast<int64_t>(wt) * a.H + static_cast<int64_t>(vv) * kVec + e;
                    *d = fmaf(a.coef, sum, *d);
                }
            }
            __syncthreads();
        }
    }
}

// The pages' backward: every masked, scaled gradient vector is added into its
// table row with vector float atomics (fast, but the order of the additions,
// and so the rounding, varies from run to run).
template <typename T, typename I>
__global__ void __launch_bounds__(kThreads)
emb_atomic_kernel(float* __restrict__ dE, const T* __restrict__ dy,
                  const uint8_t* __restrict__ mask, const int32_t* __restrict__ tokens,
                  uint64_t nv, int64_t vocab, float coef, const __grid_constant__ FastDiv by_nvr) {
    pdl_enter();
    const I n = static_cast<I>(nv);
    const I S = static_cast<I>(gridDim.x) * kThreads;
    for (I v = static_cast<I>(blockIdx.x) * kThreads + threadIdx.x; v < n; v += S) {
        uint64_t i;
        if (sizeof(I) == 4)
            i = fdiv(static_cast<uint32_t>(v), by_nvr);
        else
            i = static_cast<uint64_t>(v) / by_nvr.d;
        const uint32_t cv = static_cast<uint32_t>(static_cast<uint64_t>(v) - i * by_nvr.d);
        const int32_t w = tokens[i];
        if (w < 0 || static_cast<int64_t>(w) >= vocab) continue;
        const uint32_t bits = mask[v];
        if (bits == 0) continue;
        float g[kVec];
        load8f<T>(dy + static_cast<size_t>(v) * kVec, g);
#pragma unroll
        for (int j = 0; j < kVec; ++j) g[j] = ((bits >> j) & 1u) ? coef * g[j] : 0.f;
        float* dst = dE + (static_cast<size_t>(w) * by_nvr.d + cv) * kVec;
        asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(dst), "f"(g[0]),
                     "f"(g[1]), "f"(g[2]), "f"(g[3])
                     : "memory");
        asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(dst + 4), "f"(g[4]),
                     "f"(g[5]), "f"(g[6]), "f"(g[7])
                     : "memory");
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
cudaError_t fwd_impl(void* y, uint8_t* mask, const int32_t* tokens, const void* E, const void* P,
                     int64_t batch, int64_t seq, int64_t H, int64_t vocab, float s,
                     const DropoutRng& rng, cudaStream_t st) {
    EmbFwdArgs a;
    a.nvr = static_cast<uint32_t>(H / kVec);
    a.nv = static_cast<uint64_t>(batch * seq) * a.nvr;
    a.seq = static_cast<uint32_t>(seq);
    a.vocab = vocab;
    a.s = s;
    a.thr = rng.thr;
    a.scale = rng.scale;
    a.ks = philox_schedule(PhiloxKey{static_cast<uint32_t>(rng.seed),
                                     static_cast<uint32_t>(rng.seed >> 32)});
    a.off_lo = static_cast<uint32_t>(rng.offset);
    a.off_hi = static_cast<uint32_t>(rng.offset >> 32);
    a.by_nvr = make_fastdiv(a.nvr);
    a.by_seq = make_fastdiv(a.seq);
    a.mask_tail = static_cast<int>(((a.nv + 3) / 4) * 4 - a.nv);
    static const int occ = occupancy(emb_fwd_kernel<T, uint64_t>);
    const int64_t want = static_cast<int64_t>((a.nv + kThreads - 1) / kThreads);
    const int64_t grid = std::max<int64_t>(1, std::min<int64_t>(want, int64_t{sm_count()} * occ));
    const bool narrow = a.nv + static_cast<uint64_t>(grid) * kThreads < (uint64_t{1} << 31);
    auto kern = narrow ? emb_fwd_kernel<T, uint32_t> : emb_fwd_kernel<T, uint64_t>;
    return launch_pdl(kern, dim3(static_cast<unsigned>(grid)), dim3(kThreads), 0, st,
                      static_cast<T*>(y), mask, tokens, static_cast<const T*>(E),
                      static_cast<const T*>(P), a);
}

}  // namespace

cudaError_t launch_embedding_fwd(DType dt, void* y, uint8_t* mask, const int32_t* tokens,
                                 const void* E, const void* P, int64_t batch, int64_t seq,
                                 int64_t H, int64_t vocab, float s, const DropoutRng& rng,
                                 cudaStream_t st) {
    if (dt == DType::F16)
        return fwd_impl<__half>(y, mask, tokens, E, P, batch, seq, H, vocab, s, rng, st);
    return fwd_impl<float>(y, mask, tokens, E, P, batch, seq, H, vocab, s, rng, st);
}

template <typename T>
cudaError_t atomic_impl(float* dE, const void* dy, const uint8_t* mask, const int32_t* tokens,
                        int64_t ntok, int64_t H, int64_t vocab, float coef, cudaStream_t st) {
    const uint64_t nv = static_cast<uint64_t>(ntok) * static_cast<uint64_t>(H / kVec);
    static const int occ = occupancy(emb_atomic_kernel<T, uint64_t>);
    const int64_t want = static_cast<int64_t>((nv + kThreads - 1) / kThreads);
    const int64_t grid = std::max<int64_t>(1, std::min<int64_t>(want, int64_t{sm_count()} * occ));
    const bool narrow = nv + static_cast<uint64_t>(grid) * kThreads < (uint64_t{1} << 31);
    auto kern = narrow ? emb_atomic_kernel<T, uint32_t> : emb_atomic_kernel<T, uint64_t>;
    return launch_pdl(kern, dim3(static_cast<unsigned>(grid)), dim3(kThreads), 0, st, dE,
                      static_cast<const T*>(dy), mask, tokens, nv, vocab, coef,
                      make_fastdiv(static_cast<uint32_t>(H / kVec)));
}

cudaError_t launch_embedding_bwd_atomic(DType dt, float* dE, const void* dy, const uint8_t* mask,
                                        const int32_t* tokens, int64_t T, int64_t H,
                                        int64_t vocab, float coef, cudaStream_t st) {
    if (dt == DType::F16) return atomic_impl<__half>(dE, dy, mask, tokens, T, H, vocab, coef, st);
    return atomic_impl<float>(dE, dy, mask, tokens, T, H, vocab, coef, st);
}

namespace {

template <typename T, typename ID, int NB>
cudaError_t det_launch(float* dE, const void* dy, const uint8_t* mask, const int32_t* tokens,
                       const EmbBwdArgs& a, cudaStream_t st) {
    static int done[kMaxDevices] = {};
    auto kern = emb_det_kernel<T, ID, NB>;
    constexpr int step = IdScan<ID>::kStep, W = kDetWarps;
    const size_t smem = static_cast<size_t>((a.T + step - 1) / step * step) * sizeof(ID);
    if (smem > 16 * 1024) {
        const cudaError_t e = allow_max_dynamic_smem(kern, done);
        if (e != cudaSuccess) return e;
    }
    const dim3 grid(static_cast<unsigned>((a.T + W - 1) / W));
    return launch_pdl(kern, grid, dim3(32 * W), smem, st, dE, static_cast<const T*>(dy), mask,
                      tokens, a);
}

template <typename T, typename ID>
cudaError_t det_dispatch(float* dE, const void* dy, const uint8_t* mask, const int32_t* tokens,
                         const EmbBwdArgs& a, cudaStream_t st) {
    // Column vectors per lane per pass of a light sum: one pass up to 160
    // vectors (1280 columns), four per pass beyond.
    if (a.nvr <= 96) return det_launch<T, ID, 3>(dE, dy, mask, tokens, a, st);
    if (a.nvr > 128 && a.nvr <= 160) return det_launch<T, ID, 5>(dE, dy, mask, tokens, a, st);
    return det_launch<T, ID, 4>(dE, dy, mask, tokens, a, st);
}

}  // namespace

cudaError_t launch_embedding_bwd(DType dt, float* dE, const void* dy, const uint8_t* mask,
                                 const int32_t* tokens, int64_t T, int64_t H, int64_t vocab,
                                 float coef, cudaStream_t st) {
    EmbBwdArgs a;
    a.T = static_cast<int>(T);
    a.nvr = static_cast<int>(H / kVec);
    a.H = H;
    a.vocab = vocab;
    a.coef = coef;
    const bool narrow = vocab <= 0xFFFF;  // every valid id below the 16-bit sentinel
    if (dt == DType::F16)
        return narrow ? det_dispatch<__half, uint16_t>(dE, dy, mask, tokens, a, st)
                      : det_dispatch<__half, uint32_t>(dE, dy, mask, tokens, a, st);
    return narrow ? det_dispatch<float, uint16_t>(dE, dy, mask, tokens, a, st)
                  : det_dispatch<float, uint32_t>(dE, dy, mask, tokens, a, st);
}

}  // namespace ls
