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
// float atomics, one pass).  The other mode is deterministic: the warp of the
// first token with each id adds that id's rows in index order and adds the
// total into dE[w] -- each row of dE has exactly one writer, so no atomics.
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

constexpr int kOwnerBlk = 3;  // column vectors per lane per pass over the matches
constexpr int kIdsPerLane = 8;
constexpr int kIdStep = 32 * kIdsPerLane;  // ids a warp compares per ballot

// Deterministic backward without a sort: one warp per token j.  The warp
// returns unless j is the first token with its id w; the owner then walks the
// tokens from j on, and for every token i with id w, in increasing i, adds
// bit * dy[i] into FP32 registers, and finally adds coef times the sum into
// dE[w].  Each row of dE has one writer and a fixed order of additions, so the
// bits are the same on every run.  The ids (which stay in L1) are compared
// 256 per step, load q of lane l reading id base + 32q + l (each load a
// coalesced 128 bytes), so a scan over the batch is a short chain of
// independent loads; the matches are taken load by load and lane by lane,
// i.e. in increasing index.  Column vectors go kOwnerBlk per lane per pass
// (one pass for H <= 768); four CTAs per SM keep a whole 4096-token batch
// resident in one wave.  The owner asks L2 for its dE row and its own dy row
// before it scans, so those reads overlap the scan.
template <typename T>
__global__ void __launch_bounds__(kThreads, min_ctas<T>(4))
emb_owner_kernel(float* __restrict__ dE, const T* __restrict__ dy,
                 const uint8_t* __restrict__ mask, const int32_t* __restrict__ tokens,
                 const __grid_constant__ EmbBwdArgs a) {
    pdl_enter();
    const int j = static_cast<int>((static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x) >> 5);
    const int lane = threadIdx.x & 31;
    if (j >= a.T) return;  // whole warps
    const int32_t w = tokens[j];
    if (w < 0 || static_cast<int64_t>(w) >= a.vocab) return;  // no table row: no gradient
    // This lane's ids of the step at `base`, restricted to [lo, hi), as a bit
    // mask of matches with w (ids outside the range are never loaded).
    auto matches = [&](int base, int lo, int hi) {
        int32_t t[kIdsPerLane];
#pragma unroll
        for (int q = 0; q < kIdsPerLane; ++q) {
            const int k = base + q * 32 + lane;
            t[q] = (k >= lo && k < hi) ? tokens[k] : -1;
        }
        uint32_t my = 0;
#pragma unroll
        for (int q = 0; q < kIdsPerLane; ++q) my |= static_cast<uint32_t>(t[q] == w) << q;
        return my;
    };
    for (int base = 0; base < j; base += kIdStep)  // an earlier token with id w?
        if (__ballot_sync(0xffffffffu, matches(base, 0, j) != 0)) return;
    for (int cv = lane; cv < a.nvr; cv += 32) {
        prefetch_l2(dE + static_cast<int64_t>(w) * a.H + static_cast<int64_t>(cv) * kVec);
        prefetch_l2(dy + static_cast<int64_t>(j) * a.H + static_cast<int64_t>(cv) * kVec);
    }
    const int first = j - j % kIdStep;
    int end = a.T;  // after the first pass: one past the id's last token
    for (int cb = 0; cb < a.nvr; cb += 32 * kOwnerBlk) {
        float acc[kOwnerBlk][kVec];
#pragma unroll
        for (int b = 0; b < kOwnerBlk; ++b)
#pragma unroll
            for (int q = 0; q < kVec; ++q) acc[b][q] = 0.f;
        int last = j;
        for (int base = first; base < end; base += kIdStep) {
            const uint32_t my = matches(base, j, end);
            if (!__ballot_sync(0xffffffffu, my != 0)) continue;
#pragma unroll 1
            for (int ld = 0; ld < kIdsPerLane; ++ld) {  // warp-uniform: loads, then lanes, in order
                uint32_t lanes = __ballot_sync(0xffffffffu, (my >> ld) & 1u);
                while (lanes) {
                    const int64_t i = base + ld * 32 + __ffs(lanes) - 1;
                    lanes &= lanes - 1;
                    last = static_cast<int>(i);
                    Raw8<T> g[kOwnerBlk];
                    uint32_t bits[kOwnerBlk];
#pragma unroll
                    for (int b = 0; b < kOwnerBlk; ++b) {
                        const int cv = cb + b * 32 + lane;
                        bits[b] = 0u;
                        if (cv < a.nvr) {
                            const int64_t e = i * a.H + static_cast<int64_t>(cv) * kVec;
                            g[b] = load8<T>(dy + e);
                            bits[b] = mask[e >> 3];
                        }
                    }
#pragma unroll
                    for (int b = 0; b < kOwnerBlk; ++b) {
                        if (cb + b * 32 + lane >= a.nvr) continue;
                        float f[kVec];
                        unpack(g[b], f);
#pragma unroll
                        for (int q = 0; q < kVec; ++q)
                            if ((bits[b] >> q) & 1u) acc[b][q] += f[q];
                    }
                }
            }
        }
        end = last + 1;  // later passes stop at the id's last token
#pragma unroll
        for (int b = 0; b < kOwnerBlk; ++b) {
            const int cv = cb + b * 32 + lane;
            if (cv >= a.nvr) continue;
            float* dst = dE + static_cast<int64_t>(w) * a.H + static_cast<int64_t>(cv) * kVec;
            float4 d0 = *reinterpret_cast<float4*>(dst), d1 = *reinterpret_cast<float4*>(dst + 4);
            d0.x = fmaf(a.coef, acc[b][0], d0.x); d0.y = fmaf(a.coef, acc[b][1], d0.y);
            d0.z = fmaf(a.coef, acc[b][2], d0.z); d0.w = fmaf(a.coef, acc[b][3], d0.w);
            d1.x = fmaf(a.coef, acc[b][4], d1.x); d1.y = fmaf(a.coef, acc[b][5], d1.y);
            d1.z = fmaf(a.coef, acc[b][6], d1.z); d1.w = fmaf(a.coef, acc[b][7], d1.w);
            *reinterpret_cast<float4*>(dst) = d0;
            *reinterpret_cast<float4*>(dst + 4) = d1;
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

cudaError_t launch_embedding_bwd(DType dt, float* dE, const void* dy, const uint8_t* mask,
                                 const int32_t* tokens, int64_t T, int64_t H, int64_t vocab,
                                 float coef, cudaStream_t st) {
    EmbBwdArgs a;
    a.T = static_cast<int>(T);
    a.nvr = static_cast<int>(H / kVec);
    a.H = H;
    a.vocab = vocab;
    a.coef = coef;
    const dim3 grid(static_cast<unsigned>((T * 32 + kThreads - 1) / kThreads));
    if (dt == DType::F16)
        return launch_pdl(emb_owner_kernel<__half>, grid, dim3(kThreads), 0, st, dE,
                          static_cast<const __half*>(dy), mask, tokens, a);
    return launch_pdl(emb_owner_kernel<float>, grid, dim3(kThreads), 0, st, dE,
                      static_cast<const float*>(dy), mask, tokens, a);
}

}  // namespace ls
