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
// float atomics, one pass).  The other mode is deterministic: one CTA sorts the (id, index) pairs of the batch in shared memory (a bitonic
// sort of unique 64-bit keys, so equal ids stay in index order); then a warp
// per run of equal ids adds that id's rows in index order and adds the total
// into dE[w] -- each row of dE has exactly one writer, so no atomics.
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
// Sort: keys (id << 32 | index), ids outside [0, vocab) replaced by 2^32 - 1
// so that they sort last and are skipped.  n2 = the power of two >= T.
constexpr int kSortThreads = 1024;

__global__ void __launch_bounds__(kSortThreads)
emb_sort_kernel(uint64_t* __restrict__ sorted, const int32_t* __restrict__ tokens, int T, int n2,
                int64_t vocab) {
    extern __shared__ uint64_t keys[];
    pdl_enter();
    for (int k = threadIdx.x; k < n2; k += kSortThreads) {
        uint64_t key = ~uint64_t{0};  // padding: after every real key
        if (k < T) {
            const int32_t w = tokens[k];
            const uint32_t id = (w >= 0 && static_cast<int64_t>(w) < vocab)
                                    ? static_cast<uint32_t>(w)
                                    : 0xFFFFFFFFu;
            key = (static_cast<uint64_t>(id) << 32) | static_cast<uint32_t>(k);
        }
        keys[k] = key;
    }
    __syncthreads();
    // Bitonic sort, ascending.
    for (int size = 2; size <= n2; size <<= 1) {
        for (int stride = size >> 1; stride > 0; stride >>= 1) {
            for (int t = threadIdx.x; t < n2 / 2; t += kSortThreads) {
                const int lo = 2 * t - (t & (stride - 1));
                const int hi = lo + stride;
                const bool up = (lo & size) == 0;
                const uint64_t a = keys[lo], b = keys[hi];
                if ((a > b) == up) {
                    keys[lo] = b;
                    keys[hi] = a;
                }
            }
            __syncthreads();
        }
    }
    for (int k = threadIdx.x; k < T; k += kSortThreads) sorted[k] = keys[k];
}

// The same sort for n2 <= 4096 with four keys per thread (n2/4 threads):
// stages whose partners lie in one thread compare in registers, stages whose
// partners lie in one warp exchange by shuffle, and only the stages with
// partners 128 or more positions apart go through shared memory -- 15
// shared-memory stages for 4096 keys instead of 78.
constexpr int kRegKeys = 4;
constexpr int kRegSortMax = kSortThreads * kRegKeys;  // 4096

__device__ __forceinline__ void cas(uint64_t& mine, uint64_t other, bool keep_min) {
    mine = keep_min ? (other < mine ? other : mine) : (other > mine ? other : mine);
}

__global__ void __launch_bounds__(kSortThreads)
emb_sort_reg_kernel(uint64_t* __restrict__ sorted, const int32_t* __restrict__ tokens, int T,
                    int n2, int64_t vocab) {
    __shared__ uint64_t keys[kRegSortMax];
    pdl_enter();
    const int t = threadIdx.x;
    const int lane = t & 31;
    uint64_t k[kRegKeys];
#pragma unroll
    for (int q = 0; q < kRegKeys; ++q) {
        const int p = kRegKeys * t + q;
        uint64_t key = ~uint64_t{0};
        if (p < T) {
            const int32_t w = tokens[p];
            const uint32_t id = (w >= 0 && static_cast<int64_t>(w) < vocab)
                                    ? static_cast<uint32_t>(w)
                                    : 0xFFFFFFFFu;
            key = (static_cast<uint64_t>(id) << 32) | static_cast<uint32_t>(p);
        }
        k[q] = key;
    }
    for (int size = 2; size <= n2; size <<= 1) {
        for (int stride = size >> 1; stride > 0; stride >>= 1) {
            if (stride < kRegKeys) {
                // partners in this thread: (0,1),(2,3) or (0,2),(1,3); the
                // direction is that of the pair's lower position
                auto cx = [&](uint64_t& a, uint64_t& b, int q_lo) {
                    const bool up = ((kRegKeys * t + q_lo) & size) == 0;
                    if ((a > b) == up) {
                        const uint64_t c = a;
                        a = b;
                        b = c;
                    }
                };
                if (stride == 1) {
                    cx(k[0], k[1], 0);
                    cx(k[2], k[3], 2);
                } else {
                    cx(k[0], k[2], 0);
                    cx(k[1], k[3], 1);
                }
            } else if (stride < 32 * kRegKeys) {
                // partners in this warp: lane ^ (stride / kRegKeys), same slot
                const int lm = stride / kRegKeys;
#pragma unroll
                for (int q = 0; q < kRegKeys; ++q) {
                    const int p = kRegKeys * t + q;
                    const uint64_t other = __shfl_xor_sync(0xffffffffu, k[q], lm);
                    const bool lower = (p & stride) == 0, up = (p & size) == 0;
                    cas(k[q], other, lower == up);
                }
            } else {
                // partners in other warps: through shared memory
#pragma unroll
                for (int q = 0; q < kRegKeys; ++q) keys[kRegKeys * t + q] = k[q];
                __syncthreads();
#pragma unroll
                for (int q = 0; q < kRegKeys; ++q) {
                    const int p = kRegKeys * t + q;
                    const uint64_t other = keys[p ^ stride];
                    const bool lower = (p & stride) == 0, up = (p & size) == 0;
                    cas(k[q], other, lower == up);
                }
                __syncthreads();
            }
        }
    }
    (void)lane;
#pragma unroll
    for (int q = 0; q < kRegKeys; ++q) {
        const int p = kRegKeys * t + q;
        if (p < T) sorted[p] = k[q];
    }
}

struct EmbBwdArgs {
    int T;
    int nvr;     // H / 8
    int64_t H;
    float coef;  // s / (1 - p)
};

// One warp per sorted position; the warp at the head of a run of equal ids
// adds the run's rows in index order and adds the total into dE[id].
template <typename T>
__global__ void __launch_bounds__(kThreads)
emb_accum_kernel(float* __restrict__ dE, const T* __restrict__ dy,
                 const uint8_t* __restrict__ mask, const uint64_t* __restrict__ sorted,
                 const __grid_constant__ EmbBwdArgs a) {
    pdl_enter();
    const int j = static_cast<int>((static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x) >> 5);
    const int lane = threadIdx.x & 31;
    if (j >= a.T) return;
    const uint64_t key = sorted[j];
    const uint32_t id = static_cast<uint32_t>(key >> 32);
    if (id == 0xFFFFFFFFu) return;                                  // invalid ids sort last
    if (j > 0 && static_cast<uint32_t>(sorted[j - 1] >> 32) == id) return;  // not a run head
    int end = j + 1;
    while (end < a.T && static_cast<uint32_t>(sorted[end] >> 32) == id) ++end;
    for (int cv = lane; cv < a.nvr; cv += 32) {
        float acc[kVec];
#pragma unroll
        for (int q = 0; q < kVec; ++q) acc[q] = 0.f;
        for (int r = j; r < end; ++r) {
            const int64_t i = static_cast<int64_t>(static_cast<uint32_t>(sorted[r]));
            const int64_t e = i * a.H + static_cast<int64_t>(cv) * kVec;
            const uint32_t bits = mask[e >> 3];
            float g[kVec];
            load8f<T>(dy + e, g);
#pragma unroll
            for (int q = 0; q < kVec; ++q)
                if ((bits >> q) & 1u) acc[q] += g[q];
        }
        float* dst = dE + static_cast<int64_t>(id) * a.H + static_cast<int64_t>(cv) * kVec;
        float4 d0 = *reinterpret_cast<float4*>(dst), d1 = *reinterpret_cast<float4*>(dst + 4);
        d0.x = fmaf(a.coef, acc[0], d0.x); d0.y = fmaf(a.coef, acc[1], d0.y);
        d0.z = fmaf(a.coef, acc[2], d0.z); d0.w = fmaf(a.coef, acc[3], d0.w);
        d1.x = fmaf(a.coef, acc[4], d1.x); d1.y = fmaf(a.coef, acc[5], d1.y);
        d1.z = fmaf(a.coef, acc[6], d1.z); d1.w = fmaf(a.coef, acc[7], d1.w);
        *reinterpret_cast<float4*>(dst) = d0;
        *reinterpret_cast<float4*>(dst + 4) = d1;
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
                                 float coef, uint64_t* sorted, cudaStream_t st) {
    int n2 = 1;
    while (n2 < T) n2 <<= 1;
    cudaError_t e;
    if (n2 <= kRegSortMax) {
        // n2/4 threads, at least one warp (padding keys fill the rest)
        const int n2r = std::max(n2, 32 * kRegKeys);
        e = launch_pdl(emb_sort_reg_kernel, dim3(1), dim3(n2r / kRegKeys), 0, st, sorted, tokens,
                       static_cast<int>(T), n2r, vocab);
    } else {
        const size_t smem = static_cast<size_t>(n2) * sizeof(uint64_t);
        e = cudaFuncSetAttribute(emb_sort_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(smem));
        if (e != cudaSuccess) return e;
        e = launch_pdl(emb_sort_kernel, dim3(1), dim3(kSortThreads), smem, st, sorted, tokens,
                       static_cast<int>(T), n2, vocab);
    }
    if (e != cudaSuccess) return e;
    EmbBwdArgs a;
    a.T = static_cast<int>(T);
    a.nvr = static_cast<int>(H / kVec);
    a.H = H;
    a.coef = coef;
    const dim3 grid(static_cast<unsigned>((T * 32 + kThreads - 1) / kThreads));
    if (dt == DType::F16)
        return launch_pdl(emb_accum_kernel<__half>, grid, dim3(kThreads), 0, st, dE,
                          static_cast<const __half*>(dy), mask, sorted, a);
    return launch_pdl(emb_accum_kernel<float>, grid, dim3(kThreads), 0, st, dE,
                      static_cast<const float*>(dy), mask, sorted, a);
}

}  // namespace ls
