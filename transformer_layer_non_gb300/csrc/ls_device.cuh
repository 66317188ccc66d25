// ls_device.cuh -- device building blocks shared by the operator kernels:
// 8-element vector I/O (one 16-byte access for FP16, two for FP32), FP32
// conversion in registers, the Philox-4x32-10 counter-based generator, and
// shuffle reductions over a group of lanes.
#pragma once

#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace ls {

constexpr int kVec = 8;  // elements per vector access, both dtypes

// Minimum resident CTAs per SM asked of the compiler: the FP16 figure, one
// fewer for FP32 storage (whose vectors take twice the registers).
template <typename T> __host__ __device__ constexpr int min_ctas(int for_fp16) {
    return sizeof(T) == 2 ? for_fp16 : (for_fp16 > 1 ? for_fp16 - 1 : 1);
}

// ---------------------------------------------------------------------------
// Division of a 31-bit numerator by a fixed divisor d >= 1 as a multiply and
// a shift (Granlund & Montgomery, "Division by invariant integers using
// multiplication", PLDI 1994): with l = ceil(log2 d) and m = floor(2^(31+l)/d)
// + 1 (at most 2^32), floor(n/d) = floor(n*m / 2^(31+l)) for 0 <= n < 2^31.
// ---------------------------------------------------------------------------
struct FastDiv {
    uint64_t m;
    uint32_t shift;  // 31 + l
    uint32_t d;
};
inline FastDiv make_fastdiv(uint32_t d) {
    uint32_t l = 0;
    while ((uint64_t{1} << l) < d) ++l;
    FastDiv f;
    f.shift = 31 + l;
    f.m = ((uint64_t{1} << f.shift) / d) + 1;
    f.d = d;
    return f;
}
__host__ __device__ __forceinline__ uint32_t fdiv(uint32_t n, const FastDiv& f) {
    return static_cast<uint32_t>((static_cast<uint64_t>(n) * f.m) >> f.shift);
}
__host__ __device__ __forceinline__ uint32_t fmod_(uint32_t n, const FastDiv& f) {
    return n - fdiv(n, f) * f.d;
}

// ---------------------------------------------------------------------------
// 8-element vectors.  Raw8<T> keeps the loaded bits (4 registers for FP16,
// 8 for FP32) so that many loads can be in flight before any conversion.
// ---------------------------------------------------------------------------
// Asks L2 to fetch the line holding p (a valid global address); no register
// is written, so the later load finds the line in L2.
__device__ __forceinline__ void prefetch_l2(const void* p) {
    asm volatile("prefetch.global.L2 [%0];" ::"l"(p));
}

// Prefetches issued before griddepcontrol.wait.  Until the wait returns, a
// kernel must not read memory that the previous grid on the stream may still
// be writing.  An L2 prefetch reads nothing into the program: it only moves a
// line into L2, the device's point of coherence, where the previous grid's
// writes land as well, and the kernel's own loads after the wait see those
// writes.  So a kernel may prefetch the lines of its first inputs before the
// wait: while the previous grid drains, their DRAM round trip is under way
// (measured on GB300: LayerNorm forward at 4096 x 768, 4.08 -> 3.26 us).
// Addresses must lie inside the input (a prefetch outside an allocation is
// not an error, but nothing here relies on that).

// Prefetch of a small parameter vector (bias, gamma, beta: `bytes` bytes from
// p) into L2, one request per 128-byte line, by the first CTA only.  Kernels
// that read such a vector after their rows' loads issue this at their start,
// so that the other CTAs' reads find the lines in L2 instead of paying a DRAM
// round trip on the row's critical path.  (Measured on GB300: the same
// prefetch from every CTA is slower than none -- hundreds of requests for
// the same lines queue at one L2 slice ahead of the rows' own loads.)
__device__ __forceinline__ void prefetch_params_l2(const void* p, size_t bytes) {
    if (blockIdx.x != 0) return;
    const char* c = static_cast<const char*>(p);
    for (size_t off = static_cast<size_t>(threadIdx.x) * 128; off < bytes;
         off += static_cast<size_t>(blockDim.x) * 128)
        prefetch_l2(c + off);
}

template <typename T> struct Raw8;
template <> struct Raw8<__half> { uint4 v; };
template <> struct Raw8<float> { float4 a, b; };

// Plain C++ accesses: the compiler schedules them freely but never moves them
// across the barrier/wait instructions, whose asm carries a memory clobber.
__device__ __forceinline__ uint4 ld16(const void* p) { return *reinterpret_cast<const uint4*>(p); }
__device__ __forceinline__ void st16(void* p, uint4 v) { *reinterpret_cast<uint4*>(p) = v; }

__device__ __forceinline__ uint4 f2u4(float4 f) {
    return make_uint4(__float_as_uint(f.x), __float_as_uint(f.y), __float_as_uint(f.z),
                      __float_as_uint(f.w));
}
__device__ __forceinline__ float4 u2f4(uint4 u) {
    return make_float4(__uint_as_float(u.x), __uint_as_float(u.y), __uint_as_float(u.z),
                       __uint_as_float(u.w));
}

template <typename T> __device__ __forceinline__ Raw8<T> load8(const T* p);
template <> __device__ __forceinline__ Raw8<__half> load8<__half>(const __half* p) {
    return Raw8<__half>{ld16(p)};
}
template <> __device__ __forceinline__ Raw8<float> load8<float>(const float* p) {
    return Raw8<float>{u2f4(ld16(p)), u2f4(ld16(p + 4))};
}

template <typename T> __device__ __forceinline__ void store8(T* p, const Raw8<T>& r);
template <> __device__ __forceinline__ void store8<__half>(__half* p, const Raw8<__half>& r) {
    st16(p, r.v);
}
template <> __device__ __forceinline__ void store8<float>(float* p, const Raw8<float>& r) {
    st16(p, f2u4(r.a));
    st16(p + 4, f2u4(r.b));
}

__device__ __forceinline__ float2 h2f(uint32_t u) {
    __half2 h = *reinterpret_cast<__half2*>(&u);
    return __half22float2(h);
}
__device__ __forceinline__ uint32_t f2h(float a, float b) {
    __half2 h = __floats2half2_rn(a, b);  // round to nearest even
    return *reinterpret_cast<uint32_t*>(&h);
}

__device__ __forceinline__ void unpack(const Raw8<__half>& r, float (&f)[8]) {
    float2 t;
    t = h2f(r.v.x); f[0] = t.x; f[1] = t.y;
    t = h2f(r.v.y); f[2] = t.x; f[3] = t.y;
    t = h2f(r.v.z); f[4] = t.x; f[5] = t.y;
    t = h2f(r.v.w); f[6] = t.x; f[7] = t.y;
}
__device__ __forceinline__ void unpack(const Raw8<float>& r, float (&f)[8]) {
    f[0] = r.a.x; f[1] = r.a.y; f[2] = r.a.z; f[3] = r.a.w;
    f[4] = r.b.x; f[5] = r.b.y; f[6] = r.b.z; f[7] = r.b.w;
}
template <typename T> __device__ __forceinline__ Raw8<T> pack(const float (&f)[8]);
template <> __device__ __forceinline__ Raw8<__half> pack<__half>(const float (&f)[8]) {
    return Raw8<__half>{make_uint4(f2h(f[0], f[1]), f2h(f[2], f[3]), f2h(f[4], f[5]),
                                   f2h(f[6], f[7]))};
}
template <> __device__ __forceinline__ Raw8<float> pack<float>(const float (&f)[8]) {
    return Raw8<float>{make_float4(f[0], f[1], f[2], f[3]), make_float4(f[4], f[5], f[6], f[7])};
}

// Maximum of the 8 elements of a vector (exact: max never rounds).  FP16 takes
// the packed half2 maximum.
__device__ __forceinline__ float vmax8(const Raw8<__half>& r) {
    const __half2 a = __hmax2(*reinterpret_cast<const __half2*>(&r.v.x),
                              *reinterpret_cast<const __half2*>(&r.v.y));
    const __half2 b = __hmax2(*reinterpret_cast<const __half2*>(&r.v.z),
                              *reinterpret_cast<const __half2*>(&r.v.w));
    const __half2 c = __hmax2(a, b);
    return fmaxf(__low2float(c), __high2float(c));
}
__device__ __forceinline__ float vmax8(const Raw8<float>& r) {
    return fmaxf(fmaxf(fmaxf(r.a.x, r.a.y), fmaxf(r.a.z, r.a.w)),
                 fmaxf(fmaxf(r.b.x, r.b.y), fmaxf(r.b.z, r.b.w)));
}

// ---------------------------------------------------------------------------
// Mixed-precision arithmetic on FP16 operands with FP32 results (PTX
// fma.rn.f32.f16 and sub.rn.f32.f16, sm_100 and later), which saves the
// separate conversions.  FP16 values convert to FP32 exactly and a product of
// two FP16 values is exact in FP32, so each result equals the FP32 operation
// on the converted operands, rounded once: the same bits as convert-then-
// compute.
// ---------------------------------------------------------------------------
// acc + a[0]*b[0] + ... + a[7]*b[7], accumulated in that order.
__device__ __forceinline__ float dot8_acc(const Raw8<__half>& a, const Raw8<__half>& b,
                                          float acc) {
    const uint32_t aw[4] = {a.v.x, a.v.y, a.v.z, a.v.w};
    const uint32_t bw[4] = {b.v.x, b.v.y, b.v.z, b.v.w};
#pragma unroll
    for (int k = 0; k < 4; ++k)
        asm("{\n\t.reg .f16 al, ah, bl, bh;\n\t"
            "mov.b32 {al, ah}, %1;\n\tmov.b32 {bl, bh}, %2;\n\t"
            "fma.rn.f32.f16 %0, al, bl, %0;\n\tfma.rn.f32.f16 %0, ah, bh, %0;\n\t}"
            : "+f"(acc)
            : "r"(aw[k]), "r"(bw[k]));
    return acc;
}
__device__ __forceinline__ float dot8_acc(const Raw8<float>& a, const Raw8<float>& b,
                                          float acc) {
    float x[8], y[8];
    unpack(a, x);
    unpack(b, y);
#pragma unroll
    for (int j = 0; j < 8; ++j) acc = fmaf(x[j], y[j], acc);
    return acc;
}
// t[j] = a[j] + c[j].
__device__ __forceinline__ void add8(const Raw8<__half>& a, const float (&c)[8], float (&t)[8]) {
    const uint32_t aw[4] = {a.v.x, a.v.y, a.v.z, a.v.w};
#pragma unroll
    for (int k = 0; k < 4; ++k)
        asm("{\n\t.reg .f16 al, ah;\n\tmov.b32 {al, ah}, %2;\n\t"
            "add.rn.f32.f16 %0, al, %3;\n\tadd.rn.f32.f16 %1, ah, %4;\n\t}"
            : "=f"(t[2 * k]), "=f"(t[2 * k + 1])
            : "r"(aw[k]), "f"(c[2 * k]), "f"(c[2 * k + 1]));
}
__device__ __forceinline__ void add8(const Raw8<float>& a, const float (&c)[8], float (&t)[8]) {
    unpack(a, t);
#pragma unroll
    for (int j = 0; j < 8; ++j) t[j] += c[j];
}
// t[j] = a[j] - c.
__device__ __forceinline__ void sub8(const Raw8<__half>& a, float c, float (&t)[8]) {
    const uint32_t aw[4] = {a.v.x, a.v.y, a.v.z, a.v.w};
#pragma unroll
    for (int k = 0; k < 4; ++k)
        asm("{\n\t.reg .f16 al, ah;\n\tmov.b32 {al, ah}, %2;\n\t"
            "sub.rn.f32.f16 %0, al, %3;\n\tsub.rn.f32.f16 %1, ah, %3;\n\t}"
            : "=f"(t[2 * k]), "=f"(t[2 * k + 1])
            : "r"(aw[k]), "f"(c));
}
__device__ __forceinline__ void sub8(const Raw8<float>& a, float c, float (&t)[8]) {
    unpack(a, t);
#pragma unroll
    for (int j = 0; j < 8; ++j) t[j] -= c;
}

// t[j] = a[j] * b[j], exact for FP16 operands (their product fits FP32), as
// fma.rn.f32.f16 with a zero addend.
__device__ __forceinline__ void mul8(const Raw8<__half>& a, const Raw8<__half>& b, float (&t)[8]) {
    const uint32_t aw[4] = {a.v.x, a.v.y, a.v.z, a.v.w};
    const uint32_t bw[4] = {b.v.x, b.v.y, b.v.z, b.v.w};
#pragma unroll
    for (int k = 0; k < 4; ++k)
        asm("{\n\t.reg .f16 al, ah, bl, bh;\n\t"
            "mov.b32 {al, ah}, %2;\n\tmov.b32 {bl, bh}, %3;\n\t"
            "fma.rn.f32.f16 %0, al, bl, 0f00000000;\n\tfma.rn.f32.f16 %1, ah, bh, 0f00000000;\n\t}"
            : "=f"(t[2 * k]), "=f"(t[2 * k + 1])
            : "r"(aw[k]), "r"(bw[k]));
}
__device__ __forceinline__ void mul8(const Raw8<float>& a, const Raw8<float>& b, float (&t)[8]) {
    float x[8], y[8];
    unpack(a, x);
    unpack(b, y);
#pragma unroll
    for (int j = 0; j < 8; ++j) t[j] = x[j] * y[j];
}

// ---------------------------------------------------------------------------
// Packed FP32 pairs (PTX add/mul/fma .rn.f32x2, sm_100 and later): one
// instruction does the same operation on two lanes, each rounded as the scalar
// operation would be.
// ---------------------------------------------------------------------------
__device__ __forceinline__ float2 fma2(float2 a, float2 b, float2 c) {
    float2 d;
    asm("{\n\t.reg .b64 ra, rb, rc, rd;\n\t"
        "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\tmov.b64 rc, {%6, %7};\n\t"
        "fma.rn.f32x2 rd, ra, rb, rc;\n\tmov.b64 {%0, %1}, rd;\n\t}"
        : "=f"(d.x), "=f"(d.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
    return d;
}
__device__ __forceinline__ float2 mul2(float2 a, float2 b) {
    float2 d;
    asm("{\n\t.reg .b64 ra, rb, rd;\n\t"
        "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
        "mul.rn.f32x2 rd, ra, rb;\n\tmov.b64 {%0, %1}, rd;\n\t}"
        : "=f"(d.x), "=f"(d.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
    return d;
}
__device__ __forceinline__ float2 add2(float2 a, float2 b) {
    float2 d;
    asm("{\n\t.reg .b64 ra, rb, rd;\n\t"
        "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
        "add.rn.f32x2 rd, ra, rb;\n\tmov.b64 {%0, %1}, rd;\n\t}"
        : "=f"(d.x), "=f"(d.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
    return d;
}

template <typename T> __device__ __forceinline__ Raw8<T> zero8();
template <> __device__ __forceinline__ Raw8<__half> zero8<__half>() {
    return Raw8<__half>{make_uint4(0, 0, 0, 0)};
}
template <> __device__ __forceinline__ Raw8<float> zero8<float>() {
    return Raw8<float>{make_float4(0.f, 0.f, 0.f, 0.f), make_float4(0.f, 0.f, 0.f, 0.f)};
}

template <typename T> __device__ __forceinline__ void load8f(const T* p, float (&f)[8]) {
    unpack(load8<T>(p), f);
}
template <typename T> __device__ __forceinline__ void store8f(T* p, const float (&f)[8]) {
    store8<T>(p, pack<T>(f));
}

// ---------------------------------------------------------------------------
// Philox-4x32-10 (Salmon, Moraes, Dror, Shaw, SC'11).  One call maps a
// 128-bit counter and a 64-bit key to 128 random bits.  Round: with the two
// 32x32->64 products M0*c0 and M1*c2,
//   c <- (hi(M1*c2) ^ c1 ^ k0, lo(M1*c2), hi(M0*c0) ^ c3 ^ k1, lo(M0*c0)),
// and the key is bumped by the Weyl constants between rounds.
// ---------------------------------------------------------------------------
struct PhiloxKey {
    uint32_t k0, k1;
};

// The ten round keys of one 64-bit key (key + r * Weyl constant).  Computed
// once per thread from kernel arguments, so they are the same in every thread
// and every call.
struct PhiloxSchedule {
    uint32_t k0[10], k1[10];
};

__host__ __device__ __forceinline__ PhiloxSchedule philox_schedule(PhiloxKey key) {
    constexpr uint32_t W0 = 0x9E3779B9u, W1 = 0xBB67AE85u;
    PhiloxSchedule s;
#pragma unroll
    for (int r = 0; r < 10; ++r) {
        s.k0[r] = key.k0 + static_cast<uint32_t>(r) * W0;
        s.k1[r] = key.k1 + static_cast<uint32_t>(r) * W1;
    }
    return s;
}

__device__ __forceinline__ uint4 philox4x32_10(uint4 c, const PhiloxSchedule& ks) {
    constexpr uint32_t M0 = 0xD2511F53u, M1 = 0xCD9E8D57u;
#pragma unroll
    for (int round = 0; round < 10; ++round) {
        const uint64_t p0 = static_cast<uint64_t>(M0) * c.x;
        const uint64_t p1 = static_cast<uint64_t>(M1) * c.z;
        c = make_uint4(static_cast<uint32_t>(p1 >> 32) ^ c.y ^ ks.k0[round],
                       static_cast<uint32_t>(p1),
                       static_cast<uint32_t>(p0 >> 32) ^ c.w ^ ks.k1[round],
                       static_cast<uint32_t>(p0));
    }
    return c;
}

// Dropout keep bits of the 8 consecutive elements starting at flat index i
// (i a multiple of 4), given as its counter block b = i >> 2 = (lo, hi):
// element i+j draws word j&3 of counter block b+(j>>2).  Bit j of the result is
// set iff element i+j is kept (word >= thr).
__device__ __forceinline__ uint32_t keep_bits8_blk(uint32_t lo, uint32_t hi, uint32_t thr,
                                                   const PhiloxSchedule& ks, uint32_t off_lo,
                                                   uint32_t off_hi) {
    const uint4 a = philox4x32_10(make_uint4(lo, hi, off_lo, off_hi), ks);
    const uint32_t lo1 = lo + 1u;
    const uint4 b = philox4x32_10(make_uint4(lo1, hi + (lo1 == 0u ? 1u : 0u), off_lo, off_hi), ks);
    return (a.x >= thr ? 1u : 0u) | (a.y >= thr ? 2u : 0u) | (a.z >= thr ? 4u : 0u) |
           (a.w >= thr ? 8u : 0u) | (b.x >= thr ? 16u : 0u) | (b.y >= thr ? 32u : 0u) |
           (b.z >= thr ? 64u : 0u) | (b.w >= thr ? 128u : 0u);
}
__device__ __forceinline__ uint32_t keep_bits8(uint64_t i, uint32_t thr, const PhiloxSchedule& ks,
                                               uint32_t off_lo, uint32_t off_hi) {
    const uint64_t blk = i >> 2;
    return keep_bits8_blk(static_cast<uint32_t>(blk), static_cast<uint32_t>(blk >> 32), thr, ks,
                          off_lo, off_hi);
}

// e^x as 2^(x * log2 e), with 2^y from the PTX ex2.approx instruction (relative
// error about 2^-22; results below 2^-126 flush to zero).
__device__ __forceinline__ float exp2_approx(float y) {
    float r;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(y));
    return r;
}

// ---------------------------------------------------------------------------
// Reductions over groups of W consecutive lanes (W a power of two <= 32).
// ---------------------------------------------------------------------------
template <int W> __device__ __forceinline__ float group_sum(float v) {
#pragma unroll
    for (int o = W / 2; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}
template <int W> __device__ __forceinline__ float group_max(float v) {
#pragma unroll
    for (int o = W / 2; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}
// Both members of the pair reduced with one exchange per step: the single
// synchronisation point of the one-pass statistics.
template <int W> __device__ __forceinline__ float2 group_sum2(float2 v) {
#pragma unroll
    for (int o = W / 2; o > 0; o >>= 1) {
        v.x += __shfl_xor_sync(0xffffffffu, v.x, o);
        v.y += __shfl_xor_sync(0xffffffffu, v.y, o);
    }
    return v;
}

}  // namespace ls

namespace ls {

// ---------------------------------------------------------------------------
// Programmatic dependent launch.  Every kernel is launched with programmatic
// stream serialisation, so the next kernel on the stream may be scheduled
// while this one drains.  A kernel therefore waits for its predecessor's
// completion (and memory flush) before its first global access, then lets its
// own successor launch.  Launched without the attribute, both are no-ops.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void pdl_enter() {
    pdl_wait();
    pdl_trigger();
}

// Lets `kernel` use up to the device's opt-in maximum of dynamic shared
// memory.  The attribute is set once per kernel and device (`done` is the
// caller's per-kernel table, indexed by device), not on every launch: setting
// it is a driver call that stream capture for profiling ranges does not
// accept, and it costs host time on every eager call.
constexpr int kMaxDevices = 64;
template <typename K>
inline cudaError_t allow_max_dynamic_smem(K kernel, int (&done)[kMaxDevices]) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < kMaxDevices && __atomic_load_n(&done[dev], __ATOMIC_ACQUIRE)) return e;
    int optin = 0;
    e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    // The kernel's own static shared memory counts against the same limit.
    cudaFuncAttributes fa;
    if (e == cudaSuccess) e = cudaFuncGetAttributes(&fa, kernel);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 optin - static_cast<int>(fa.sharedSizeBytes));
    if (e == cudaSuccess && dev >= 0 && dev < kMaxDevices)
        __atomic_store_n(&done[dev], 1, __ATOMIC_RELEASE);
    return e;
}

template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                              cudaStream_t stream, Args... args) {
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

}  // namespace ls

namespace ls {

// ---------------------------------------------------------------------------
// Bulk copies (TMA, non-tensor form) into shared memory, completed on an
// mbarrier.  Both addresses must be 16-byte aligned and the size a multiple
// of 16 bytes; every caller copies whole 16-byte vectors of 16-byte-aligned
// rows.
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
                 : "memory");
}
__device__ __forceinline__ void mbar_init_fence() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
// One arrival that also expects `bytes` of transactions (0 completes the phase).
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
                 "r"(bytes)
                 : "memory");
}
// Waits for the phase with the given parity to complete; the thread sleeps
// (up to kWaitHintNs) instead of spinning.  Returns whether it completed.
constexpr uint32_t kWaitHintNs = 2000;
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(smem_u32(bar)), "r"(parity), "r"(kWaitHintNs)
        : "memory");
    return done != 0;
}
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes,
                                         uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
            "r"(smem_u32(dst)),
        "l"(src), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}
// Orders this thread's earlier generic-proxy accesses to shared memory before
// later async-proxy (bulk copy) accesses to it.
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ uint4 lds16(const void* p) { return *reinterpret_cast<const uint4*>(p); }
template <typename T> __device__ __forceinline__ Raw8<T> load8_smem(const T* p);
template <> __device__ __forceinline__ Raw8<__half> load8_smem<__half>(const __half* p) {
    return Raw8<__half>{lds16(p)};
}
template <> __device__ __forceinline__ Raw8<float> load8_smem<float>(const float* p) {
    return Raw8<float>{u2f4(lds16(p)), u2f4(lds16(p + 4))};
}

// Device-side failure flags of the kernels in one translation unit (each
// unit that includes this header has its own word; ls_check_device_errors
// collects them).  Bit 0: a bulk-copy wait ran out of time.
constexpr unsigned int kDevErrWaitTimeout = 1u;
namespace {
__device__ unsigned int g_device_error = 0;
}
__device__ __forceinline__ void flag_device_error(unsigned int bits) {
    atomicOr(&g_device_error, bits);
}
// Host: read and clear this unit's flags (synchronous copy).
static inline cudaError_t take_device_error_word(unsigned int* out) {
    unsigned int v = 0;
    cudaError_t e = cudaMemcpyFromSymbol(&v, g_device_error, sizeof(v));
    if (e == cudaSuccess && v != 0) {
        const unsigned int zero = 0;
        e = cudaMemcpyToSymbol(g_device_error, &zero, sizeof(zero));
    }
    *out = v;
    return e;
}

// Polls of an mbarrier before a wait is declared failed.  Each poll sleeps up
// to kWaitHintNs, so a wait is bounded to about a second, and even polls that
// return at once span milliseconds -- far beyond any bulk copy's latency.
constexpr uint32_t kWaitPolls = 1u << 19;

// An S-stage ring of shared-memory buffers owned by one warp.  Lane 0 arms a
// stage and issues its bulk copies; all lanes wait on the stage's barrier; the
// k-th use of stage k % S completes phase (k / S) & 1.
template <int S>
struct WarpRing {
    uint64_t* bar;
    unsigned char* buf;
    uint32_t stage_bytes;
    uint32_t pending;  // bit s: a copy into stage s was issued and not yet waited for

    __device__ __forceinline__ void init(uint64_t* bars, unsigned char* data, uint32_t sb) {
        bar = bars;
        buf = data;
        stage_bytes = sb;
        pending = 0;
        if ((threadIdx.x & 31) == 0) {
#pragma unroll
            for (int s = 0; s < S; ++s) mbar_init(bar + s, 1);
            mbar_init_fence();
        }
        __syncwarp();
    }
    __device__ __forceinline__ unsigned char* stage(int s) const { return buf + s * stage_bytes; }

    // Arm stage s for n0 + n1 bytes: n0 from src0 to the stage start, n1 from
    // src1 to the stage at byte offset off1.  n0 = n1 = 0 completes the phase
    // at once (the row has nothing to read).  Called by every lane.
    // The caller's earlier reads of stage s must have completed (their values
    // used) and the warp synchronised before it re-arms the stage.
    __device__ __forceinline__ void issue(int s, const void* src0, uint32_t n0, const void* src1,
                                          uint32_t n1, uint32_t off1) {
        if ((threadIdx.x & 31) == 0) {
            mbar_arrive_expect_tx(bar + s, n0 + n1);
            if (n0) bulk_g2s(stage(s), src0, n0, bar + s);
            if (n1) bulk_g2s(stage(s) + off1, src1, n1, bar + s);
        }
        pending |= 1u << s;
    }

    // Bounded wait for stage s; false (and the failure flagged) on timeout.
    __device__ __forceinline__ bool wait(int s, uint32_t parity) {
        for (uint32_t i = 0; i < kWaitPolls; ++i) {
            if (mbar_try_wait(bar + s, parity)) {
                pending &= ~(1u << s);
                return true;
            }
        }
        flag_device_error(kDevErrWaitTimeout);
        return false;
    }

    // After a failed wait: wait (bounded again) for every copy still in flight
    // into this warp's stages, so none lands after the CTA has exited.
    __device__ __forceinline__ void drain(const uint32_t (&parity_of)[S]) {
#pragma unroll
        for (int s = 0; s < S; ++s) {
            if (pending & (1u << s)) {
                for (uint32_t i = 0; i < kWaitPolls; ++i)
                    if (mbar_try_wait(bar + s, parity_of[s])) break;
            }
        }
        pending = 0;
    }
};

}  // namespace ls

