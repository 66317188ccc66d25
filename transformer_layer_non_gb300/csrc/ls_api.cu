// ls_api.cu -- the C ABI declared in include/ls_ops.h.  Every entry point
// validates its arguments on the host (returning before anything is enqueued
// on an error), then hands the call to a launcher in ls_internal.h.  Nothing
// here allocates device memory or synchronises; per-thread state is the
// message of the last error and, once a reduction stream is set, that
// stream's events and the workspaces its pending reductions read.
#include <math.h>
#include <stdarg.h>
#include <stdio.h>
#include <string.h>

#include <algorithm>
#include <atomic>

#include "../../include/ls_ops.h"
#include "ls_internal.h"

namespace {

thread_local char g_last_error[512] = "";

ls_status fail(ls_status st, const char* fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_last_error, sizeof(g_last_error), fmt, ap);
    va_end(ap);
    return st;
}

ls_status ok() {
    g_last_error[0] = '\0';
    return LS_OK;
}

ls_status from_cuda(cudaError_t e, const char* what) {
    if (e == cudaSuccess) return ok();
    return fail(LS_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// ----------------------------------------------------------------------------
// Column reductions on a second stream.  The backward entries with a bias,
// gamma or beta gradient run a main kernel (dx and per-tile partial sums in
// the workspace) and then the fixed-order reduction of the partial sums.
// Only the gradient depends on the reduction, so with a reduction stream set
// the reduction is forked onto it (an event recorded after the main kernel)
// and the caller's next kernel follows the main kernel directly.  Each fork
// remembers the workspace it reads and an event recorded after it; a later
// backward call whose workspace overlaps a pending one first makes its own
// stream wait for that event, so sharing one workspace stays correct (and
// merely does not overlap).  ls_join_reductions ends all of it.
// ----------------------------------------------------------------------------
constexpr int kMaxPendingReductions = 16;

struct PendingReduction {
    uintptr_t lo, hi;  // workspace bytes [lo, hi) the reduction reads
    int ev;            // index into ReductionState::done
};

struct ReductionState {
    cudaStream_t side = nullptr;
    bool active = false;  // a reduction stream is set
    int device = -1;      // the device the events belong to
    cudaEvent_t fork = nullptr, join = nullptr;
    cudaEvent_t done[kMaxPendingReductions] = {};
    bool used[kMaxPendingReductions] = {};
    PendingReduction pend[kMaxPendingReductions];
    int npend = 0;
    bool forked = false;  // a fork since the last join
};

thread_local ReductionState t_red;

cudaError_t make_event(cudaEvent_t* ev) {
    if (*ev) return cudaSuccess;
    return cudaEventCreateWithFlags(ev, cudaEventDisableTiming);
}

// Drops pending entry i (its event slot becomes free).
void drop_pending(int i) {
    ReductionState& r = t_red;
    r.used[r.pend[i].ev] = false;
    r.pend[i] = r.pend[r.npend - 1];
    --r.npend;
}

// Before a backward call writes partial sums into [ws, ws + bytes) on s:
// order s after every pending reduction that reads an overlapping range.
cudaError_t guard_workspace(cudaStream_t s, const void* ws, size_t bytes) {
    ReductionState& r = t_red;
    if (r.npend == 0 || !ws || bytes == 0) return cudaSuccess;
    const uintptr_t lo = reinterpret_cast<uintptr_t>(ws), hi = lo + bytes;
    for (int i = 0; i < r.npend; ++i)
        if (lo < r.pend[i].hi && r.pend[i].lo < hi) {
            const cudaError_t e = cudaStreamWaitEvent(s, r.done[r.pend[i].ev], 0);
            if (e != cudaSuccess) return e;
        }
    return cudaSuccess;
}

// Launches a column reduction fn(stream) that reads [ws, ws + bytes): on s,
// or forked onto the reduction stream after s's work so far.
template <typename F>
cudaError_t launch_reduction(cudaStream_t s, const void* ws, size_t bytes, F fn,
                             bool inline_only = false) {
    ReductionState& r = t_red;
    if (!r.active || inline_only) return fn(s);
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev != r.device) return cudaErrorInvalidResourceHandle;  // events of another device
    if (r.npend == kMaxPendingReductions) {
        // Full: order s after the oldest pending reduction and forget it.
        e = cudaStreamWaitEvent(s, r.done[r.pend[0].ev], 0);
        if (e != cudaSuccess) return e;
        drop_pending(0);
    }
    int slot = 0;
    while (r.used[slot]) ++slot;
    e = cudaEventRecord(r.fork, s);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(r.side, r.fork, 0);
    if (e == cudaSuccess) e = fn(r.side);
    if (e == cudaSuccess) e = cudaEventRecord(r.done[slot], r.side);
    if (e != cudaSuccess) return e;
    const uintptr_t lo = reinterpret_cast<uintptr_t>(ws), hi = lo + bytes;
    // Pending reductions inside this range are implied by the new one (the
    // reduction stream runs in order).
    for (int i = 0; i < r.npend;)
        if (lo <= r.pend[i].lo && r.pend[i].hi <= hi)
            drop_pending(i);
        else
            ++i;
    r.used[slot] = true;
    r.pend[r.npend++] = PendingReduction{lo, hi, slot};
    r.forked = true;
    return cudaSuccess;
}

// A byte range [p, p+n) of one argument.
struct Span {
    const char* name;
    const void* p;
    size_t n;
};

bool overlaps(const Span& a, const Span& b) {
    if (!a.p || !b.p || a.n == 0 || b.n == 0) return false;
    const uintptr_t a0 = reinterpret_cast<uintptr_t>(a.p), b0 = reinterpret_cast<uintptr_t>(b.p);
    return a0 < b0 + b.n && b0 < a0 + a.n;
}

// Outputs may coincide exactly with an input of the same size (in place);
// every other overlap involving an output is an error.
ls_status check_overlaps(const Span* outs, int nout, const Span* ins, int nin) {
    for (int i = 0; i < nout; ++i) {
        for (int j = i + 1; j < nout; ++j)
            if (overlaps(outs[i], outs[j]))
                return fail(LS_ERR_INVALID_ARGUMENT, "outputs %s and %s overlap", outs[i].name,
                            outs[j].name);
        for (int j = 0; j < nin; ++j) {
            if (!overlaps(outs[i], ins[j])) continue;
            if (outs[i].p == ins[j].p && outs[i].n == ins[j].n) continue;  // exact alias
            return fail(LS_ERR_INVALID_ARGUMENT, "output %s partially overlaps input %s",
                        outs[i].name, ins[j].name);
        }
    }
    return LS_OK;
}

ls_status check_dtype(ls_dtype dt, ls::DType* out) {
    if (dt == LS_F16) { *out = ls::DType::F16; return LS_OK; }
    if (dt == LS_F32) { *out = ls::DType::F32; return LS_OK; }
    return fail(LS_ERR_INVALID_ARGUMENT, "unknown dtype %d", static_cast<int>(dt));
}

size_t elem_size(ls::DType dt) { return dt == ls::DType::F16 ? 2 : 4; }

// Common checks of a [rows, cols] activation.
ls_status check_shape(int64_t rows, int64_t cols, int64_t max_cols) {
    if (rows < 0) return fail(LS_ERR_INVALID_ARGUMENT, "rows = %lld < 0", (long long)rows);
    if (cols <= 0) return fail(LS_ERR_INVALID_ARGUMENT, "cols = %lld <= 0", (long long)cols);
    if (cols % 8 != 0)
        return fail(LS_ERR_MISALIGNED, "cols = %lld is not a multiple of 8", (long long)cols);
    if (cols > max_cols)
        return fail(LS_ERR_UNSUPPORTED_SHAPE, "cols = %lld exceeds %lld", (long long)cols,
                    (long long)max_cols);
    // Keep every flat element index below 2^62 and every grid dimension legal.
    if (rows > (int64_t{1} << 40) || rows * cols > (int64_t{1} << 46))
        return fail(LS_ERR_UNSUPPORTED_SHAPE, "too many elements (%lld x %lld)", (long long)rows,
                    (long long)cols);
    return LS_OK;
}

ls_status check_ptr(const void* p, const char* name, bool required) {
    if (!p) {
        if (required) return fail(LS_ERR_INVALID_ARGUMENT, "%s is NULL", name);
        return LS_OK;
    }
    if (!aligned16(p)) return fail(LS_ERR_MISALIGNED, "%s is not 16-byte aligned", name);
    return LS_OK;
}

ls_status check_p(float p, ls::DropoutRng* rng, uint64_t seed, uint64_t offset) {
    if (!(p >= 0.f && p < 1.f))
        return fail(LS_ERR_INVALID_ARGUMENT, "dropout probability p = %g is not in [0, 1)",
                    static_cast<double>(p));
    double t = floor(static_cast<double>(p) * 4294967296.0);
    if (t > 4294967295.0) t = 4294967295.0;
    rng->thr = static_cast<uint32_t>(t);
    rng->scale = 1.0f / (1.0f - p);
    rng->seed = seed;
    rng->offset = offset;
    return LS_OK;
}

size_t mask_bytes(int64_t rows, int64_t cols) {
    return static_cast<size_t>((rows * cols + 31) / 32) * 4;
}

// Dropout ops accept any cols % 8 == 0 whose vector count fits a grid row.
constexpr int64_t kMaxDropoutCols = int64_t{1} << 22;

#define LS_TRY(expr)                         \
    do {                                     \
        ls_status _st = (expr);              \
        if (_st != LS_OK) return _st;        \
    } while (0)

}  // namespace

int ls::sm_count() {
    static std::atomic<int> cache[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return 1;
    if (dev >= 64) {
        int n = 0;
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
        return n > 0 ? n : 1;
    }
    int n = cache[dev].load(std::memory_order_relaxed);
    if (n > 0) return n;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
        n = 1;
    cache[dev].store(n, std::memory_order_relaxed);
    return n;
}

void ls::set_last_error_message(const char* fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_last_error, sizeof(g_last_error), fmt, ap);
    va_end(ap);
}

// The library is built with hidden visibility; only the C ABI is exported.
#pragma GCC visibility push(default)
extern "C" {

const char* ls_status_string(ls_status status) {
    switch (status) {
        case LS_OK: return "LS_OK";
        case LS_ERR_INVALID_ARGUMENT: return "LS_ERR_INVALID_ARGUMENT";
        case LS_ERR_MISALIGNED: return "LS_ERR_MISALIGNED";
        case LS_ERR_UNSUPPORTED_SHAPE: return "LS_ERR_UNSUPPORTED_SHAPE";
        case LS_ERR_WORKSPACE_TOO_SMALL: return "LS_ERR_WORKSPACE_TOO_SMALL";
        case LS_ERR_CUDA: return "LS_ERR_CUDA";
    }
    return "unknown ls_status";
}

const char* ls_last_error(void) { return g_last_error; }

int ls_version(void) { return 10000; }

ls_status ls_check_device_errors(uint32_t* flags) {
    if (!flags) return fail(LS_ERR_INVALID_ARGUMENT, "flags is NULL");
    *flags = 0;
    cudaError_t e = cudaDeviceSynchronize();
    if (e != cudaSuccess) return from_cuda(e, "ls_check_device_errors: synchronise");
    unsigned int a = 0, b = 0, c = 0;
    e = ls::softmax_take_device_error(&a);
    if (e == cudaSuccess) e = ls::layernorm_take_device_error(&b);
    if (e == cudaSuccess) e = ls::dropout_take_device_error(&c);
    if (e != cudaSuccess) return from_cuda(e, "ls_check_device_errors: read flags");
    *flags = a | b | c;
    return ok();
}

ls_status ls_selftest_wait_timeout(uint32_t polls, void* stream) {
    if (polls == 0 || polls > (1u << 19))
        return fail(LS_ERR_INVALID_ARGUMENT, "polls = %u is not in [1, 2^19]", polls);
    return from_cuda(ls::launch_wait_timeout_selftest(polls, static_cast<cudaStream_t>(stream)),
                     "ls_selftest_wait_timeout launch");
}

ls_status ls_set_reduction_stream(void* reduce_stream) {
    ReductionState& r = t_red;
    if (r.forked)
        return fail(LS_ERR_INVALID_ARGUMENT,
                    "ls_set_reduction_stream: reductions are pending on the previous reduction "
                    "stream; call ls_join_reductions first");
    if (!reduce_stream) {
        r.active = false;
        r.side = nullptr;
        return ok();
    }
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess && r.device >= 0 && dev != r.device) {
        // Events of another device: release them and start over.
        cudaEventDestroy(r.fork);
        cudaEventDestroy(r.join);
        for (cudaEvent_t& ev : r.done) {
            if (ev) cudaEventDestroy(ev);
            ev = nullptr;
        }
        r.fork = r.join = nullptr;
    }
    if (e == cudaSuccess) e = make_event(&r.fork);
    if (e == cudaSuccess) e = make_event(&r.join);
    for (int i = 0; e == cudaSuccess && i < kMaxPendingReductions; ++i) e = make_event(&r.done[i]);
    if (e != cudaSuccess) return from_cuda(e, "ls_set_reduction_stream");
    r.device = dev;
    r.side = static_cast<cudaStream_t>(reduce_stream);
    r.active = true;
    return ok();
}

ls_status ls_join_reductions(void* stream) {
    ReductionState& r = t_red;
    if (!r.forked) return ok();
    cudaError_t e = cudaEventRecord(r.join, r.side);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(static_cast<cudaStream_t>(stream), r.join, 0);
    if (e != cudaSuccess) return from_cuda(e, "ls_join_reductions");
    while (r.npend > 0) drop_pending(r.npend - 1);
    r.forked = false;
    return ok();
}

size_t ls_colreduce_workspace_bytes(int64_t rows, int64_t cols) {
    if (rows <= 0 || cols <= 0 || cols % 8 != 0) return 0;
    const size_t a = ls::dropout_bwd_plan(rows, cols).bytes();
    const size_t b = cols <= ls::kMaxRowLen
                         ? std::max(ls::layernorm_bwd_plan(rows, cols, 2).bytes(),
                                    ls::layernorm_bwd_plan(rows, cols, 4).bytes())
                         : 0;
    return std::max(a, b);
}

ls_status ls_bias_dropout_residual_fwd(ls_dtype dtype, void* out, uint32_t* mask_bits,
                                       const void* x, const void* bias, const void* residual,
                                       int64_t rows, int64_t cols, float p, uint64_t seed,
                                       uint64_t offset, void* stream) {
    ls::DType dt;
    LS_TRY(check_dtype(dtype, &dt));
    LS_TRY(check_shape(rows, cols, kMaxDropoutCols));
    ls::DropoutRng rng;
    LS_TRY(check_p(p, &rng, seed, offset));
    if (rows == 0) return ok();
    LS_TRY(check_ptr(out, "out", true));
    LS_TRY(check_ptr(mask_bits, "mask_bits", false));
    LS_TRY(check_ptr(x, "x", true));
    LS_TRY(check_ptr(bias, "bias", true));
    LS_TRY(check_ptr(residual, "residual", true));
    const size_t nb = static_cast<size_t>(rows * cols) * elem_size(dt);
    const Span outs[] = {{"out", out, nb}, {"mask_bits", mask_bits, mask_bytes(rows, cols)}};
    const Span ins[] = {{"x", x, nb}, {"residual", residual, nb},
                        {"bias", bias, static_cast<size_t>(cols) * elem_size(dt)}};
    LS_TRY(check_overlaps(outs, 2, ins, 3));
    return from_cuda(ls::launch_dropout_fwd(dt, false, out, reinterpret_cast<uint8_t*>(mask_bits),
                                            x, bias, residual, rows, cols, rng,
                                            static_cast<cudaStream_t>(stream)),
                     "ls_bias_dropout_residual_fwd launch");
}

static ls_status dropout_bwd_common(const char* fn, ls_dtype dtype, void* dx, void* dbias,
                                    const void* dout, const uint32_t* mask_bits, bool regen_ok,
                                    int64_t rows, int64_t cols, float p, uint64_t seed,
                                    uint64_t offset, void* workspace, size_t workspace_bytes,
                                    void* stream) {
    ls::DType dt;
    LS_TRY(check_dtype(dtype, &dt));
    LS_TRY(check_shape(rows, cols, kMaxDropoutCols));
    ls::DropoutRng rng;
    LS_TRY(check_p(p, &rng, seed, offset));
    if (rows == 0) {
        // The bias gradient of an empty batch is zero.
        if (dbias) {
            LS_TRY(check_ptr(dbias, "dbias", true));
            return from_cuda(cudaMemsetAsync(dbias, 0, static_cast<size_t>(cols) * elem_size(dt),
                                             static_cast<cudaStream_t>(stream)),
                             fn);
        }
        return ok();
    }
    LS_TRY(check_ptr(dx, "dx", true));
    LS_TRY(check_ptr(dbias, "dbias", false));
    LS_TRY(check_ptr(dout, "dout", true));
    LS_TRY(check_ptr(mask_bits, "mask_bits", !regen_ok));
    const ls::ColReducePlan plan = ls::dropout_bwd_plan(rows, cols);
    if (dbias) {
        LS_TRY(check_ptr(workspace, "workspace", true));
        if (workspace_bytes < plan.bytes())
            return fail(LS_ERR_WORKSPACE_TOO_SMALL, "%s: workspace of %zu bytes, need %zu", fn,
                        workspace_bytes, plan.bytes());
    }
    const size_t nb = static_cast<size_t>(rows * cols) * elem_size(dt);
    const size_t bb = static_cast<size_t>(cols) * elem_size(dt);
    const Span outs[] = {{"dx", dx, nb}, {"dbias", dbias, bb},
                         {"workspace", dbias ? workspace : nullptr, plan.bytes()}};
    const Span ins[] = {{"dout", dout, nb}, {"mask_bits", mask_bits, mask_bytes(rows, cols)}};
    LS_TRY(check_overlaps(outs, 3, ins, 2));
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    float* partial = dbias ? static_cast<float*>(workspace) : nullptr;
    cudaError_t e = guard_workspace(s, partial, plan.bytes());
    if (e == cudaSuccess)
        e = ls::launch_dropout_bwd(dt, dx, partial, dout,
                                   reinterpret_cast<const uint8_t*>(mask_bits), rows, cols, rng,
                                   s);
    if (e == cudaSuccess && dbias)
        e = launch_reduction(s, partial, plan.bytes(), [&](cudaStream_t rs) {
            return ls::launch_colreduce(dt, dbias, nullptr, cols, partial, plan.parts, cols, rs);
        });
    return from_cuda(e, fn);
}

ls_status ls_bias_dropout_residual_bwd(ls_dtype dtype, void* dx, void* dbias, const void* dout,
                                       const uint32_t* mask_bits, int64_t rows, int64_t cols,
                                       float p, uint64_t seed, uint64_t offset, void* workspace,
                                       size_t workspace_bytes, void* stream) {
    return dropout_bwd_common("ls_bias_dropout_residual_bwd", dtype, dx, dbias, dout, mask_bits,
                              true, rows, cols, p, seed, offset, workspace, workspace_bytes,
                              stream);
}

ls_status ls_bias_relu_dropout_fwd(ls_dtype dtype, void* out, uint32_t* mask_bits, const void* x,
                                   const void* bias, int64_t rows, int64_t cols, float p,
                                   uint64_t seed, uint64_t offset, void* stream) {
    ls::DType dt;
    LS_TRY(check_dtype(dtype, &dt));
    LS_TRY(check_shape(rows, cols, kMaxDropoutCols));
    ls::DropoutRng rng;
    LS_TRY(check_p(p, &rng, seed, offset));
    if (rows == 0) return ok();
    LS_TRY(check_ptr(out, "out", true));
    LS_TRY(check_ptr(mask_bits, "mask_bits", true));
    LS_TRY(check_ptr(x, "x", true));
    LS_TRY(check_ptr(bias, "bias", true));
    const size_t nb = static_cast<size_t>(rows * cols) * elem_size(dt);
    const Span outs[] = {{"out", out, nb}, {"mask_bits", mask_bits, mask_bytes(rows, cols)}};
    const Span ins[] = {{"x", x, nb}, {"bias", bias, static_cast<size_t>(cols) * elem_size(dt)}};
    LS_TRY(check_overlaps(outs, 2, ins, 2));
    return from_cuda(ls::launch_dropout_fwd(dt, true, out, reinterpret_cast<uint8_t*>(mask_bits),
                                            x, bias, nullptr, rows, cols, rng,
                                            static_cast<cudaStream_t>(stream)),
                     "ls_bias_relu_dropout_fwd launch");
}

ls_status ls_bias_relu_dropout_bwd(ls_dtype dtype, void* dx, void* dbias, const void* dout,
                                   const uint32_t* mask_bits, int64_t rows, int64_t cols, float p,
                                   void* workspace, size_t workspace_bytes, void* stream) {
    return dropout_bwd_common("ls_bias_relu_dropout_bwd", dtype, dx, dbias, dout, mask_bits,
                              false, rows, cols, p, 0, 0, workspace, workspace_bytes, stream);
}

ls_status ls_layernorm_fwd(ls_dtype dtype, void* y, float* mean, float* rstd, const void* x,
                           const void* gamma, const void* beta, int64_t rows, int64_t cols,
                           float eps, void* stream) {
    ls::DType dt;
    LS_TRY(check_dtype(dtype, &dt));
    LS_TRY(check_shape(rows, cols, ls::kMaxRowLen));
    if (!(eps >= 0.f) || isinf(eps))
        return fail(LS_ERR_INVALID_ARGUMENT, "eps = %g must be finite and >= 0",
                    static_cast<double>(eps));
    if (rows == 0) return ok();
    LS_TRY(check_ptr(y, "y", true));
    LS_TRY(check_ptr(mean, "mean", false));
    LS_TRY(check_ptr(rstd, "rstd", false));
    LS_TRY(check_ptr(x, "x", true));
    LS_TRY(check_ptr(gamma, "gamma", true));
    LS_TRY(check_ptr(beta, "beta", true));
    const size_t nb = static_cast<size_t>(rows * cols) * elem_size(dt);
    const size_t pb = static_cast<size_t>(cols) * elem_size(dt);
    const size_t sb = static_cast<size_t>(rows) * sizeof(float);
    const Span outs[] = {{"y", y, nb}, {"mean", mean, sb}, {"rstd", rstd, sb}};
    const Span ins[] = {{"x", x, nb}, {"gamma", gamma, pb}, {"beta", beta, pb}};
    LS_TRY(check_overlaps(outs, 3, ins, 3));
    return from_cuda(ls::launch_layernorm_fwd(dt, y, mean, rstd, x, gamma, beta, rows, cols, eps,
                                              static_cast<cudaStream_t>(stream)),
                     "ls_layernorm_fwd launch");
}

ls_status ls_layernorm_bwd(ls_dtype dtype, void* dx, void* dgamma, void* dbeta, const void* dy,
                           const void* x, const void* gamma, const float* mean, const float* rstd,
                           int64_t rows, int64_t cols, void* workspace, size_t workspace_bytes,
                           void* stream) {
    return ls::layernorm_bwd_entry(dtype, dx, dgamma, dbeta, dy, x, gamma, mean, rstd, rows, cols,
                                   workspace, workspace_bytes, stream, false);
}

}  // extern "C"
#pragma GCC visibility pop

ls_status ls::layernorm_bwd_entry(ls_dtype dtype, void* dx, void* dgamma, void* dbeta,
                                  const void* dy, const void* x, const void* gamma,
                                  const float* mean, const float* rstd, int64_t rows,
                                  int64_t cols, void* workspace, size_t workspace_bytes,
                                  void* stream, bool inline_reduction) {
    ls::DType dt;
    LS_TRY(check_dtype(dtype, &dt));
    LS_TRY(check_shape(rows, cols, ls::kMaxRowLen));
    if ((dgamma == nullptr) != (dbeta == nullptr))
        return fail(LS_ERR_INVALID_ARGUMENT, "dgamma and dbeta must both be given or both NULL");
    const size_t pb = static_cast<size_t>(cols) * elem_size(dt);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (rows == 0) {
        if (dgamma) {
            LS_TRY(check_ptr(dgamma, "dgamma", true));
            LS_TRY(check_ptr(dbeta, "dbeta", true));
            cudaError_t e = cudaMemsetAsync(dgamma, 0, pb, s);
            if (e == cudaSuccess) e = cudaMemsetAsync(dbeta, 0, pb, s);
            return from_cuda(e, "ls_layernorm_bwd");
        }
        return ok();
    }
    LS_TRY(check_ptr(dx, "dx", true));
    LS_TRY(check_ptr(dgamma, "dgamma", false));
    LS_TRY(check_ptr(dbeta, "dbeta", false));
    LS_TRY(check_ptr(dy, "dy", true));
    LS_TRY(check_ptr(x, "x", true));
    LS_TRY(check_ptr(gamma, "gamma", true));
    LS_TRY(check_ptr(mean, "mean", true));
    LS_TRY(check_ptr(rstd, "rstd", true));
    const ls::ColReducePlan plan = ls::layernorm_bwd_plan(rows, cols, elem_size(dt));
    if (dgamma) {
        LS_TRY(check_ptr(workspace, "workspace", true));
        if (workspace_bytes < plan.bytes())
            return fail(LS_ERR_WORKSPACE_TOO_SMALL, "ls_layernorm_bwd: workspace of %zu bytes, need %zu",
                        workspace_bytes, plan.bytes());
    }
    const size_t nb = static_cast<size_t>(rows * cols) * elem_size(dt);
    const size_t sb = static_cast<size_t>(rows) * sizeof(float);
    const Span outs[] = {{"dx", dx, nb}, {"dgamma", dgamma, pb}, {"dbeta", dbeta, pb},
                         {"workspace", dgamma ? workspace : nullptr, plan.bytes()}};
    const Span ins[] = {{"dy", dy, nb},       {"x", x, nb},       {"gamma", gamma, pb},
                        {"mean", mean, sb},   {"rstd", rstd, sb}};
    LS_TRY(check_overlaps(outs, 4, ins, 5));
    float* partial = dgamma ? static_cast<float*>(workspace) : nullptr;
    cudaError_t e = guard_workspace(s, partial, plan.bytes());
    if (e == cudaSuccess)
        e = ls::launch_layernorm_bwd(dt, dx, partial, dy, x, gamma, mean, rstd, rows, cols, s);
    if (e == cudaSuccess && dgamma) {
        // Each partial row is [dgamma part | dbeta part]: one reduction of
        // 2*cols columns, the first half to dgamma and the second to dbeta.
        e = launch_reduction(s, partial, plan.bytes(), [&](cudaStream_t rs) {
            return ls::launch_colreduce(dt, dgamma, dbeta, cols, partial, plan.parts, plan.width,
                                        rs);
        }, inline_reduction);
    }
    return from_cuda(e, "ls_layernorm_bwd launch");
}

#pragma GCC visibility push(default)
extern "C" {

static ls_status softmax_common(const char* fn, ls_dtype dtype, int64_t batch, int64_t heads,
                                int64_t q_len, int64_t k_len, const int32_t* key_len,
                                ls::DType* dt, int64_t* nrows) {
    LS_TRY(check_dtype(dtype, dt));
    if (batch < 0 || heads < 0 || q_len < 0)
        return fail(LS_ERR_INVALID_ARGUMENT, "%s: negative batch/heads/q_len", fn);
    if (k_len <= 0) return fail(LS_ERR_INVALID_ARGUMENT, "%s: k_len = %lld <= 0", fn, (long long)k_len);
    if (k_len % 8 != 0)
        return fail(LS_ERR_MISALIGNED, "%s: k_len = %lld is not a multiple of 8", fn, (long long)k_len);
    if (k_len > ls::kMaxSoftmaxRowLen)
        return fail(LS_ERR_UNSUPPORTED_SHAPE, "%s: k_len = %lld exceeds %lld", fn,
                    (long long)k_len, (long long)ls::kMaxSoftmaxRowLen);
    if (q_len > (int64_t{1} << 30) || batch > (int64_t{1} << 30) || heads > (int64_t{1} << 30))
        return fail(LS_ERR_UNSUPPORTED_SHAPE, "%s: dimension too large", fn);
    const double n = static_cast<double>(batch) * heads * q_len;
    if (n * k_len > static_cast<double>(int64_t{1} << 46) || n >= static_cast<double>(1u << 31))
        return fail(LS_ERR_UNSUPPORTED_SHAPE, "%s: too many elements", fn);
    *nrows = batch * heads * q_len;
    if (key_len && (reinterpret_cast<uintptr_t>(key_len) & 3u))
        return fail(LS_ERR_MISALIGNED, "%s: key_len is not 4-byte aligned", fn);
    return LS_OK;
}

ls_status ls_softmax_fwd(ls_dtype dtype, void* y, const void* x, int64_t batch, int64_t heads,
                         int64_t q_len, int64_t k_len, const int32_t* key_len, int causal,
                         void* stream) {
    ls::DType dt;
    int64_t nrows;
    LS_TRY(softmax_common("ls_softmax_fwd", dtype, batch, heads, q_len, k_len, key_len, &dt, &nrows));
    if (nrows == 0) return ok();
    LS_TRY(check_ptr(y, "y", true));
    LS_TRY(check_ptr(x, "x", true));
    const size_t nb = static_cast<size_t>(nrows * k_len) * elem_size(dt);
    const Span outs[] = {{"y", y, nb}};
    const Span ins[] = {{"x", x, nb}, {"key_len", key_len, static_cast<size_t>(batch) * 4}};
    LS_TRY(check_overlaps(outs, 1, ins, 2));
    const ls::SoftmaxShape sh{batch, heads, q_len, k_len, key_len, causal ? 1 : 0};
    return from_cuda(ls::launch_softmax_fwd(dt, y, x, sh, static_cast<cudaStream_t>(stream)),
                     "ls_softmax_fwd launch");
}

ls_status ls_softmax_bwd(ls_dtype dtype, void* dx, const void* y, const void* dy, int64_t batch,
                         int64_t heads, int64_t q_len, int64_t k_len, const int32_t* key_len,
                         int causal, void* stream) {
    ls::DType dt;
    int64_t nrows;
    LS_TRY(softmax_common("ls_softmax_bwd", dtype, batch, heads, q_len, k_len, key_len, &dt, &nrows));
    if (nrows == 0) return ok();
    LS_TRY(check_ptr(dx, "dx", true));
    LS_TRY(check_ptr(y, "y", true));
    LS_TRY(check_ptr(dy, "dy", true));
    const size_t nb = static_cast<size_t>(nrows * k_len) * elem_size(dt);
    const Span outs[] = {{"dx", dx, nb}};
    const Span ins[] = {{"y", y, nb}, {"dy", dy, nb},
                        {"key_len", key_len, static_cast<size_t>(batch) * 4}};
    LS_TRY(check_overlaps(outs, 1, ins, 3));
    const ls::SoftmaxShape sh{batch, heads, q_len, k_len, key_len, causal ? 1 : 0};
    return from_cuda(ls::launch_softmax_bwd(dt, dx, y, dy, sh, static_cast<cudaStream_t>(stream)),
                     "ls_softmax_bwd launch");
}

ls_status ls_adam_update(ls_dtype dtype, void* param, const void* grad, float* exp_avg,
                         float* exp_avg_sq, int64_t n, float lr, float beta1, float beta2,
                         float eps, float weight_decay, int64_t step, float grad_scale,
                         void* stream) {
    ls::DType dt;
    LS_TRY(check_dtype(dtype, &dt));
    if (n < 0) return fail(LS_ERR_INVALID_ARGUMENT, "n = %lld < 0", (long long)n);
    if (n > (int64_t{1} << 46))
        return fail(LS_ERR_UNSUPPORTED_SHAPE, "n = %lld is too large", (long long)n);
    if (step < 1) return fail(LS_ERR_INVALID_ARGUMENT, "step = %lld < 1", (long long)step);
    if (!(lr >= 0.f) || !isfinite(lr))
        return fail(LS_ERR_INVALID_ARGUMENT, "lr = %g is not finite and >= 0", (double)lr);
    if (!(beta1 >= 0.f && beta1 < 1.f) || !(beta2 >= 0.f && beta2 < 1.f))
        return fail(LS_ERR_INVALID_ARGUMENT, "betas (%g, %g) are not in [0, 1)", (double)beta1,
                    (double)beta2);
    if (!(eps >= 0.f) || !isfinite(eps))
        return fail(LS_ERR_INVALID_ARGUMENT, "eps = %g is not finite and >= 0", (double)eps);
    if (!(weight_decay >= 0.f) || !isfinite(weight_decay))
        return fail(LS_ERR_INVALID_ARGUMENT, "weight_decay = %g is not finite and >= 0",
                    (double)weight_decay);
    if (!isfinite(grad_scale))
        return fail(LS_ERR_INVALID_ARGUMENT, "grad_scale = %g is not finite", (double)grad_scale);
    if (n == 0) return ok();
    LS_TRY(check_ptr(param, "param", true));
    LS_TRY(check_ptr(grad, "grad", true));
    LS_TRY(check_ptr(exp_avg, "exp_avg", true));
    LS_TRY(check_ptr(exp_avg_sq, "exp_avg_sq", true));
    const size_t pb = static_cast<size_t>(n) * elem_size(dt);
    const size_t fb = static_cast<size_t>(n) * sizeof(float);
    // param, exp_avg and exp_avg_sq are updated in place: none may overlap
    // another or the gradient.
    if (param == grad) return fail(LS_ERR_INVALID_ARGUMENT, "param and grad are the same buffer");
    const Span outs[] = {{"param", param, pb}, {"exp_avg", exp_avg, fb},
                         {"exp_avg_sq", exp_avg_sq, fb}};
    const Span ins[] = {{"grad", grad, pb}};
    LS_TRY(check_overlaps(outs, 3, ins, 1));
    const ls::AdamHyper h{lr, beta1, beta2, eps, weight_decay, grad_scale, step};
    return from_cuda(ls::launch_adam(dt, param, grad, exp_avg, exp_avg_sq, n, h,
                                     static_cast<cudaStream_t>(stream)),
                     "ls_adam_update launch");
}

static ls_status qkv_common(ls_dtype dtype, int64_t batch, int64_t seq, int64_t heads,
                            int64_t head_dim, ls::DType* dt, int64_t* rows, int64_t* cols) {
    LS_TRY(check_dtype(dtype, dt));
    if (batch < 0 || seq < 0 || heads < 0)
        return fail(LS_ERR_INVALID_ARGUMENT, "batch, seq and heads must be >= 0");
    if (head_dim <= 0) return fail(LS_ERR_INVALID_ARGUMENT, "head_dim = %lld <= 0", (long long)head_dim);
    if (head_dim % 8 != 0)
        return fail(LS_ERR_MISALIGNED, "head_dim = %lld is not a multiple of 8", (long long)head_dim);
    if (seq > INT32_MAX || heads > INT32_MAX || heads * head_dim > kMaxDropoutCols)
        return fail(LS_ERR_UNSUPPORTED_SHAPE, "seq = %lld, heads x head_dim = %lld x %lld too large",
                    (long long)seq, (long long)heads, (long long)head_dim);
    *rows = batch * seq;
    *cols = 3 * heads * head_dim;
    if (*cols == 0) *cols = 8;  // heads == 0: nothing to move; keep the shape checks happy
    return check_shape(*rows, *cols, 3 * kMaxDropoutCols);
}

ls_status ls_bias_reshape_qkv_fwd(ls_dtype dtype, void* q_k_v, const void* qkv, const void* bias,
                                  int64_t batch, int64_t seq, int64_t heads, int64_t head_dim,
                                  void* stream) {
    ls::DType dt;
    int64_t rows, cols;
    LS_TRY(qkv_common(dtype, batch, seq, heads, head_dim, &dt, &rows, &cols));
    if (rows == 0 || heads == 0) return ok();
    LS_TRY(check_ptr(q_k_v, "q_k_v", true));
    LS_TRY(check_ptr(qkv, "qkv", true));
    LS_TRY(check_ptr(bias, "bias", true));
    const size_t nb = static_cast<size_t>(rows * cols) * elem_size(dt);
    const size_t bb = static_cast<size_t>(cols) * elem_size(dt);
    // The reshape moves every element: the output may not overlap an input at all.
    const Span out{"q_k_v", q_k_v, nb}, in0{"qkv", qkv, nb}, in1{"bias", bias, bb};
    if (overlaps(out, in0) || overlaps(out, in1))
        return fail(LS_ERR_INVALID_ARGUMENT, "q_k_v overlaps qkv or bias (no in-place reshape)");
    return from_cuda(ls::launch_qkv_fwd(dt, q_k_v, qkv, bias, batch, seq, heads, head_dim,
                                        static_cast<cudaStream_t>(stream)),
                     "ls_bias_reshape_qkv_fwd launch");
}

ls_status ls_bias_reshape_qkv_bwd(ls_dtype dtype, void* dqkv, void* dbias, const void* dq_k_v,
                                  int64_t batch, int64_t seq, int64_t heads, int64_t head_dim,
                                  void* workspace, size_t workspace_bytes, void* stream) {
    ls::DType dt;
    int64_t rows, cols;
    LS_TRY(qkv_common(dtype, batch, seq, heads, head_dim, &dt, &rows, &cols));
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const size_t bb = static_cast<size_t>(cols) * elem_size(dt);
    if (rows == 0 || heads == 0) {
        if (dbias && heads > 0) {
            LS_TRY(check_ptr(dbias, "dbias", true));
            return from_cuda(cudaMemsetAsync(dbias, 0, bb, s), "ls_bias_reshape_qkv_bwd");
        }
        return ok();
    }
    LS_TRY(check_ptr(dqkv, "dqkv", true));
    LS_TRY(check_ptr(dbias, "dbias", false));
    LS_TRY(check_ptr(dq_k_v, "dq_k_v", true));
    const ls::ColReducePlan plan = ls::dropout_bwd_plan(rows, cols);
    if (dbias) {
        LS_TRY(check_ptr(workspace, "workspace", true));
        if (workspace_bytes < plan.bytes())
            return fail(LS_ERR_WORKSPACE_TOO_SMALL,
                        "ls_bias_reshape_qkv_bwd: workspace of %zu bytes, need %zu",
                        workspace_bytes, plan.bytes());
    }
    const size_t nb = static_cast<size_t>(rows * cols) * elem_size(dt);
    const Span outs[] = {{"dqkv", dqkv, nb}, {"dbias", dbias, bb},
                         {"workspace", dbias ? workspace : nullptr, plan.bytes()}};
    const Span in{"dq_k_v", dq_k_v, nb};
    for (const Span& o : outs)
        if (overlaps(o, in))
            return fail(LS_ERR_INVALID_ARGUMENT, "%s overlaps dq_k_v (no in-place reshape)",
                        o.name);
    LS_TRY(check_overlaps(outs, 3, nullptr, 0));
    float* partial = dbias ? static_cast<float*>(workspace) : nullptr;
    cudaError_t e = guard_workspace(s, partial, plan.bytes());
    if (e == cudaSuccess)
        e = ls::launch_qkv_bwd(dt, dqkv, partial, dq_k_v, batch, seq, heads, head_dim, s);
    if (e == cudaSuccess && dbias)
        e = launch_reduction(s, partial, plan.bytes(), [&](cudaStream_t rs) {
            return ls::launch_colreduce(dt, dbias, nullptr, cols, partial, plan.parts, cols, rs);
        });
    return from_cuda(e, "ls_bias_reshape_qkv_bwd launch");
}

ls_status ls_softmax_dropout_fwd(ls_dtype dtype, void* y, void* y_drop, uint32_t* mask_bits,
                                 const void* x, int64_t batch, int64_t heads, int64_t q_len,
                                 int64_t k_len, const int32_t* key_len, int causal, float p,
                                 uint64_t seed, uint64_t offset, void* stream) {
    ls::DType dt;
    int64_t nrows;
    LS_TRY(softmax_common("ls_softmax_dropout_fwd", dtype, batch, heads, q_len, k_len, key_len,
                          &dt, &nrows));
    ls::DropoutRng rng;
    LS_TRY(check_p(p, &rng, seed, offset));
    if (nrows == 0) return ok();
    LS_TRY(check_ptr(y, "y", true));
    LS_TRY(check_ptr(y_drop, "y_drop", true));
    LS_TRY(check_ptr(mask_bits, "mask_bits", true));
    LS_TRY(check_ptr(x, "x", true));
    const size_t nb = static_cast<size_t>(nrows * k_len) * elem_size(dt);
    const Span outs[] = {{"y", y, nb}, {"y_drop", y_drop, nb},
                         {"mask_bits", mask_bits, mask_bytes(nrows, k_len)}};
    const Span ins[] = {{"x", x, nb}, {"key_len", key_len, static_cast<size_t>(batch) * 4}};
    LS_TRY(check_overlaps(outs, 3, ins, 2));
    const ls::SoftmaxShape sh{batch, heads, q_len, k_len, key_len, causal ? 1 : 0};
    return from_cuda(ls::launch_softmax_dropout_fwd(dt, y, y_drop,
                                                    reinterpret_cast<uint8_t*>(mask_bits), x, sh,
                                                    rng, static_cast<cudaStream_t>(stream)),
                     "ls_softmax_dropout_fwd launch");
}

ls_status ls_softmax_dropout_bwd(ls_dtype dtype, void* dx, const void* y, const void* dy_drop,
                                 const uint32_t* mask_bits, int64_t batch, int64_t heads,
                                 int64_t q_len, int64_t k_len, const int32_t* key_len, int causal,
                                 float p, void* stream) {
    ls::DType dt;
    int64_t nrows;
    LS_TRY(softmax_common("ls_softmax_dropout_bwd", dtype, batch, heads, q_len, k_len, key_len,
                          &dt, &nrows));
    ls::DropoutRng rng;
    LS_TRY(check_p(p, &rng, 0, 0));
    if (nrows == 0) return ok();
    LS_TRY(check_ptr(dx, "dx", true));
    LS_TRY(check_ptr(y, "y", true));
    LS_TRY(check_ptr(dy_drop, "dy_drop", true));
    LS_TRY(check_ptr(mask_bits, "mask_bits", true));
    const size_t nb = static_cast<size_t>(nrows * k_len) * elem_size(dt);
    const Span outs[] = {{"dx", dx, nb}};
    const Span ins[] = {{"y", y, nb}, {"dy_drop", dy_drop, nb},
                        {"mask_bits", mask_bits, mask_bytes(nrows, k_len)},
                        {"key_len", key_len, static_cast<size_t>(batch) * 4}};
    LS_TRY(check_overlaps(outs, 1, ins, 4));
    const ls::SoftmaxShape sh{batch, heads, q_len, k_len, key_len, causal ? 1 : 0};
    return from_cuda(ls::launch_softmax_dropout_bwd(dt, dx, y, dy_drop,
                                                    reinterpret_cast<const uint8_t*>(mask_bits),
                                                    sh, rng.scale,
                                                    static_cast<cudaStream_t>(stream)),
                     "ls_softmax_dropout_bwd launch");
}

static ls_status ce_common(const char* fn, ls_dtype dtype, int64_t rows, int64_t vocab,
                           float eps, ls::DType* dt) {
    LS_TRY(check_dtype(dtype, dt));
    if (rows < 0) return fail(LS_ERR_INVALID_ARGUMENT, "%s: rows = %lld < 0", fn, (long long)rows);
    if (vocab <= 0)
        return fail(LS_ERR_INVALID_ARGUMENT, "%s: vocab = %lld <= 0", fn, (long long)vocab);
    if (vocab % 8 != 0)
        return fail(LS_ERR_MISALIGNED, "%s: vocab = %lld is not a multiple of 8", fn,
                    (long long)vocab);
    if (vocab > (int64_t{1} << 28) || rows >= (int64_t{1} << 31))
        return fail(LS_ERR_UNSUPPORTED_SHAPE, "%s: %lld rows of %lld logits too large", fn,
                    (long long)rows, (long long)vocab);
    if (!(eps >= 0.f && eps < 1.f))
        return fail(LS_ERR_INVALID_ARGUMENT, "%s: label_smoothing = %g is not in [0, 1)", fn,
                    (double)eps);
    return LS_OK;
}

ls_status ls_cross_entropy_fwd(ls_dtype dtype, float* loss, float* lse, const void* logits,
                               const int32_t* target, int64_t rows, int64_t vocab,
                               float label_smoothing, int32_t ignore_index, void* stream) {
    ls::DType dt;
    LS_TRY(ce_common("ls_cross_entropy_fwd", dtype, rows, vocab, label_smoothing, &dt));
    if (rows == 0) return ok();
    LS_TRY(check_ptr(loss, "loss", true));
    LS_TRY(check_ptr(lse, "lse", false));
    LS_TRY(check_ptr(logits, "logits", true));
    if (!target) return fail(LS_ERR_INVALID_ARGUMENT, "target is NULL");
    if (reinterpret_cast<uintptr_t>(target) & 3u)
        return fail(LS_ERR_MISALIGNED, "target is not 4-byte aligned");
    const size_t rb = static_cast<size_t>(rows) * 4;
    const Span outs[] = {{"loss", loss, rb}, {"lse", lse, rb}};
    const Span ins[] = {{"logits", logits, static_cast<size_t>(rows * vocab) * elem_size(dt)},
                        {"target", target, rb}};
    LS_TRY(check_overlaps(outs, 2, ins, 2));
    return from_cuda(ls::launch_cross_entropy_fwd(dt, loss, lse, logits, target, rows, vocab,
                                                  label_smoothing, ignore_index,
                                                  static_cast<cudaStream_t>(stream)),
                     "ls_cross_entropy_fwd launch");
}

ls_status ls_cross_entropy_bwd(ls_dtype dtype, void* dlogits, const void* logits,
                               const int32_t* target, const float* lse, const float* dloss,
                               int64_t rows, int64_t vocab, float label_smoothing,
                               int32_t ignore_index, void* stream) {
    ls::DType dt;
    LS_TRY(ce_common("ls_cross_entropy_bwd", dtype, rows, vocab, label_smoothing, &dt));
    if (rows == 0) return ok();
    LS_TRY(check_ptr(dlogits, "dlogits", true));
    LS_TRY(check_ptr(logits, "logits", true));
    LS_TRY(check_ptr(lse, "lse", true));
    LS_TRY(check_ptr(dloss, "dloss", false));
    if (!target) return fail(LS_ERR_INVALID_ARGUMENT, "target is NULL");
    if (reinterpret_cast<uintptr_t>(target) & 3u)
        return fail(LS_ERR_MISALIGNED, "target is not 4-byte aligned");
    const size_t rb = static_cast<size_t>(rows) * 4;
    const size_t nb = static_cast<size_t>(rows * vocab) * elem_size(dt);
    const Span outs[] = {{"dlogits", dlogits, nb}};
    const Span ins[] = {{"logits", logits, nb}, {"target", target, rb}, {"lse", lse, rb},
                        {"dloss", dloss, rb}};
    LS_TRY(check_overlaps(outs, 1, ins, 4));
    return from_cuda(ls::launch_cross_entropy_bwd(dt, dlogits, logits, target, lse, dloss, rows,
                                                  vocab, label_smoothing, ignore_index,
                                                  static_cast<cudaStream_t>(stream)),
                     "ls_cross_entropy_bwd launch");
}

static ls_status emb_common(const char* fn, ls_dtype dtype, int64_t batch, int64_t seq,
                            int64_t hidden, int64_t vocab, float scale, ls::DType* dt) {
    LS_TRY(check_dtype(dtype, dt));
    if (batch < 0 || seq < 0 || vocab < 0)
        return fail(LS_ERR_INVALID_ARGUMENT, "%s: negative batch/seq/vocab", fn);
    LS_TRY(check_shape(batch * seq, hidden, kMaxDropoutCols));
    if (seq > INT32_MAX || vocab > INT32_MAX)
        return fail(LS_ERR_UNSUPPORTED_SHAPE, "%s: seq or vocab too large", fn);
    if (!isfinite(scale)) return fail(LS_ERR_INVALID_ARGUMENT, "%s: scale is not finite", fn);
    return LS_OK;
}

ls_status ls_embedding_fwd(ls_dtype dtype, void* y, uint32_t* mask_bits, const int32_t* tokens,
                           const void* token_table, const void* pos_table, int64_t batch,
                           int64_t seq, int64_t hidden, int64_t vocab, int64_t max_positions,
                           float scale, float p, uint64_t seed, uint64_t offset, void* stream) {
    ls::DType dt;
    LS_TRY(emb_common("ls_embedding_fwd", dtype, batch, seq, hidden, vocab, scale, &dt));
    ls::DropoutRng rng;
    LS_TRY(check_p(p, &rng, seed, offset));
    if (max_positions < seq)
        return fail(LS_ERR_INVALID_ARGUMENT, "max_positions = %lld < seq = %lld",
                    (long long)max_positions, (long long)seq);
    const int64_t T = batch * seq;
    if (T == 0) return ok();
    LS_TRY(check_ptr(y, "y", true));
    LS_TRY(check_ptr(mask_bits, "mask_bits", false));
    LS_TRY(check_ptr(token_table, "token_table", vocab > 0));
    LS_TRY(check_ptr(pos_table, "pos_table", true));
    if (!tokens) return fail(LS_ERR_INVALID_ARGUMENT, "tokens is NULL");
    if (reinterpret_cast<uintptr_t>(tokens) & 3u)
        return fail(LS_ERR_MISALIGNED, "tokens is not 4-byte aligned");
    const size_t es = elem_size(dt);
    const Span outs[] = {{"y", y, static_cast<size_t>(T * hidden) * es},
                         {"mask_bits", mask_bits, mask_bytes(T, hidden)}};
    const Span ins[] = {{"tokens", tokens, static_cast<size_t>(T) * 4},
                        {"token_table", token_table, static_cast<size_t>(vocab * hidden) * es},
                        {"pos_table", pos_table, static_cast<size_t>(max_positions * hidden) * es}};
    LS_TRY(check_overlaps(outs, 2, ins, 3));
    return from_cuda(ls::launch_embedding_fwd(dt, y, reinterpret_cast<uint8_t*>(mask_bits),
                                              tokens, token_table, pos_table, batch, seq, hidden,
                                              vocab, scale, rng,
                                              static_cast<cudaStream_t>(stream)),
                     "ls_embedding_fwd launch");
}

size_t ls_embedding_workspace_bytes(int64_t tokens) {
    (void)tokens;  // the deterministic backward needs no scratch
    return 0;
}

ls_status ls_embedding_bwd(ls_dtype dtype, float* d_token_table, const void* dy,
                           const uint32_t* mask_bits, const int32_t* tokens, int64_t batch,
                           int64_t seq, int64_t hidden, int64_t vocab, float scale, float p,
                           int deterministic, void* workspace, size_t workspace_bytes,
                           void* stream) {
    ls::DType dt;
    LS_TRY(emb_common("ls_embedding_bwd", dtype, batch, seq, hidden, vocab, scale, &dt));
    ls::DropoutRng rng;
    LS_TRY(check_p(p, &rng, 0, 0));
    const int64_t T = batch * seq;
    if (T == 0 || vocab == 0) return ok();
    if (!deterministic) {
        LS_TRY(check_ptr(d_token_table, "d_token_table", true));
        LS_TRY(check_ptr(dy, "dy", true));
        LS_TRY(check_ptr(mask_bits, "mask_bits", true));
        if (!tokens) return fail(LS_ERR_INVALID_ARGUMENT, "tokens is NULL");
        if (reinterpret_cast<uintptr_t>(tokens) & 3u)
            return fail(LS_ERR_MISALIGNED, "tokens is not 4-byte aligned");
        const Span outs[] = {
            {"d_token_table", d_token_table, static_cast<size_t>(vocab * hidden) * 4}};
        const Span ins[] = {{"dy", dy, static_cast<size_t>(T * hidden) * elem_size(dt)},
                            {"mask_bits", mask_bits, mask_bytes(T, hidden)},
                            {"tokens", tokens, static_cast<size_t>(T) * 4}};
        LS_TRY(check_overlaps(outs, 1, ins, 3));
        const float c = static_cast<float>(static_cast<double>(scale) * rng.scale);
        return from_cuda(ls::launch_embedding_bwd_atomic(
                             dt, d_token_table, dy, reinterpret_cast<const uint8_t*>(mask_bits),
                             tokens, T, hidden, vocab, c, static_cast<cudaStream_t>(stream)),
                         "ls_embedding_bwd launch");
    }
    if (T > ls::kEmbeddingMaxTokens)
        return fail(LS_ERR_UNSUPPORTED_SHAPE,
                    "ls_embedding_bwd: %lld tokens in one call; at most %lld (split the batch: "
                    "calls on one stream accumulate in order)",
                    (long long)T, (long long)ls::kEmbeddingMaxTokens);
    LS_TRY(check_ptr(d_token_table, "d_token_table", true));
    LS_TRY(check_ptr(dy, "dy", true));
    LS_TRY(check_ptr(mask_bits, "mask_bits", true));
    if (!tokens) return fail(LS_ERR_INVALID_ARGUMENT, "tokens is NULL");
    if (reinterpret_cast<uintptr_t>(tokens) & 3u)
        return fail(LS_ERR_MISALIGNED, "tokens is not 4-byte aligned");
    (void)workspace;  // none needed (ls_embedding_workspace_bytes is 0)
    (void)workspace_bytes;
    const size_t es = elem_size(dt);
    const Span outs[] = {{"d_token_table", d_token_table, static_cast<size_t>(vocab * hidden) * 4}};
    const Span ins[] = {{"dy", dy, static_cast<size_t>(T * hidden) * es},
                        {"mask_bits", mask_bits, mask_bytes(T, hidden)},
                        {"tokens", tokens, static_cast<size_t>(T) * 4}};
    LS_TRY(check_overlaps(outs, 1, ins, 3));
    const float coef = static_cast<float>(static_cast<double>(scale) * rng.scale);
    return from_cuda(ls::launch_embedding_bwd(dt, d_token_table, dy,
                                              reinterpret_cast<const uint8_t*>(mask_bits), tokens,
                                              T, hidden, vocab, coef,
                                              static_cast<cudaStream_t>(stream)),
                     "ls_embedding_bwd launch");
}

}  // extern "C"
#pragma GCC visibility pop
