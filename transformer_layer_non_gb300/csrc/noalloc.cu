// noalloc.cu -- LayerNorm backward for callers that cannot allocate device
// memory.
//
// ls_layernorm_bwd asks its caller for a device workspace to hold the FP32
// partial sums of the gamma/beta gradients.  Some callers have no way to
// provide one: a plugin running inside a host application that owns every
// device allocation, or a code path where calling cudaMalloc is not allowed
// (it would synchronise the device or fail while a graph is being captured).
// ls_layernorm_bwd_noalloc gives them the same computation with the scratch
// kept in a fixed, file-scope device array instead.  The array is
// kNoAllocScratchBytes large and every GPU that loads the library holds it
// until the process exits.
//
// Nothing here allocates: the array is part of the library's device image,
// its device address is looked up in the current context on every call, and
// the call then goes through the ordinary LayerNorm backward path with that
// address as workspace and its column reduction kept on the caller's stream.
#include "../../include/ls_ops.h"
#include "ls_internal.h"

namespace {

constexpr size_t kNoAllocScratchBytes = LS_NOALLOC_SCRATCH_BYTES;

// The shared scratch.  In host code this name is only a host-side stand-in
// for the symbol, never a device address: the address comes from
// cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

// Device address of the scratch array in the current context.  A __device__
// array exists once per context that has loaded the library's module, so the
// address belongs to the context, not to the device: it is looked up on every
// call (a query that allocates nothing), never cached, and so stays right in
// a second context on the same device and after cudaDeviceReset.
cudaError_t scratch_address(void** out) {
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return e;
    if (p == nullptr) return cudaErrorInvalidSymbol;
    *out = p;
    return cudaSuccess;
}

}  // namespace

#pragma GCC visibility push(default)
extern "C" ls_status ls_layernorm_bwd_noalloc(ls_dtype dtype, void* dx, void* dgamma,
                                              void* dbeta, const void* dy, const void* x,
                                              const void* gamma, const float* mean,
                                              const float* rstd, int64_t rows, int64_t cols,
                                              void* stream) {
    const bool param_grads = dgamma != nullptr || dbeta != nullptr;
    // Without parameter gradients, or for an empty batch, no scratch is used;
    // the shared LayerNorm backward path validates the arguments and does the work.
    if (!param_grads || rows == 0)
        return ls::layernorm_bwd_entry(dtype, dx, dgamma, dbeta, dy, x, gamma, mean, rstd, rows,
                                       cols, nullptr, 0, stream, /*inline_reduction=*/true);
    // Reject shapes whose partial sums do not fit, before touching the GPU.
    if (rows > 0 && cols > 0 && cols % 8 == 0 && cols <= ls::kMaxRowLen) {
        const size_t need = ls::layernorm_bwd_plan(rows, cols, dtype == LS_F32 ? 4 : 2).bytes();
        if (need > kNoAllocScratchBytes) {
            ls::set_last_error_message(
                "ls_layernorm_bwd_noalloc: rows=%lld cols=%lld need %zu bytes of scratch; the "
                "built-in scratch holds %zu bytes (use ls_layernorm_bwd with a workspace)",
                static_cast<long long>(rows), static_cast<long long>(cols), need,
                kNoAllocScratchBytes);
            return LS_ERR_UNSUPPORTED_SHAPE;
        }
    }
    void* scratch = nullptr;
    const cudaError_t e = scratch_address(&scratch);
    if (e != cudaSuccess) {
        ls::set_last_error_message("ls_layernorm_bwd_noalloc: scratch set-up failed: %s (%s)",
                                   cudaGetErrorName(e), cudaGetErrorString(e));
        return LS_ERR_CUDA;
    }
    // The column reduction stays on `stream` even when a reduction stream is
    // set: the scratch is shared by every host thread, and a reduction forked
    // onto another stream would still be reading it when a call from another
    // thread, ordered only on `stream`, overwrites it.
    return ls::layernorm_bwd_entry(dtype, dx, dgamma, dbeta, dy, x, gamma, mean, rstd, rows, cols,
                                   scratch, kNoAllocScratchBytes, stream,
                                   /*inline_reduction=*/true);
}
#pragma GCC visibility pop
