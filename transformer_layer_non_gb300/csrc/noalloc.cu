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
// its device address is looked up once per device, and the call then goes
// through the ordinary ls_layernorm_bwd path with that address as workspace.
#include <mutex>

#include "../../include/ls_ops.h"
#include "ls_internal.h"

namespace {

constexpr size_t kNoAllocScratchBytes = LS_NOALLOC_SCRATCH_BYTES;

// The shared scratch.  In host code this name is only a host-side stand-in
// for the symbol, never a device address: the address comes from
// cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 256;
std::mutex g_setup_mutex;
void* g_scratch_addr[kMaxDevices] = {};  // per device, set on the first call there

// Device address of the scratch array on the current device (set-up on the
// first call per device, with that device current).
cudaError_t scratch_address(void** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_setup_mutex);
    if (g_scratch_addr[dev] == nullptr) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess) return e;
        if (p == nullptr) return cudaErrorInvalidSymbol;
        g_scratch_addr[dev] = p;
    }
    *out = g_scratch_addr[dev];
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
    // ls_layernorm_bwd validates the arguments and does the work.
    if (!param_grads || rows == 0)
        return ls_layernorm_bwd(dtype, dx, dgamma, dbeta, dy, x, gamma, mean, rstd, rows, cols,
                                nullptr, 0, stream);
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
    return ls_layernorm_bwd(dtype, dx, dgamma, dbeta, dy, x, gamma, mean, rstd, rows, cols,
                            scratch, kNoAllocScratchBytes, stream);
}
#pragma GCC visibility pop
