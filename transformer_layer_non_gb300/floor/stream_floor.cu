// stream_floor.cu -- the benchmark's reference kernel (not part of the operator
// library): a plain streaming pass that reads `read_vecs` 16-byte vectors from
// src and writes `write_vecs` to dst, one vector per thread, launched the way
// the operator kernels are (programmatic dependent launch: it waits for its
// predecessor's completion before its first access and then releases its own
// successor).  Like the operator kernels, each thread first prefetches its
// source line into L2 before the wait (a prefetch is not a read of the
// predecessor's data: it only moves the line into L2, where the
// predecessor's writes land too), so the CTAs resident while the predecessor
// drains have their DRAM round trip under way.  Chained back to back over
// L2-cold buffers, its time per launch is what a dependent launch moving those
// bytes costs with no arithmetic at all: the floor each operator's time is
// compared with.
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace {

__global__ void __launch_bounds__(256)
stream_floor_kernel(uint4* __restrict__ dst, const uint4* __restrict__ src, uint64_t read_vecs,
                    uint64_t write_vecs, uint32_t never) {
    const uint64_t i = static_cast<uint64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (i < read_vecs) asm volatile("prefetch.global.L2 [%0];" ::"l"(src + i));
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    uint4 v = make_uint4(0, 0, 0, 0);
    if (i < read_vecs) v = src[i];
    if (i < write_vecs) {
        dst[i] = v;
    } else if (v.x == never && v.y == never && v.z == never && v.w == never) {
        // Reads past the written range are kept live by a store whose
        // condition the caller makes false (`never` is absent from src).
        dst[0] = v;
    }
}

}  // namespace

#pragma GCC visibility push(default)
extern "C" int lsf_stream(void* dst, const void* src, uint64_t read_vecs, uint64_t write_vecs,
                          uint32_t never, void* stream) {
    const uint64_t n = read_vecs > write_vecs ? read_vecs : write_vecs;
    if (n == 0) return 0;
    if ((n + 255) / 256 > 0x7fffffffull) return static_cast<int>(cudaErrorInvalidValue);
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>((n + 255) / 256));
    cfg.blockDim = dim3(256);
    cfg.stream = static_cast<cudaStream_t>(stream);
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return static_cast<int>(cudaLaunchKernelEx(&cfg, stream_floor_kernel, static_cast<uint4*>(dst),
                                               static_cast<const uint4*>(src), read_vecs,
                                               write_vecs, never));
}
#pragma GCC visibility pop
