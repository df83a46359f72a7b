// Test helper: a kernel launched right after a forward call with
// programmatic stream serialization, so that it may start before the forward
// grid ends. It waits for the grids it depends on (griddepcontrol.wait) and
// then copies the forward pass's output, which must by then be complete.
#include <cuda_runtime.h>
#include <cstdint>

__global__ void successor_copy(const uint16_t* __restrict__ src, uint16_t* __restrict__ dst, size_t n) {
    asm volatile("griddepcontrol.wait;" ::: "memory");
    for (size_t i = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; i < n;
         i += static_cast<size_t>(gridDim.x) * blockDim.x)
        dst[i] = src[i];
}

extern "C" int launch_successor_copy(const void* src, void* dst, size_t n, void* stream) {
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(256, 1, 1);
    cfg.blockDim = dim3(256, 1, 1);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = static_cast<cudaStream_t>(stream);
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const cudaError_t e = cudaLaunchKernelEx(&cfg, successor_copy, static_cast<const uint16_t*>(src),
                                             static_cast<uint16_t*>(dst), n);
    return e == cudaSuccess ? 0 : static_cast<int>(e);
}
