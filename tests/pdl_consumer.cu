// Test helper: a consumer kernel launched with programmatic stream
// serialization that copies its input WITHOUT waiting for the preceding grid
// (no griddepcontrol.wait), as a consumer that reads before its wait does.
// Built by tests/test_hold_gpu.py with nvcc; not part of the library.
#include <cuda_runtime.h>

__global__ void copy_early(const int *src, int *dst, int n) {
    for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n; i += gridDim.x * blockDim.x) dst[i] = src[i];
}

extern "C" int launch_copy_early(const int *src, int *dst, int n, void *stream) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(64, 1, 1);
    cfg.blockDim = dim3(256, 1, 1);
    cfg.stream = static_cast<cudaStream_t>(stream);
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr.val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    return static_cast<int>(cudaLaunchKernelEx(&cfg, copy_early, src, dst, n));
}
