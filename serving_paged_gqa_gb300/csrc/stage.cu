// Copy kernel of the serving step (pkv_serve_step): moves the packed step input from page-locked host memory, read
// through its device-visible address over the host link, into device memory. Enqueueing one launch costs the host
// about 3 us; a small cudaMemcpyAsync from page-locked memory cost about 9 us on a GB300's Grace host.
#include <cuda_runtime.h>

#include <algorithm>

#include "pkv_internal.h"
#include "pkv_ptx.cuh"

namespace pkv {
namespace {

__global__ void __launch_bounds__(256) stage_copy_kernel(const uint4* __restrict__ src, uint4* __restrict__ dst,
                                                         size_t n16) {
    // the decode launched after this grid may start its set-up now; it reads the copied input only after waiting
    // for this grid's completion
    grid_launch_dependents();
    for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n16; i += (size_t)gridDim.x * blockDim.x)
        dst[i] = src[i];
}

}  // namespace

int launch_stage_copy(const void* src, void* dst, size_t bytes, void* stream) {
    const size_t n16 = bytes / 16;
    if (n16 == 0) return cudaSuccess;
    const int grid = (int)std::min<size_t>(64, (n16 + 255) / 256);
    stage_copy_kernel<<<grid, 256, 0, static_cast<cudaStream_t>(stream)>>>(static_cast<const uint4*>(src),
                                                                          static_cast<uint4*>(dst), n16);
    return cudaGetLastError();
}

}  // namespace pkv
