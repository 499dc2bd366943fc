// launch_pdl.cuh -- host-side launch with programmatic dependent launch
// (internal to the library; not part of the run-time compiled sources).
#pragma once

#include <cuda_runtime.h>

#include <utility>

namespace attnres {

// Launch `kern` on `stream` allowed to start while the kernel before it on the
// stream is still running (programmatic stream serialization).  The kernel
// must call pdl_wait() before its first global memory access; launched after
// anything but a kernel, or outside a stream of kernels, it behaves as an
// ordinary launch.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                       Args&&... args) {
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

}  // namespace attnres
