// Kernel launches with the programmatic-stream-serialization attribute.
#pragma once

#include <cuda_runtime.h>

#include <utility>

namespace pcp {

// False when PCP_DISABLE_PDL is set in the environment (read once).
bool pdl_enabled();

// Launch `kernel` as a programmatic dependent of the previous kernel on
// `stream` (it must call pdl_wait() before touching global memory).  If the
// runtime refuses the attribute, the kernel is launched plainly.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t stream, Args&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl_enabled() ? 1 : 0;
    cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
    if (e != cudaSuccess && cfg.numAttrs == 1) {
        (void)cudaGetLastError();
        cfg.numAttrs = 0;
        e = cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
    }
    return e;
}

}  // namespace pcp
