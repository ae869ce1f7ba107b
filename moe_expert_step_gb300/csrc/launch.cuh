// Host-side launch helper: every kernel goes out with programmatic stream
// serialisation allowed (see pdl_trigger / pdl_wait in common.cuh), and
// per-device one-time dynamic shared-memory opt-in.
#pragma once
#include <cuda_runtime.h>

namespace moestep {

// Whether launches carry the programmatic-dependent-launch attribute (cleared
// only while a graph that cannot hold programmatic edges is captured).
extern bool g_launch_pdl;

template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                              Args... args) {
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = g_launch_pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kern, static_cast<KArgs>(args)...);
}

// Raise a kernel's dynamic shared-memory limit once per device, so repeated
// calls make no attribute calls (the opt-in is needed whenever static plus
// dynamic shared memory exceeds 48 KiB).  `done` is the caller's per-kernel
// record (one static array per kernel instantiation).
template <typename K>
inline cudaError_t ensure_smem(K kern, size_t bytes, int (&done)[64]) {
    if (bytes == 0) return cudaSuccess;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (done[dev] >= static_cast<int>(bytes)) return cudaSuccess;
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(bytes));
    if (e == cudaSuccess) done[dev] = static_cast<int>(bytes);
    return e;
}

}  // namespace moestep
