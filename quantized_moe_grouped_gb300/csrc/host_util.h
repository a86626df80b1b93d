// host_util.h -- host-side helpers shared by the qmoe entry points.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "qmoe.h"

namespace qmoe {

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
inline bool aligned4(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }
inline bool aligned8(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 7u) == 0; }

// Number of SMs of the current device (cached per device ordinal).
inline int device_sm_count() {
    static std::mutex mu;
    static int cache[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
    std::lock_guard<std::mutex> g(mu);
    if (cache[dev] == 0) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
        cache[dev] = n;
    }
    return cache[dev];
}

inline qmoe_status_t launch_status() {
    return cudaPeekAtLastError() == cudaSuccess ? QMOE_OK : QMOE_ERR_CUDA;
}

// Launch with programmatic stream serialisation: the kernel may begin while
// the previous kernel on the stream is still running; it must execute
// griddepcontrol.wait (pdl_wait) before it reads or writes memory the previous
// kernel touches, and may signal griddepcontrol.launch_dependents so that the
// next kernel can begin early in turn.
template <typename... KArgs, typename... Args>
inline qmoe_status_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                                Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, static_cast<KArgs>(args)...) == cudaSuccess ? QMOE_OK : QMOE_ERR_CUDA;
}

}  // namespace qmoe
