// gemm_w8a8_noalloc.cu -- FP8 W8A8 grouped GEMM with the sum over top_k, for
// callers that cannot allocate device memory.
//
// The TOKEN_SUM layout needs an fp32 [M, N] accumulation buffer.  The regular
// entry point takes it from the caller; this one uses a fixed array compiled
// into the library instead, so a caller that has no allocator at hand -- for
// example code running inside a memory-pool-managed runtime that forbids
// cudaMalloc on its hot path, or a plugin that only receives its input and
// output buffers -- can still run the fused sum.
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "host_util.h"
#include "qmoe.h"

namespace {

// Shared by every call on a device, kept until the process exits.
static __device__ __align__(256) float g_token_sum_scratch[QMOE_NOALLOC_ACCUM_MAX_ELEMS];

// Device address of the array, looked up once per device with that device
// current (the host-side name of the array is not a device address).
float* scratch_for_current_device(qmoe_status_t* st) {
    static std::mutex mu;
    static float* addr[64] = {nullptr};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
        *st = QMOE_ERR_CUDA;
        return nullptr;
    }
    std::lock_guard<std::mutex> g(mu);
    if (addr[dev] == nullptr) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_token_sum_scratch) != cudaSuccess || p == nullptr) {
            *st = QMOE_ERR_CUDA;
            return nullptr;
        }
        addr[dev] = static_cast<float*>(p);
    }
    *st = QMOE_OK;
    return addr[dev];
}

}  // namespace

extern "C" qmoe_status_t qmoe_moe_gemm_w8a8_token_sum_noalloc(const qmoe_gemm_args* args, qmoe_stream_t stream) {
    if (!args || args->struct_size < sizeof(qmoe_gemm_args)) return QMOE_ERR_INVALID_ARG;
    if (args->out_layout != QMOE_OUT_TOKEN_SUM) return QMOE_ERR_INVALID_ARG;
    if (args->M < 0 || args->N < 0) return QMOE_ERR_INVALID_ARG;
    if (args->M * args->N > static_cast<int64_t>(QMOE_NOALLOC_ACCUM_MAX_ELEMS)) return QMOE_ERR_UNSUPPORTED;
    qmoe_status_t st = QMOE_OK;
    float* scratch = scratch_for_current_device(&st);
    if (st != QMOE_OK) return st;
    qmoe_gemm_args a = *args;
    a.accum = scratch;  // zeroed (first M*N floats) on the stream by the regular path
    return qmoe_moe_gemm_w8a8(&a, stream);
}
