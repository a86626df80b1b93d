// gemm_w8a8_noalloc.cu -- FP8 W8A8 grouped GEMM with the sum over top_k, for
// callers that cannot allocate device memory.
//
// The TOKEN_SUM layout needs an fp32 [M, N] accumulation buffer.  The regular
// entry point takes it from the caller; this one uses a fixed array compiled
// into the library instead, so a caller that has no allocator at hand -- for
// example code running inside a memory-pool-managed runtime that forbids
// cudaMalloc on its hot path, or a plugin that only receives its input and
// output buffers -- can still run the fused sum.
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "host_util.h"
#include "qmoe.h"

namespace {

// Shared by every call on a device, kept until the process exits.
static __device__ __align__(256) float g_token_sum_scratch[QMOE_NOALLOC_ACCUM_MAX_ELEMS];

typedef CUresult (*CtxGetCurrentFn)(CUcontext*);
typedef CUresult (*CtxGetIdFn)(CUcontext, unsigned long long*);

// Identity of the current CUDA context (0 when it cannot be read).  A context
// destroyed and created again (cudaDeviceReset, or the primary context
// released and retained) gets a new id, and the array a new address.
unsigned long long current_context_id() {
    static CtxGetCurrentFn get_current = nullptr;
    static CtxGetIdFn get_id = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_current = reinterpret_cast<CtxGetCurrentFn>(f);
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_id = reinterpret_cast<CtxGetIdFn>(f);
    });
    CUcontext ctx = nullptr;
    unsigned long long id = 0;
    if (!get_current || !get_id || get_current(&ctx) != CUDA_SUCCESS || !ctx || get_id(ctx, &id) != CUDA_SUCCESS)
        return 0;
    return id;
}

// Device address of the array in the current device's context (the host-side
// name of the array is not a device address).  Looked up once per device with
// that device current, and again whenever the device's context has changed
// since (a reset unloads the library's module; an address kept from before
// would point at memory that is no longer mapped).  When the context id cannot
// be read, the address is looked up on every call.
float* scratch_for_current_device(qmoe_status_t* st) {
    static std::mutex mu;
    static float* addr[64] = {nullptr};
    static unsigned long long ctx_of[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
        *st = QMOE_ERR_CUDA;
        return nullptr;
    }
    std::lock_guard<std::mutex> g(mu);
    const unsigned long long ctx = current_context_id();
    if (addr[dev] == nullptr || ctx == 0 || ctx != ctx_of[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_token_sum_scratch) != cudaSuccess || p == nullptr) {
            addr[dev] = nullptr;
            *st = QMOE_ERR_CUDA;
            return nullptr;
        }
        addr[dev] = static_cast<float*>(p);
        ctx_of[dev] = current_context_id();  // the lookup has made the device's context current
    }
    *st = QMOE_OK;
    return addr[dev];
}

}  // namespace

extern "C" qmoe_status_t qmoe_moe_gemm_w8a8_token_sum_noalloc(const qmoe_gemm_args* args, qmoe_stream_t stream) {
    if (!args || args->struct_size < sizeof(qmoe_gemm_args)) return QMOE_ERR_INVALID_ARG;
    if (args->out_layout != QMOE_OUT_TOKEN_SUM) return QMOE_ERR_INVALID_ARG;
    if (args->M < 0 || args->N < 0) return QMOE_ERR_INVALID_ARG;
    // M * N <= the array's size, checked without forming a product that could overflow
    if (args->N > 0 && args->M > static_cast<int64_t>(QMOE_NOALLOC_ACCUM_MAX_ELEMS) / args->N)
        return QMOE_ERR_UNSUPPORTED;
    qmoe_status_t st = QMOE_OK;
    float* scratch = scratch_for_current_device(&st);
    if (st != QMOE_OK) return st;
    qmoe_gemm_args a = *args;
    a.accum = scratch;  // zeroed (first M*N floats) on the stream by the regular path
    return qmoe_moe_gemm_w8a8(&a, stream);
}
