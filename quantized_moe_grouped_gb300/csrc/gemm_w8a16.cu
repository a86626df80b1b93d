// gemm_w8a16.cu -- INT8 W8A16 grouped GEMM entry point (in-kernel int8 -> bf16,
// tcgen05 kind::f16 with bf16 operands).
#include "gemm_kernel.cuh"

extern "C" qmoe_status_t qmoe_moe_gemm_w8a16(const qmoe_gemm_args* args, qmoe_stream_t stream) {
    return qmoe::run_moe_gemm<true>(args, stream);
}
