// gemm_w8a8.cu -- FP8 e4m3 W8A8 grouped GEMM entry point (tcgen05 kind::f8f6f4).
#include "gemm_kernel.cuh"

extern "C" qmoe_status_t qmoe_moe_gemm_w8a8(const qmoe_gemm_args* args, qmoe_stream_t stream) {
    return qmoe::run_moe_gemm<false>(args, stream);
}
