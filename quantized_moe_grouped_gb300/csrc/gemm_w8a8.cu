// gemm_w8a8.cu -- FP8 e4m3 W8A8 grouped GEMM entry point (tcgen05 kind::f8f6f4),
// and the bf16 rounding pass of the TOKEN_SUM layout shared by both precisions.
#include "gemm_kernel.cuh"

namespace qmoe {

// out = bf16(accum), 8 elements per step (n % 8 == 0, 16-byte aligned), else 1.
// Each thread has four steps' loads in flight before it converts them.
__global__ void token_sum_finalize_kernel(const float* __restrict__ accum, uint16_t* __restrict__ out, int64_t n) {
    pdl_launch_dependents();
    pdl_wait();  // the GEMM's sums are complete
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    const int64_t i0 = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x;
    if ((n & 7) == 0) {
        const float4* a4 = reinterpret_cast<const float4*>(accum);
        uint4* o4 = reinterpret_cast<uint4*>(out);
        const int64_t n8 = n / 8;
        int64_t i = i0;
        for (; i + 3 * stride < n8; i += 4 * stride) {
            float4 a[4], b[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                a[u] = __ldcs(a4 + 2 * (i + u * stride));
                b[u] = __ldcs(a4 + 2 * (i + u * stride) + 1);
            }
#pragma unroll
            for (int u = 0; u < 4; ++u)
                o4[i + u * stride] = make_uint4(pack_bf16x2(a[u].x, a[u].y), pack_bf16x2(a[u].z, a[u].w),
                                                pack_bf16x2(b[u].x, b[u].y), pack_bf16x2(b[u].z, b[u].w));
        }
        for (; i < n8; i += stride) {
            const float4 a = __ldcs(a4 + 2 * i), b = __ldcs(a4 + 2 * i + 1);
            o4[i] = make_uint4(pack_bf16x2(a.x, a.y), pack_bf16x2(a.z, a.w), pack_bf16x2(b.x, b.y),
                               pack_bf16x2(b.z, b.w));
        }
    } else {
        for (int64_t i = i0; i < n; i += stride) out[i] = static_cast<uint16_t>(pack_bf16x2(accum[i], 0.0f) & 0xFFFFu);
    }
}

// accum[0, n) = 0 before a TOKEN_SUM GEMM adds into it (n % 4 == 0, 16-byte
// aligned); launched like the GEMM so that it can start under the previous
// kernel's tail.
__global__ void token_sum_zero_kernel(float* __restrict__ accum, int64_t n) {
    pdl_launch_dependents();
    pdl_wait();  // earlier users of accum are complete
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    float4* a4 = reinterpret_cast<float4*>(accum);
    const float4 z = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
    for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < n / 4; i += stride) a4[i] = z;
}

// Per-token quantisation of the fp32 h rows (defined in align_quant.cu).
qmoe_status_t launch_quant_h_token(const float* h, const float* amax, int64_t rows, int64_t I, uint8_t* q,
                                   float* scale, cudaStream_t st);

qmoe_status_t launch_token_sum_finalize(const float* accum, uint16_t* out, int64_t n, cudaStream_t st) {
    if (n <= 0) return QMOE_OK;
    const int sms = device_sm_count();
    const int64_t work = (n & 7) == 0 ? n / 8 : n;
    int64_t blocks = (work + 255) / 256;
    const int64_t cap = static_cast<int64_t>(sms > 0 ? sms : 132) * 8;
    if (blocks > cap) blocks = cap;
    return launch_pdl(token_sum_finalize_kernel, dim3(static_cast<unsigned>(blocks)), dim3(256), 0, st, accum, out, n);
}

qmoe_status_t launch_token_sum_zero(float* accum, int64_t n, cudaStream_t st) {
    if (n <= 0) return QMOE_OK;
    const int sms = device_sm_count();
    int64_t blocks = (n / 4 + 255) / 256;
    const int64_t cap = static_cast<int64_t>(sms > 0 ? sms : 132) * 8;
    if (blocks > cap) blocks = cap;
    return launch_pdl(token_sum_zero_kernel, dim3(static_cast<unsigned>(blocks)), dim3(256), 0, st, accum, n);
}

}  // namespace qmoe

extern "C" qmoe_status_t qmoe_moe_gemm_w8a8(const qmoe_gemm_args* args, qmoe_stream_t stream) {
    return qmoe::run_moe_gemm<false>(args, stream);
}

extern "C" qmoe_status_t qmoe_debug_moe_gemm_tile(const qmoe_gemm_args* args, int32_t weights, int32_t tile,
                                                  qmoe_stream_t stream) {
    if (tile < qmoe::kTileAuto || tile > qmoe::kTilePair) return QMOE_ERR_INVALID_ARG;
    const qmoe::GemmTile t = static_cast<qmoe::GemmTile>(tile);
    switch (weights) {
        case 0: return qmoe::run_moe_gemm<false>(args, stream, nullptr, false, t);
        case 1: return qmoe::run_moe_gemm<true>(args, stream, nullptr, false, t);
        case 2: return qmoe::run_moe_gemm<true, true>(args, stream, nullptr, false, t);
        default: return QMOE_ERR_INVALID_ARG;
    }
}

extern "C" qmoe_status_t qmoe_moe_gemm_w8a8_silu_mxfp8(const qmoe_gemm_args* args, uint8_t* q, uint8_t* sf,
                                                      int64_t sf_ld, const int32_t* sf_padded_offsets,
                                                      qmoe_stream_t stream) {
    const qmoe::SwiGluOut so{q, sf, sf_ld, sf_padded_offsets, nullptr, nullptr};
    return qmoe::run_moe_gemm<false>(args, stream, &so);
}

extern "C" qmoe_status_t qmoe_moe_gemm_w8a8_silu_fp8_token(const qmoe_gemm_args* args, uint8_t* q, float* scale,
                                                          float* h_scratch, qmoe_stream_t stream) {
    if (!args || args->struct_size < sizeof(qmoe_gemm_args)) return QMOE_ERR_INVALID_ARG;
    if (args->M < 0 || args->top_k < 1 || args->N % 256 != 0) return QMOE_ERR_INVALID_ARG;
    const int64_t T = args->M * args->top_k;
    if (T == 0) return qmoe::run_moe_gemm<false>(args, stream, nullptr, true);  // nothing to write
    if (!q || !scale || !h_scratch || !qmoe::aligned16(q) || !qmoe::aligned16(h_scratch)) return QMOE_ERR_INVALID_ARG;
    const int64_t I = args->N / 2;
    float* amax = h_scratch + T * I;  // the row maxima follow the h rows
    const qmoe::SwiGluOut so{nullptr, nullptr, 0, nullptr, h_scratch, amax};
    qmoe_status_t r = qmoe::run_moe_gemm<false>(args, stream, &so, true);
    if (r != QMOE_OK) return r;
    if (cudaMemsetAsync(amax, 0, static_cast<size_t>(T) * sizeof(float), stream) != cudaSuccess) return QMOE_ERR_CUDA;
    r = qmoe::run_moe_gemm<false>(args, stream, &so);
    if (r != QMOE_OK) return r;
    return qmoe::launch_quant_h_token(h_scratch, amax, T, I, q, scale, stream);
}
