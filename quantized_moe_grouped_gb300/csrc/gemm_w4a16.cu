// gemm_w4a16.cu -- INT4 weight-only ("int4wo") grouped GEMM entry point and
// its weight quantiser: packed int4 weights with one fp32 scale per output
// channel and 128-wide group of K, turned into bf16 (q * scale, exact for the
// quantiser's 5-bit scales) by the converter warps ahead of a tcgen05
// kind::f16 MMA on bf16 activations.
#include "gemm_kernel.cuh"

namespace qmoe {

constexpr int kI4QuantThreads = 128;

// One thread per (row, 128-wide group): scale = amax/7 (IEEE division) rounded
// up to the nearest value with at most 5 significant bits (1 for an all-zero
// group), so that q * scale for |q| <= 7 has at most 8 significant bits and
// the converters' bf16 rounding of it is exact; q = clamp(rint(x/scale), -7, 7),
// nibbles packed low-first.
__global__ void __launch_bounds__(kI4QuantThreads)
    quant_rows_int4_kernel(const float* __restrict__ w, int64_t rows, int64_t cols, uint8_t* __restrict__ q,
                           float* __restrict__ scale) {
    const int64_t G = cols / 128;
    const int64_t g = blockIdx.x * static_cast<int64_t>(kI4QuantThreads) + threadIdx.x;
    if (g >= rows * G) return;
    const int64_t r = g / G;
    const int64_t grp = g - r * G;
    const float4* src = reinterpret_cast<const float4*>(w + r * cols + grp * 128);
    float a = 0.0f;
#pragma unroll 8
    for (int i = 0; i < 32; ++i) {
        const float4 t = src[i];
        a = fmaxf(a, fmaxf(fmaxf(fabsf(t.x), fabsf(t.y)), fmaxf(fabsf(t.z), fabsf(t.w))));
    }
    float s = 1.0f;
    if (a != 0.0f) {
        uint32_t b = __float_as_uint(__fdiv_rn(a, 7.0f));
        if (b & 0x7FFFFu) b = (b | 0x7FFFFu) + 1u;  // clear the 19 low fraction bits, rounding up
        s = __uint_as_float(b);
    }
    scale[g] = s;
    uint4* dst = reinterpret_cast<uint4*>(q + r * (cols / 2) + grp * 64);
#pragma unroll
    for (int v = 0; v < 4; ++v) {  // 32 values -> 16 bytes
        uint32_t word[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const float4 x0 = src[v * 8 + 2 * j];
            const float4 x1 = src[v * 8 + 2 * j + 1];
            const float xs[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
            uint32_t wv = 0u;
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                const float f = fminf(fmaxf(rintf(__fdiv_rn(xs[k], s)), -7.0f), 7.0f);
                wv |= (static_cast<uint32_t>(static_cast<int>(f)) & 0xFu) << (4 * k);
            }
            word[j] = wv;
        }
        dst[v] = make_uint4(word[0], word[1], word[2], word[3]);
    }
}

}  // namespace qmoe

using namespace qmoe;

extern "C" {

qmoe_status_t qmoe_quant_weight_int4(const float* w, int64_t rows, int64_t cols, uint8_t* q, float* scale,
                                     qmoe_stream_t stream) {
    if (rows < 0 || cols < 128 || cols % 128 != 0) return QMOE_ERR_INVALID_ARG;
    if (rows == 0) return QMOE_OK;
    if (!w || !q || !scale || !aligned16(w) || !aligned16(q)) return QMOE_ERR_INVALID_ARG;
    const int64_t items = rows * (cols / 128);
    const int64_t blocks = (items + kI4QuantThreads - 1) / kI4QuantThreads;
    if (blocks > 0x7FFFFFFF) return QMOE_ERR_UNSUPPORTED;
    quant_rows_int4_kernel<<<static_cast<unsigned>(blocks), kI4QuantThreads, 0, stream>>>(w, rows, cols, q, scale);
    return launch_status();
}

qmoe_status_t qmoe_moe_gemm_w4a16(const qmoe_gemm_args* args, qmoe_stream_t stream) {
    return run_moe_gemm<true, true>(args, stream);
}

}  // extern "C"
