// mx_quant.cu -- MXFP8 quantisers for block-scaled operands ("[PyTorch] Let
// GroupedLinear accept MXFP8 input and gradient", Description and the
// two-expert example): weights in 1x32 blocks along K, and columnwise 32x1
// blocks.  Block rule: e = the smallest integer with 448 * 2^e >= amax
// (mx_block_exponent), byte e + 127, codes e4m3(x * 2^-e) with an exact
// power-of-two multiply.
#include "common.cuh"
#include "host_util.h"

namespace qmoe {

constexpr int kMxqThreads = 256;

// One thread per (row, 32-wide block) of fp32 rows; thread b == 0 of a row
// also zeroes the row's pad columns.
__global__ void __launch_bounds__(kMxqThreads)
    mx_rows_f32_kernel(const float* __restrict__ w, int64_t rows, int64_t cols, uint8_t* __restrict__ q,
                       uint8_t* __restrict__ sf, int64_t sf_ld) {
    const int64_t nblk = cols / 32;
    const int64_t g = blockIdx.x * static_cast<int64_t>(kMxqThreads) + threadIdx.x;
    if (g >= rows * nblk) return;
    const int64_t r = g / nblk;
    const int64_t b = g - r * nblk;
    const float4* src = reinterpret_cast<const float4*>(w + r * cols + b * 32);
    float v[32];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const float4 t = src[i];
        v[4 * i] = t.x;
        v[4 * i + 1] = t.y;
        v[4 * i + 2] = t.z;
        v[4 * i + 3] = t.w;
    }
    float a = 0.0f;
#pragma unroll
    for (int i = 0; i < 32; ++i) a = fmaxf(a, fabsf(v[i]));
    const int ex = mx_block_exponent(a);
    const float mul = pow2_neg(ex);
    uint32_t o[8];
#pragma unroll
    for (int i = 0; i < 8; ++i)
        o[i] = e4m3x4(__fmul_rn(v[4 * i], mul), __fmul_rn(v[4 * i + 1], mul), __fmul_rn(v[4 * i + 2], mul),
                      __fmul_rn(v[4 * i + 3], mul));
    uint8_t* qr = q + r * cols + b * 32;
    *reinterpret_cast<uint4*>(qr) = make_uint4(o[0], o[1], o[2], o[3]);
    *reinterpret_cast<uint4*>(qr + 16) = make_uint4(o[4], o[5], o[6], o[7]);
    uint8_t* sfr = sf + r * sf_ld;
    sfr[b] = static_cast<uint8_t>(ex + 127);
    if (b == 0)
        for (int64_t c = nblk; c < sf_ld; ++c) sfr[c] = 0;
}

// Columnwise: one thread per (32-row block rb, group of 8 columns) of the
// [sf_rows, sf_ld] factor grid.  Each row of the block is one 16-byte load of
// 8 bf16 (a warp reads 512 contiguous bytes per row); a first pass takes the 8
// column amaxes, a second re-reads the rows (from L1) and writes 8 codes per
// row.  Groups outside the data write zero factors.  cols % 8 == 0 and
// ldx % 8 == 0 (16-byte rows) on this path.
__global__ void __launch_bounds__(kMxqThreads)
    mx_cols_bf16_kernel(const uint16_t* __restrict__ x, int64_t rows, int64_t cols, int64_t ldx,
                        uint8_t* __restrict__ q, uint8_t* __restrict__ sf, int64_t sf_rows, int64_t sf_ld) {
    const int64_t groups = sf_ld / 8;
    const int64_t g = blockIdx.x * static_cast<int64_t>(kMxqThreads) + threadIdx.x;
    if (g >= sf_rows * groups) return;
    const int64_t rb = g / groups;
    const int64_t c0 = (g - rb * groups) * 8;
    const int64_t nrb = (rows + 31) / 32;
    uint8_t* sfp = sf + rb * sf_ld + c0;
    if (rb >= nrb || c0 >= cols) {
        *reinterpret_cast<uint2*>(sfp) = make_uint2(0u, 0u);
        return;
    }
    const int64_t r0 = rb * 32;
    const int n = static_cast<int>(rows - r0 < 32 ? rows - r0 : 32);
    const uint16_t* xp = x + r0 * ldx + c0;
    float a[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    for (int i = 0; i < n; ++i) {
        const uint4 w = *reinterpret_cast<const uint4*>(xp + i * ldx);
        a[0] = fmaxf(a[0], fabsf(bf16_lo(w.x)));
        a[1] = fmaxf(a[1], fabsf(bf16_hi(w.x)));
        a[2] = fmaxf(a[2], fabsf(bf16_lo(w.y)));
        a[3] = fmaxf(a[3], fabsf(bf16_hi(w.y)));
        a[4] = fmaxf(a[4], fabsf(bf16_lo(w.z)));
        a[5] = fmaxf(a[5], fabsf(bf16_hi(w.z)));
        a[6] = fmaxf(a[6], fabsf(bf16_lo(w.w)));
        a[7] = fmaxf(a[7], fabsf(bf16_hi(w.w)));
    }
    float mul[8];
    uint32_t e8[2] = {0u, 0u};
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        const int ex = mx_block_exponent(a[k]);
        mul[k] = pow2_neg(ex);
        e8[k >> 2] |= static_cast<uint32_t>(ex + 127) << (8 * (k & 3));
    }
    *reinterpret_cast<uint2*>(sfp) = make_uint2(e8[0], e8[1]);
    uint8_t* qp = q + r0 * cols + c0;
    for (int i = 0; i < n; ++i) {
        const uint4 w = *reinterpret_cast<const uint4*>(xp + i * ldx);
        const uint32_t lo = e4m3x4(__fmul_rn(bf16_lo(w.x), mul[0]), __fmul_rn(bf16_hi(w.x), mul[1]),
                                   __fmul_rn(bf16_lo(w.y), mul[2]), __fmul_rn(bf16_hi(w.y), mul[3]));
        const uint32_t hi = e4m3x4(__fmul_rn(bf16_lo(w.z), mul[4]), __fmul_rn(bf16_hi(w.z), mul[5]),
                                   __fmul_rn(bf16_lo(w.w), mul[6]), __fmul_rn(bf16_hi(w.w), mul[7]));
        *reinterpret_cast<uint2*>(qp + i * cols) = make_uint2(lo, hi);
    }
}

// Columnwise for shapes the vector path does not take (cols or ldx not a
// multiple of 8): one thread per factor (rb, c).
__global__ void __launch_bounds__(kMxqThreads)
    mx_cols_bf16_scalar_kernel(const uint16_t* __restrict__ x, int64_t rows, int64_t cols, int64_t ldx,
                               uint8_t* __restrict__ q, uint8_t* __restrict__ sf, int64_t sf_rows, int64_t sf_ld) {
    const int64_t g = blockIdx.x * static_cast<int64_t>(kMxqThreads) + threadIdx.x;
    if (g >= sf_rows * sf_ld) return;
    const int64_t rb = g / sf_ld;
    const int64_t c = g - rb * sf_ld;
    const int64_t nrb = (rows + 31) / 32;
    if (rb >= nrb || c >= cols) {
        sf[g] = 0;
        return;
    }
    const int64_t r0 = rb * 32;
    const int n = static_cast<int>(rows - r0 < 32 ? rows - r0 : 32);
    float a = 0.0f;
    for (int i = 0; i < n; ++i) a = fmaxf(a, fabsf(__uint_as_float(static_cast<uint32_t>(x[(r0 + i) * ldx + c]) << 16)));
    const int ex = mx_block_exponent(a);
    const float mul = pow2_neg(ex);
    sf[g] = static_cast<uint8_t>(ex + 127);
    for (int i = 0; i < n; ++i)
        q[(r0 + i) * cols + c] = static_cast<uint8_t>(
            e4m3x2(__fmul_rn(__uint_as_float(static_cast<uint32_t>(x[(r0 + i) * ldx + c]) << 16), mul), 0.0f) & 0xFFu);
}

// Tiled weight factors: one thread per 16-byte row (e, nb, kb, h, i) of the
// 1 KB blocks; its four 4-byte words are the factors of weight rows
// nb*256 + h*128 + 32c + i (c = 0..3) for K blocks 4kb .. 4kb+3, or 2^0
// (0x7F bytes) past N.
__global__ void __launch_bounds__(kMxqThreads)
    mx_weight_sf_tiled_kernel(const uint8_t* __restrict__ sf, int64_t E, int64_t N, int64_t NB, int64_t KB,
                              int64_t sf_ld, uint8_t* __restrict__ out) {
    const int64_t g = blockIdx.x * static_cast<int64_t>(kMxqThreads) + threadIdx.x;
    if (g >= E * NB * KB * 64) return;
    const int64_t blk = g >> 6;  // (e * NB + nb) * KB + kb
    const int row = static_cast<int>(g & 63);  // h * 32 + i
    const int64_t kb = blk % KB;
    const int64_t enb = blk / KB;
    const int64_t nb = enb % NB;
    const int64_t e = enb / NB;
    const int h = row >> 5, i = row & 31;
    uint32_t w[4];
#pragma unroll
    for (int c = 0; c < 4; ++c) {
        const int64_t n = nb * 256 + h * 128 + 32 * c + i;
        w[c] = (n < N) ? *reinterpret_cast<const uint32_t*>(sf + (e * N + n) * sf_ld + 4 * kb) : 0x7F7F7F7Fu;
    }
    *reinterpret_cast<uint4*>(out + blk * 1024 + h * 512 + i * 16) = make_uint4(w[0], w[1], w[2], w[3]);
}

}  // namespace qmoe

using namespace qmoe;

extern "C" {

qmoe_status_t qmoe_quant_weight_mxfp8(const float* w, int64_t rows, int64_t cols, uint8_t* q, uint8_t* sf,
                                      int64_t sf_ld, qmoe_stream_t stream) {
    if (rows < 0 || cols < 32 || cols % 32 != 0 || sf_ld < (cols / 32 + 3) / 4 * 4) return QMOE_ERR_INVALID_ARG;
    if (rows == 0) return QMOE_OK;
    if (!w || !q || !sf || !aligned16(w) || !aligned16(q)) return QMOE_ERR_INVALID_ARG;
    const int64_t items = rows * (cols / 32);
    const int64_t blocks = (items + kMxqThreads - 1) / kMxqThreads;
    if (blocks > 0x7FFFFFFF) return QMOE_ERR_UNSUPPORTED;
    mx_rows_f32_kernel<<<static_cast<unsigned>(blocks), kMxqThreads, 0, stream>>>(w, rows, cols, q, sf, sf_ld);
    return launch_status();
}

qmoe_status_t qmoe_quant_mxfp8_colwise(const uint16_t* x, int64_t rows, int64_t cols, int64_t ldx, uint8_t* q,
                                       uint8_t* sf, int64_t sf_rows, int64_t sf_ld, qmoe_stream_t stream) {
    if (rows < 0 || cols < 1 || ldx < cols || sf_ld < cols || sf_rows < (rows + 31) / 32) return QMOE_ERR_INVALID_ARG;
    if (rows == 0 && sf_rows == 0) return QMOE_OK;
    if ((rows > 0 && (!x || !q)) || !sf) return QMOE_ERR_INVALID_ARG;
    const bool vec = cols % 8 == 0 && ldx % 8 == 0 && sf_ld % 8 == 0 && aligned16(x) && aligned8(q) && aligned8(sf);
    const int64_t items = vec ? sf_rows * (sf_ld / 8) : sf_rows * sf_ld;
    const int64_t blocks = (items + kMxqThreads - 1) / kMxqThreads;
    if (blocks > 0x7FFFFFFF) return QMOE_ERR_UNSUPPORTED;
    if (vec)
        mx_cols_bf16_kernel<<<static_cast<unsigned>(blocks), kMxqThreads, 0, stream>>>(x, rows, cols, ldx, q, sf,
                                                                                      sf_rows, sf_ld);
    else
        mx_cols_bf16_scalar_kernel<<<static_cast<unsigned>(blocks), kMxqThreads, 0, stream>>>(x, rows, cols, ldx, q,
                                                                                             sf, sf_rows, sf_ld);
    return launch_status();
}

int64_t qmoe_mx_weight_sf_tiled_bytes(int64_t E, int64_t N, int64_t K) {
    if (E < 1 || N < 1 || K < 1) return -1;
    return E * ((N + 255) / 256) * ((K + 127) / 128) * 1024;
}

qmoe_status_t qmoe_mx_weight_sf_tiled(const uint8_t* sf, int64_t E, int64_t N, int64_t K, int64_t sf_ld, uint8_t* out,
                                      qmoe_stream_t stream) {
    if (E < 1 || N < 1 || K < 32 || K % 32 != 0) return QMOE_ERR_INVALID_ARG;
    const int64_t NB = (N + 255) / 256, KB = (K + 127) / 128;
    if (sf_ld < 4 * KB || sf_ld % 4 != 0 || !sf || !out || !aligned4(sf) || !aligned16(out))
        return QMOE_ERR_INVALID_ARG;
    const int64_t items = E * NB * KB * 64;
    const int64_t blocks = (items + kMxqThreads - 1) / kMxqThreads;
    if (blocks > 0x7FFFFFFF) return QMOE_ERR_UNSUPPORTED;
    mx_weight_sf_tiled_kernel<<<static_cast<unsigned>(blocks), kMxqThreads, 0, stream>>>(sf, E, N, NB, KB, sf_ld, out);
    return launch_status();
}

}  // extern "C"
