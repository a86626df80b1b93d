/*
 * qmoe.h -- C ABI of libqmoe.so: the quantized Mixture-of-Experts expert-FFN
 * grouped GEMM path on one GB300 (sm_103a).
 *
 * The problem: tokens A[M, K] are routed to top_k of E experts
 * (topk_ids[M, top_k], routing weights topk_weights[M, top_k]); slot
 * s = m*top_k + j of token m goes to expert e = topk_ids[m, j] and produces
 *     out[m, j, :] = w[m, j] * dequant(Aq[m]) . dequant(Wq[e])^T
 * in FP8-e4m3 W8A8 (dynamic per-token activation scales, per-output-channel
 * weight scales) or INT8 W8A16 (per-channel int8 weights against bf16
 * activations), the two precisions benchmarked in "Tianxing/moe
 * quantization" (ROCm/triton PR 693, tables "FP8_W8A8 Benchmark" and
 * "INT8_W8A16 Benchmark", columns M K N E top_k).
 *
 * Conventions shared by every entry point
 *  - Tensor pointers are DEVICE pointers owned by the caller.  The library
 *    allocates no device memory and keeps no mutable global state except a
 *    per-device cache of attributes (SM count) and of kernel attributes.
 *  - Every call is asynchronous on the given stream (a cudaStream_t; NULL is
 *    the legacy default stream).  Nothing inside synchronises the host.
 *  - Arguments that can be checked on the host are checked before anything is
 *    launched; a failed check returns QMOE_ERR_INVALID_ARG or
 *    QMOE_ERR_UNSUPPORTED and launches nothing.  A failed launch returns
 *    QMOE_ERR_CUDA (the CUDA error is left for cudaGetLastError()).
 *  - Errors found on the device are OR-ed into *d_status (an int32 the caller
 *    zeroes and reads after its own synchronisation; may be NULL):
 *    QMOE_DEV_INVALID_EXPERT for an expert id outside [0, E),
 *    QMOE_DEV_TIMEOUT when a bounded wait inside a kernel gave up (the kernel
 *    then returns early; its outputs are undefined).
 *  - bf16 tensors are passed as uint16_t bit patterns; e4m3 and E8M0 as bytes.
 *  - Sizes are int64_t unless they are small counts (E, top_k, BM).  Row
 *    strides (ld*) are in elements.
 */
#ifndef QMOE_H
#define QMOE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* qmoe_stream_t; /* == cudaStream_t */

typedef enum {
    QMOE_OK = 0,
    QMOE_ERR_INVALID_ARG = 1,
    QMOE_ERR_UNSUPPORTED = 2,
    QMOE_ERR_CUDA = 3
} qmoe_status_t;

#define QMOE_DEV_INVALID_EXPERT 1
#define QMOE_DEV_TIMEOUT 2

/* activation scale modes */
#define QMOE_SCALE_PER_TOKEN 0 /* one fp32 scale per A row */
#define QMOE_SCALE_MX_1X32 1   /* one E8M0 byte per 32 elements along K */
#define QMOE_SCALE_PER_ROW 0   /* weights: one fp32 scale per output channel */
/* A row layouts.  GROUPED and PADDED rows reach the GEMM as TMA boxes and are
 * the fast layouts; TOKEN_GATHER rows are gathered by cp.async warps inside the
 * GEMM (measured on the FP8 decode shape: 1.02x the padded time at M=64,
 * 1.3x at M=512 with BM=128). */
#define QMOE_A_TOKEN_GATHER 0 /* slot s reads A row s / top_k ([M, K])        */
#define QMOE_A_GROUPED 1      /* slot s reads its compact expert-grouped row ([T, K]) */
#define QMOE_A_PADDED 2       /* slot at padded sorted position p reads row p
                                 ([qmoe_align_max_padded(T,E,BM), K], written by
                                 qmoe_quant_act_fp8_sorted)                      */
/* output layouts */
#define QMOE_OUT_SLOT 0      /* out[s, :] of [T, N] == [M, top_k, N]                  */
#define QMOE_OUT_GROUPED 1   /* out[compact row of s, :] of [T, N] (expert-contiguous) */
#define QMOE_OUT_TOKEN_SUM 2 /* out[m, :] = sum_j of slot m*top_k+j; [M, N]            */

const char* qmoe_status_string(qmoe_status_t st);
int qmoe_version(void);

/* ------------------------------------------------------------------------ */
/* moe_align_block_size                                                     */
/* ------------------------------------------------------------------------ */
/* Capacity (entries) that sorted_ids must have for T slots, E experts and
 * tile size BM: T + E*(BM-1), rounded up to a multiple of BM.  expert_ids
 * needs capacity/BM entries.  Returns -1 for invalid sizes. */
int64_t qmoe_align_max_padded(int64_t T, int32_t E, int32_t BM);

/* Sorts the T = M*top_k token-slots by expert and pads every expert's group
 * to a multiple of the tile size BM (integer work; one kernel launch).
 * The grouped GEMM needs its rows grouped by expert and each group padded to
 * its tile: this is the reading of the grouped ("fused") MoE kernel whose
 * benchmarks "Tianxing/moe quantization" prints, made explicit.
 *   topk_ids       [T]   int32, row-major [M, top_k], values in [0, E)
 *   sorted_ids     [cap] int32 out: expert e's slots, ascending s, start at
 *                  padded_offsets[e]; pad entries hold the sentinel T
 *   expert_ids     [cap/BM] int32 out: expert of block b, -1 past the end
 *   num_post_padded[1]  int32 out: sum_e roundup(cnt_e, BM)
 *   expert_offsets [E+1] int32 out: exclusive prefix sum of cnt_e
 *   padded_offsets [E+1] int32 out: exclusive prefix sum of roundup(cnt_e, BM)
 * Slots with an id outside [0, E) are dropped and flag QMOE_DEV_INVALID_EXPERT.
 * Limits: 1 <= E <= 256, 1 <= BM <= 1024, 0 <= T < 2^31 - E*BM. */
qmoe_status_t qmoe_moe_align_block_size(const int32_t* topk_ids, int64_t T, int32_t E, int32_t BM,
                                        int32_t* sorted_ids, int32_t* expert_ids,
                                        int32_t* num_post_padded, int32_t* expert_offsets,
                                        int32_t* padded_offsets, int32_t* d_status,
                                        qmoe_stream_t stream);

/* ------------------------------------------------------------------------ */
/* quantisers                                                               */
/* ------------------------------------------------------------------------ */
/* Dynamic per-token FP8 activation quantisation (the "fp8dq" recipe of
 * "Enabling MOE Quantization using linear decomposition", pytorch/ao PR 2043,
 * Summary): for each row r of the bf16 matrix x[rows, cols] (row stride ldx),
 * amax = max|x|, scale[r] = amax/448 (IEEE fp32 division; 1 if amax == 0),
 * q[r, c] = e4m3(x/scale) with round-to-nearest-even and saturation to +-448.
 *   q [rows, cols] bytes (row stride cols), scale [rows] fp32.
 * cols >= 1.  16-byte aligned rows (ldx % 8 == 0, x 16-B aligned, cols % 8 ==
 * 0) take the vector path; other shapes are accepted and give identical bytes. */
qmoe_status_t qmoe_quant_act_fp8(const uint16_t* x, int64_t rows, int64_t cols, int64_t ldx,
                                 uint8_t* q, float* scale, qmoe_stream_t stream);

/* The same per-token quantisation, with the rows written in the padded sorted
 * order of the grouped GEMM: for every padded position p < *num_post_padded
 * with s = sorted_ids[p] < T, row p of q (and scale[p]) is the quantised token
 * row x[s / top_k]; pad positions get zero codes and scale 0; rows at or past
 * *num_post_padded are not written.  This fuses the per-slot row gather into
 * the quantiser, so the GEMM reads its activation tiles as contiguous boxes
 * (QMOE_A_PADDED).  q holds cap = qmoe_align_max_padded(T, E, BM) rows of
 * cols bytes; scale cap floats.  Limits: cols % 16 == 0, ldx % 8 == 0,
 * x and q 16-byte aligned. */
qmoe_status_t qmoe_quant_act_fp8_sorted(const uint16_t* x, int64_t M, int64_t cols, int64_t ldx,
                                        const int32_t* sorted_ids, const int32_t* num_post_padded,
                                        int32_t top_k, int64_t cap, uint8_t* q, float* scale,
                                        qmoe_stream_t stream);

/* moe_align_block_size and qmoe_quant_act_fp8_sorted in one launch (for
 * T = M*top_k <= 4096; larger T issues the two launches).  Outputs are those
 * of the two calls -- identical align outputs, identical codes and scales at
 * every valid padded position -- except that pad rows of q and scale are not
 * written (the grouped GEMM never stores results of pad rows).  Each token row
 * is quantised once and copied to its top_k positions.  Limits as for the two
 * calls, with top_k <= 8. */
qmoe_status_t qmoe_moe_align_quant_fp8(const uint16_t* x, int64_t M, int64_t cols, int64_t ldx,
                                       const int32_t* topk_ids, int32_t top_k, int32_t E, int32_t BM,
                                       int32_t* sorted_ids, int32_t* expert_ids, int32_t* num_post_padded,
                                       int32_t* expert_offsets, int32_t* padded_offsets, uint8_t* q, float* scale,
                                       int32_t* d_status, qmoe_stream_t stream);

/* bf16 token rows copied into the padded sorted order of the grouped GEMM
 * (the activation operand of qmoe_moe_gemm_w8a16 with QMOE_A_PADDED): row p <
 * *num_post_padded of out is x[sorted_ids[p] / top_k], or zeros for a pad
 * position; rows at or past *num_post_padded are not written.  out holds
 * cap = qmoe_align_max_padded(T, E, BM) rows of cols bf16.  Limits: cols % 8
 * == 0, ldx % 8 == 0, x and out 16-byte aligned. */
qmoe_status_t qmoe_gather_sorted_bf16(const uint16_t* x, int64_t M, int64_t cols, int64_t ldx,
                                      const int32_t* sorted_ids, const int32_t* num_post_padded, int32_t top_k,
                                      int64_t cap, uint16_t* out, qmoe_stream_t stream);

/* Router (the step in front of the grouped GEMM; the "top_k" column of the
 * "Tianxing/moe quantization" tables): fp32 logits [M, E] -> softmax -> the
 * top_k experts -> weights renormalised to sum to one.  Softmax is strictly
 * increasing, so the selected experts are the top_k logits and their
 * renormalised weights are the softmax over the selected logits alone; per
 * token, in fp32: e_1..e_k = the top_k logits in descending order, ties to
 * the lower expert id; p_j = exp(l_{e_j} - l_{e_1}) (the same fixed exp as
 * qmoe_silu_mul_quant); S = sum of p_j in that order; w_j = p_j / S (IEEE).
 *   logits [M, E] fp32, finite, row-major; topk_ids [M, top_k] int32;
 *   topk_weights [M, top_k] fp32 (device memory, caller-owned).
 * Limits: 1 <= E <= 256, 1 <= top_k <= min(E, 8); else
 * QMOE_ERR_INVALID_ARG before any launch. */
qmoe_status_t qmoe_moe_router_topk(const float* logits, int64_t M, int32_t E, int32_t top_k, int32_t* topk_ids,
                                   float* topk_weights, qmoe_stream_t stream);

/* Router + moe_align_block_size + per-token quantisation in padded sorted
 * order, the decode-sized front of the grouped GEMM: one launch for M <= 64
 * (every CTA routes all M tokens itself), two for larger M with
 * T = M*top_k <= 4096 (the router, then align + quantisation in one launch),
 * three for larger T.  Outputs are those of
 * qmoe_moe_router_topk followed by qmoe_moe_align_quant_fp8 (pad rows of q and
 * scale not written).  Limits as there. */
qmoe_status_t qmoe_moe_route_align_quant_fp8(const float* logits, const uint16_t* x, int64_t M, int64_t cols,
                                             int64_t ldx, int32_t E, int32_t top_k, int32_t BM, int32_t* topk_ids,
                                             float* topk_weights, int32_t* sorted_ids, int32_t* expert_ids,
                                             int32_t* num_post_padded, int32_t* expert_offsets,
                                             int32_t* padded_offsets, uint8_t* q, float* scale, int32_t* d_status,
                                             qmoe_stream_t stream);

/* Per-output-channel weight quantisation, the same rule on fp32 rows: every
 * (expert, output channel) row of W[E, N, K] is one row (rows = E*N).
 * fp8: scale = amax/448, e4m3 codes; int8: scale = amax/127,
 * q = clamp(rint(w/scale), -127, 127) (the "int8wo" recipe of the same page). */
qmoe_status_t qmoe_quant_weight_fp8(const float* w, int64_t rows, int64_t cols,
                                    uint8_t* q, float* scale, qmoe_stream_t stream);
qmoe_status_t qmoe_quant_weight_int8(const float* w, int64_t rows, int64_t cols,
                                     int8_t* q, float* scale, qmoe_stream_t stream);

/* INT4 weight-only quantisation (the "int4wo" recipe named in "Enabling MOE
 * Quantization using linear decomposition", Summary; the pages do not define
 * it -- this library reads it as symmetric groups of 128 along K): every
 * fp32 row of cols (a multiple of 128) values, per 128-wide group
 * scale = amax/7 (IEEE division) rounded up to the nearest fp32 value with at
 * most 5 significant bits (1 for an all-zero group), so that every
 * dequantised weight q * scale is exactly a bf16 number;
 * q = clamp(rint(w/scale), -7, 7), two's-complement nibbles packed two per
 * byte with element 2j in the low nibble of byte j.
 *   q [rows, cols/2] bytes and w 16-byte aligned; scale [rows, cols/128] fp32. */
qmoe_status_t qmoe_quant_weight_int4(const float* w, int64_t rows, int64_t cols, uint8_t* q, float* scale,
                                     qmoe_stream_t stream);

/* MXFP8 weights ("[PyTorch] Let GroupedLinear accept MXFP8 input and
 * gradient", Description: block-scaled operands): every row of fp32 W
 * (rows = E*N, cols = K, K % 32 == 0) in 1x32 blocks along K; per block
 * e = the smallest integer with 448 * 2^e >= amax (clamped to [-127, 127];
 * 0 for an all-zero block), byte e + 127 at sf[row * sf_ld + k/32], codes
 * e4m3(w * 2^-e).  sf_ld >= roundup(K/32, 4); the columns past K/32 are
 * written as zero.  q [rows, K] e4m3, 16-byte aligned; w 16-byte aligned. */
qmoe_status_t qmoe_quant_weight_mxfp8(const float* w, int64_t rows, int64_t cols, uint8_t* q, uint8_t* sf,
                                      int64_t sf_ld, qmoe_stream_t stream);

/* Plain MXFP8 quantisation of bf16 rows (the "MXFP8 input" of the same page,
 * quantised as one concatenated tensor): the rowwise rule of
 * qmoe_quant_weight_mxfp8 on x [rows, I] (I % 32 == 0, ldx >= I, ldx % 8 == 0)
 * with the per-expert scale-factor layout of qmoe_silu_mul_quant's MX mode:
 * row r of expert e has its factors at sf row sf_padded_offsets[e] + (r -
 * expert_offsets[e]), each expert's block padded with zero rows to
 * sf_padded_offsets[e+1], row stride sf_ld >= roundup(I/32, 4) (pad columns
 * zero).  q [rows, I]. */
qmoe_status_t qmoe_quant_mxfp8(const uint16_t* x, int64_t rows, int64_t I, int64_t ldx, uint8_t* q, uint8_t* sf,
                               int64_t sf_ld, const int32_t* expert_offsets, const int32_t* sf_padded_offsets,
                               int32_t E, int32_t* d_status, qmoe_stream_t stream);

/* Columnwise MXFP8 (the colwise scaling factors of the same page: a [128,
 * 128] tensor has colwise factors of shape [4, 128]): in every column, blocks
 * of 32 consecutive rows (the last block holds the rows that are left) with
 * the same rule; factor of block rb of column c at sf[rb * sf_ld + c], codes
 * q[r * cols + c] = e4m3(x[r, c] * 2^-e) (same shape as x).  sf_rows >=
 * ceil(rows/32) and sf_ld >= cols; every factor outside the blocks is written
 * as zero (the page pads the block rows to a multiple of 4). */
qmoe_status_t qmoe_quant_mxfp8_colwise(const uint16_t* x, int64_t rows, int64_t cols, int64_t ldx, uint8_t* q,
                                       uint8_t* sf, int64_t sf_rows, int64_t sf_ld, qmoe_stream_t stream);

/* MXFP8 weight factors rearranged, once per weight matrix, into the order the
 * grouped GEMM streams them: one contiguous 1024-byte block per 256 weight
 * rows x 128 K columns, block ((e * NB + nb) * KB + kb) * 1024 with
 * NB = ceil(N/256), KB = ceil(K/128); inside a block, byte
 * h*512 + i*16 + c*4 + b is the factor of weight row nb*256 + h*128 + 32c + i
 * (h < 2, i < 32, c < 4) for K block 4kb + b (b < 4), and 127 (2^0) for rows
 * at or past N.  Each 512-byte half is the 32 x 16-byte matrix that
 * tcgen05.cp 32x128b.warpx4 copies into TMEM for the block-scaled MMA, so the
 * GEMM moves a stage's weight factors with one bulk copy.
 *   sf: [E*N, sf_ld] from qmoe_quant_weight_mxfp8 (sf_ld >= 4*KB, a multiple
 *   of 4, 4-byte aligned); out: qmoe_mx_weight_sf_tiled_bytes(E, N, K) bytes,
 *   16-byte aligned.  K % 32 == 0. */
int64_t qmoe_mx_weight_sf_tiled_bytes(int64_t E, int64_t N, int64_t K);
qmoe_status_t qmoe_mx_weight_sf_tiled(const uint8_t* sf, int64_t E, int64_t N, int64_t K, int64_t sf_ld, uint8_t* out,
                                      qmoe_stream_t stream);

/* ------------------------------------------------------------------------ */
/* grouped GEMM                                                             */
/* ------------------------------------------------------------------------ */
typedef struct {
    size_t struct_size;            /* sizeof(qmoe_gemm_args), for ABI evolution */
    /* activations */
    const void* a;                 /* e4m3 bytes (w8a8) or bf16 bits (w8a16)     */
    int64_t lda;                   /* row stride in elements                      */
    const float* a_scale;          /* PER_TOKEN: [rows of A] fp32 (w8a8 only)     */
    int32_t a_scale_mode;          /* QMOE_SCALE_*                                 */
    const uint8_t* a_sf;           /* MX: E8M0 [sf rows, a_sf_ld]                 */
    int64_t a_sf_ld;
    const int32_t* a_sf_padded_offsets; /* MX: [E+1] first sf row of each expert */
    int32_t a_layout;              /* QMOE_A_*                                     */
    /* weights W[E, N, K] (K contiguous) */
    const void* w;                 /* e4m3 bytes (w8a8) or int8 (w8a16)           */
    const float* w_scale;          /* [E, N] fp32 per output channel              */
    /* metadata from qmoe_moe_align_block_size with the same BM */
    const int32_t* sorted_ids;
    const int32_t* expert_ids;
    const int32_t* num_post_padded;
    const int32_t* expert_offsets;
    const int32_t* padded_offsets;
    const float* topk_weights;     /* [T] fp32 or NULL (no routing-weight multiply) */
    /* output, bf16 */
    uint16_t* out;
    int32_t out_layout;            /* QMOE_OUT_*                                   */
    int64_t M, N, K;
    int32_t E, top_k, BM;
    int32_t* d_status;
    /* QMOE_OUT_TOKEN_SUM only: fp32 [M, N] scratch owned by the caller (16-byte
     * aligned).  The library zeroes it, adds every routed slot result into it
     * in fp32, and writes out = bf16(accum) with a second launch. */
    float* accum;
    /* Weight scales.  QMOE_SCALE_PER_ROW (0): w_scale [E, N] fp32 per output
     * channel.  QMOE_SCALE_MX_1X32: MXFP8 weights (qmoe_quant_weight_mxfp8);
     * w_sf holds their E8M0 factors in the tiled order of
     * qmoe_mx_weight_sf_tiled (16-byte aligned); w_scale is then optional (an
     * extra fp32 factor per output channel, or NULL).  FP8 GEMM with MX
     * activations only. */
    int32_t w_scale_mode;
    const uint8_t* w_sf;
} qmoe_gemm_args;

/* FP8 W8A8 grouped GEMM (tables "FP8_W8A8 Benchmark" / "Model Results" of
 * "Tianxing/moe quantization"):
 *   out = w[s] * a_scale * w_scale[e, n] * sum_k e4m3(A)[k] * e4m3(W[e, n])[k]
 * with fp32 accumulation on the tensor cores and a bf16 (RNE) result.
 * Limits: K % 16 == 0, N % 16 == 0, 1 <= E <= 256, 1 <= top_k <= E,
 * BM in {16, 32, 64, 128, 256}, a and w 16-byte aligned, lda % 16 == 0.
 * TOKEN_SUM (the routing-weighted sum over the top_k slots of a token) needs
 * args->accum: the slot results are added into it with fp32 atomics and a
 * second launch rounds the sums to bf16 into out[M, N].  For top_k == 2 the
 * result does not depend on the order of the additions (0 + a + b == 0 + b + a
 * in IEEE arithmetic); for larger top_k the fp32 rounding order may vary.
 * QMOE_SCALE_MX_1X32 (the MXFP8 intermediate of qmoe_silu_mul_quant): A holds
 * e4m3 codes in compact grouped rows (QMOE_A_GROUPED) and a_sf their E8M0
 * scales, row r of expert e at sf row a_sf_padded_offsets[e] + (r -
 * expert_offsets[e]), one byte per 32 elements along K (row stride a_sf_ld, a
 * multiple of 4 and >= roundup(K/32, 4)); a_scale is unused.  The scales are
 * applied inside the tensor-core MMA (block-scaled kind::mxf8f6f4).  Needs
 * K % 32 == 0 and BM >= 128 (else QMOE_ERR_UNSUPPORTED).  With MX activations
 * the weights may be MXFP8 too (w_scale_mode QMOE_SCALE_MX_1X32): both
 * operands then carry their block scales into the MMA; MX weights with
 * per-token activations return QMOE_ERR_UNSUPPORTED. */
qmoe_status_t qmoe_moe_gemm_w8a8(const qmoe_gemm_args* args, qmoe_stream_t stream);

/* INT4 W4A16 grouped GEMM (weight-only int4 against bf16 activations):
 *   out = w[s] * sum_k a_bf16[k] * (q4[e, n, k] * scale[e, n, k/128])
 * with fp32 accumulation and a bf16 result.  args->w holds the packed int4
 * weights [E, N, K/2] of qmoe_quant_weight_int4 and args->w_scale their group
 * scales [E, N, K/128]; the converter warps form each bf16 weight as the fp32
 * product q * scale rounded to bf16 (RN) before the tensor-core MMA, which is
 * exact for the scales qmoe_quant_weight_int4 writes (other scales: the
 * product is rounded to bf16).
 * Activation and output layouts as qmoe_moe_gemm_w8a16.  Limits: K % 128 == 0,
 * BM in {64, 128, 256} (else QMOE_ERR_UNSUPPORTED), w_scale_mode PER_ROW. */
qmoe_status_t qmoe_moe_gemm_w4a16(const qmoe_gemm_args* args, qmoe_stream_t stream);

/* FP8 W8A8 grouped GEMM with the TOKEN_SUM layout that allocates nothing.
 * The pages have no counterpart to this entry point; it exists for callers
 * that cannot call cudaMalloc (allocator-managed runtimes that forbid it on
 * their hot path, plugins that only receive input and output buffers), which
 * therefore cannot provide args->accum.  It computes exactly what
 * qmoe_moe_gemm_w8a8 computes for QMOE_OUT_TOKEN_SUM, but the fp32
 * accumulation buffer is a fixed array of QMOE_NOALLOC_ACCUM_MAX_ELEMS floats
 * (16 MiB) compiled into the library: every GPU that loads the library holds
 * it until the process exits.  args->accum is ignored.
 *  - args->out_layout must be QMOE_OUT_TOKEN_SUM (else QMOE_ERR_INVALID_ARG);
 *    M*N above QMOE_NOALLOC_ACCUM_MAX_ELEMS returns QMOE_ERR_UNSUPPORTED and
 *    launches nothing.
 *  - The first call on a device looks up the array's device address (with
 *    that device current); make that first call before any stream capture.
 *    The address is kept per device and looked up again when the device's
 *    context has changed (after cudaDeviceReset, for example, the array has
 *    a new address); make the first call after such a reset before any
 *    stream capture too.
 *  - All calls share the one array: the first M*N floats are zeroed on the
 *    stream at every call, but calls whose work overlaps on the GPU (other
 *    streams, other host threads) race on it and must be serialised by the
 *    caller.
 *  - No cudaMalloc, cudaFree or allocating library call is made. */
#define QMOE_NOALLOC_ACCUM_MAX_ELEMS (4u << 20)
qmoe_status_t qmoe_moe_gemm_w8a8_token_sum_noalloc(const qmoe_gemm_args* args, qmoe_stream_t stream);

/* INT8 W8A16 grouped GEMM (table "INT8_W8A16 Benchmark"): int8 weights are
 * converted exactly to bf16 inside the kernel (offset-binary magic-number
 * conversion after the int8->fp16 trick of the "INT8 quantization support"
 * issue, casper-hansen/AutoAWQ 45, moved to fp32/bf16), multiplied with the
 * bf16 activations on the tensor cores with fp32 accumulation, and the
 * per-channel scale is applied in the epilogue:
 *   out = w[s] * w_scale[e, n] * sum_k A[k] * q[e, n, k].
 * Limits as for w8a8, with lda % 8 == 0 and a_scale unused. */
qmoe_status_t qmoe_moe_gemm_w8a16(const qmoe_gemm_args* args, qmoe_stream_t stream);

/* ------------------------------------------------------------------------ */
/* SwiGLU + requantisation                                                  */
/* ------------------------------------------------------------------------ */
/* y[rows, 2I] bf16 (row stride ldy) holds gate (first I columns) and up (last
 * I columns); h = silu(gate) * up in fp32 (silu(g) = g / (1 + exp(-g)),
 * with exp evaluated by a fixed fp32 Cody-Waite + degree-7 Taylor sequence so
 * that the result is reproducible bit for bit; silu(g) is within 3 ulp of
 * the exact value for g in [-87.3, 89], and is -0 for g < -88.72, where
 * exp(-g) overflows fp32 and the exact value is below 2.7e-37), then
 *  mode QMOE_SCALE_PER_TOKEN: scale[r] = amax_r/448, q = e4m3(h/scale);
 *  mode QMOE_SCALE_MX_1X32:   per 1x32 block along the row, e = smallest
 *    integer with 448*2^e >= block amax (clamped to [-127, 127], 0 for an
 *    all-zero block), sf byte e+127, q = e4m3(h*2^-e).
 * MX rows are the expert-grouped compact rows: expert e owns rows
 * [expert_offsets[e], expert_offsets[e+1]); its rowwise scale factors are
 * written at sf rows sf_padded_offsets[e] + (r - expert_offsets[e]), and its
 * pad rows up to sf_padded_offsets[e+1] and the pad columns past I/32 are
 * zeroed -- the per-expert scale-factor padding of "[PyTorch] Let
 * GroupedLinear accept MXFP8 input and gradient" (TransformerEngine PR 2099,
 * the two-expert [64,128] example), done in the same launch.
 *   q [rows, I] bytes; scale [rows] fp32 (PER_TOKEN); sf [.., sf_ld] (MX).
 * Limits: I % 8 == 0 (I % 32 == 0 for MX), ldy % 8 == 0, y 16-B aligned,
 * sf_ld >= I/32, 1 <= E <= 256 (MX). */
qmoe_status_t qmoe_silu_mul_quant(const uint16_t* y, int64_t rows, int64_t I, int64_t ldy,
                                  int32_t mode, uint8_t* q, float* scale, uint8_t* sf,
                                  int64_t sf_ld, const int32_t* expert_offsets,
                                  const int32_t* sf_padded_offsets, int32_t E,
                                  int32_t* d_status, qmoe_stream_t stream);

/* SReLU + requantisation, the second fused activation of "[PyTorch] Let
 * GroupedLinear accept MXFP8 input and gradient" (Description: "SReLU + MXFP8
 * Quantization"): y[rows, I] bf16 (not gated), h = relu(y)^2 in fp32 (exact
 * for bf16 inputs), then the same per-token or MX 1x32 requantisation, scale
 * layout and per-expert scale-factor padding as qmoe_silu_mul_quant.  Limits
 * as there, with ldy >= I. */
qmoe_status_t qmoe_srelu_quant(const uint16_t* y, int64_t rows, int64_t I, int64_t ldy, int32_t mode, uint8_t* q,
                               float* scale, uint8_t* sf, int64_t sf_ld, const int32_t* expert_offsets,
                               const int32_t* sf_padded_offsets, int32_t E, int32_t* d_status,
                               qmoe_stream_t stream);

/* FP8 up projection with SwiGLU + MXFP8 in the GEMM epilogue: the fused
 * activation + MXFP8 quantisation of "[PyTorch] Let GroupedLinear accept
 * MXFP8 input and gradient" (TransformerEngine PR 2099, Description) moved
 * into the producing GEMM.  The result is the same as
 *   qmoe_moe_gemm_w8a8(args) with out_layout QMOE_OUT_GROUPED -> y bf16 [T, N]
 *   qmoe_silu_mul_quant(y, rows = T, I = N/2, mode QMOE_SCALE_MX_1X32, ...)
 * bit for bit, but y never reaches memory: each bf16 value is rounded exactly
 * as that GEMM stores it and the SwiGLU and the 1x32 block factors are
 * computed from it in registers.  args describes the [gate | up] projection
 * (w [E, N, K] with gate rows [0, N/2) and up rows [N/2, N), per-row
 * w_scale, per-token a_scale, any activation layout); args->out and
 * args->accum are unused (out may be NULL) and out_layout must be
 * QMOE_OUT_GROUPED.  Outputs, as qmoe_silu_mul_quant's MX mode with
 * I = N/2: q [T, I] e4m3 codes in compact grouped rows (16-byte aligned) and
 * sf [.., sf_ld] E8M0 factors, row r of expert e at sf row
 * sf_padded_offsets[e] + (r - expert_offsets[e]); the expert's pad rows up to
 * sf_padded_offsets[e+1] and the columns past I/32 are zeroed.
 * sf_padded_offsets must be the padded_offsets of the BM = 128 align the GEMM
 * uses.  Limits: BM == 128, N % 256 == 0, sf_ld >= N/64, FP8 per-token
 * activations and per-row weights (MX operands: QMOE_ERR_UNSUPPORTED). */
qmoe_status_t qmoe_moe_gemm_w8a8_silu_mxfp8(const qmoe_gemm_args* args, uint8_t* q, uint8_t* sf, int64_t sf_ld,
                                           const int32_t* sf_padded_offsets, qmoe_stream_t stream);

/* The same fused [gate | up] projection with the per-token requantisation:
 * the result is that of qmoe_moe_gemm_w8a8 (QMOE_OUT_GROUPED) followed by
 * qmoe_silu_mul_quant(mode QMOE_SCALE_PER_TOKEN), bit for bit.  A row's scale
 * needs the amax of all its I = N/2 values, so the GEMM epilogue writes
 * h = silu(y_gate) * y_up in fp32 (y rounded to bf16 exactly as the GEMM
 * stores it) and reduces each row's amax |h|; a second launch forms
 * scale[r] = amax_r/448 (1 for an all-zero row) and q = e4m3(h/scale).
 *   q [T, I] e4m3 codes and scale [T] fp32, compact grouped rows.
 *   h_scratch: caller-owned fp32 scratch of T*I + T floats (16-byte aligned),
 *   overwritten (h, then the T row maxima, zeroed on the stream first).
 * args as for qmoe_moe_gemm_w8a8_silu_mxfp8 (out unused, out_layout
 * QMOE_OUT_GROUPED, BM == 128, N % 256 == 0, FP8 per-token operands).  Host
 * errors return before anything is launched. */
qmoe_status_t qmoe_moe_gemm_w8a8_silu_fp8_token(const qmoe_gemm_args* args, uint8_t* q, float* scale,
                                               float* h_scratch, qmoe_stream_t stream);

/* ------------------------------------------------------------------------ */
/* element-level hooks used by the exhaustive tests                         */
/* ------------------------------------------------------------------------ */
/* e4m3 codes of n fp32 values with the same conversion the kernels use. */
qmoe_status_t qmoe_debug_e4m3_encode(const float* x, uint8_t* q, int64_t n, qmoe_stream_t stream);
/* bf16 bit patterns of n int8 values through the in-kernel W8A16 operand
 * conversion (4 values per 32-bit word; n % 4 == 0, 4-byte aligned). */
qmoe_status_t qmoe_debug_int8_to_bf16(const int8_t* x, uint16_t* y, int64_t n, qmoe_stream_t stream);
/* h = silu(g) * u through the kernels' fp32 sequence, n values. */
qmoe_status_t qmoe_debug_silu_mul(const float* g, const float* u, float* h, int64_t n,
                                  qmoe_stream_t stream);
/* Failure-detection check: one thread waits, through the bounded wait every
 * GEMM pipeline wait uses, on an mbarrier nothing arrives at; after limit_ns
 * (at most 1 s) it gives up and ORs QMOE_DEV_TIMEOUT into *d_status.  The
 * kernel returns normally and the context stays usable. */
qmoe_status_t qmoe_debug_wait_timeout(int32_t* d_status, int64_t limit_ns, qmoe_stream_t stream);
/* q = x / s through the correctly rounded division by a row scale (like IEEE
 * fp32 division; the int8 weight quantiser's), n values. */
qmoe_status_t qmoe_debug_div_by_scale(const float* x, float s, float* q, int64_t n, qmoe_stream_t stream);
/* q[i] = the e4m3 code the quantisers write for x[i] / s (what
 * qmoe_quant_act_fp8 and the other per-row quantisers compute per value from
 * the row scale s), n values: the exhaustive check of that code path. */
qmoe_status_t qmoe_debug_quant_by_scale(const float* x, float s, uint8_t* q, int64_t n, qmoe_stream_t stream);
/* y[i] = 1/d[i] with the reciprocal the SiLU uses (correctly rounded, for
 * d >= 1): the exhaustive check of that sequence. */
qmoe_status_t qmoe_debug_rcp_ge1(const float* d, float* y, int64_t n, qmoe_stream_t stream);
/* A grouped GEMM with its tile family chosen by the caller, so that tests and
 * timings can run each family on any shape.  weights: 0 = qmoe_moe_gemm_w8a8,
 * 1 = qmoe_moe_gemm_w8a16, 2 = qmoe_moe_gemm_w4a16 (same arguments and
 * checks).  tile 0 = the library's own choice (exactly that entry point),
 * 1 = one CTA per tile, 2 = CTA pairs (two SMs per 256 x 256 tile through
 * tcgen05 cta_group::2; GROUPED or PADDED activation rows, per-token FP8
 * activation scales with BM >= 128 or bf16 activations, else
 * QMOE_ERR_UNSUPPORTED).  Any other weights or tile value returns
 * QMOE_ERR_INVALID_ARG. */
qmoe_status_t qmoe_debug_moe_gemm_tile(const qmoe_gemm_args* args, int32_t weights, int32_t tile,
                                       qmoe_stream_t stream);

#ifdef __cplusplus
}
#endif
#endif /* QMOE_H */
