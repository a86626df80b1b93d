/*
 * qmoe_oracle.c -- plain, slow CPU oracle for the quantized MoE grouped GEMM path.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the library path may call, link or
 * load this file; only the tests, the smoke check and the benchmark's
 * CPU-baseline leg do.  It shares no code, header, table or constant
 * generator with the CUDA sources.
 *
 * Build: gcc -O2 -std=gnu11 -ffp-contract=off -fno-fast-math -fopenmp -shared -fPIC
 * (contraction is off so that every fp32 expression below rounds exactly as
 * written: one rounding per operation, fmaf only where it is spelled out).
 *
 * What it follows:
 *  - The grouped GEMM: tokens A[M,K] routed to top_k of E experts,
 *    out[m,j,:] = w[m,j] * dequant(Aq[m]) . dequant(Wq[e = topk_ids[m,j]])^T,
 *    in the two precisions benchmarked by "Tianxing/moe quantization"
 *    (ROCm/triton PR 693): FP8_W8A8 and INT8_W8A16 (tables "FP8_W8A8 Benchmark"
 *    and "INT8_W8A16 Benchmark", columns M, K, N, E, top_k).  Dequantisation is
 *    to fp64 and the sum is a dense per-token expert loop.
 *  - Dynamic per-token activation quantisation and per-channel weight
 *    quantisation (the "fp8dq" and "int8wo" recipes listed in "Enabling MOE
 *    Quantization using linear decomposition", pytorch/ao PR 2043, Summary):
 *    per row amax -> scale = amax/448 -> e4m3, or amax/127 -> int8.
 *  - SwiGLU + MXFP8 1x32 requantisation with per-expert row padding of the
 *    rowwise scale factors to 128 rows, as described in "[PyTorch] Let
 *    GroupedLinear accept MXFP8 input and gradient" (TransformerEngine PR 2099,
 *    Description and the two-expert [64,128] example).
 *  - Number formats from the OCP 8-bit floating point (E4M3) and OCP
 *    Microscaling (E8M0) specifications.
 *
 * Readings where the pages are silent (stated once here, used below):
 *  - e4m3 encode: round-to-nearest-even, saturating to +-448, sign of zero kept.
 *  - scale = amax / 448 with IEEE fp32 division; amax == 0 gives scale 1.
 *  - element code = e4m3(x / scale), IEEE fp32 division then e4m3 rounding.
 *  - MX block exponent: smallest integer e with 448 * 2^e >= amax (clamped to
 *    [-127, 127]); amax == 0 gives e = 0; code = e4m3(h * 2^-e).
 *  - SiLU uses one fixed fp32 operation sequence for exp (Cody-Waite range
 *    reduction, Cody & Waite 1980, plus a degree-7 Taylor polynomial) so that
 *    both implementations of the path produce identical fp32 h.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* ------------------------------------------------------------------------- */
/* bit helpers                                                                */
/* ------------------------------------------------------------------------- */
static float f32_from_bits(uint32_t u) { float f; memcpy(&f, &u, 4); return f; }
static uint32_t bits_from_f32(float f) { uint32_t u; memcpy(&u, &f, 4); return u; }

int orc_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

void orc_set_num_threads(int n) {
#ifdef _OPENMP
    if (n > 0) omp_set_num_threads(n);
#else
    (void)n;
#endif
}

/* ------------------------------------------------------------------------- */
/* bf16: the upper half of an fp32 word, rounded to nearest even              */
/* ------------------------------------------------------------------------- */
uint16_t orc_bf16_from_f32(float x) {
    uint32_t u = bits_from_f32(x);
    uint32_t lsb = (u >> 16) & 1u;
    u += 0x7FFFu + lsb;
    return (uint16_t)(u >> 16);
}

float orc_bf16_to_f32(uint16_t h) { return f32_from_bits((uint32_t)h << 16); }

/* orc_bf16_from_f32 over an array (marshalling only). */
void orc_bf16_from_f32_array(const float* x, int64_t n, uint16_t* h) {
    for (int64_t i = 0; i < n; ++i) h[i] = orc_bf16_from_f32(x[i]);
}

/* ------------------------------------------------------------------------- */
/* OCP E4M3: 1 sign, 4 exponent (bias 7), 3 mantissa bits; no infinities;    */
/* S.1111.111 is NaN; largest finite 1.75 * 2^8 = 448; subnormals m * 2^-9.  */
/* ------------------------------------------------------------------------- */
double orc_e4m3_to_f64(uint8_t b) {
    int s = b >> 7, e = (b >> 3) & 0xF, m = b & 7;
    double v;
    if (e == 15 && m == 7) return NAN;
    if (e == 0) v = ldexp((double)m, -9);            /* (m/8) * 2^(1-7) */
    else v = ldexp((double)(8 + m), e - 10);         /* (1 + m/8) * 2^(e-7) */
    return s ? -v : v;
}

uint8_t orc_e4m3_from_f32(float xf) {
    uint8_t sign = signbit(xf) ? 0x80 : 0x00;
    if (isnan(xf)) return (uint8_t)(sign | 0x7F);
    double a = fabs((double)xf);                     /* exact */
    if (a >= 448.0) return (uint8_t)(sign | 0x7E);   /* saturate (and +-inf) */
    if (a < ldexp(1.0, -6)) {
        /* subnormal grid, spacing 2^-9; q == 8 is the smallest normal, code 0x08 */
        double q = rint(ldexp(a, 9));                /* a * 2^9 is exact; rint = RNE */
        return (uint8_t)(sign | (uint8_t)q);
    }
    int ex;
    double fr = frexp(a, &ex);                       /* a = fr * 2^ex, fr in [0.5, 1) */
    int E = ex - 1;                                  /* a = (2 fr) * 2^E            */
    double q = rint(ldexp(fr, 4));                   /* (2 fr) * 8, RNE, in [8, 16] */
    if (q == 16.0) { q = 8.0; E += 1; }
    int biased = E + 7;
    if (biased > 15 || (biased == 15 && (int)q - 8 == 7)) return (uint8_t)(sign | 0x7E);
    return (uint8_t)(sign | (uint8_t)((biased << 3) | ((int)q - 8)));
}

/* OCP E8M0: value 2^(b - 127); 0xFF is NaN. */
double orc_e8m0_to_f64(uint8_t b) {
    if (b == 0xFF) return NAN;
    return ldexp(1.0, (int)b - 127);
}

/* Smallest integer e with 448 * 2^e >= a, clamped to [-127, 127]; a == 0 -> 0.
 * Write a = m * 2^Ea with m in [1, 2).  448 = 1.75 * 2^8, so the bound holds
 * at e = Ea - 8 exactly when m <= 1.75, and otherwise first at e = Ea - 7. */
int orc_mx_scale_exponent(float a) {
    if (a == 0.0f) return 0;
    int ex;
    double fr = frexp((double)a, &ex);
    int Ea = ex - 1;
    double m = 2.0 * fr;
    int e = (m <= 1.75) ? Ea - 8 : Ea - 7;
    if (e < -127) e = -127;
    if (e > 127) e = 127;
    return e;
}

/* orc_mx_scale_exponent over an array (marshalling only). */
void orc_mx_scale_exponent_array(const float* a, int64_t n, int32_t* e) {
    for (int64_t i = 0; i < n; ++i) e[i] = orc_mx_scale_exponent(a[i]);
}

/* ------------------------------------------------------------------------- */
/* moe_align_block_size: sort token-slots by expert, pad each expert's group */
/* to a multiple of the tile size BM.                                        */
/*   slots s = 0..T-1 (s = m*top_k + j), expert e = topk_ids[s]              */
/*   cnt_e = #slots of e; padded_e = roundup(cnt_e, BM)                      */
/*   expert_offsets[e] = sum_{e'<e} cnt_e' ; padded_offsets[e] = sum padded   */
/*   sorted_ids[padded_offsets[e] + i] = i-th slot of e in ascending s        */
/*   pad entries hold the sentinel T; expert_ids[b] = expert owning block b, */
/*   -1 for blocks at or past num_post_padded.                               */
/* Returns 0, or 1 if some id is outside [0, E) (such slots are dropped).    */
/* ------------------------------------------------------------------------- */
int orc_moe_align(const int32_t* topk_ids, int64_t T, int32_t E, int32_t BM,
                  int32_t* sorted_ids, int64_t sorted_cap,
                  int32_t* expert_ids, int64_t blocks_cap,
                  int32_t* num_post_padded, int32_t* expert_offsets, int32_t* padded_offsets) {
    int bad = 0;
    int64_t* cnt = (int64_t*)calloc((size_t)E, sizeof(int64_t));
    int64_t* cursor = (int64_t*)calloc((size_t)E, sizeof(int64_t));
    for (int64_t s = 0; s < T; ++s) {
        int32_t e = topk_ids[s];
        if (e < 0 || e >= E) { bad = 1; continue; }
        cnt[e] += 1;
    }
    int64_t off = 0, poff = 0;
    for (int32_t e = 0; e < E; ++e) {
        expert_offsets[e] = (int32_t)off;
        padded_offsets[e] = (int32_t)poff;
        off += cnt[e];
        poff += (cnt[e] + BM - 1) / BM * BM;
    }
    expert_offsets[E] = (int32_t)off;
    padded_offsets[E] = (int32_t)poff;
    *num_post_padded = (int32_t)poff;
    for (int64_t i = 0; i < sorted_cap; ++i) sorted_ids[i] = (int32_t)T;
    for (int64_t s = 0; s < T; ++s) {                /* ascending s: stable */
        int32_t e = topk_ids[s];
        if (e < 0 || e >= E) continue;
        sorted_ids[padded_offsets[e] + cursor[e]] = (int32_t)s;
        cursor[e] += 1;
    }
    for (int64_t b = 0; b < blocks_cap; ++b) expert_ids[b] = -1;
    for (int32_t e = 0; e < E; ++e)
        for (int64_t p = padded_offsets[e]; p < padded_offsets[e + 1]; p += BM)
            expert_ids[p / BM] = e;
    free(cnt);
    free(cursor);
    return bad;
}

/* ------------------------------------------------------------------------- */
/* Per-row FP8 quantisation: amax -> scale = amax/448 -> e4m3(x/scale).       */
/* Used for dynamic per-token activations (bf16 input) and per-output-channel */
/* weights (fp32 input, one row per (expert, output channel)).                */
/* ------------------------------------------------------------------------- */
static void quant_row_fp8(const float* x, int64_t cols, uint8_t* q, float* scale) {
    float amax = 0.0f;
    for (int64_t c = 0; c < cols; ++c) {
        float a = fabsf(x[c]);
        if (a > amax) amax = a;
    }
    float s = (amax == 0.0f) ? 1.0f : amax / 448.0f;
    *scale = s;
    for (int64_t c = 0; c < cols; ++c) q[c] = orc_e4m3_from_f32(x[c] / s);
}

void orc_quant_rows_fp8_f32(const float* x, int64_t rows, int64_t cols, int64_t ldx,
                            uint8_t* q, float* scale) {
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < rows; ++r) quant_row_fp8(x + r * ldx, cols, q + r * cols, scale + r);
}

void orc_quant_rows_fp8_bf16(const uint16_t* x, int64_t rows, int64_t cols, int64_t ldx,
                             uint8_t* q, float* scale) {
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < rows; ++r) {
        float* tmp = (float*)malloc((size_t)cols * sizeof(float));
        for (int64_t c = 0; c < cols; ++c) tmp[c] = orc_bf16_to_f32(x[r * ldx + c]);
        quant_row_fp8(tmp, cols, q + r * cols, scale + r);
        free(tmp);
    }
}

/* Symmetric per-row INT8: scale = amax/127, q = clamp(rint(x/scale), -127, 127). */
void orc_quant_rows_int8_f32(const float* x, int64_t rows, int64_t cols, int64_t ldx,
                             int8_t* q, float* scale) {
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < rows; ++r) {
        const float* xr = x + r * ldx;
        float amax = 0.0f;
        for (int64_t c = 0; c < cols; ++c) {
            float a = fabsf(xr[c]);
            if (a > amax) amax = a;
        }
        float s = (amax == 0.0f) ? 1.0f : amax / 127.0f;
        scale[r] = s;
        for (int64_t c = 0; c < cols; ++c) {
            float v = rintf(xr[c] / s);
            if (v > 127.0f) v = 127.0f;
            if (v < -127.0f) v = -127.0f;
            q[r * cols + c] = (int8_t)v;
        }
    }
}

/* Symmetric INT4 in groups of 128 along the row (the "int4wo" weight-only
 * recipe named in "Enabling MOE Quantization using linear decomposition",
 * Summary; group size, symmetric range and scale format are this build's
 * reading): per group s0 = amax/7 (IEEE division), and the stored scale is s0
 * rounded up to the nearest fp32 value with at most 5 significant bits (1 for
 * an all-zero group), so that every dequantised weight q * scale (|q| <= 7,
 * at most 3 significant bits) has at most 8 significant bits and is a bf16
 * number, the operand format of a weight-only GEMM on bf16 activations;
 * q = clamp(rint(x/scale), -7, 7); two's-complement nibbles packed two per
 * byte, element 2j in the low nibble of byte j.  q is [rows, cols/2] bytes,
 * scale [rows, cols/128]. */
static float round_up_5bits(float s) {
    uint32_t b;
    memcpy(&b, &s, 4);
    if (b & 0x7FFFFu) b = (b | 0x7FFFFu) + 1u;  /* clear 19 low fraction bits, rounding up */
    memcpy(&s, &b, 4);
    return s;
}

void orc_quant_rows_int4_f32(const float* x, int64_t rows, int64_t cols, uint8_t* q, float* scale) {
    const int64_t G = cols / 128;
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < rows; ++r) {
        for (int64_t g = 0; g < G; ++g) {
            const float* xg = x + r * cols + g * 128;
            float amax = 0.0f;
            for (int64_t c = 0; c < 128; ++c) {
                float a = fabsf(xg[c]);
                if (a > amax) amax = a;
            }
            float s = (amax == 0.0f) ? 1.0f : round_up_5bits(amax / 7.0f);
            scale[r * G + g] = s;
            for (int64_t c = 0; c < 128; c += 2) {
                int v[2];
                for (int t = 0; t < 2; ++t) {
                    float f = rintf(xg[c + t] / s);
                    if (f > 7.0f) f = 7.0f;
                    if (f < -7.0f) f = -7.0f;
                    v[t] = (int)f;
                }
                q[r * (cols / 2) + (g * 128 + c) / 2] = (uint8_t)((v[0] & 0xF) | ((v[1] & 0xF) << 4));
            }
        }
    }
}

/* Value of nibble k of a packed INT4 row (two's complement). */
static int int4_at(const uint8_t* row, int64_t k) {
    int n = (row[k / 2] >> ((k & 1) * 4)) & 0xF;
    return (n >= 8) ? n - 16 : n;
}

/* ------------------------------------------------------------------------- */
/* exp in a fixed fp32 operation sequence.                                     */
/*  clamp x to [-104, 89]; n = rint(x * log2(e));                              */
/*  r = x - n*ln2 with ln2 split as hi + lo (hi = ln2 in fp32 with its low 12 */
/*  bits cleared, so n*hi is exact for |n| < 2^12; lo = fp32(ln2 - hi));      */
/*  p = sum_{k=0..7} r^k / k! by Horner with fused multiply-adds;             */
/*  result = (p * 2^n1) * 2^n2 with n1 = trunc(n/2), n2 = n - n1, so that the  */
/*  over- and underflow of the final scaling round like any fp32 product.     */
/* ------------------------------------------------------------------------- */
#define ORC_LOG2E   0x1.715476p+0f
#define ORC_LN2_HI  0x1.62ep-1f
#define ORC_LN2_LO  0x1.0bfbe8p-15f

float orc_exp_f32(float x) {
    /* Taylor coefficients 1/k!, rounded to fp32 */
    const float c[8] = {1.0f, 1.0f, 0.5f, 0x1.555556p-3f, 0x1.555556p-5f,
                        0x1.111112p-7f, 0x1.6c16c2p-10f, 0x1.a01a02p-13f};
    if (x < -104.0f) x = -104.0f;
    if (x > 89.0f) x = 89.0f;
    float t = x * ORC_LOG2E;
    float n = rintf(t);
    float r = fmaf(-n, ORC_LN2_HI, x);
    r = fmaf(-n, ORC_LN2_LO, r);
    float p = c[7];
    for (int k = 6; k >= 0; --k) p = fmaf(p, r, c[k]);
    int ni = (int)n;
    int n1 = ni / 2;                                 /* C division truncates */
    int n2 = ni - n1;
    float s1 = f32_from_bits((uint32_t)(n1 + 127) << 23);
    float s2 = f32_from_bits((uint32_t)(n2 + 127) << 23);
    float y = p * s1;
    return y * s2;
}

/* SwiGLU element: silu(g) * u with silu(g) = g * sigmoid(g) = g / (1 + exp(-g)),
 * evaluated as t = exp(-g); sig = 1/(1+t); h = (g*sig)*u  (all fp32, RN). */
float orc_silu_mul_f32(float g, float u) {
    float t = orc_exp_f32(-g);
    float den = 1.0f + t;
    float sig = 1.0f / den;
    float gs = g * sig;
    return gs * u;
}

/* Squared ReLU (the SReLU of "[PyTorch] Let GroupedLinear accept MXFP8 input
 * and gradient", Description): relu(x)^2 = x*x for x > 0, else 0.  For a bf16
 * x the fp32 product is exact. */
float orc_srelu_f32(float x) { return (x > 0.0f) ? x * x : 0.0f; }

/* h for one row.  act 0: SwiGLU of a fused gate|up row y[2I] (gate = first I
 * columns); act 1: SReLU of a plain row y[I]. */
static void act_row(int act, const uint16_t* yr, int64_t I, float* h) {
    for (int64_t i = 0; i < I; ++i)
        h[i] = (act == 0)   ? orc_silu_mul_f32(orc_bf16_to_f32(yr[i]), orc_bf16_to_f32(yr[I + i]))
               : (act == 1) ? orc_srelu_f32(orc_bf16_to_f32(yr[i]))
                            : orc_bf16_to_f32(yr[i]);  /* act 2: no activation (plain MXFP8 input) */
}

/* activation + per-token requantisation: h -> row amax -> scale -> e4m3(h/scale). */
static void act_quant_token(int act, const uint16_t* y, int64_t R, int64_t I, int64_t ldy,
                            uint8_t* q, float* scale) {
#pragma omp parallel for schedule(dynamic, 16)
    for (int64_t r = 0; r < R; ++r) {
        float* h = (float*)malloc((size_t)I * sizeof(float));
        act_row(act, y + r * ldy, I, h);
        quant_row_fp8(h, I, q + r * I, scale + r);
        free(h);
    }
}

void orc_silu_mul_quant_token(const uint16_t* y, int64_t R, int64_t I, int64_t ldy,
                              uint8_t* q, float* scale) {
    act_quant_token(0, y, R, I, ldy, q, scale);
}

void orc_srelu_quant_token(const uint16_t* y, int64_t R, int64_t I, int64_t ldy, uint8_t* q, float* scale) {
    act_quant_token(1, y, R, I, ldy, q, scale);
}

/* silu_mul_quant, MX mode: for each 1x32 block of h along the row, exponent
 * e (see orc_mx_scale_exponent), scale byte e+127, codes e4m3(h * 2^-e).
 * Rows are the expert-grouped compact rows r (expert e owns rows
 * [expert_offsets[e], expert_offsets[e+1])).  The rowwise scale matrix has
 * sf_padded_offsets[E] rows of sf_ld bytes: row r of expert e is stored at
 * sf_padded_offsets[e] + (r - expert_offsets[e]); every other byte (pad rows
 * of each expert, pad columns past I/32) is 0.  sf must hold
 * sf_padded_offsets[E] * sf_ld bytes. */
static void act_quant_mx(int act, const uint16_t* y, int64_t R, int64_t I, int64_t ldy,
                         const int32_t* expert_offsets, const int32_t* sf_padded_offsets, int32_t E,
                         uint8_t* q, uint8_t* sf, int64_t sf_ld) {
    memset(sf, 0, (size_t)sf_padded_offsets[E] * (size_t)sf_ld);
    int64_t nblk = I / 32;
#pragma omp parallel for schedule(dynamic, 16)
    for (int64_t r = 0; r < R; ++r) {
        int32_t e = 0;
        while (e < E && !(r >= expert_offsets[e] && r < expert_offsets[e + 1])) ++e;
        if (e >= E) continue;                          /* row not owned by any expert */
        int64_t srow = (int64_t)sf_padded_offsets[e] + (r - expert_offsets[e]);
        float* h = (float*)malloc((size_t)I * sizeof(float));
        act_row(act, y + r * ldy, I, h);
        for (int64_t b = 0; b < nblk; ++b) {
            float amax = 0.0f;
            for (int64_t k = 0; k < 32; ++k) {
                float a = fabsf(h[b * 32 + k]);
                if (a > amax) amax = a;
            }
            int ex = orc_mx_scale_exponent(amax);
            sf[srow * sf_ld + b] = (uint8_t)(ex + 127);
            float mul = ldexpf(1.0f, -ex);             /* exact power of two */
            for (int64_t k = 0; k < 32; ++k) q[r * I + b * 32 + k] = orc_e4m3_from_f32(h[b * 32 + k] * mul);
        }
        free(h);
    }
}

void orc_silu_mul_quant_mx(const uint16_t* y, int64_t R, int64_t I, int64_t ldy,
                           const int32_t* expert_offsets, const int32_t* sf_padded_offsets, int32_t E,
                           uint8_t* q, uint8_t* sf, int64_t sf_ld) {
    act_quant_mx(0, y, R, I, ldy, expert_offsets, sf_padded_offsets, E, q, sf, sf_ld);
}

void orc_srelu_quant_mx(const uint16_t* y, int64_t R, int64_t I, int64_t ldy,
                        const int32_t* expert_offsets, const int32_t* sf_padded_offsets, int32_t E,
                        uint8_t* q, uint8_t* sf, int64_t sf_ld) {
    act_quant_mx(1, y, R, I, ldy, expert_offsets, sf_padded_offsets, E, q, sf, sf_ld);
}

/* Plain MXFP8 quantisation of bf16 rows ("MXFP8 input" of "[PyTorch] Let
 * GroupedLinear accept MXFP8 input and gradient"): the MX rows above with no
 * activation, rowwise factors padded per expert to 128 rows. */
void orc_quant_mxfp8_rows(const uint16_t* y, int64_t R, int64_t I, int64_t ldy,
                          const int32_t* expert_offsets, const int32_t* sf_padded_offsets, int32_t E,
                          uint8_t* q, uint8_t* sf, int64_t sf_ld) {
    act_quant_mx(2, y, R, I, ldy, expert_offsets, sf_padded_offsets, E, q, sf, sf_ld);
}

/* Columnwise MXFP8 (the colwise scaling factors of the same page, Description:
 * a [128, 128] tensor has colwise factors [4, 128]; a [64, 128] one [4, 128],
 * its two blocks of rows padded to 4): in each column, blocks of 32
 * consecutive rows (the last block holds the rows that are left); per block
 * the MX rule on its amax gives e, the byte e + 127 goes to sf[rb * sf_ld + c]
 * and every element of the block becomes e4m3(x * 2^-e) in place.  sf has
 * sf_rows >= ceil(R/32) rows of sf_ld >= C bytes; entries outside the blocks
 * are zero. */
void orc_quant_mxfp8_cols_bf16(const uint16_t* x, int64_t R, int64_t C, int64_t ldx, uint8_t* q,
                               uint8_t* sf, int64_t sf_rows, int64_t sf_ld) {
    memset(sf, 0, (size_t)sf_rows * (size_t)sf_ld);
    int64_t nrb = (R + 31) / 32;
#pragma omp parallel for schedule(static)
    for (int64_t c = 0; c < C; ++c) {
        for (int64_t rb = 0; rb < nrb; ++rb) {
            int64_t r1 = (rb + 1) * 32 < R ? (rb + 1) * 32 : R;
            float amax = 0.0f;
            for (int64_t r = rb * 32; r < r1; ++r) {
                float a = fabsf(orc_bf16_to_f32(x[r * ldx + c]));
                if (a > amax) amax = a;
            }
            int ex = orc_mx_scale_exponent(amax);
            sf[rb * sf_ld + c] = (uint8_t)(ex + 127);
            float mul = ldexpf(1.0f, -ex);
            for (int64_t r = rb * 32; r < r1; ++r) q[r * C + c] = orc_e4m3_from_f32(orc_bf16_to_f32(x[r * ldx + c]) * mul);
        }
    }
}

/* MXFP8 weights: each of the R rows of C values (R = E*N weight rows, C = K)
 * in 1x32 blocks along the row with the same rule; sf[row * sf_ld + c/32],
 * columns past C/32 zero.  C is a multiple of 32. */
void orc_quant_rows_mxfp8_f32(const float* w, int64_t R, int64_t C, uint8_t* q, uint8_t* sf, int64_t sf_ld) {
    memset(sf, 0, (size_t)R * (size_t)sf_ld);
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < R; ++r) {
        for (int64_t b = 0; b < C / 32; ++b) {
            float amax = 0.0f;
            for (int64_t k = 0; k < 32; ++k) {
                float a = fabsf(w[r * C + b * 32 + k]);
                if (a > amax) amax = a;
            }
            int ex = orc_mx_scale_exponent(amax);
            sf[r * sf_ld + b] = (uint8_t)(ex + 127);
            float mul = ldexpf(1.0f, -ex);
            for (int64_t k = 0; k < 32; ++k) q[r * C + b * 32 + k] = orc_e4m3_from_f32(w[r * C + b * 32 + k] * mul);
        }
    }
}

/* MXFP8 weight factors in the tiled order the grouped GEMM reads (one
 * contiguous 1024-byte block per 256 weight rows x 128 K columns): block
 * ((e * NB + nb) * KB + kb) * 1024 with NB = ceil(N/256), KB = ceil(K/128);
 * inside it byte h*512 + i*16 + c*4 + b holds the factor of weight row
 * nb*256 + h*128 + 32c + i (h in 0..1, i in 0..31, c in 0..3) for K block
 * 4kb + b (b in 0..3), and 127 (2^0) for rows at or past N.  sf is
 * [E*N, sf_ld] with sf_ld >= 4*KB. */
void orc_mx_weight_sf_tiled(const uint8_t* sf, int64_t E, int64_t N, int64_t K, int64_t sf_ld, uint8_t* out) {
    const int64_t NB = (N + 255) / 256, KB = (K + 127) / 128;
    for (int64_t e = 0; e < E; ++e)
        for (int64_t nb = 0; nb < NB; ++nb)
            for (int64_t kb = 0; kb < KB; ++kb) {
                uint8_t* blk = out + ((e * NB + nb) * KB + kb) * 1024;
                for (int h = 0; h < 2; ++h)
                    for (int i = 0; i < 32; ++i)
                        for (int c = 0; c < 4; ++c)
                            for (int b = 0; b < 4; ++b) {
                                const int64_t n = nb * 256 + h * 128 + 32 * c + i;
                                blk[h * 512 + i * 16 + c * 4 + b] =
                                    (n < N) ? sf[(e * N + n) * sf_ld + 4 * kb + b] : (uint8_t)127;
                            }
            }
}

/* ------------------------------------------------------------------------- */
/* Router: softmax over the E logits of a token -> top-k -> renormalise (the  */
/* router sits in front of the grouped GEMM; the "top_k" column of the        */
/* "Tianxing/moe quantization" tables).  Softmax is strictly increasing, so   */
/* its top-k are the top-k logits, and the renormalised weights of the        */
/* selected experts are the softmax over the selected logits alone:           */
/*   e_1..e_k = the k largest logits in descending order, ties to the lower   */
/*   expert id (exact comparisons);  p_j = exp(l_{e_j} - l_{e_1}) with the    */
/*   fixed exp;  S = sum of p_j in selection order;  w_j = p_j / S  (fp32).   */
/* ------------------------------------------------------------------------- */
void orc_router_topk(const float* logits, int64_t M, int32_t E, int32_t k, int32_t* ids, float* w) {
#pragma omp parallel for schedule(static)
    for (int64_t m = 0; m < M; ++m) {
        const float* l = logits + m * E;
        int* taken = (int*)calloc((size_t)E, sizeof(int));
        float p[8];
        for (int j = 0; j < k; ++j) {
            int best = -1;
            for (int e = 0; e < E; ++e)
                if (!taken[e] && (best < 0 || l[e] > l[best])) best = e;
            taken[best] = 1;
            ids[m * k + j] = best;
        }
        const float top = l[ids[m * k]];
        float S = 0.0f;
        for (int j = 0; j < k; ++j) {
            p[j] = orc_exp_f32(l[ids[m * k + j]] - top);
            S = S + p[j];
        }
        for (int j = 0; j < k; ++j) w[m * k + j] = p[j] / S;
        free(taken);
    }
}

/* ------------------------------------------------------------------------- */
/* Grouped GEMM, dense per-token expert loop in fp64.                         */
/* For each listed slot s (slots[i]):                                          */
/*   e   = topk_ids[s]                                                         */
/*   a   = dequant(A[a_row[s], :])           (fp64)                            */
/*   out[i, n] = w[s] * sum_k a[k] * dequant(W[e, n, k])   for n < N          */
/* with w[s] = 1 when topk_w is NULL.  Layout of the result (slot order,      */
/* grouped order, sum over top_k) is left to the caller, which places rows.   */
/*                                                                            */
/* a_kind 0: e4m3 codes with one fp32 scale per A row (a_scale[row]);          */
/* a_kind 1: e4m3 codes with E8M0 scales per 1x32 block,                       */
/*           a_sf[a_sf_row[row] * a_sf_ld + k/32];                             */
/* a_kind 2: bf16 bit patterns (exact).                                        */
/* w_kind 0: e4m3 codes, w_kind 1: int8; both times w_scale[e*N + n];         */
/* w_kind 2: e4m3 codes with E8M0 scales per 1x32 block along K,               */
/*           w_sf[(e*N + n) * w_sf_ld + k/32] (times w_scale[e*N + n] if given).*/
/* w_kind 3: packed INT4 rows of K/2 bytes with one fp32 scale per group of    */
/*           128 along K, w_scale[(e*N + n) * (K/128) + k/128]; dequantised   */
/*           as q * scale in fp64 like every other kind.                      */
/* ------------------------------------------------------------------------- */
void orc_moe_gemm(int a_kind, const void* a, int64_t lda, const float* a_scale,
                  const uint8_t* a_sf, int64_t a_sf_ld, const int64_t* a_sf_row,
                  int w_kind, const void* w, const float* w_scale,
                  const uint8_t* w_sf, int64_t w_sf_ld,
                  const int32_t* topk_ids, const float* topk_w,
                  const int64_t* slots, int64_t n_slots, const int64_t* a_row,
                  int64_t N, int64_t K, double* out) {
    double lut[256];
    for (int b = 0; b < 256; ++b) lut[b] = orc_e4m3_to_f64((uint8_t)b);
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t i = 0; i < n_slots; ++i) {
        int64_t s = slots[i];
        int32_t e = topk_ids[s];
        int64_t ra = a_row[s];
        double* arow = (double*)malloc((size_t)K * sizeof(double));
        for (int64_t k = 0; k < K; ++k) {
            if (a_kind == 0) {
                arow[k] = lut[((const uint8_t*)a)[ra * lda + k]] * (double)a_scale[ra];
            } else if (a_kind == 1) {
                arow[k] = lut[((const uint8_t*)a)[ra * lda + k]] *
                          orc_e8m0_to_f64(a_sf[a_sf_row[ra] * a_sf_ld + k / 32]);
            } else {
                arow[k] = (double)orc_bf16_to_f32(((const uint16_t*)a)[ra * lda + k]);
            }
        }
        double ws = topk_w ? (double)topk_w[s] : 1.0;
        for (int64_t n = 0; n < N; ++n) {
            const int64_t wrow = ((int64_t)e * N + n) * K;
            const double sw = (w_scale && w_kind != 3) ? (double)w_scale[(int64_t)e * N + n] : 1.0;
            double acc = 0.0;
            if (w_kind == 3) {
                const uint8_t* wq = (const uint8_t*)w + ((int64_t)e * N + n) * (K / 2);
                const float* gs = w_scale + ((int64_t)e * N + n) * (K / 128);
                for (int64_t k = 0; k < K; ++k) acc += arow[k] * ((double)int4_at(wq, k) * (double)gs[k / 128]);
            } else if (w_kind == 0) {
                const uint8_t* wq = (const uint8_t*)w + wrow;
                for (int64_t k = 0; k < K; ++k) acc += arow[k] * (lut[wq[k]] * sw);
            } else if (w_kind == 2) {
                const uint8_t* wq = (const uint8_t*)w + wrow;
                const uint8_t* ws = w_sf + ((int64_t)e * N + n) * w_sf_ld;
                for (int64_t k = 0; k < K; ++k) acc += arow[k] * (lut[wq[k]] * orc_e8m0_to_f64(ws[k / 32]) * sw);
            } else {
                const int8_t* wq = (const int8_t*)w + wrow;
                for (int64_t k = 0; k < K; ++k) acc += arow[k] * ((double)wq[k] * sw);
            }
            out[i * N + n] = ws * acc;
        }
        free(arow);
    }
}

/* ------------------------------------------------------------------------- */
/* Array forms of the element functions above, for exhaustive comparisons.   */
/* ------------------------------------------------------------------------- */
void orc_e4m3_from_f32_array(const float* x, int64_t n, uint8_t* q) {
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; ++i) q[i] = orc_e4m3_from_f32(x[i]);
}

void orc_exp_f32_array(const float* x, int64_t n, float* y) {
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; ++i) y[i] = orc_exp_f32(x[i]);
}

void orc_silu_mul_f32_array(const float* g, const float* u, int64_t n, float* h) {
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; ++i) h[i] = orc_silu_mul_f32(g[i], u[i]);
}
