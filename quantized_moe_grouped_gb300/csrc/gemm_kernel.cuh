// gemm_kernel.cuh -- persistent grouped GEMM for the MoE expert FFN on sm_103a.
//
// Two tile shapes share one warp-specialised kernel template:
//
//  * swapped (BM 16 or 32): one tile = 128 output channels n of one expert x
//    BN sorted slots (one BM block, BN == BM).  The weight rows are the MMA
//    "A" operand (M = 128) and the slot activations the "B" operand (N = BN),
//    so a handful of slots per expert still fills the tensor-core M dimension
//    while the kernel streams W at HBM rate.
//  * wide (BM >= 64): one tile = 128 sorted slots (MMA M) x 256 output
//    channels (MMA N), or at BM = 64 64 slots (M = 64 MMAs; the decode tile:
//    32 KB of weights per stage, where a fixed cost per ring stage made the
//    swapped tile's 16 KB stages the bound).  Per byte of weights it gathers a
//    quarter of the activation bytes the swapped shape would need at BN = 256.
//
// D lives in TMEM (fp32), double-buffered so the epilogue of one tile overlaps
// the main loop of the next.
//
// Warp roles (one CTA per SM, persistent over tiles, static round robin):
//   warp 0      TMA producer: weight tile W[e, n0:n0+WR, k0:k0+BK] -> smem ring,
//               and the activation tile when its rows are contiguous (GROUPED
//               compact rows or PADDED sorted rows)
//   warp 1      TMEM owner + single-thread tcgen05.mma issuer
//   warps 2-3   activation gather for TOKEN_GATHER: the tile's token rows with
//               16-byte cp.async into the 128-byte-swizzled K-major layout
//   warps 4-7   epilogue: TMEM -> registers, x w_scale[e,n] x a_scale x w[s],
//               bf16 store (TOKEN_SUM: fp32 vector atomic add into the
//               caller's accumulation buffer, rounded to bf16 by a second launch)
//   warps 8+    W8A16: int8 -> bf16 converters (raw ring -> main ring), two
//               groups (eight warps each for the wide tile, four for the
//               swapped one) taking alternate stages
//   warp  2     MX: the scale writer (activation factors -> shared memory;
//               the MMA thread copies them into TMEM), warps 8-11 a second
//               epilogue group
//   W4A16 (kI4): the converters also apply each row's scale per 128-wide
//               group of K while turning packed int4 into bf16
//
// Every wait is bounded (mbar_wait); on a timeout the CTA raises an abort
// flag, all roles leave their loops, copies in flight are drained and TMEM is
// released before the kernel returns with QMOE_DEV_TIMEOUT set.
#pragma once

#include "common.cuh"
#include "host_util.h"

#include <string.h>

#include <mutex>

namespace qmoe {

struct GemmParams {
    const uint8_t* a;            // activation base (bytes)
    int64_t lda_bytes;
    int64_t a_row_bytes;         // valid bytes per activation row (K * element size)
    const float* a_scale;        // per-row activation scale, or nullptr
    const int32_t* sorted_ids;
    const int32_t* expert_ids;
    const int32_t* num_post_padded;
    const int32_t* expert_offsets;
    const int32_t* padded_offsets;
    const float* topk_w;
    const float* w_scale;
    uint16_t* out;
    float* accum;                // TOKEN_SUM: fp32 [M, N] accumulation buffer
    int64_t N;
    int64_t T;
    int32_t E, top_k, a_layout, out_layout, BM;
    int32_t a_tma;               // 1: activation tiles by TMA (GROUPED / PADDED rows), 0: cp.async gather
    const uint8_t* a_sf;         // MX: E8M0 scale rows of the grouped activations
    int64_t a_sf_ld;
    const int32_t* a_sf_poff;    // MX: first scale row of each expert
    const uint8_t* w_sf;         // MX weights: E8M0 factors in 1 KB tiled blocks, or nullptr (2^0)
    const float* w_gscale;       // W4A16: fp32 scale per weight row and group of 128 along K
    int32_t w_groups;            // W4A16: K / 128
    int32_t num_k_blocks;
    int32_t* d_status;
    // SwiGLU epilogues (kAct): h = silu(gate) * up of the grouped rows, as
    // MXFP8 (kAct 1: e4m3 codes [T, N/2], E8M0 factors [rows, act_sf_ld]) or
    // as fp32 (kAct 2: act_h [T, N/2] and each row's running amax |h| in
    // act_amax [T], for the per-token quantisation that follows)
    uint8_t* act_q;
    uint8_t* act_sf;
    int64_t act_sf_ld;
    const int32_t* act_sf_poff;  // first factor row of each expert
    float* act_h;
    float* act_amax;
    // > 0: before waiting for the previous kernel, prefetch this many k-blocks of
    // the CTA's first weight tile into L2, the tile taken as if every expert had
    // one slot block (decode-sized launches; a wrong guess only costs bandwidth)
    int32_t l2_prefetch_kb;
};

constexpr int kGemmMaxE = 256;  // experts per call (the align's limit)

// kI4: W4A16 -- packed int4 weight tiles (32 bytes per row per stage) with a
// scale per 128-wide group along K, applied by the converters (wide tile only).
// kAct != 0: FP8 wide tile whose 256 weight rows are 128 gate rows
// [nb*128, +128) and the matching 128 up rows [N/2 + nb*128, +128) of a fused
// [gate | up] projection, with a SwiGLU epilogue: kAct 1 quantises h to MXFP8
// (one 1x32 block = 32 columns of one thread's row), kAct 2 writes fp32 h and
// the row amax.
template <bool kBF16, bool kWide, int BN, bool kMX = false, bool kI4 = false, int kAct = 0>
struct GemmCfg {
    // kW2 (wide, BN = 256): two 128-slot halves share every weight stage, one
    // accumulator each -- one weight pass serves both slot blocks of a 256 block
    static constexpr bool kW2 = kWide && BN == 256;
    static constexpr int kSlotRows = BN;                     // slots per tile
    static constexpr int kWRows = kWide ? 256 : 128;        // weight rows (output channels) per tile
    static constexpr int kMmaN = kWide ? 256 : BN;
    static constexpr int kBK = kBF16 ? 64 : 128;            // K elements per stage (128 bytes of MMA operand)
    static constexpr int kWBytes = kWRows * 128;
    static constexpr int kActBytes = kSlotRows * 128;
    static constexpr int kRawRowBytes = kI4 ? 32 : 64;     // raw weight bytes per row per stage
    static constexpr int kRawBytes = kBF16 ? kWRows * kRawRowBytes : 0;  // int8/int4 tile before conversion
    // Main ring: MMA operand tiles (weights -- converted to bf16 for W8A16 --
    // and activations).  W8A16 adds a separate, deeper ring of raw int8 weight
    // tiles so that the weight stream keeps many bytes in flight while the
    // converted tiles need only a few stages.
    static constexpr int kStageBytes = kWBytes + kActBytes;
    static constexpr int kStagesFit = (200 * 1024) / kStageBytes;
    static constexpr int kStages = kBF16 ? (kWide ? 3 : 4) : (kStagesFit > 8 ? 8 : kStagesFit);
    // W8A16 / W4A16: the raw ring gets what the main ring leaves of 216 KB (the raw weight
    // bytes in flight bound the decode stream: 3 -> 4 int8 stages took M = 64 at N = 14336
    // from 125 to 121 us and M = 1024 from 289 to 278 us)
    static constexpr int kRawFit = kBF16 ? (216 * 1024 - kStages * kStageBytes) / (kRawBytes > 0 ? kRawBytes : 1) : 0;
    static constexpr int kRawStages = kBF16 ? (kRawFit > 16 ? 16 : kRawFit) : 0;
    // cp.async completion lag (stages): the MMA can run kStages - kLag - 1 stages
    // ahead of the gather warps, so the lag shrinks when the ring is short.
    static constexpr int kLag = kStages >= 6 ? 3 : (kStages >= 5 ? 2 : 1);
    // TOKEN_GATHER activation gather: warps 2-3, and more warps after all the
    // others (the last two of the block, four for W8A16); MX tiles never gather
    static constexpr int kExtraGather = kMX ? 0 : (kBF16 ? 128 : 64);
    static constexpr int kBProdThreads = 64 + kExtraGather;
    // MX: two groups of four warps, one per column half; kW2: one per slot
    // half; kAct (SwiGLU epilogues): one per half of the tile's 128 h columns
    static constexpr int kEpiThreads = (kMX || kW2 || kAct != 0) ? 256 : 128;
    // MX: a stage's scales in shared memory, as 512-byte blocks of 32 x 16
    // bytes: the 128 activation rows, then the two 128-row halves of the 256
    // weight rows (MXFP8 weights only)
    static constexpr int kSfBytes = 512;
    static constexpr int kSfStageBytes = 3 * kSfBytes;
    // W8A16 converter group: 8 warps for the wide tile (256 weight rows per
    // stage), 4 for the swapped one; groups alternate stages
    static constexpr int kConvThreads = (kBF16 && kWide) ? 256 : 128;
    static constexpr int kConvGroups = kBF16 ? 2 : 1;       // converter groups alternate stages
    static constexpr int kThreads =
        (kBF16 ? 256 + 2 * kConvThreads : ((kMX || kW2 || kAct != 0) ? 384 : 256)) + kExtraGather;
    static constexpr int kFirstExtraGatherWarp = (kThreads - kExtraGather) / 32;
    static constexpr int kAccCols = kMmaN;                  // TMEM columns per accumulator
    // MX: one accumulator (256 columns), then four scale columns per stage for
    // the 128 activation rows (4-column aligned) and 8 columns of constant
    // weight scales 2^0 (8-column aligned), all copied in from shared memory
    // by the MMA thread.
    static constexpr int kAccBufs = (kMX || kW2) ? 1 : 2;   // kW2: the one buffer is both halves' accumulators
    static constexpr int kSfaCol = kAccCols;
    static constexpr int kSfbCol = (kAccCols + 4 * kStages + 7) / 8 * 8;
    static constexpr int kTmemCols = (kMX || kW2) ? 512 : (2 * kAccCols < 32 ? 32 : 2 * kAccCols);
    // MMA M: 128 rows, or 64 for the 64-slot wide tile (D row i then sits in TMEM
    // lane 32 * (i / 16) + i % 16: each warp's lane quadrant holds 16 rows in lanes 0-15)
    static constexpr int kMmaM = (kWide && BN == 64) ? 64 : 128;
    static constexpr int kRowsPerQuad = kMmaM / 4;
    static constexpr uint32_t kIdesc =
        kMX ? make_idesc_mx(128, kMmaN) : make_idesc(kBF16 ? kFmtBF16 : kFmtE4M3, kMmaM, kMmaN);
    // Tail split (plain FP8 wide tile): quarter tiles of 64 weight rows (MMA N = 64)
    static constexpr bool kTailSplit = kWide && !kBF16 && !kMX && kAct == 0 && !kW2;
    static constexpr int kQRows = 64;
    static constexpr uint32_t kIdescQ = make_idesc(kFmtE4M3, kMmaM, kQRows);
    static_assert(!kMX || (kWide && !kBF16), "MX scales: FP8 wide tile only");
    static_assert(!kI4 || (kBF16 && kWide), "W4A16: wide bf16 tile only");
    static_assert(!kWide || BN == 128 || BN == 256 || BN == 64, "wide tile: 64, 128 or 256 slots");
    static_assert(!(kWide && BN == 64) || (!kMX && kAct == 0), "64-slot wide tile: per-row scales, plain epilogue");
    static_assert(!kW2 || (!kBF16 && !kMX), "two-half tile: FP8 with per-row scales only");
    static_assert(kAct == 0 || (kWide && BN == 128 && !kBF16 && !kMX), "SwiGLU epilogue: FP8 wide 128-slot tile only");
    static_assert(!kMX || kSfbCol + 8 * kStages <= 512, "TMEM columns");  // per-stage weight scales
    static constexpr int kDynSmem =
        kStages * kStageBytes + kRawStages * kRawBytes + (kMX ? kStages * kSfStageBytes + kSfBytes : 0) + 1024;
    static_assert(kStages >= 2, "need at least two pipeline stages");
    static_assert(!kBF16 || kRawStages >= 2, "need at least two raw weight stages");
    static_assert(kMmaN % 16 == 0 && kMmaN >= 16 && kMmaN <= 256, "MMA N must be a multiple of 16 in [16, 256]");
    static_assert(kActBytes % 1024 == 0 && kWBytes % 1024 == 0 && kRawBytes % 1024 == 0, "1 KB tile alignment");
};

// Waits with a time limit but without honouring the abort flag (used for the
// final drains, which must finish even after an abort).
QMOE_DI bool mbar_wait_drain(uint64_t* bar, uint32_t parity, int32_t* d_status) {
    int dummy = 0;
    return mbar_wait(bar, parity, &dummy, d_status);
}

// L2 prefetch of one box of a tiled tensor map (no shared memory, no barrier).
QMOE_DI void tma_prefetch_l2_3d(const CUtensorMap* map, int x, int y, int z) {
    asm volatile("cp.async.bulk.prefetch.tensor.3d.L2.global.tile [%0, {%1, %2, %3}];" ::"l"(
                     reinterpret_cast<uint64_t>(map)),
                 "r"(x), "r"(y), "r"(z)
                 : "memory");
}

QMOE_DI uint32_t pack_bf16x2(float lo, float hi) {
    const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<const uint32_t*>(&v);
}

QMOE_DI void red_add_f32x2(float* dst, float a, float b) {
    asm volatile("red.global.add.v2.f32 [%0], {%1, %2};" ::"l"(dst), "f"(a), "f"(b) : "memory");
}
QMOE_DI void red_add_f32x4(float* dst, float a, float b, float c, float d) {
    asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(dst), "f"(a), "f"(b), "f"(c), "f"(d)
                 : "memory");
}

// 32 TMEM lanes x 32 consecutive 32-bit columns per warp.
QMOE_DI void tmem_ld32(uint32_t taddr, float (&v)[32]) {
    uint32_t r[32];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
        "%15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
          "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
          "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

// 32 columns of this warp's 32 TMEM lanes, without the wait: the caller issues
// several, then tmem_wait_ld_regs on each set before using the values.
QMOE_DI void tmem_ld32_nowait(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
        "%15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
          "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
          "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr));
}
QMOE_DI void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
// Ties the registers of an earlier tmem_ld32_nowait to a point after
// tmem_wait_ld, so that no use of them is scheduled before the wait.
QMOE_DI void tmem_wait_ld_regs(uint32_t (&r)[32]) {
    asm volatile(""
                 : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]), "+r"(r[7]),
                   "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]), "+r"(r[14]),
                   "+r"(r[15]), "+r"(r[16]), "+r"(r[17]), "+r"(r[18]), "+r"(r[19]), "+r"(r[20]), "+r"(r[21]),
                   "+r"(r[22]), "+r"(r[23]), "+r"(r[24]), "+r"(r[25]), "+r"(r[26]), "+r"(r[27]), "+r"(r[28]),
                   "+r"(r[29]), "+r"(r[30]), "+r"(r[31]));
}

template <bool kBF16, bool kWide, int BN, bool kMX, bool kI4, int kAct>
__global__ void __launch_bounds__(GemmCfg<kBF16, kWide, BN, kMX, kI4, kAct>::kThreads, 1)
    moe_gemm_kernel(const __grid_constant__ CUtensorMap tmap_w, const __grid_constant__ CUtensorMap tmap_a,
                    const __grid_constant__ CUtensorMap tmap_wq, const GemmParams p) {
    using C = GemmCfg<kBF16, kWide, BN, kMX, kI4, kAct>;
    constexpr int S = C::kStages;
    constexpr int SR = C::kSlotRows;
    constexpr int WR = C::kWRows;
    extern __shared__ uint8_t smem_raw[];
    constexpr int R = C::kRawStages > 0 ? C::kRawStages : 1;
    __shared__ uint64_t bar_full[S], bar_empty[S], bar_conv[S], bar_raw_full[R], bar_raw_empty[R];
    __shared__ uint64_t bar_tfull[2], bar_tempty[2], bar_drain;
    __shared__ uint32_t s_tmem_base;
    __shared__ int s_abort;
    __shared__ int32_t s_brow[SR];                 // activation producers: source row of each slot row (-1: zero)
    __shared__ float s_cscale[kWide ? 1 : SR];     // swapped epilogue: a_scale * routing weight per column
    __shared__ int32_t s_crow[kWide ? 1 : SR];     // swapped epilogue: output row per column (-1: padding)
    __shared__ float s_wsc[kWide ? WR : 1];        // wide epilogue: w_scale per column
    __shared__ int32_t s_poff[kGemmMaxE + 1];      // padded_offsets: first padded position of each expert
    __shared__ int32_t s_ppre[C::kW2 ? kGemmMaxE + 1 : 1];  // kW2: tile pairs of the experts before e

    const uint32_t raw_addr = smem_u32(smem_raw);
    uint8_t* smem = smem_raw + (((raw_addr + 1023u) & ~1023u) - raw_addr);
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    // MX scale staging: S stage buffers, then the constant weight-scale block
    auto sf_smem = [&](int s) {
        return smem + S * C::kStageBytes + C::kRawStages * C::kRawBytes + s * C::kSfStageBytes;
    };

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            // arrivals: the TMA thread (weights and/or activation tile), or the 64 gather threads;
            // MX adds the 32 lanes of the scale warp
            mbar_init(&bar_full[s], (p.a_tma ? 1 : (kBF16 ? 0 : 1) + C::kBProdThreads) + (kMX ? 32 : 0));
            mbar_init(&bar_empty[s], 1);
            mbar_init(&bar_conv[s], C::kConvThreads);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&bar_tfull[i], 1);
            mbar_init(&bar_tempty[i], C::kEpiThreads);
        }
        for (int r = 0; r < R; ++r) {
            mbar_init(&bar_raw_full[r], 1);
            mbar_init(&bar_raw_empty[r], C::kConvThreads);
        }
        mbar_init(&bar_drain, 1);
        s_abort = 0;
        fence_mbar_init();
    }
    if constexpr (kMX) {  // weight scales 2^0: E8M0 byte 127 everywhere
        if (threadIdx.x < C::kSfBytes / 4) reinterpret_cast<uint32_t*>(sf_smem(S))[threadIdx.x] = 0x7F7F7F7Fu;
        fence_proxy_async_smem();
    }
    if (warp == 1) tmem_alloc(&s_tmem_base, C::kTmemCols);
    // Everything above touches only this CTA's own resources and overlaps the
    // previous kernel on the stream; from here on the kernel reads the align
    // outputs, activations and weights and writes its outputs.
    pdl_launch_dependents();
    if (p.l2_prefetch_kb > 0 && threadIdx.x == 0) {
        // the weights are not written by the previous kernel: while it finishes,
        // bring the likely first weight tile into L2 (expert-major order with one
        // slot block per expert: tile t = expert t / n_blocks, weight block t % n_blocks)
        const int nbk = static_cast<int>((p.N + WR - 1) / WR);
        const int e0 = static_cast<int>(blockIdx.x) / nbk;
        const int nb0 = static_cast<int>(blockIdx.x) % nbk;
        if (e0 < p.E)
            for (int kb = 0; kb < p.l2_prefetch_kb && kb < p.num_k_blocks; ++kb)
                tma_prefetch_l2_3d(&tmap_w, kb * C::kBK, nb0 * WR, e0);
    }
    pdl_wait();
    for (int i = threadIdx.x; i <= p.E; i += blockDim.x) s_poff[i] = p.padded_offsets[i];
    if (C::kW2 && warp == 0) {
        // s_ppre[i] = sum over experts e < i of ceil(128-slot blocks of e / 2), a warp scan per 32 experts
        int base = 0;
        for (int c = 0; c <= p.E; c += 32) {
            const int i = c + lane;
            const int v = i < p.E ? ((p.padded_offsets[i + 1] - p.padded_offsets[i]) / 128 + 1) / 2 : 0;
            int x = v;
#pragma unroll
            for (int d = 1; d < 32; d <<= 1) {
                const int y = __shfl_up_sync(0xFFFFFFFFu, x, d);
                if (lane >= d) x += y;
            }
            if (i <= p.E) s_ppre[i] = base + x - v;
            base += __shfl_sync(0xFFFFFFFFu, x, 31);
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = s_tmem_base;
    volatile int* abort = &s_abort;

    const int n_blocks = static_cast<int>((p.N + WR - 1) / WR);
    const int num_tiles = C::kW2 ? s_ppre[p.E] * n_blocks : s_poff[p.E] / SR * n_blocks;
    constexpr int SRB = C::kW2 ? 128 : SR;  // padded rows per unit of the slot-block index sb
    const int nkb = p.num_k_blocks;
    auto w_tile = [&](int s) { return smem + s * C::kStageBytes; };
    auto act_tile = [&](int s) { return smem + s * C::kStageBytes + C::kWBytes; };
    auto raw_tile = [&](int r) { return smem + S * C::kStageBytes + r * C::kRawBytes; };
    // Tile order: expert by expert (expert e owns the slot blocks
    // [s_poff[e], s_poff[e+1]) / SR); inside an expert, weight block major and
    // slot block fastest.  The slot blocks that share a weight tile run at the
    // same time (one HBM read of the tile), and while an expert's weight tiles
    // stream its activation rows stay in L2.  Returns the expert, or -1 when
    // the tile is to be skipped: (tiles narrower than BM) a tile whose first
    // slot is padding -- valid slots precede the padding inside an expert's
    // region, so the whole tile is padding then.
    //
    // kW2: the tiles of an expert are the pairs of consecutive 128-slot blocks
    // of its region (the last pair may hold one block), numbered like the
    // blocks above; sb is then the index of the pair's first 128-slot block.
    auto tile_expert = [&](int tile, int& sb, int& nb) {
        if constexpr (C::kW2) {
            int lo = 0, hi = p.E - 1;
            while (lo < hi) {
                const int mid = (lo + hi + 1) >> 1;
                if (s_ppre[mid] * n_blocks <= tile) lo = mid;
                else hi = mid - 1;
            }
            const int np = s_ppre[lo + 1] - s_ppre[lo];
            const int local = tile - s_ppre[lo] * n_blocks;
            nb = local / np;
            sb = s_poff[lo] / 128 + 2 * (local % np);
            return lo;
        }
        int lo = 0, hi = p.E - 1;
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (s_poff[mid] / SR * n_blocks <= tile) lo = mid;
            else hi = mid - 1;
        }
        const int sb0 = s_poff[lo] / SR;
        const int nsb = s_poff[lo + 1] / SR - sb0;
        const int local = tile - sb0 * n_blocks;
        nb = local / nsb;
        sb = sb0 + local % nsb;
        if (SR < p.BM && p.sorted_ids[sb * SR] >= p.T) return -1;
        return lo;
    };
    // kW2: whether the tile's second 128-slot block lies in expert e's region
    // and holds a valid slot (valid slots precede the padding in a region)
    auto second_half = [&](int e, int sb) {
        return sb + 1 < s_poff[e + 1] / 128 && p.sorted_ids[(sb + 1) * 128] < p.T;
    };
    // Tail split (kTailSplit): when the last partial wave of the round robin
    // holds at most a quarter of the CTAs' worth of tiles, each of those tiles
    // runs as four quarter tiles of 64 weight rows (loaded through tmap_wq, MMA
    // N = 64), so the launch ends about a quarter of a tile's time after the
    // full waves instead of a whole tile's.  Every role walks the same work
    // items: items below full_tiles are the tiles above, item full_tiles + 4i + q
    // is quarter q of tile full_tiles + i.  qt = -1 for a whole tile.
    const int grid_n = static_cast<int>(gridDim.x);
    const int tail_r = (C::kTailSplit && num_tiles % grid_n != 0 && 4 * (num_tiles % grid_n) <= grid_n)
                           ? num_tiles % grid_n
                           : 0;
    const int full_tiles = num_tiles - tail_r;
    const int num_work = full_tiles + 4 * tail_r;
    auto work_tile = [&](int w, int& sb, int& nb, int& qt) {
        qt = -1;
        if (w >= full_tiles) {
            qt = (w - full_tiles) & 3;
            w = full_tiles + ((w - full_tiles) >> 2);
        }
        return tile_expert(w, sb, nb);
    };

    if (warp == 0) {
        // ------------------------------------------------ TMA producer ---
        if (lane == 0) {
            int it = 0;
            bool ok = true;
            // MXFP8 weights add the stage's 1 KB block of tiled weight factors
            const uint32_t tx = C::kWBytes + (p.a_tma ? C::kActBytes : 0) + (kMX && p.w_sf ? 2 * C::kSfBytes : 0);
            for (int tile = blockIdx.x; ok && tile < num_work; tile += gridDim.x) {
                int sb, nb;
                int qt;
                const int e = work_tile(tile, sb, nb, qt);
                if (e < 0) continue;
                // first activation row of the tile: padded position, or compact grouped row
                const int arow0 = (p.a_layout == QMOE_A_PADDED)
                                      ? sb * SRB
                                      : p.expert_offsets[e] + (sb * SRB - p.padded_offsets[e]);
                for (int kb = 0; kb < nkb; ++kb, ++it) {
                    if constexpr (kBF16) {  // raw int8 weights into their own ring
                        const int r = it % R;
                        const uint32_t rph = (it / R) & 1;
                        if (!mbar_wait(&bar_raw_empty[r], rph ^ 1, abort, p.d_status)) { ok = false; break; }
                        mbar_arrive_expect_tx(&bar_raw_full[r], C::kRawBytes);
                        tma_load_3d(&tmap_w, &bar_raw_full[r], raw_tile(r), kb * C::kRawRowBytes, nb * WR, e);
                    } else {
                        const int s = it % S;
                        const uint32_t ph = (it / S) & 1;
                        if (!mbar_wait(&bar_empty[s], ph ^ 1, abort, p.d_status)) { ok = false; break; }
                        // a quarter tile brings a quarter of the weight rows
                        mbar_arrive_expect_tx(&bar_full[s], qt < 0 ? tx : tx - (C::kWBytes - C::kWBytes / 4));
                        if constexpr (kAct != 0) {  // gate rows, then the matching up rows
                            tma_load_3d(&tmap_w, &bar_full[s], w_tile(s), kb * C::kBK, nb * 128, e);
                            tma_load_3d(&tmap_w, &bar_full[s], w_tile(s) + 128 * 128, kb * C::kBK,
                                        static_cast<int>(p.N / 2) + nb * 128, e);
                        } else if (C::kTailSplit && qt >= 0) {
                            tma_load_3d(&tmap_wq, &bar_full[s], w_tile(s), kb * C::kBK, nb * WR + qt * C::kQRows, e);
                        } else {
                            tma_load_3d(&tmap_w, &bar_full[s], w_tile(s), kb * C::kBK, nb * WR, e);
                        }
                        if (p.a_tma) tma_load_2d(&tmap_a, &bar_full[s], act_tile(s), kb * C::kBK, arow0);
                        if (kMX && p.w_sf)
                            bulk_load(sf_smem(s) + C::kSfBytes,
                                      p.w_sf + ((static_cast<int64_t>(e) * n_blocks + nb) * nkb + kb) * 2 * C::kSfBytes,
                                      2 * C::kSfBytes, &bar_full[s]);
                    }
                }
            }
            if (!ok) {  // let copies already issued land before the CTA can exit
                const uint64_t t0 = global_timer_ns();
                while (global_timer_ns() - t0 < 2000000ull) {}
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------ MMA issuer ---
        if (lane == 0) {
            int it = 0, tcount = 0;
            bool ok = true;
            if (kMX && !p.w_sf) {  // per-channel weights: constant block scales 2^0, two 4-column copies
                const uint64_t sd = desc_rows16_noswizzle(smem_u32(sf_smem(S)));
                tmem_cp_32x128b_x4(tmem_base + C::kSfbCol, sd);
                tmem_cp_32x128b_x4(tmem_base + C::kSfbCol + 4, sd);
            }
            for (int tile = blockIdx.x; ok && tile < num_work; tile += gridDim.x) {
                int sb, nb;
                int qt;
                const int e = work_tile(tile, sb, nb, qt);
                if (e < 0) continue;
                const int acc = tcount % C::kAccBufs;
                const uint32_t aph = (tcount / C::kAccBufs) & 1;
                if (!mbar_wait(&bar_tempty[acc], aph ^ 1, abort, p.d_status)) break;
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * C::kAccCols);
                const bool half2 = C::kW2 && second_half(e, sb);  // kW2: accumulator at columns +256
                for (int kb = 0; kb < nkb; ++kb, ++it) {
                    const int s = it % S;
                    const uint32_t ph = (it / S) & 1;
                    if (!mbar_wait(&bar_full[s], ph, abort, p.d_status)) { ok = false; break; }
                    if (kBF16 && !mbar_wait(&bar_conv[s], ph, abort, p.d_status)) { ok = false; break; }
                    tc_fence_after();
                    if constexpr (kMX) {  // this stage's scales, ahead of its MMAs in the same pipe
                        tmem_cp_32x128b_x4(tmem_base + C::kSfaCol + 4 * s, desc_rows16_noswizzle(smem_u32(sf_smem(s))));
                        if (p.w_sf) {  // weight rows 0-127 -> columns +0..3, rows 128-255 -> +4..7
                            tmem_cp_32x128b_x4(tmem_base + C::kSfbCol + 8 * s,
                                               desc_rows16_noswizzle(smem_u32(sf_smem(s) + C::kSfBytes)));
                            tmem_cp_32x128b_x4(tmem_base + C::kSfbCol + 8 * s + 4,
                                               desc_rows16_noswizzle(smem_u32(sf_smem(s) + 2 * C::kSfBytes)));
                        }
                    }
                    const uint64_t dw = desc_kmajor_sw128(smem_u32(w_tile(s)));
                    const uint64_t dx = desc_kmajor_sw128(smem_u32(act_tile(s)));
                    const uint64_t da = kWide ? dx : dw;
                    const uint64_t db = kWide ? dw : dx;
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        if (kMX)
                            // scale byte k of each 4-byte scale word: A's id at bits 29-30, B's at bits 4-5
                            mma_mxf8(d_tmem, da + 2 * k, db + 2 * k,
                                     C::kIdesc | (static_cast<uint32_t>(k) << 29) | (static_cast<uint32_t>(k) << 4),
                                     tmem_base + C::kSfaCol + 4 * s, tmem_base + C::kSfbCol + (p.w_sf ? 8 * s : 0),
                                     (kb | k) != 0);
                        else if (kBF16) mma_f16(d_tmem, da + 2 * k, db + 2 * k, C::kIdesc, (kb | k) != 0);
                        else mma_f8f6f4(d_tmem, da + 2 * k, db + 2 * k, (C::kTailSplit && qt >= 0) ? C::kIdescQ : C::kIdesc,
                                        (kb | k) != 0);
                    }
                    if constexpr (C::kW2) {
                        if (half2) {
                            const uint64_t dx2 = desc_kmajor_sw128(smem_u32(act_tile(s) + 128 * 128));
#pragma unroll
                            for (int k = 0; k < 4; ++k)
                                mma_f8f6f4(d_tmem + 256, dx2 + 2 * k, dw + 2 * k, C::kIdesc, (kb | k) != 0);
                        }
                    }
                    tc_commit(&bar_empty[s]);
                }
                if (!ok) break;
                tc_commit(&bar_tfull[acc]);
                ++tcount;
            }
            tc_commit(&bar_drain);  // every MMA issued above has completed once this fires
            mbar_wait_drain(&bar_drain, 0, p.d_status);
        }
    } else if (kMX && warp == 2) {
        // ------------------------- activation scales -> shared memory (MX) ---
        // A stage's scales for the 128 tile rows as the 32 rows of 16 bytes the
        // TMEM copy takes: row i holds, for c = 0..3, the four bytes of tile
        // row 32c + i, one per 32-wide K block of the stage (TMEM lane i, column
        // c, byte k for the stage's k-th MMA); the copy replicates the 32 rows
        // into every lane quadrant.  Scale words are loaded kPf stages before
        // their slot frees, so their latency stays off the MMA's path.
        int it = 0;
        bool ok = true;
        for (int tile = blockIdx.x; ok && tile < num_work; tile += gridDim.x) {
            int sb, nb;
            int qt;
            const int e = work_tile(tile, sb, nb, qt);
            if (e < 0) continue;
            const int cnt = p.expert_offsets[e + 1] - p.expert_offsets[e];
            const uint8_t* sfrow[4];
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                const int i = sb * SR + c * 32 + lane - s_poff[e];  // local row of tile row 32c + lane
                sfrow[c] = (i < cnt) ? p.a_sf + (static_cast<int64_t>(p.a_sf_poff[e]) + i) * p.a_sf_ld : nullptr;
            }
            constexpr int kPf = 4;
            uint32_t pf[kPf][4];
            auto load_stage = [&](int kb, uint32_t* v) {
#pragma unroll
                for (int c = 0; c < 4; ++c)
                    v[c] = (sfrow[c] && kb < nkb) ? __ldg(reinterpret_cast<const uint32_t*>(sfrow[c] + kb * 4))
                                                  : 0x7F7F7F7Fu;
            };
#pragma unroll
            for (int j = 0; j < kPf; ++j) load_stage(j, pf[j]);
            for (int kb0 = 0; ok && kb0 < nkb; kb0 += kPf) {
#pragma unroll
                for (int j = 0; j < kPf; ++j) {
                    if (kb0 + j >= nkb) break;
                    const int s = it % S;
                    const uint32_t ph = (it / S) & 1;
                    if (!mbar_wait(&bar_empty[s], ph ^ 1, abort, p.d_status)) ok = false;
                    ok = __all_sync(0xFFFFFFFFu, ok);
                    if (!ok) break;
                    *reinterpret_cast<uint4*>(sf_smem(s) + 16 * lane) = make_uint4(pf[j][0], pf[j][1], pf[j][2], pf[j][3]);
                    fence_proxy_async_smem();
                    mbar_arrive(&bar_full[s]);
                    load_stage(kb0 + j + kPf, pf[j]);
                    ++it;
                }
            }
        }
    } else if (warp < 4 && kBF16 && p.a_tma) {
        // ------------------- W8A16: activation tiles by TMA (own thread) ---
        if (warp == 2 && lane == 0) {
            int it = 0;
            bool ok = true;
            for (int tile = blockIdx.x; ok && tile < num_work; tile += gridDim.x) {
                int sb, nb;
                int qt;
                const int e = work_tile(tile, sb, nb, qt);
                if (e < 0) continue;
                const int arow0 = (p.a_layout == QMOE_A_PADDED)
                                      ? sb * SR
                                      : p.expert_offsets[e] + (sb * SR - p.padded_offsets[e]);
                for (int kb = 0; kb < nkb; ++kb, ++it) {
                    const int s = it % S;
                    const uint32_t ph = (it / S) & 1;
                    if (!mbar_wait(&bar_empty[s], ph ^ 1, abort, p.d_status)) { ok = false; break; }
                    mbar_arrive_expect_tx(&bar_full[s], C::kActBytes);
                    tma_load_2d(&tmap_a, &bar_full[s], act_tile(s), kb * C::kBK, arow0);
                }
            }
            if (!ok) {
                const uint64_t t0 = global_timer_ns();
                while (global_timer_ns() - t0 < 2000000ull) {}
            }
        }
    } else if (warp < 4 || (C::kExtraGather > 0 && warp >= C::kFirstExtraGatherWarp)) {
        // ------------------------------- activation gather (TOKEN_GATHER) ---
        const int pt = warp < 4 ? threadIdx.x - 64 : 64 + threadIdx.x - 32 * C::kFirstExtraGatherWarp;
        int it = 0;
        bool ok = !p.a_tma;
        for (int tile = blockIdx.x; ok && tile < num_work; tile += gridDim.x) {
            if (*abort) break;
            int sb, nb;
            int qt;
            const int e = work_tile(tile, sb, nb, qt);
            if (e < 0) continue;
            named_bar_sync(1, C::kBProdThreads);
            for (int j = pt; j < SR; j += C::kBProdThreads) {
                const int pos = sb * SR + j;
                const int s = p.sorted_ids[pos];
                int row = -1;
                if (s >= 0 && s < p.T)
                    row = (p.a_layout == QMOE_A_TOKEN_GATHER) ? s / p.top_k
                                                              : p.expert_offsets[e] + (pos - p.padded_offsets[e]);
                s_brow[j] = row;
            }
            named_bar_sync(1, C::kBProdThreads);
            for (int kb = 0; kb < nkb; ++kb, ++it) {
                const int s = it % S;
                const uint32_t ph = (it / S) & 1;
                if (!mbar_wait(&bar_empty[s], ph ^ 1, abort, p.d_status)) { ok = false; break; }
                uint8_t* dst_tile = act_tile(s);
                const int64_t k0 = static_cast<int64_t>(kb) * 128;
                for (int idx = pt; idx < SR * 8; idx += C::kBProdThreads) {
                    const int r = idx >> 3, c = idx & 7;
                    const int row = s_brow[r];
                    const int64_t kbyte = k0 + c * 16;
                    const bool valid = row >= 0 && kbyte < p.a_row_bytes;
                    const uint8_t* src = valid ? p.a + row * p.lda_bytes + kbyte : p.a;
                    cp_async_16(dst_tile + r * 128 + ((c ^ (r & 7)) << 4), src, valid ? 16u : 0u);
                }
                cp_async_commit();
                if (it >= C::kLag) {
                    cp_async_wait<C::kLag>();
                    fence_proxy_async_smem();
                    mbar_arrive(&bar_full[(it - C::kLag) % S]);
                }
            }
        }
        cp_async_wait<0>();
        fence_proxy_async_smem();
        for (int j = (it > C::kLag ? it - C::kLag : 0); j < it; ++j) mbar_arrive(&bar_full[j % S]);
    } else if (warp < 8 || kMX || C::kW2 || kAct != 0) {
        // ------------------------------------------------- epilogue ---
        const int et = threadIdx.x - 128;
        const int q = warp & 3;  // TMEM lane quadrant of this warp
        const int hs = C::kW2 ? (warp - 4) >> 2 : 0;  // kW2: slot half (accumulator) of this group
        int tcount = 0;
        for (int tile = blockIdx.x; tile < num_work; tile += gridDim.x) {
            if (*abort) break;
            int sb, nb;
            int qt;
            const int e = work_tile(tile, sb, nb, qt);
            if (e < 0) continue;
            const int acc = tcount % C::kAccBufs;
            const uint32_t aph = (tcount / C::kAccBufs) & 1;
            const uint32_t t_base =
                tmem_base + (static_cast<uint32_t>(q * 32) << 16) + static_cast<uint32_t>(acc * C::kAccCols + hs * 256);
            if constexpr (kWide) {
                // lane = slot row, columns = 256 output channels
                named_bar_sync(2, C::kEpiThreads);
                for (int c = et; c < WR; c += C::kEpiThreads) {
                    const int64_t n = kAct == 0 ? static_cast<int64_t>(nb) * WR + (qt >= 0 ? qt * C::kQRows : 0) + c
                                            : (c < 128 ? 0 : p.N / 2) + static_cast<int64_t>(nb) * 128 + (c & 127);
                    s_wsc[c] = (n < p.N) ? (p.w_scale ? p.w_scale[static_cast<int64_t>(e) * p.N + n] : 1.0f) : 0.0f;
                }
                named_bar_sync(2, C::kEpiThreads);
                const int pos = sb * SRB + hs * 128 + q * C::kRowsPerQuad + lane;
                const bool in_tile = (!C::kW2 || hs == 0 || second_half(e, sb)) && lane < C::kRowsPerQuad;
                const int s = in_tile ? p.sorted_ids[pos] : -1;
                const bool valid = s >= 0 && s < p.T;
                float rs = 0.0f;
                int64_t orow = 0;
                if (valid) {
                    const int m = s / p.top_k;
                    const int compact = p.expert_offsets[e] + (pos - p.padded_offsets[e]);
                    const int arow = (p.a_layout == QMOE_A_TOKEN_GATHER) ? m
                                     : (p.a_layout == QMOE_A_GROUPED ? compact : pos);
                    rs = (p.a_scale ? p.a_scale[arow] : 1.0f) * (p.topk_w ? p.topk_w[s] : 1.0f);
                    orow = (p.out_layout == QMOE_OUT_SLOT) ? s : (p.out_layout == QMOE_OUT_GROUPED ? compact : m);
                }
                if (!mbar_wait(&bar_tfull[acc], aph, abort, p.d_status)) break;
                tc_fence_after();
                // first output channel of the tile (a quarter tile starts qt * 64 rows in)
                const int64_t nbase = static_cast<int64_t>(nb) * WR + (qt >= 0 ? qt * C::kQRows : 0);
                const int ncols = qt >= 0 ? C::kQRows : WR;  // accumulator columns of this tile
                const int64_t col0 = orow * p.N + nbase;
                const int64_t n_left = p.N - nbase;
                const bool tsum = p.out_layout == QMOE_OUT_TOKEN_SUM;
                // scale and write 8 consecutive output channels starting at column cc
                auto emit8 = [&](int cc, const float* v) {
                    float x[8];
#pragma unroll
                    for (int i = 0; i < 8; ++i) x[i] = v[i] * s_wsc[cc + i] * rs;
                    if (tsum) {
                        red_add_f32x4(p.accum + col0 + cc, x[0], x[1], x[2], x[3]);
                        red_add_f32x4(p.accum + col0 + cc + 4, x[4], x[5], x[6], x[7]);
                    } else {
                        uint4 o;
                        o.x = pack_bf16x2(x[0], x[1]);
                        o.y = pack_bf16x2(x[2], x[3]);
                        o.z = pack_bf16x2(x[4], x[5]);
                        o.w = pack_bf16x2(x[6], x[7]);
                        *reinterpret_cast<uint4*>(p.out + col0 + cc) = o;
                    }
                };
                if constexpr (kMX) {
                    // One accumulator: read this warp's 128 columns out in one go
                    // and hand the accumulator back to the MMA before the stores.
                    const int h = (warp - 4) >> 2;  // column half of this group
                    uint32_t r[4][32];
#pragma unroll
                    for (int j = 0; j < 4; ++j) tmem_ld32_nowait(t_base + h * 128 + 32 * j, r[j]);
                    tmem_wait_ld();
#pragma unroll
                    for (int j = 0; j < 4; ++j) tmem_wait_ld_regs(r[j]);
                    tc_fence_before();
                    mbar_arrive(&bar_tempty[acc]);
                    if (valid) {
#pragma unroll
                        for (int j = 0; j < 4; ++j) {
#pragma unroll
                            for (int g = 0; g < 4; ++g) {
                                const int cc = h * 128 + 32 * j + g * 8;
                                if (cc < n_left) {
                                    float v[8];
#pragma unroll
                                    for (int i = 0; i < 8; ++i) v[i] = __uint_as_float(r[j][g * 8 + i]);
                                    emit8(cc, v);
                                }
                            }
                        }
                    }
                } else if constexpr (kAct == 1) {
                    // y = bf16(acc * w_scale * row scale), rounded exactly as
                    // the plain epilogue stores it, then h = silu(y_gate) * y_up
                    // in fp32 and each 1x32 block's E8M0 factor and e4m3 codes,
                    // the same operations as the SwiGLU + MXFP8 kernel applies to
                    // the stored y.  Padding rows of the expert get factor 0.
                    const int64_t I = p.N / 2;
                    const int64_t local = pos - p.padded_offsets[e];
                    uint8_t* sfr = p.act_sf + (static_cast<int64_t>(p.act_sf_poff[e]) + local) * p.act_sf_ld;
                    uint8_t* qr = p.act_q + (static_cast<int64_t>(p.expert_offsets[e]) + local) * I +
                                  static_cast<int64_t>(nb) * 128;
                    auto bf16r = [](float x) { return __bfloat162float(__float2bfloat16_rn(x)); };
                    const int j0 = 2 * ((warp - 4) >> 2);  // this group's two 32-column blocks
#pragma unroll 1
                    for (int j = j0; j < j0 + 2; ++j) {
                        float vg[32], vu[32];
                        tmem_ld32(t_base + 32 * j, vg);
                        tmem_ld32(t_base + 128 + 32 * j, vu);
                        if (j == j0 + 1) {  // accumulator read out: the MMA may reuse it
                            tc_fence_before();
                            mbar_arrive(&bar_tempty[acc]);
                        }
                        if (!valid) {
                            sfr[nb * 4 + j] = 0;
                            continue;
                        }
                        float amax = 0.0f;
#pragma unroll
                        for (int i = 0; i < 32; i += 2) {
                            const float g0 = bf16r(vg[i] * s_wsc[32 * j + i] * rs);
                            const float g1 = bf16r(vg[i + 1] * s_wsc[32 * j + i + 1] * rs);
                            const float u0 = bf16r(vu[i] * s_wsc[128 + 32 * j + i] * rs);
                            const float u1 = bf16r(vu[i + 1] * s_wsc[128 + 32 * j + i + 1] * rs);
                            silu_mul2(g0, g1, u0, u1, vg[i], vg[i + 1]);
                            amax = fmaxf(amax, fmaxf(fabsf(vg[i]), fabsf(vg[i + 1])));
                        }
                        const int ex = mx_block_exponent(amax);
                        const float mul = pow2_neg(ex);
                        sfr[nb * 4 + j] = static_cast<uint8_t>(ex + 127);
                        uint32_t o[8];
#pragma unroll
                        for (int i = 0; i < 8; ++i)
                            o[i] = e4m3x4(__fmul_rn(vg[4 * i], mul), __fmul_rn(vg[4 * i + 1], mul),
                                          __fmul_rn(vg[4 * i + 2], mul), __fmul_rn(vg[4 * i + 3], mul));
                        *reinterpret_cast<uint4*>(qr + 32 * j) = make_uint4(o[0], o[1], o[2], o[3]);
                        *reinterpret_cast<uint4*>(qr + 32 * j + 16) = make_uint4(o[4], o[5], o[6], o[7]);
                    }
                    if (nb == n_blocks - 1 && j0 == 0)  // factor columns past I/32 (row padding of the factor matrix)
                        for (int64_t c = I / 32; c < p.act_sf_ld; ++c) sfr[c] = 0;
                } else if constexpr (kAct == 2) {
                    // y and h as for kAct 1; h goes to act_h in fp32 and the
                    // amax |h| of this group's 64 columns of the row into
                    // act_amax[row] by an integer max on the bit patterns
                    // (monotone for floats >= 0)
                    const int64_t I = p.N / 2;
                    const int64_t compact = p.expert_offsets[e] + (pos - p.padded_offsets[e]);
                    float* hr = p.act_h + compact * I + static_cast<int64_t>(nb) * 128;
                    auto bf16r = [](float x) { return __bfloat162float(__float2bfloat16_rn(x)); };
                    float amax = 0.0f;
                    const int j0 = 2 * ((warp - 4) >> 2);  // this group's two 32-column blocks
#pragma unroll 1
                    for (int j = j0; j < j0 + 2; ++j) {
                        float vg[32], vu[32];
                        tmem_ld32(t_base + 32 * j, vg);
                        tmem_ld32(t_base + 128 + 32 * j, vu);
                        if (j == j0 + 1) {  // accumulator read out: the MMA may reuse it
                            tc_fence_before();
                            mbar_arrive(&bar_tempty[acc]);
                        }
                        if (!valid) continue;
#pragma unroll
                        for (int i = 0; i < 32; i += 2) {
                            const float g0 = bf16r(vg[i] * s_wsc[32 * j + i] * rs);
                            const float g1 = bf16r(vg[i + 1] * s_wsc[32 * j + i + 1] * rs);
                            const float u0 = bf16r(vu[i] * s_wsc[128 + 32 * j + i] * rs);
                            const float u1 = bf16r(vu[i + 1] * s_wsc[128 + 32 * j + i + 1] * rs);
                            silu_mul2(g0, g1, u0, u1, vg[i], vg[i + 1]);
                            amax = fmaxf(amax, fmaxf(fabsf(vg[i]), fabsf(vg[i + 1])));
                        }
#pragma unroll
                        for (int i = 0; i < 32; i += 4)
                            *reinterpret_cast<float4*>(hr + 32 * j + i) = make_float4(vg[i], vg[i + 1], vg[i + 2], vg[i + 3]);
                    }
                    if (valid) atomicMax(reinterpret_cast<int*>(p.act_amax) + compact, __float_as_int(amax));
                } else {
                    for (int c0 = 0; c0 < ncols; c0 += 32) {
                        float v[32];
                        tmem_ld32(t_base + c0, v);
                        if (c0 + 32 == ncols) {  // accumulator read out: the MMA may reuse it while the stores finish
                            tc_fence_before();
                            mbar_arrive(&bar_tempty[acc]);
                        }
                        if (!valid) continue;
#pragma unroll
                        for (int g = 0; g < 4; ++g) {
                            const int cc = c0 + g * 8;
                            if (cc >= n_left) break;
                            emit8(cc, v + g * 8);
                        }
                    }
                }
            } else {
                // lane = output channel, columns = BN slots
                const bool even = (lane & 1) == 0;
                named_bar_sync(2, C::kEpiThreads);
                for (int j = et; j < SR; j += C::kEpiThreads) {
                    const int pos = sb * SR + j;
                    const int s = p.sorted_ids[pos];
                    if (s < 0 || s >= p.T) {
                        s_crow[j] = -1;
                        s_cscale[j] = 0.0f;
                    } else {
                        const int m = s / p.top_k;
                        const int compact = p.expert_offsets[e] + (pos - p.padded_offsets[e]);
                        const int arow = (p.a_layout == QMOE_A_TOKEN_GATHER) ? m
                                         : (p.a_layout == QMOE_A_GROUPED ? compact : pos);
                        const float sa = p.a_scale ? p.a_scale[arow] : 1.0f;
                        const float wr = p.topk_w ? p.topk_w[s] : 1.0f;
                        s_cscale[j] = sa * wr;
                        s_crow[j] = (p.out_layout == QMOE_OUT_SLOT) ? s
                                                                    : (p.out_layout == QMOE_OUT_GROUPED ? compact : m);
                    }
                }
                named_bar_sync(2, C::kEpiThreads);
                if (!mbar_wait(&bar_tfull[acc], aph, abort, p.d_status)) break;
                tc_fence_after();
                const int64_t n = static_cast<int64_t>(nb) * WR + q * 32 + lane;
                const float sw = (n < p.N) ? p.w_scale[static_cast<int64_t>(e) * p.N + n] : 0.0f;
                const int64_t nn = even ? n : n - 1;
                for (int c0 = 0; c0 < SR; c0 += 16) {
                    float v[16];
                    tmem_ld16(t_base + c0, v);
#pragma unroll
                    for (int i = 0; i < 16; i += 2) {
                        const int j = c0 + i;
                        const float v0 = v[i] * sw * s_cscale[j];
                        const float v1 = v[i + 1] * sw * s_cscale[j + 1];
                        const float o0 = __shfl_xor_sync(0xFFFFFFFFu, v0, 1);
                        const float o1 = __shfl_xor_sync(0xFFFFFFFFu, v1, 1);
                        // even lane: column j at (n, n+1); odd lane: column j+1 at (n-1, n)
                        const int col = even ? j : j + 1;
                        const int row = s_crow[col];
                        if (row >= 0 && nn < p.N) {
                            const float lo = even ? v0 : o1, hi = even ? o0 : v1;
                            const int64_t off = static_cast<int64_t>(row) * p.N + nn;
                            if (p.out_layout == QMOE_OUT_TOKEN_SUM) red_add_f32x2(p.accum + off, lo, hi);
                            else *reinterpret_cast<uint32_t*>(p.out + off) = pack_bf16x2(lo, hi);
                        }
                    }
                }
            }
            if constexpr (!kWide) {
                tc_fence_before();
                mbar_arrive(&bar_tempty[acc]);
            }
            ++tcount;
        }
    } else {
        // ---------------------------------- int8 -> bf16 converters ---
        if (kBF16) {
            const int group = (warp - 8) / (C::kConvThreads / 32);
            const int ct = threadIdx.x - 256 - group * C::kConvThreads;
            int it = 0;
            bool ok = true;
            for (int tile = blockIdx.x; ok && tile < num_work; tile += gridDim.x) {
                int sb, nb;
                int qt;
                const int e = work_tile(tile, sb, nb, qt);
                if (e < 0) continue;
                for (int kb = 0; kb < nkb; ++kb, ++it) {
                    if ((it & 1) != group) continue;
                    const int s = it % S;
                    const uint32_t ph = (it / S) & 1;
                    const int r = it % R;
                    const uint32_t rph = (it / R) & 1;
                    // raw tile landed, and the MMA is done with the previous use of slot s
                    if (!mbar_wait(&bar_raw_full[r], rph, abort, p.d_status)) { ok = false; break; }
                    if (!mbar_wait(&bar_empty[s], ph ^ 1, abort, p.d_status)) { ok = false; break; }
                    const uint8_t* raw = raw_tile(r);
                    uint8_t* dst = w_tile(s);
                    if constexpr (kI4) {
                        // two threads per 32-byte row (32 int4 each), each with the
                        // row's scale for this stage's 128-wide group (kb / 2)
                        const int c2 = ct & 1;
                        constexpr int kRows4 = C::kConvThreads / 2;
#pragma unroll
                        for (int i = 0; i < WR / kRows4; ++i) {
                            const int rr = (ct >> 1) + kRows4 * i;
                            const int64_t n = static_cast<int64_t>(nb) * WR + rr;
                            const float sc = (n < p.N) ? __ldg(p.w_gscale + (static_cast<int64_t>(e) * p.N + n) *
                                                                               p.w_groups + (kb >> 1))
                                                       : 0.0f;
                            const uint4 w = *reinterpret_cast<const uint4*>(raw + rr * 32 + c2 * 16);
                            uint32_t o[4][4];
                            int4x8_to_bf16x8_scaled(w.x, sc, o[0]);
                            int4x8_to_bf16x8_scaled(w.y, sc, o[1]);
                            int4x8_to_bf16x8_scaled(w.z, sc, o[2]);
                            int4x8_to_bf16x8_scaled(w.w, sc, o[3]);
#pragma unroll
                            for (int t = 0; t < 4; ++t)
                                *reinterpret_cast<uint4*>(dst + rr * 128 + (((4 * c2 + t) ^ (rr & 7)) << 4)) =
                                    make_uint4(o[t][0], o[t][1], o[t][2], o[t][3]);
                        }
                        fence_proxy_async_smem();
                        mbar_arrive(&bar_conv[s]);
                        mbar_arrive(&bar_raw_empty[r]);
                        continue;
                    }
                    const int c = ct & 3;
                    constexpr int kRowsPerPass = C::kConvThreads / 4;  // four threads per 64-byte row
#pragma unroll
                    for (int i = 0; i < WR / kRowsPerPass; ++i) {
                        const int r = (ct >> 2) + kRowsPerPass * i;
                        const uint4 w = *reinterpret_cast<const uint4*>(raw + r * 64 + c * 16);
                        uint4 o0, o1;
                        int8x4_to_bf16x4(w.x, o0.x, o0.y);
                        int8x4_to_bf16x4(w.y, o0.z, o0.w);
                        int8x4_to_bf16x4(w.z, o1.x, o1.y);
                        int8x4_to_bf16x4(w.w, o1.z, o1.w);
                        *reinterpret_cast<uint4*>(dst + r * 128 + (((2 * c) ^ (r & 7)) << 4)) = o0;
                        *reinterpret_cast<uint4*>(dst + r * 128 + (((2 * c + 1) ^ (r & 7)) << 4)) = o1;
                    }
                    fence_proxy_async_smem();
                    mbar_arrive(&bar_conv[s]);
                    mbar_arrive(&bar_raw_empty[r]);
                }
            }
        }
    }

    __syncwarp();
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, C::kTmemCols);
    }
}

// ---------------------------------------------------------------- host ---
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

inline EncodeTiledFn encode_tiled_fn() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(f);
    });
    return fn;
}

// Weight map over W[E][N][K] bytes: box {box_k, box_rows, 1}.
inline bool make_weight_map(CUtensorMap* map, const void* w, int64_t E, int64_t N, int64_t K, int box_k, int box_rows,
                            bool swizzle128) {
    EncodeTiledFn enc = encode_tiled_fn();
    if (!enc) return false;
    cuuint64_t dims[3] = {static_cast<cuuint64_t>(K), static_cast<cuuint64_t>(N), static_cast<cuuint64_t>(E)};
    cuuint64_t strides[2] = {static_cast<cuuint64_t>(K), static_cast<cuuint64_t>(N * K)};
    cuuint32_t box[3] = {static_cast<cuuint32_t>(box_k), static_cast<cuuint32_t>(box_rows), 1u};
    cuuint32_t estr[3] = {1u, 1u, 1u};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(w), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Activation map over A[rows][K] (1- or 2-byte elements): box {128 bytes, box_rows}, 128-byte swizzle.
inline bool make_act_map(CUtensorMap* map, const void* a, int64_t rows, int64_t K, int64_t lda, int elem,
                         int box_rows) {
    EncodeTiledFn enc = encode_tiled_fn();
    if (!enc) return false;
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(K), static_cast<cuuint64_t>(rows)};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(lda * elem)};
    cuuint32_t box[2] = {static_cast<cuuint32_t>(128 / elem), static_cast<cuuint32_t>(box_rows)};
    cuuint32_t estr[2] = {1u, 1u};
    return enc(map, elem == 1 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_UINT16, 2,
               const_cast<void*>(a), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
               CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <bool kBF16, bool kWide, int BN, bool kMX = false, bool kI4 = false, int kAct = 0>
inline qmoe_status_t launch_gemm(const void* w, int64_t E, int64_t N, int64_t K, const GemmParams& p,
                                 int64_t max_padded, int64_t a_rows, int64_t lda, cudaStream_t st) {
    using C = GemmCfg<kBF16, kWide, BN, kMX, kI4, kAct>;
    static std::mutex mu;
    static bool attr_set[64] = {false};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return QMOE_ERR_CUDA;
    {
        std::lock_guard<std::mutex> g(mu);
        if (!attr_set[dev]) {
            if (cudaFuncSetAttribute(moe_gemm_kernel<kBF16, kWide, BN, kMX, kI4, kAct>,
                                     cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     C::kDynSmem) != cudaSuccess)
                return QMOE_ERR_CUDA;
            attr_set[dev] = true;
        }
    }
    CUtensorMap map, amap;
    // rows of K weight bytes (FP8, INT8) or K/2 (packed INT4); box: one stage's bytes per row
    // (kAct: 128-row boxes, the gate and up halves of a tile loaded separately)
    if (!make_weight_map(&map, w, E, N, kI4 ? K / 2 : K, kBF16 ? C::kRawRowBytes : C::kBK, kAct ? 128 : C::kWRows,
                         !kBF16))
        return QMOE_ERR_CUDA;
    memset(&amap, 0, sizeof(amap));
    if (p.a_tma && !make_act_map(&amap, p.a, a_rows, K, lda, kBF16 ? 2 : 1, C::kSlotRows)) return QMOE_ERR_CUDA;
    CUtensorMap mapq;  // quarter-tile weight boxes (tail split)
    memset(&mapq, 0, sizeof(mapq));
    if (C::kTailSplit && !make_weight_map(&mapq, w, E, N, K, C::kBK, C::kQRows, true)) return QMOE_ERR_CUDA;
    const int sms = device_sm_count();
    if (sms <= 0) return QMOE_ERR_CUDA;
    // (kW2: the last pair of an expert may hold a single 128-slot block)
    const int64_t max_tiles = ((max_padded + C::kSlotRows - 1) / C::kSlotRows + (C::kW2 ? E : 0)) *
                              ((N + C::kWRows - 1) / C::kWRows);
    // (tail split: up to four CTAs per tile when all tiles fit in a quarter of a wave)
    const int64_t max_work = max_tiles * (C::kTailSplit ? 4 : 1);
    const int64_t grid = max_work < sms ? max_work : sms;
    if (grid <= 0) return QMOE_OK;
    return launch_pdl(moe_gemm_kernel<kBF16, kWide, BN, kMX, kI4, kAct>, dim3(static_cast<unsigned>(grid)),
                      dim3(C::kThreads), C::kDynSmem, st, map, amap, mapq, p);
}

// out[i] = bf16(accum[i]) for the TOKEN_SUM layout (defined in gemm_w8a8.cu).
qmoe_status_t launch_token_sum_finalize(const float* accum, uint16_t* out, int64_t n, cudaStream_t st);
qmoe_status_t launch_token_sum_zero(float* accum, int64_t n, cudaStream_t st);

// FP8 GEMM on CTA pairs (tcgen05 cta_group::2, defined in gemm_pair.cu): per-row
// scales, activation tiles by TMA (GROUPED / PADDED rows), BM >= 128.
qmoe_status_t launch_gemm_pair(const void* w, int64_t E, int64_t N, int64_t K, const GemmParams& p,
                               int64_t max_padded, int64_t a_rows, int64_t lda, cudaStream_t st);

// INT8 / INT4 weight-only GEMM on CTA pairs (defined in gemm_pair_a16.cu): bf16
// activation tiles by TMA (GROUPED / PADDED rows).
qmoe_status_t launch_gemm_pair_a16(bool int4, const void* w, int64_t E, int64_t N, int64_t K, const GemmParams& p,
                                   int64_t max_padded, int64_t a_rows, int64_t lda, cudaStream_t st);

// Tile family of the GEMMs: the library's choice, or one forced by a test.
enum GemmTile { kTileAuto = 0, kTileOneSm = 1, kTilePair = 2 };

// Outputs of the SwiGLU epilogues: MXFP8 codes and factors
// (qmoe_moe_gemm_w8a8_silu_mxfp8), or, with h set, fp32 h and the row amax
// that qmoe_moe_gemm_w8a8_silu_fp8_token quantises per token afterwards.
struct SwiGluOut {
    uint8_t* q;
    uint8_t* sf;
    int64_t sf_ld;
    const int32_t* sf_poff;
    float* h;
    float* amax;
};

// Shared argument checks and dispatch for both precisions;
// check_only: validate the arguments and return without launching anything.
template <bool kBF16, bool kI4 = false>
inline qmoe_status_t run_moe_gemm(const qmoe_gemm_args* a, cudaStream_t st, const SwiGluOut* so = nullptr,
                                  bool check_only = false, GemmTile tile = kTileAuto) {
    static_assert(!kI4 || kBF16, "W4A16 is a bf16-activation GEMM");
    if (kI4 && a && a->struct_size >= sizeof(qmoe_gemm_args)) {
        // packed int4 weights with a scale per 128-wide group of K: wide tile only
        if (a->BM != 64 && a->BM != 128 && a->BM != 256) return QMOE_ERR_UNSUPPORTED;
        if (a->K % 128 != 0 || a->w_scale_mode != QMOE_SCALE_PER_ROW) return QMOE_ERR_INVALID_ARG;
    }
    if (!a || a->struct_size < sizeof(qmoe_gemm_args)) return QMOE_ERR_INVALID_ARG;
    if (a->M < 0 || a->N < 16 || a->N % 16 != 0 || a->K < 16 || a->K % 16 != 0) return QMOE_ERR_INVALID_ARG;
    if (a->E < 1 || a->E > kGemmMaxE || a->top_k < 1 || a->top_k > a->E) return QMOE_ERR_INVALID_ARG;
    if (a->BM != 16 && a->BM != 32 && a->BM != 64 && a->BM != 128 && a->BM != 256) return QMOE_ERR_UNSUPPORTED;
    if (a->a_layout != QMOE_A_TOKEN_GATHER && a->a_layout != QMOE_A_GROUPED && a->a_layout != QMOE_A_PADDED)
        return QMOE_ERR_INVALID_ARG;
    if (a->out_layout < QMOE_OUT_SLOT || a->out_layout > QMOE_OUT_TOKEN_SUM) return QMOE_ERR_INVALID_ARG;
    const int64_t elem = kBF16 ? 2 : 1;
    if (a->lda < a->K || (a->lda * elem) % 16 != 0) return QMOE_ERR_INVALID_ARG;
    const bool mx = !kBF16 && a->a_scale_mode == QMOE_SCALE_MX_1X32;
    const bool wmx = a->w_scale_mode == QMOE_SCALE_MX_1X32;
    if (a->w_scale_mode != QMOE_SCALE_PER_ROW && !wmx) return QMOE_ERR_INVALID_ARG;
    if (wmx) {  // MXFP8 weights: FP8 GEMM with MX activations only
        if (kBF16 || !mx) return QMOE_ERR_UNSUPPORTED;
        if (!a->w_sf || !aligned16(a->w_sf)) return QMOE_ERR_INVALID_ARG;
    }
    if (kBF16) {
        if (a->a_scale_mode != QMOE_SCALE_PER_TOKEN) return QMOE_ERR_UNSUPPORTED;
    } else if (mx) {
        // MX activations: grouped rows (as written by qmoe_silu_mul_quant), wide tile only
        if (a->a_layout != QMOE_A_GROUPED || a->BM < 128) return QMOE_ERR_UNSUPPORTED;
        if (a->K % 32 != 0 || !a->a_sf || !a->a_sf_padded_offsets || a->a_sf_ld < (a->K / 32 + 3) / 4 * 4 ||
            a->a_sf_ld % 4 != 0 || !aligned4(a->a_sf))
            return QMOE_ERR_INVALID_ARG;
    } else {
        if (a->a_scale_mode != QMOE_SCALE_PER_TOKEN || !a->a_scale) return QMOE_ERR_INVALID_ARG;
    }
    const int64_t T = a->M * a->top_k;
    if (T >= (int64_t(1) << 30) || a->N * a->K * a->E >= (int64_t(1) << 40)) return QMOE_ERR_UNSUPPORTED;
    if (T == 0) return QMOE_OK;
    if (!a->a || !a->w || (!a->w_scale && !wmx) || (!a->out && !so) || !a->sorted_ids || !a->expert_ids ||
        !a->num_post_padded || !a->expert_offsets || !a->padded_offsets)
        return QMOE_ERR_INVALID_ARG;
    if (!aligned16(a->a) || !aligned16(a->w) || (a->out && !aligned16(a->out))) return QMOE_ERR_INVALID_ARG;
    if (so) {  // fused [gate | up] projection of grouped rows: FP8 per-row scales, 128-slot tiles
        if (kBF16 || mx || wmx) return QMOE_ERR_UNSUPPORTED;
        if (a->out_layout != QMOE_OUT_GROUPED || a->BM != 128 || a->N % 256 != 0) return QMOE_ERR_INVALID_ARG;
        if (so->h ? (!aligned16(so->h) || !so->amax || !aligned4(so->amax))
                  : (!so->q || !so->sf || !so->sf_poff || !aligned16(so->q) || so->sf_ld < a->N / 64))
            return QMOE_ERR_INVALID_ARG;
    }
    // CTA-pair tile: per-row (FP8, INT8) or per-group (INT4) weight scales, per-token or bf16
    // activations in contiguous rows; FP8 with BM >= 128
    const bool pair_ok = !mx && !wmx && !so && a->a_layout != QMOE_A_TOKEN_GATHER && (kBF16 || a->BM >= 128);
    if (tile == kTilePair && !pair_ok) return QMOE_ERR_UNSUPPORTED;
    // The library's choice (measured on the Mixtral-shaped projections, E = 8, with
    // two k-blocks per pair stage): the pair tile for long K from 256 slots per
    // expert on average (down projections, M = 1024-4096: 150 / 212 / 339 us against
    // 183 / 259 / 349 at N = 4096, K = 14336), and at short K for about one 128-slot
    // block per expert (the decode GEMM at M = 512: 101 against 106 us) and from 512
    // slots per expert (up projections at M = 2048-4096: 567 / 1007 against 596 /
    // 1049 us at N = 32768, K = 6144; even at N = 28672, K = 4096); elsewhere the
    // one-SM tiles are as fast or faster.
    const int64_t slots_per_expert = a->M * a->top_k / a->E;
    const bool pair_auto =
        (a->K >= 8192 && slots_per_expert >= 256) ||
        (a->K < 8192 && ((slots_per_expert >= 96 && slots_per_expert <= 160) || slots_per_expert >= 512));
    // INT8 / INT4 weights: the pair tile from 1024 slots per expert (M = 4096 at N = 14336:
    // W8A16 870 -> 854 us, W4A16 1016 -> 943 us); at decode its 256 x 32 MMAs issue at
    // about 170 cycles each and the one-SM wide tile is faster (125 against 184 us at M = 64)
    const bool pair_auto_a16 = slots_per_expert >= 1024;
    const bool use_pair = pair_ok && (tile == kTilePair || (tile == kTileAuto && (kBF16 ? pair_auto_a16 : pair_auto)));
    if (check_only) return QMOE_OK;

    const bool tsum = a->out_layout == QMOE_OUT_TOKEN_SUM;
    if (tsum) {
        if (!a->accum || !aligned16(a->accum)) return QMOE_ERR_INVALID_ARG;
        const qmoe_status_t rz = launch_token_sum_zero(a->accum, a->M * a->N, st);
        if (rz != QMOE_OK) return rz;
    }
    GemmParams p{};  // every field set below; value-initialised so that none can be left undefined
    p.a = static_cast<const uint8_t*>(a->a);
    p.lda_bytes = a->lda * elem;
    p.a_row_bytes = a->K * elem;
    p.a_scale = (kBF16 || mx) ? nullptr : a->a_scale;
    p.a_sf = mx ? a->a_sf : nullptr;
    p.a_sf_ld = mx ? a->a_sf_ld : 0;
    p.a_sf_poff = mx ? a->a_sf_padded_offsets : nullptr;
    p.sorted_ids = a->sorted_ids;
    p.expert_ids = a->expert_ids;
    p.num_post_padded = a->num_post_padded;
    p.expert_offsets = a->expert_offsets;
    p.padded_offsets = a->padded_offsets;
    p.topk_w = a->topk_weights;
    p.w_scale = kI4 ? nullptr : a->w_scale;   // W4A16: the group scales are applied by the converters
    p.w_gscale = kI4 ? a->w_scale : nullptr;
    p.w_groups = kI4 ? static_cast<int32_t>(a->K / 128) : 0;
    p.w_sf = wmx ? a->w_sf : nullptr;
    p.out = a->out;
    p.accum = a->accum;
    p.N = a->N;
    p.T = T;
    p.E = a->E;
    p.top_k = a->top_k;
    p.a_layout = a->a_layout;
    p.out_layout = a->out_layout;
    p.BM = a->BM;
    p.a_tma = a->a_layout != QMOE_A_TOKEN_GATHER;
    p.num_k_blocks = static_cast<int32_t>((a->K + (kBF16 ? 63 : 127)) / (kBF16 ? 64 : 128));
    p.d_status = a->d_status;
    p.act_q = so ? so->q : nullptr;
    p.act_sf = so ? so->sf : nullptr;
    p.act_sf_ld = so ? so->sf_ld : 0;
    p.act_sf_poff = so ? so->sf_poff : nullptr;
    p.act_h = so ? so->h : nullptr;
    p.act_amax = so ? so->amax : nullptr;
    // decode-sized FP8 launches (at most one slot block per expert on average):
    // about 256 KB of weights per CTA prefetched into L2 ahead of the wait (measured:
    // 128 KB 5641, 256 KB 5652, 512 KB 5646 GB/s on the decode sweep)
    {
        const int64_t slot_rows = a->BM >= 128 ? 128 : a->BM;
        const int64_t w_stage = (a->BM >= 64 ? 256 : 128) * 128;  // weight rows of the tile x 128 bytes
        p.l2_prefetch_kb = (!kBF16 && !mx && !so && T <= slot_rows * a->E) ? static_cast<int32_t>(262144 / w_stage) : 0;
    }
    const int64_t max_padded = (T + static_cast<int64_t>(a->E) * (a->BM - 1) + a->BM - 1) / a->BM * a->BM;
    const int64_t a_rows = a->a_layout == QMOE_A_PADDED ? max_padded : (a->a_layout == QMOE_A_GROUPED ? T : a->M);
    // the kernel numbers its tiles (slot blocks x weight blocks) with 32-bit ints
    if (max_padded / 16 * ((a->N + 127) / 128) >= (int64_t(1) << 31)) return QMOE_ERR_UNSUPPORTED;
    qmoe_status_t r;
    if (use_pair) {
        r = kBF16 ? launch_gemm_pair_a16(kI4, a->w, a->E, a->N, a->K, p, max_padded, a_rows, a->lda, st)
                  : launch_gemm_pair(a->w, a->E, a->N, a->K, p, max_padded, a_rows, a->lda, st);
        if (r != QMOE_OK || !tsum) return r;
        return launch_token_sum_finalize(a->accum, a->out, a->M * a->N, st);
    }
    if constexpr (kI4) {
        r = a->BM == 64
                ? launch_gemm<true, true, 64, false, true>(a->w, a->E, a->N, a->K, p, max_padded, a_rows, a->lda, st)
                : launch_gemm<true, true, 128, false, true>(a->w, a->E, a->N, a->K, p, max_padded, a_rows, a->lda, st);
        if (r != QMOE_OK || !tsum) return r;
        return launch_token_sum_finalize(a->accum, a->out, a->M * a->N, st);
    }
    if constexpr (!kBF16) {
        if (so && so->h)
            return launch_gemm<false, true, 128, false, false, 2>(a->w, a->E, a->N, a->K, p, max_padded, a_rows, a->lda,
                                                                  st);
        if (so)
            return launch_gemm<false, true, 128, false, false, 1>(a->w, a->E, a->N, a->K, p, max_padded, a_rows, a->lda,
                                                                  st);
        if (mx) {
            r = launch_gemm<false, true, 128, true>(a->w, a->E, a->N, a->K, p, max_padded, a_rows, a->lda, st);
            if (r != QMOE_OK || !tsum) return r;
            return launch_token_sum_finalize(a->accum, a->out, a->M * a->N, st);
        }
    }

    if constexpr (!kBF16) {
        // long K (e.g. a down projection): one weight pass for two 128-slot
        // blocks, which halves the weight-operand reads per MMA; at short K the
        // single accumulator buffer costs more than that saves
        if (a->BM >= 128 && p.a_tma && a->K >= 8192) {
            r = launch_gemm<false, true, 256>(a->w, a->E, a->N, a->K, p, max_padded, a_rows, a->lda, st);
            if (r != QMOE_OK || !tsum) return r;
            return launch_token_sum_finalize(a->accum, a->out, a->M * a->N, st);
        }
    }
    switch (a->BM) {
        case 16: r = launch_gemm<kBF16, false, 16>(a->w, a->E, a->N, a->K, p, max_padded, a_rows, a->lda, st); break;
        case 32: r = launch_gemm<kBF16, false, 32>(a->w, a->E, a->N, a->K, p, max_padded, a_rows, a->lda, st); break;
        case 64:  // the 64-slot wide tile (M = 64 MMAs, 256 weight rows each)
            r = launch_gemm<kBF16, true, 64, false, kI4>(a->w, a->E, a->N, a->K, p, max_padded, a_rows, a->lda, st);
            break;
        default: r = launch_gemm<kBF16, true, 128>(a->w, a->E, a->N, a->K, p, max_padded, a_rows, a->lda, st); break;
    }
    if (r != QMOE_OK || !tsum) return r;
    return launch_token_sum_finalize(a->accum, a->out, a->M * a->N, st);
}

}  // namespace qmoe
