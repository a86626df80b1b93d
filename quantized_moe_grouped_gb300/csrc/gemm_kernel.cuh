// gemm_kernel.cuh -- persistent grouped GEMM for the MoE expert FFN on sm_103a.
//
// One tile = 128 output channels n of one expert e  x  BN sorted slots (one
// BM-block of the align output, BN == BM).  The expert weight rows are the
// MMA "A" operand (M = 128) and the slot activations the "B" operand
// (N = BN), so small slot counts (decode) keep the tensor-core M dimension
// full while the kernel streams W at HBM rate.  D = W_tile . A_slots^T
// lives in TMEM (fp32), double-buffered so the epilogue of one tile overlaps
// the main loop of the next.
//
// Warp roles (one CTA per SM, persistent over tiles, static round robin):
//   warp 0      TMA producer: W[e, n0:n0+128, k0:k0+BK] -> smem ring
//   warp 1      TMEM owner + single-thread tcgen05.mma issuer
//   warps 2-3   activation producers: gather the BN slot rows (token rows
//               for TOKEN_GATHER, compact rows for GROUPED) with 16-byte
//               cp.async into the 128-byte-swizzled K-major layout
//   warps 4-7   epilogue: TMEM -> registers, x w_scale[e,n] x a_scale x w[s],
//               bf16, store (or bf16x2 atomic add for TOKEN_SUM)
//   warps 8-11  (W8A16 only) int8 -> bf16 converters, smem -> smem
//
// Every wait is bounded (common.cuh: mbar_wait); on a timeout the CTA raises
// an abort flag, all roles leave their loops, copies in flight are drained
// and TMEM is released before the kernel returns with QMOE_DEV_TIMEOUT set.
#pragma once

#include "common.cuh"
#include "host_util.h"

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
    int64_t N;
    int64_t T;
    int32_t E, top_k, a_layout, out_layout;
    int32_t num_k_blocks;
    int32_t* d_status;
};

template <bool kBF16, int BN>
struct GemmCfg {
    static constexpr int kBK = kBF16 ? 64 : 128;            // K elements per stage (128 bytes of MMA operand)
    static constexpr int kWBytes = 128 * 128;                // MMA-A tile: 128 rows x 128 bytes
    static constexpr int kBBytes = BN * 128;                 // MMA-B tile: BN rows x 128 bytes
    static constexpr int kRawBytes = kBF16 ? 128 * 64 : 0;   // int8 weight tile before conversion
    static constexpr int kWLoadBytes = kBF16 ? kRawBytes : kWBytes;
    static constexpr int kStageBytes = kWBytes + kBBytes + kRawBytes;
    static constexpr int kStagesRaw = (200 * 1024) / kStageBytes;
    static constexpr int kStages = kStagesRaw > 8 ? 8 : kStagesRaw;
    static constexpr int kLag = kStages - 1 < 3 ? kStages - 1 : 3;  // cp.async completion lag (stages)
    static constexpr int kBProdThreads = 64;
    static constexpr int kEpiThreads = 128;
    static constexpr int kConvThreads = 128;
    static constexpr int kThreads = kBF16 ? 384 : 256;
    static constexpr int kTmemCols = 2 * BN < 32 ? 32 : 2 * BN;
    static constexpr uint32_t kIdesc = make_idesc(kBF16 ? kFmtBF16 : kFmtE4M3, 128, BN);
    static constexpr int kDynSmem = kStages * kStageBytes + 1024;
    static_assert(kStages >= 2, "need at least two pipeline stages");
    static_assert(BN % 16 == 0 && BN >= 16 && BN <= 256, "MMA N must be a multiple of 16 in [16, 256]");
    static_assert(kBBytes % 1024 == 0 && kWBytes % 1024 == 0 && kRawBytes % 1024 == 0, "1 KB tile alignment");
};

// Waits with a time limit but without honouring the abort flag (used for the
// final drains, which must finish even after an abort).
QMOE_DI bool mbar_wait_drain(uint64_t* bar, uint32_t parity, int32_t* d_status) {
    int dummy = 0;
    return mbar_wait(bar, parity, &dummy, d_status);
}

QMOE_DI uint32_t pack_bf16x2(float lo, float hi) {
    const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<const uint32_t*>(&v);
}

QMOE_DI void red_add_bf16x2(uint16_t* dst, uint32_t v) {
    asm volatile("red.global.add.noftz.bf16x2 [%0], %1;" ::"l"(dst), "r"(v) : "memory");
}

template <bool kBF16, int BN>
__global__ void __launch_bounds__(GemmCfg<kBF16, BN>::kThreads, 1)
    moe_gemm_kernel(const __grid_constant__ CUtensorMap tmap_w, const GemmParams p) {
    using C = GemmCfg<kBF16, BN>;
    constexpr int S = C::kStages;
    extern __shared__ uint8_t smem_raw[];
    __shared__ uint64_t bar_full[S], bar_empty[S], bar_conv[S];
    __shared__ uint64_t bar_tfull[2], bar_tempty[2], bar_drain;
    __shared__ uint32_t s_tmem_base;
    __shared__ int s_abort;
    __shared__ int32_t s_brow[BN];   // activation producers: source row of each B row (-1: zero)
    __shared__ float s_cscale[BN];   // epilogue: a_scale * routing weight of each column
    __shared__ int32_t s_crow[BN];   // epilogue: output row of each column (-1: padding)

    const uint32_t raw_addr = smem_u32(smem_raw);
    uint8_t* smem = smem_raw + (((raw_addr + 1023u) & ~1023u) - raw_addr);
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(&bar_full[s], 1 + C::kBProdThreads);
            mbar_init(&bar_empty[s], 1);
            mbar_init(&bar_conv[s], C::kConvThreads);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&bar_tfull[i], 1);
            mbar_init(&bar_tempty[i], C::kEpiThreads);
        }
        mbar_init(&bar_drain, 1);
        s_abort = 0;
        fence_mbar_init();
    }
    if (warp == 1) tmem_alloc(&s_tmem_base, C::kTmemCols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = s_tmem_base;
    volatile int* abort = &s_abort;

    const int num_sb = *p.num_post_padded / BN;
    const int n_blocks = static_cast<int>((p.N + 127) / 128);
    const int num_tiles = num_sb * n_blocks;
    const int nkb = p.num_k_blocks;
    auto w_tile = [&](int s) { return smem + s * C::kStageBytes; };
    auto b_tile = [&](int s) { return smem + s * C::kStageBytes + C::kWBytes; };
    auto raw_tile = [&](int s) { return smem + s * C::kStageBytes + C::kWBytes + C::kBBytes; };
    auto tile_expert = [&](int tile) {
        const int e = p.expert_ids[tile % num_sb];
        return (e >= 0 && e < p.E) ? e : -1;
    };

    if (warp == 0) {
        // ------------------------------------------------ TMA producer ---
        if (lane == 0) {
            int it = 0;
            bool ok = true;
            for (int tile = blockIdx.x; ok && tile < num_tiles; tile += gridDim.x) {
                const int e = tile_expert(tile);
                if (e < 0) continue;
                const int nb = tile / num_sb;
                for (int kb = 0; kb < nkb; ++kb, ++it) {
                    const int s = it % S;
                    const uint32_t ph = (it / S) & 1;
                    if (!mbar_wait(&bar_empty[s], ph ^ 1, abort, p.d_status)) { ok = false; break; }
                    mbar_arrive_expect_tx(&bar_full[s], C::kWLoadBytes);
                    tma_load_3d(&tmap_w, &bar_full[s], kBF16 ? raw_tile(s) : w_tile(s), kb * C::kBK, nb * 128, e);
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
            for (int tile = blockIdx.x; ok && tile < num_tiles; tile += gridDim.x) {
                if (tile_expert(tile) < 0) continue;
                const int acc = tcount & 1;
                const uint32_t aph = (tcount >> 1) & 1;
                if (!mbar_wait(&bar_tempty[acc], aph ^ 1, abort, p.d_status)) break;
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * BN);
                for (int kb = 0; kb < nkb; ++kb, ++it) {
                    const int s = it % S;
                    const uint32_t ph = (it / S) & 1;
                    if (!mbar_wait(&bar_full[s], ph, abort, p.d_status)) { ok = false; break; }
                    if (kBF16 && !mbar_wait(&bar_conv[s], ph, abort, p.d_status)) { ok = false; break; }
                    tc_fence_after();
                    const uint64_t da = desc_kmajor_sw128(smem_u32(w_tile(s)));
                    const uint64_t db = desc_kmajor_sw128(smem_u32(b_tile(s)));
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        if (kBF16) mma_f16(d_tmem, da + 2 * k, db + 2 * k, C::kIdesc, (kb | k) != 0);
                        else mma_f8f6f4(d_tmem, da + 2 * k, db + 2 * k, C::kIdesc, (kb | k) != 0);
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
    } else if (warp < 4) {
        // ------------------------------------- activation producers ---
        const int pt = threadIdx.x - 64;
        int it = 0;
        bool ok = true;
        for (int tile = blockIdx.x; ok && tile < num_tiles; tile += gridDim.x) {
            if (*abort) break;
            const int e = tile_expert(tile);
            if (e < 0) continue;
            const int sb = tile % num_sb;
            named_bar_sync(1, C::kBProdThreads);
            for (int j = pt; j < BN; j += C::kBProdThreads) {
                const int pos = sb * BN + j;
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
                uint8_t* dst_tile = b_tile(s);
                const int64_t k0 = static_cast<int64_t>(kb) * 128;
                for (int idx = pt; idx < BN * 8; idx += C::kBProdThreads) {
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
    } else if (warp < 8) {
        // ------------------------------------------------- epilogue ---
        const int et = threadIdx.x - 128;
        const int q = warp & 3;  // TMEM lane quadrant of this warp
        const bool even = (lane & 1) == 0;
        int tcount = 0;
        for (int tile = blockIdx.x; tile < num_tiles; tile += gridDim.x) {
            if (*abort) break;
            const int e = tile_expert(tile);
            if (e < 0) continue;
            const int sb = tile % num_sb;
            const int nb = tile / num_sb;
            const int acc = tcount & 1;
            const uint32_t aph = (tcount >> 1) & 1;
            named_bar_sync(2, C::kEpiThreads);
            for (int j = et; j < BN; j += C::kEpiThreads) {
                const int pos = sb * BN + j;
                const int s = p.sorted_ids[pos];
                if (s < 0 || s >= p.T) {
                    s_crow[j] = -1;
                    s_cscale[j] = 0.0f;
                } else {
                    const int m = s / p.top_k;
                    const int compact = p.expert_offsets[e] + (pos - p.padded_offsets[e]);
                    const int arow = (p.a_layout == QMOE_A_TOKEN_GATHER) ? m : compact;
                    const float sa = p.a_scale ? p.a_scale[arow] : 1.0f;
                    const float wr = p.topk_w ? p.topk_w[s] : 1.0f;
                    s_cscale[j] = sa * wr;
                    s_crow[j] = (p.out_layout == QMOE_OUT_SLOT) ? s : (p.out_layout == QMOE_OUT_GROUPED ? compact : m);
                }
            }
            named_bar_sync(2, C::kEpiThreads);
            if (!mbar_wait(&bar_tfull[acc], aph, abort, p.d_status)) break;
            tc_fence_after();
            const int64_t n = static_cast<int64_t>(nb) * 128 + q * 32 + lane;
            const float sw = (n < p.N) ? p.w_scale[static_cast<int64_t>(e) * p.N + n] : 0.0f;
            const uint32_t t_row = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + static_cast<uint32_t>(acc * BN);
            const int64_t nn = even ? n : n - 1;
            for (int c0 = 0; c0 < BN; c0 += 16) {
                float v[16];
                tmem_ld16(t_row + c0, v);
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
                        const uint32_t packed = even ? pack_bf16x2(v0, o0) : pack_bf16x2(o1, v1);
                        uint16_t* dst = p.out + static_cast<int64_t>(row) * p.N + nn;
                        if (p.out_layout == QMOE_OUT_TOKEN_SUM) red_add_bf16x2(dst, packed);
                        else *reinterpret_cast<uint32_t*>(dst) = packed;
                    }
                }
            }
            tc_fence_before();
            mbar_arrive(&bar_tempty[acc]);
            ++tcount;
        }
    } else {
        // ---------------------------------- int8 -> bf16 converters ---
        if (kBF16) {
            const int ct = threadIdx.x - 256;
            int it = 0;
            bool ok = true;
            for (int tile = blockIdx.x; ok && tile < num_tiles; tile += gridDim.x) {
                if (tile_expert(tile) < 0) continue;
                for (int kb = 0; kb < nkb; ++kb, ++it) {
                    const int s = it % S;
                    const uint32_t ph = (it / S) & 1;
                    if (!mbar_wait(&bar_full[s], ph, abort, p.d_status)) { ok = false; break; }
                    const uint8_t* raw = raw_tile(s);
                    uint8_t* dst = w_tile(s);
                    const int c = ct & 3;
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const int r = (ct >> 2) + 32 * i;
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

// Weight map over W[E][N][K] bytes: box {box_k, 128, 1}.
inline bool make_weight_map(CUtensorMap* map, const void* w, int64_t E, int64_t N, int64_t K, int box_k,
                            bool swizzle128) {
    EncodeTiledFn enc = encode_tiled_fn();
    if (!enc) return false;
    cuuint64_t dims[3] = {static_cast<cuuint64_t>(K), static_cast<cuuint64_t>(N), static_cast<cuuint64_t>(E)};
    cuuint64_t strides[2] = {static_cast<cuuint64_t>(K), static_cast<cuuint64_t>(N * K)};
    cuuint32_t box[3] = {static_cast<cuuint32_t>(box_k), 128u, 1u};
    cuuint32_t estr[3] = {1u, 1u, 1u};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(w), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <bool kBF16, int BN>
inline qmoe_status_t launch_gemm(const CUtensorMap& map, const GemmParams& p, int64_t max_tiles, cudaStream_t st) {
    using C = GemmCfg<kBF16, BN>;
    static std::mutex mu;
    static bool attr_set[64] = {false};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return QMOE_ERR_CUDA;
    {
        std::lock_guard<std::mutex> g(mu);
        if (!attr_set[dev]) {
            if (cudaFuncSetAttribute(moe_gemm_kernel<kBF16, BN>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     C::kDynSmem) != cudaSuccess)
                return QMOE_ERR_CUDA;
            attr_set[dev] = true;
        }
    }
    const int sms = device_sm_count();
    if (sms <= 0) return QMOE_ERR_CUDA;
    const int64_t grid = max_tiles < sms ? max_tiles : sms;
    if (grid <= 0) return QMOE_OK;
    moe_gemm_kernel<kBF16, BN><<<static_cast<unsigned>(grid), C::kThreads, C::kDynSmem, st>>>(map, p);
    return launch_status();
}

// Shared argument checks and dispatch for both precisions.
template <bool kBF16>
inline qmoe_status_t run_moe_gemm(const qmoe_gemm_args* a, cudaStream_t st) {
    if (!a || a->struct_size < sizeof(qmoe_gemm_args)) return QMOE_ERR_INVALID_ARG;
    if (a->M < 0 || a->N < 16 || a->N % 16 != 0 || a->K < 16 || a->K % 16 != 0) return QMOE_ERR_INVALID_ARG;
    if (a->E < 1 || a->E > 256 || a->top_k < 1 || a->top_k > a->E) return QMOE_ERR_INVALID_ARG;
    if (a->BM != 16 && a->BM != 32 && a->BM != 64 && a->BM != 128 && a->BM != 256) return QMOE_ERR_UNSUPPORTED;
    if (a->a_layout != QMOE_A_TOKEN_GATHER && a->a_layout != QMOE_A_GROUPED) return QMOE_ERR_INVALID_ARG;
    if (a->out_layout < QMOE_OUT_SLOT || a->out_layout > QMOE_OUT_TOKEN_SUM) return QMOE_ERR_INVALID_ARG;
    const int64_t elem = kBF16 ? 2 : 1;
    if (a->lda < a->K || (a->lda * elem) % 16 != 0) return QMOE_ERR_INVALID_ARG;
    if (kBF16) {
        if (a->a_scale_mode != QMOE_SCALE_PER_TOKEN) return QMOE_ERR_UNSUPPORTED;
    } else {
        if (a->a_scale_mode == QMOE_SCALE_MX_1X32) return QMOE_ERR_UNSUPPORTED;
        if (a->a_scale_mode != QMOE_SCALE_PER_TOKEN || !a->a_scale) return QMOE_ERR_INVALID_ARG;
    }
    const int64_t T = a->M * a->top_k;
    if (T >= (int64_t(1) << 30) || a->N * a->K * a->E >= (int64_t(1) << 40)) return QMOE_ERR_UNSUPPORTED;
    if (T == 0) return QMOE_OK;
    if (!a->a || !a->w || !a->w_scale || !a->out || !a->sorted_ids || !a->expert_ids || !a->num_post_padded ||
        !a->expert_offsets || !a->padded_offsets)
        return QMOE_ERR_INVALID_ARG;
    if (!aligned16(a->a) || !aligned16(a->w) || !aligned16(a->out)) return QMOE_ERR_INVALID_ARG;

    CUtensorMap map;
    if (!make_weight_map(&map, a->w, a->E, a->N, a->K, kBF16 ? 64 : 128, !kBF16)) return QMOE_ERR_CUDA;

    if (a->out_layout == QMOE_OUT_TOKEN_SUM) {
        if (cudaMemsetAsync(a->out, 0, static_cast<size_t>(a->M * a->N) * 2, st) != cudaSuccess) return QMOE_ERR_CUDA;
    }
    GemmParams p;
    p.a = static_cast<const uint8_t*>(a->a);
    p.lda_bytes = a->lda * elem;
    p.a_row_bytes = a->K * elem;
    p.a_scale = kBF16 ? nullptr : a->a_scale;
    p.sorted_ids = a->sorted_ids;
    p.expert_ids = a->expert_ids;
    p.num_post_padded = a->num_post_padded;
    p.expert_offsets = a->expert_offsets;
    p.padded_offsets = a->padded_offsets;
    p.topk_w = a->topk_weights;
    p.w_scale = a->w_scale;
    p.out = a->out;
    p.N = a->N;
    p.T = T;
    p.E = a->E;
    p.top_k = a->top_k;
    p.a_layout = a->a_layout;
    p.out_layout = a->out_layout;
    p.num_k_blocks = static_cast<int32_t>((a->K + (kBF16 ? 63 : 127)) / (kBF16 ? 64 : 128));
    p.d_status = a->d_status;
    const int64_t cap_padded = T + static_cast<int64_t>(a->E) * (a->BM - 1);
    const int64_t max_tiles = ((cap_padded + a->BM - 1) / a->BM) * ((a->N + 127) / 128);
    switch (a->BM) {
        case 16: return launch_gemm<kBF16, 16>(map, p, max_tiles, st);
        case 32: return launch_gemm<kBF16, 32>(map, p, max_tiles, st);
        case 64: return launch_gemm<kBF16, 64>(map, p, max_tiles, st);
        case 128: return launch_gemm<kBF16, 128>(map, p, max_tiles, st);
        default: return launch_gemm<kBF16, 256>(map, p, max_tiles, st);
    }
}

}  // namespace qmoe
