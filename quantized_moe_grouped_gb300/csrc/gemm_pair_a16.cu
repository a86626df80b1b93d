// gemm_pair_a16.cu -- INT8 / INT4 weight-only grouped GEMM (W8A16, W4A16) on
// CTA pairs (tcgen05 cta_group::2, kind::f16).
//
// One tile = 256 output channels of one expert x up to 256 of its sorted slots,
// on a cluster of two CTAs:
//   * MMA A operand (M = 256): the weight rows converted to bf16.  Each CTA
//     streams the raw int8 (int4) rows of its 128 output channels by TMA into
//     a ring of its own, and two groups of converter warps (alternate stages)
//     turn them into a 128 x 64 bf16 tile in the 128-byte-swizzled K-major
//     layout (int4: times the row's scale of the stage's 128-wide K group).
//   * MMA B operand (N = nt, the tile's valid slots rounded up to 32): the
//     bf16 activation rows, CTA r holding slots [r nt/2, (r+1) nt/2) of the
//     tile in 32-row TMA boxes (nt/64 of them, so a decode tile with a few
//     slots per expert loads a few rows, not a padded 128-row block).
//   * D: CTA r's tensor memory holds its 128 output channels x nt slots.
// Against the one-SM wide tile (128 slots x 256 channels) every SM converts
// and stores half the weight rows per 64-wide k-step for the same FLOPs, and a
// decode tile no longer reads a mostly padded 128-row activation tile per MMA.
//
// Roles, in each CTA: warp 0 raw-weight producer, warp 1 MMA issuer (CTA 0),
// warp 2 activation producer, warps 4-7 epilogue, warps 8-15 converters.
// Barriers: the raw ring is per CTA (TMA -> converters); `full` (CTA 0) takes
// both CTAs' activation boxes (CTA 1's through the cta_group::2 TMA form);
// `conv` (CTA 0) one arrival per converter warp of both CTAs (after an
// async-proxy fence; a cluster-scope release there cost each converter warp
// about 0.8 us per stage and made the tile 1.5-2x slower); the MMA commits to both CTAs' `empty`
// and `tfull`; both epilogues arrive on CTA 0's `tempty`.  Every wait is
// bounded; the CTAs meet at a cluster barrier before TMEM is released.
#include "pair_common.cuh"

namespace qmoe {
namespace pairtile {

template <bool kI4>
struct A16Cfg {
    static constexpr int kStages = 4;                    // main ring: bf16 A tile + activation boxes
    static constexpr int kBK = 64;                       // K elements per stage (128 bytes of bf16)
    static constexpr int kABytes = kRowsCta * 128;       // 16 KB converted weights
    static constexpr int kBoxRows = 32;                  // activation rows per TMA box
    static constexpr int kBoxBytes = kBoxRows * 128;     // 4 KB
    static constexpr int kBBytes = 4 * kBoxBytes;        // up to 128 rows per CTA
    static constexpr int kStageBytes = kABytes + kBBytes;
    static constexpr int kRawRowBytes = kI4 ? 32 : 64;   // raw weight bytes per row per stage
    static constexpr int kRawBytes = kRowsCta * kRawRowBytes;
    static constexpr int kRawStages = (64 * 1024) / kRawBytes;  // 8 (int8) or 16 (int4)
    static constexpr int kConvThreads = 128;             // one converter group (alternate stages)
    static constexpr int kEpiThreads = 128;
    static constexpr int kThreads = 512;                 // 16 warps
    static constexpr int kFirstConvWarp = 8;
    static constexpr int kAccCols = 256;
    static constexpr int kTmemCols = 512;
    static constexpr int kDynSmem = kStages * kStageBytes + kRawStages * kRawBytes + 1024;
    static_assert(kDynSmem + 6 * 1024 <= 227 * 1024, "shared memory");
};

template <bool kI4>
__global__ void __launch_bounds__(A16Cfg<kI4>::kThreads, 1)
    moe_gemm_pair_a16_kernel(const __grid_constant__ CUtensorMap tmap_w, const __grid_constant__ CUtensorMap tmap_a,
                             const GemmParams p) {
    using C = A16Cfg<kI4>;
    constexpr int S = C::kStages;
    constexpr int R = C::kRawStages;
    extern __shared__ uint8_t smem_raw[];
    __shared__ uint64_t bar_full[S], bar_empty[S], bar_conv[S], bar_raw_full[R], bar_raw_empty[R];
    __shared__ uint64_t bar_tfull[2], bar_tempty[2], bar_drain;
    __shared__ uint32_t s_tmem_base;
    __shared__ int s_abort;
    __shared__ int32_t s_crow[kTileSlots];
    __shared__ float s_cscale[kTileSlots];
    __shared__ int32_t s_poff[kGemmMaxE + 1];
    __shared__ int32_t s_pre[kGemmMaxE + 1];

    const uint32_t raw_addr = smem_u32(smem_raw);
    uint8_t* smem = smem_raw + (((raw_addr + 1023u) & ~1023u) - raw_addr);
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t rank = cluster_ctarank();

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(&bar_full[s], 1);    // used in CTA 0: activation producer, plus both CTAs' box bytes
            mbar_init(&bar_empty[s], 1);   // the pair's MMA commit
            mbar_init(&bar_conv[s], 2 * (C::kConvThreads / 32));  // used in CTA 0: each converter warp of both CTAs
        }
        for (int r = 0; r < R; ++r) {
            mbar_init(&bar_raw_full[r], 1);
            mbar_init(&bar_raw_empty[r], C::kConvThreads);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&bar_tfull[i], 1);
            mbar_init(&bar_tempty[i], 2 * C::kEpiThreads);
        }
        mbar_init(&bar_drain, 1);
        s_abort = 0;
        fence_mbar_init();
    }
    if (warp == 1) tmem_alloc_pair(&s_tmem_base, C::kTmemCols);
    __syncwarp();
    cluster_sync_all();
    pdl_launch_dependents();
    pdl_wait();
    for (int i = threadIdx.x; i <= p.E; i += blockDim.x) s_poff[i] = p.padded_offsets[i];
    if (warp == 0) {
        int base = 0;
        for (int c = 0; c <= p.E; c += 32) {
            const int i = c + lane;
            const int v = i < p.E ? (p.padded_offsets[i + 1] - p.padded_offsets[i] + kTileSlots - 1) / kTileSlots : 0;
            int x = v;
#pragma unroll
            for (int d = 1; d < 32; d <<= 1) {
                const int y = __shfl_up_sync(0xFFFFFFFFu, x, d);
                if (lane >= d) x += y;
            }
            if (i <= p.E) s_pre[i] = base + x - v;
            base += __shfl_sync(0xFFFFFFFFu, x, 31);
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = s_tmem_base;
    volatile int* abort = &s_abort;

    const int n_blocks = static_cast<int>((p.N + kTileRows - 1) / kTileRows);
    const int num_tiles = s_pre[p.E] * n_blocks;
    const int c0 = static_cast<int>(cluster_id_x());
    const int nc = static_cast<int>(num_clusters_x());
    const int nkb = p.num_k_blocks;
    auto a_tile = [&](int s) { return smem + s * C::kStageBytes; };
    auto b_tile = [&](int s) { return smem + s * C::kStageBytes + C::kABytes; };
    auto raw_tile = [&](int r) { return smem + S * C::kStageBytes + r * C::kRawBytes; };

    if (warp == 0) {
        // ------------------------------------- raw weight producer ---
        if (lane == 0) {
            int it = 0;
            bool ok = true;
            for (int t = c0; ok && t < num_tiles; t += nc) {
                const Tile x = decode_tile(t, p.E, n_blocks, s_pre, s_poff, p.expert_offsets);
                const int wrow = x.nb * kTileRows + static_cast<int>(rank) * kRowsCta;
                for (int kb = 0; kb < nkb; ++kb, ++it) {
                    const int r = it % R;
                    const uint32_t rph = (it / R) & 1;
                    if (!mbar_wait(&bar_raw_empty[r], rph ^ 1, abort, p.d_status)) { ok = false; break; }
                    mbar_arrive_expect_tx(&bar_raw_full[r], C::kRawBytes);
                    tma_load_3d(&tmap_w, &bar_raw_full[r], raw_tile(r), kb * C::kRawRowBytes, wrow, x.e);
                }
            }
            if (!ok) {
                const uint64_t t0 = global_timer_ns();
                while (global_timer_ns() - t0 < 2000000ull) {}
            }
        }
    } else if (warp == 2) {
        // ------------------------------------- activation producer ---
        if (lane == 0) {
            int it = 0;
            bool ok = true;
            for (int t = c0; ok && t < num_tiles; t += nc) {
                const Tile x = decode_tile(t, p.E, n_blocks, s_pre, s_poff, p.expert_offsets);
                const int half = x.nt / 2;
                const int nbox = (half + C::kBoxRows - 1) / C::kBoxRows;
                const int arow = (p.a_layout == QMOE_A_PADDED ? x.s0
                                                              : p.expert_offsets[x.e] + (x.s0 - s_poff[x.e])) +
                                 static_cast<int>(rank) * half;
                for (int kb = 0; kb < nkb; ++kb, ++it) {
                    const int s = it % S;
                    const uint32_t ph = (it / S) & 1;
                    if (!mbar_wait(&bar_empty[s], ph ^ 1, abort, p.d_status)) { ok = false; break; }
                    if (rank == 0) {
                        mbar_arrive_expect_tx(&bar_full[s], 2 * nbox * C::kBoxBytes);
                        for (int i = 0; i < nbox; ++i)
                            tma_load_2d(&tmap_a, &bar_full[s], b_tile(s) + i * C::kBoxBytes, kb * C::kBK,
                                        arow + i * C::kBoxRows);
                    } else {
                        const uint32_t bar0 = map_shared_rank(&bar_full[s], 0);
                        for (int i = 0; i < nbox; ++i)
                            tma_load_2d_to_leader(&tmap_a, bar0, b_tile(s) + i * C::kBoxBytes, kb * C::kBK,
                                                  arow + i * C::kBoxRows);
                    }
                }
            }
            if (!ok) {
                const uint64_t t0 = global_timer_ns();
                while (global_timer_ns() - t0 < 2000000ull) {}
            }
        }
    } else if (warp == 1) {
        // ------------------------------------- MMA issuer (CTA 0) ---
        if (lane == 0 && rank == 0) {
            int it = 0, tcount = 0;
            bool ok = true;
            for (int t = c0; ok && t < num_tiles; t += nc) {
                const Tile x = decode_tile(t, p.E, n_blocks, s_pre, s_poff, p.expert_offsets);
                const int acc = tcount & 1;
                const uint32_t aph = (tcount >> 1) & 1;
                if (!mbar_wait(&bar_tempty[acc], aph ^ 1, abort, p.d_status)) break;
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * C::kAccCols);
                const uint32_t idesc = make_idesc(kFmtBF16, 256, x.nt);
                for (int kb = 0; kb < nkb; ++kb, ++it) {
                    const int s = it % S;
                    const uint32_t ph = (it / S) & 1;
                    if (!mbar_wait(&bar_full[s], ph, abort, p.d_status)) { ok = false; break; }
                    if (!mbar_wait(&bar_conv[s], ph, abort, p.d_status)) { ok = false; break; }
                    tc_fence_after();
                    const uint64_t da = desc_kmajor_sw128(smem_u32(a_tile(s)));
                    const uint64_t db = desc_kmajor_sw128(smem_u32(b_tile(s)));
#pragma unroll
                    for (int k = 0; k < 4; ++k) mma_pair_f16(d_tmem, da + 2 * k, db + 2 * k, idesc, (kb | k) != 0);
                    tc_commit_pair(&bar_empty[s], 0x3);
                }
                if (!ok) break;
                tc_commit_pair(&bar_tfull[acc], 0x3);
                ++tcount;
            }
            tc_commit_pair(&bar_drain, 0x1);
            int dummy = 0;
            mbar_wait(&bar_drain, 0, &dummy, p.d_status);
        }
    } else if (warp >= 4 && warp < 8) {
        // ------------------------------------------------- epilogue ---
        // lane = output channel, columns = the tile's slots
        const int et = threadIdx.x - 128;
        const int q = warp & 3;
        const bool even = (lane & 1) == 0;
        const uint32_t tempty0 = map_shared_rank(&bar_tempty[0], 0);
        const uint32_t tempty1 = map_shared_rank(&bar_tempty[1], 0);
        int tcount = 0;
        for (int t = c0; t < num_tiles; t += nc) {
            if (*abort) break;
            const Tile x = decode_tile(t, p.E, n_blocks, s_pre, s_poff, p.expert_offsets);
            const int acc = tcount & 1;
            const uint32_t aph = (tcount >> 1) & 1;
            named_bar_sync(1, C::kEpiThreads);
            for (int j = et; j < kTileSlots; j += C::kEpiThreads) {
                int row = -1;
                float sc = 0.0f;
                if (j < x.nv) {
                    const int pos = x.s0 + j;
                    const int s = p.sorted_ids[pos];
                    if (s >= 0 && s < p.T) {
                        const int m = s / p.top_k;
                        const int compact = p.expert_offsets[x.e] + (pos - s_poff[x.e]);
                        sc = 1.0f * (p.topk_w ? p.topk_w[s] : 1.0f);
                        row = (p.out_layout == QMOE_OUT_SLOT) ? s : (p.out_layout == QMOE_OUT_GROUPED ? compact : m);
                    }
                }
                s_crow[j] = row;
                s_cscale[j] = sc;
            }
            named_bar_sync(1, C::kEpiThreads);
            const int64_t n = static_cast<int64_t>(x.nb) * kTileRows + static_cast<int64_t>(rank) * kRowsCta + q * 32 +
                              lane;
            // int4: the group scales were applied by the converters
            const float sw = (n < p.N) ? (p.w_scale ? p.w_scale[static_cast<int64_t>(x.e) * p.N + n] : 1.0f) : 0.0f;
            const int64_t nn = even ? n : n - 1;
            const bool tsum = p.out_layout == QMOE_OUT_TOKEN_SUM;
            if (!mbar_wait(&bar_tfull[acc], aph, abort, p.d_status)) break;
            tc_fence_after();
            const uint32_t t_base =
                tmem_base + (static_cast<uint32_t>(q * 32) << 16) + static_cast<uint32_t>(acc * C::kAccCols);
            for (int cb = 0; cb < x.nt; cb += 16) {
                float v[16];
                tmem_ld16(t_base + cb, v);
#pragma unroll
                for (int i = 0; i < 16; i += 2) {
                    const int j = cb + i;
                    const float v0 = v[i] * sw * s_cscale[j];
                    const float v1 = v[i + 1] * sw * s_cscale[j + 1];
                    const float o0 = __shfl_xor_sync(0xFFFFFFFFu, v0, 1);
                    const float o1 = __shfl_xor_sync(0xFFFFFFFFu, v1, 1);
                    const int col = even ? j : j + 1;
                    const int row = s_crow[col];
                    if (row >= 0 && nn < p.N) {
                        const float lo = even ? v0 : o1, hi = even ? o0 : v1;
                        const int64_t off = static_cast<int64_t>(row) * p.N + nn;
                        if (tsum) red_add_f32x2(p.accum + off, lo, hi);
                        else *reinterpret_cast<uint32_t*>(p.out + off) = pack_bf16x2(lo, hi);
                    }
                }
            }
            tc_fence_before();
            mbar_arrive_cluster(acc == 0 ? tempty0 : tempty1);
            ++tcount;
        }
    } else if (warp >= C::kFirstConvWarp) {
        // ------------------------------------- int8 / int4 -> bf16 converters ---
        const int group = (warp - C::kFirstConvWarp) / (C::kConvThreads / 32);
        const int ct = threadIdx.x - 32 * C::kFirstConvWarp - group * C::kConvThreads;
        int it = 0;
        bool ok = true;
        for (int t = c0; ok && t < num_tiles; t += nc) {
            const Tile x = decode_tile(t, p.E, n_blocks, s_pre, s_poff, p.expert_offsets);
            const int64_t row0 = static_cast<int64_t>(x.nb) * kTileRows + static_cast<int64_t>(rank) * kRowsCta;
            for (int kb = 0; kb < nkb; ++kb, ++it) {
                if ((it & 1) != group) continue;
                const int s = it % S;
                const uint32_t ph = (it / S) & 1;
                const int r = it % R;
                const uint32_t rph = (it / R) & 1;
                if (!mbar_wait(&bar_raw_full[r], rph, abort, p.d_status)) { ok = false; break; }
                if (!mbar_wait(&bar_empty[s], ph ^ 1, abort, p.d_status)) { ok = false; break; }
                const uint8_t* raw = raw_tile(r);
                uint8_t* dst = a_tile(s);
                if constexpr (kI4) {
                    // one thread per 32-byte row (64 int4), with the row's scale for this
                    // stage's 128-wide K group (kb / 2)
                    const int rr = ct;
                    const int64_t n = row0 + rr;
                    const float sc = (n < p.N) ? __ldg(p.w_gscale + (static_cast<int64_t>(x.e) * p.N + n) * p.w_groups +
                                                       (kb >> 1))
                                               : 0.0f;
#pragma unroll
                    for (int c2 = 0; c2 < 2; ++c2) {
                        const uint4 w = *reinterpret_cast<const uint4*>(raw + rr * 32 + c2 * 16);
                        uint32_t o[4][4];
                        int4x8_to_bf16x8_scaled(w.x, sc, o[0]);
                        int4x8_to_bf16x8_scaled(w.y, sc, o[1]);
                        int4x8_to_bf16x8_scaled(w.z, sc, o[2]);
                        int4x8_to_bf16x8_scaled(w.w, sc, o[3]);
#pragma unroll
                        for (int t4 = 0; t4 < 4; ++t4)
                            *reinterpret_cast<uint4*>(dst + rr * 128 + (((4 * c2 + t4) ^ (rr & 7)) << 4)) =
                                make_uint4(o[t4][0], o[t4][1], o[t4][2], o[t4][3]);
                    }
                } else {
                    // four threads per 64-byte row, 32 rows per pass
                    const int c = ct & 3;
#pragma unroll
                    for (int i = 0; i < kRowsCta / (C::kConvThreads / 4); ++i) {
                        const int rr = (ct >> 2) + (C::kConvThreads / 4) * i;
                        const uint4 w = *reinterpret_cast<const uint4*>(raw + rr * 64 + c * 16);
                        uint4 o0, o1;
                        int8x4_to_bf16x4(w.x, o0.x, o0.y);
                        int8x4_to_bf16x4(w.y, o0.z, o0.w);
                        int8x4_to_bf16x4(w.z, o1.x, o1.y);
                        int8x4_to_bf16x4(w.w, o1.z, o1.w);
                        *reinterpret_cast<uint4*>(dst + rr * 128 + (((2 * c) ^ (rr & 7)) << 4)) = o0;
                        *reinterpret_cast<uint4*>(dst + rr * 128 + (((2 * c + 1) ^ (rr & 7)) << 4)) = o1;
                    }
                }
                // the converted tile is read by the tensor core (async proxy), possibly of the partner SM
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive_cluster(map_shared_rank(&bar_conv[s], 0));
                mbar_arrive(&bar_raw_empty[r]);
            }
        }
    }

    __syncwarp();
    tc_fence_before();
    cluster_sync_all();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc_pair(tmem_base, C::kTmemCols);
    }
}

template <bool kI4>
qmoe_status_t launch_pair_a16(const void* w, int64_t E, int64_t N, int64_t K, const GemmParams& p, int64_t max_padded,
                              int64_t a_rows, int64_t lda, cudaStream_t st) {
    using C = A16Cfg<kI4>;
    static std::mutex mu;
    static bool attr_set[64] = {false};
    static int max_clusters[64] = {0};
    auto kern = moe_gemm_pair_a16_kernel<kI4>;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return QMOE_ERR_CUDA;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.blockDim = dim3(C::kThreads);
    cfg.dynamicSmemBytes = C::kDynSmem;
    cfg.stream = st;
    cfg.attrs = attr;
    {
        std::lock_guard<std::mutex> g(mu);
        if (!attr_set[dev]) {
            if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kDynSmem) != cudaSuccess)
                return QMOE_ERR_CUDA;
            const int sms = device_sm_count();
            if (sms <= 1) return QMOE_ERR_CUDA;
            cfg.gridDim = dim3(static_cast<unsigned>(sms / 2 * 2));
            cfg.numAttrs = 1;
            int n = 0;
            if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess || n <= 0) return QMOE_ERR_CUDA;
            max_clusters[dev] = n;
            attr_set[dev] = true;
        }
    }
    CUtensorMap map, amap;
    // raw weight rows: K bytes (int8) or K/2 (packed int4); box = one stage's bytes x 128 rows
    if (!make_weight_map(&map, w, E, N, kI4 ? K / 2 : K, C::kRawRowBytes, kRowsCta, false)) return QMOE_ERR_CUDA;
    if (!make_act_map(&amap, p.a, a_rows, K, lda, 2, C::kBoxRows)) return QMOE_ERR_CUDA;
    const int64_t max_tiles = ((max_padded + kTileSlots - 1) / kTileSlots + E) * ((N + kTileRows - 1) / kTileRows);
    const int64_t clusters = max_tiles < max_clusters[dev] ? max_tiles : max_clusters[dev];
    if (clusters <= 0) return QMOE_OK;
    cfg.gridDim = dim3(static_cast<unsigned>(2 * clusters));
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, kern, map, amap, p) == cudaSuccess ? QMOE_OK : QMOE_ERR_CUDA;
}

}  // namespace pairtile

// Launch of the A16 pair-tile GEMM (declared in gemm_kernel.cuh): bf16
// activation rows contiguous per tile (GROUPED or PADDED, loaded by TMA), int8
// weights with per-row scales or packed int4 weights with per-group scales.
qmoe_status_t launch_gemm_pair_a16(bool int4, const void* w, int64_t E, int64_t N, int64_t K, const GemmParams& p,
                                   int64_t max_padded, int64_t a_rows, int64_t lda, cudaStream_t st) {
    return int4 ? pairtile::launch_pair_a16<true>(w, E, N, K, p, max_padded, a_rows, lda, st)
                : pairtile::launch_pair_a16<false>(w, E, N, K, p, max_padded, a_rows, lda, st);
}

}  // namespace qmoe
