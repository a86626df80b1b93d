// gemm_pair.cu -- FP8 W8A8 grouped GEMM on CTA pairs (tcgen05 cta_group::2)
// for the large-M (prefill) shapes.
//
// One tile = 256 output channels n of one expert x up to 256 consecutive
// sorted slots of that expert, computed by a cluster of two CTAs on two SMs
// with one 256-row MMA per k-step:
//
//   * MMA A operand (M = 256): the weight rows.  CTA r loads rows
//     [n0 + 128 r, n0 + 128 r + 128) of W[e] into its own shared memory.
//   * MMA B operand (N = Nt <= 256): the activation rows of the tile's slots.
//     CTA r loads slots [s0 + r Nt/2, s0 + r Nt/2 + Nt/2) (a 128-row box, of
//     which the first Nt/2 rows are used).
//   * D: CTA r's tensor memory holds its 128 weight rows x all Nt slots.
//
// Against the one-SM wide tile (128 slots x 256 weight rows) every SM loads
// 32 KB of operands per 128-wide k-step instead of 48 KB for the same FLOPs,
// and reads a third less shared memory per MMA.  Nt is the tile's valid slot
// count rounded up to 32, so the last, partly filled slot block of an expert
// costs MMA time in proportion to its slots.
//
// Roles (each CTA: warp 0 TMA producer, warp 1 MMA issuer in CTA 0, warps
// 2-5 epilogue over the CTA's own accumulator):
//   * both producers load into their own ring; every load completes on CTA
//     0's `full` barrier (CTA 1's through the cta_group::2 form of the TMA
//     load, which may signal the partner's barrier), whose expected bytes CTA
//     0's producer sets for both; each producer also prefetches the weight box
//     one ring ahead into L2;
//   * CTA 0's MMA thread waits on `full`, issues the pair's MMAs
//     and commits them to the `empty` barrier of both CTAs (multicast commit),
//     and at the end of a tile to both CTAs' `tfull`;
//   * each epilogue reads its accumulator, then arrives on CTA 0's `tempty`
//     (256 arrivals: both CTAs' epilogue threads).
// Every wait is bounded; a CTA that gives up sets QMOE_DEV_TIMEOUT and leaves
// its loops, and its partner's waits then run out too.  Both CTAs meet at a
// cluster barrier before TMEM is released and before either exits, so no CTA
// leaves while the other can still reach its shared or tensor memory.
#include "pair_common.cuh"

namespace qmoe {
namespace pairtile {

constexpr int kBoxRows = 128;                 // activation rows loaded per CTA per k-block (B half <= 128)
constexpr int kBK = 128;                      // K bytes per k-block (one 128-byte swizzled box per operand)
constexpr int kABytes = kRowsCta * kBK;       // 16 KB of weight rows per k-block
constexpr int kBBytes = kBoxRows * kBK;       // 16 KB of activation rows per k-block
constexpr int kEpiThreads = 128;
constexpr int kThreads = 64 + kEpiThreads;
constexpr int kAccCols = 256;
constexpr bool kPfFirstPairOnly = true;       // only the first slot pair of a weight block prefetches it
// Ring of kKS k-blocks per stage: one barrier round trip per stage moves kKS x 32
// KB per CTA (the weight halves first, then the activation halves), with the
// ring's 192 KB in 6 / kKS stages; weight boxes are prefetched into L2 one ring
// ahead.  Two k-blocks per stage halve the per-stage handshakes, which bound
// the decode-sized launches (16 KB of weights per stage and CTA).
template <int kKS>
struct PairCfg {
    static constexpr int kStages = 6 / kKS;
    static constexpr int kStageBytes = kKS * (kABytes + kBBytes);
    static constexpr int kDynSmem = kStages * kStageBytes + 1024;
    static constexpr int kPfStages = kStages;  // stages prefetched ahead
};

// kAccBufs: accumulators in tensor memory (2: the epilogue of one tile
// overlaps the MMAs of the next; 1: 256 columns, one tile at a time).
template <int kAccBufs, int kKS>
__global__ void __launch_bounds__(kThreads, 1)
    moe_gemm_pair_kernel(const __grid_constant__ CUtensorMap tmap_w, const __grid_constant__ CUtensorMap tmap_a,
                         const GemmParams p) {
    using PC = PairCfg<kKS>;
    constexpr int S = PC::kStages;
    constexpr int kStageBytes = PC::kStageBytes;
    constexpr int kPfStages = PC::kPfStages;
    constexpr int kTmemCols = kAccBufs * kAccCols;
    extern __shared__ uint8_t smem_raw[];
    __shared__ uint64_t bar_full[S], bar_empty[S];
    __shared__ uint64_t bar_tfull[2], bar_tempty[2], bar_drain;
    __shared__ uint32_t s_tmem_base;
    __shared__ int s_abort;
    __shared__ int32_t s_crow[kTileSlots];     // output row of each tile column (-1: none)
    __shared__ float s_cscale[kTileSlots];     // activation scale x routing weight of each tile column
    __shared__ int32_t s_poff[kGemmMaxE + 1];  // padded_offsets
    __shared__ int32_t s_pre[kGemmMaxE + 1];   // slot pairs (256-slot tiles) of the experts before e

    const uint32_t raw_addr = smem_u32(smem_raw);
    uint8_t* smem = smem_raw + (((raw_addr + 1023u) & ~1023u) - raw_addr);
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t rank = cluster_ctarank();

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(&bar_full[s], 1);   // used in CTA 0: its producer, plus both CTAs' TMA bytes
            mbar_init(&bar_empty[s], 1);  // the pair's MMA commit
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&bar_tfull[i], 1);
            mbar_init(&bar_tempty[i], 2 * kEpiThreads);  // used in CTA 0: both CTAs' epilogue threads
        }
        mbar_init(&bar_drain, 1);
        s_abort = 0;
        fence_mbar_init();
    }
    if (warp == 1) tmem_alloc_pair(&s_tmem_base, kTmemCols);
    // the partner's barriers are initialised before any arrival reaches them
    __syncwarp();
    cluster_sync_all();
    pdl_launch_dependents();
    pdl_wait();
    for (int i = threadIdx.x; i <= p.E; i += blockDim.x) s_poff[i] = p.padded_offsets[i];
    if (warp == 0) {
        // s_pre[i] = sum over experts e < i of ceil(padded rows of e / 256), a warp scan per 32 experts
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
    const int nks = (nkb + kKS - 1) / kKS;  // stages per tile (a last k-block past K loads zeros)
    // k-block kk of stage s: weight rows (MMA A), slot rows (MMA B)
    auto a_tile = [&](int s, int kk) { return smem + s * kStageBytes + kk * kABytes; };
    auto b_tile = [&](int s, int kk) { return smem + s * kStageBytes + kKS * kABytes + kk * kBBytes; };

    if (warp == 0) {
        // ------------------------------------------------ TMA producer ---
        if (lane == 0) {
            int it = 0;
            bool ok = true;
            for (int t = c0; ok && t < num_tiles; t += nc) {
                const Tile x = decode_tile(t, p.E, n_blocks, s_pre, s_poff, p.expert_offsets);
                const int half = x.nt / 2;
                const int arow = (p.a_layout == QMOE_A_PADDED ? x.s0
                                                              : p.expert_offsets[x.e] + (x.s0 - s_poff[x.e])) +
                                 static_cast<int>(rank) * half;
                const int wrow = x.nb * kTileRows + static_cast<int>(rank) * kRowsCta;
                // the CTA's next tile, whose first weight boxes are prefetched into L2
                // while this tile's last k-blocks load
                const bool has_next = t + nc < num_tiles;
                const Tile xn = has_next ? decode_tile(t + nc, p.E, n_blocks, s_pre, s_poff, p.expert_offsets) : x;
                const int wrow_n = xn.nb * kTileRows + static_cast<int>(rank) * kRowsCta;
                for (int ks = 0; ks < nks; ++ks, ++it) {
                    const int s = it % S;
                    const uint32_t ph = (it / S) & 1;
                    if (!mbar_wait(&bar_empty[s], ph ^ 1, abort, p.d_status)) { ok = false; break; }
                    if (rank == 0) {  // both CTAs' loads complete on CTA 0's barrier
                        mbar_arrive_expect_tx(&bar_full[s], 2 * kStageBytes);
#pragma unroll
                        for (int kk = 0; kk < kKS; ++kk) {
                            tma_load_3d(&tmap_w, &bar_full[s], a_tile(s, kk), (ks * kKS + kk) * kBK, wrow, x.e);
                            tma_load_2d(&tmap_a, &bar_full[s], b_tile(s, kk), (ks * kKS + kk) * kBK, arow);
                        }
                    } else {
                        const uint32_t bar0 = map_shared_rank(&bar_full[s], 0);
#pragma unroll
                        for (int kk = 0; kk < kKS; ++kk) {
                            tma_load_3d_to_leader(&tmap_w, bar0, a_tile(s, kk), (ks * kKS + kk) * kBK, wrow, x.e);
                            tma_load_2d_to_leader(&tmap_a, bar0, b_tile(s, kk), (ks * kKS + kk) * kBK, arow);
                        }
                    }
                    const int kp = ks + kPfStages;  // the stage one ring ahead, in this tile or the next
#pragma unroll
                    for (int kk = 0; kk < kKS; ++kk) {
                        if (kp < nks) {
                            if ((!kPfFirstPairOnly || x.pr == 0) && kp * kKS + kk < nkb)
                                tma_prefetch_l2_3d_box(&tmap_w, (kp * kKS + kk) * kBK, wrow, x.e);
                        } else if (has_next && kp - nks < nks && (!kPfFirstPairOnly || xn.pr == 0) &&
                                   (kp - nks) * kKS + kk < nkb) {
                            tma_prefetch_l2_3d_box(&tmap_w, ((kp - nks) * kKS + kk) * kBK, wrow_n, xn.e);
                        }
                    }
                }
            }
            if (!ok) {  // let copies already issued land before the CTA can go on
                const uint64_t t0 = global_timer_ns();
                while (global_timer_ns() - t0 < 2000000ull) {}
            }
        }
    } else if (warp == 1) {
        if (lane == 0 && rank == 0) {
            // ------------------------------------- MMA issuer (CTA 0) ---
            int it = 0, tcount = 0;
            bool ok = true;
            for (int t = c0; ok && t < num_tiles; t += nc) {
                const Tile x = decode_tile(t, p.E, n_blocks, s_pre, s_poff, p.expert_offsets);
                const int acc = tcount % kAccBufs;
                const uint32_t aph = (tcount / kAccBufs) & 1;
                if (!mbar_wait(&bar_tempty[acc], aph ^ 1, abort, p.d_status)) break;
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * kAccCols);
                const uint32_t idesc = make_idesc(kFmtE4M3, 256, x.nt);
                for (int ks = 0; ks < nks; ++ks, ++it) {
                    const int s = it % S;
                    const uint32_t ph = (it / S) & 1;
                    if (!mbar_wait(&bar_full[s], ph, abort, p.d_status)) { ok = false; break; }
                    tc_fence_after();
#pragma unroll
                    for (int kk = 0; kk < kKS; ++kk) {
                        const uint64_t da = desc_kmajor_sw128(smem_u32(a_tile(s, kk)));
                        const uint64_t db = desc_kmajor_sw128(smem_u32(b_tile(s, kk)));
#pragma unroll
                        for (int k = 0; k < 4; ++k)
                            mma_pair_f8f6f4(d_tmem, da + 2 * k, db + 2 * k, idesc, (ks | kk | k) != 0);
                    }
                    tc_commit_pair(&bar_empty[s], 0x3);
                }
                if (!ok) break;
                tc_commit_pair(&bar_tfull[acc], 0x3);
                ++tcount;
            }
            tc_commit_pair(&bar_drain, 0x1);  // every MMA issued above has completed once this fires
            int dummy = 0;
            mbar_wait(&bar_drain, 0, &dummy, p.d_status);
        }
    } else {
        // ------------------------------------------------- epilogue ---
        // lane = weight row (output channel), columns = the tile's slots
        const int et = threadIdx.x - 64;
        const int q = warp & 3;  // TMEM lane quadrant of this warp
        const bool even = (lane & 1) == 0;
        const uint32_t tempty0 = map_shared_rank(&bar_tempty[0], 0);
        const uint32_t tempty1 = map_shared_rank(&bar_tempty[1], 0);
        int tcount = 0;
        for (int t = c0; t < num_tiles; t += nc) {
            if (*abort) break;
            const Tile x = decode_tile(t, p.E, n_blocks, s_pre, s_poff, p.expert_offsets);
            const int acc = tcount % kAccBufs;
            const uint32_t aph = (tcount / kAccBufs) & 1;
            named_bar_sync(1, kEpiThreads);
            for (int j = et; j < kTileSlots; j += kEpiThreads) {
                int row = -1;
                float sc = 0.0f;
                if (j < x.nv) {
                    const int pos = x.s0 + j;
                    const int s = p.sorted_ids[pos];
                    if (s >= 0 && s < p.T) {
                        const int m = s / p.top_k;
                        const int compact = p.expert_offsets[x.e] + (pos - s_poff[x.e]);
                        const int arow = (p.a_layout == QMOE_A_GROUPED) ? compact : pos;
                        sc = p.a_scale[arow] * (p.topk_w ? p.topk_w[s] : 1.0f);
                        row = (p.out_layout == QMOE_OUT_SLOT) ? s : (p.out_layout == QMOE_OUT_GROUPED ? compact : m);
                    }
                }
                s_crow[j] = row;
                s_cscale[j] = sc;
            }
            named_bar_sync(1, kEpiThreads);
            const int64_t n = static_cast<int64_t>(x.nb) * kTileRows + static_cast<int64_t>(rank) * kRowsCta + q * 32 +
                              lane;
            const float sw = (n < p.N) ? p.w_scale[static_cast<int64_t>(x.e) * p.N + n] : 0.0f;
            const int64_t nn = even ? n : n - 1;
            const bool tsum = p.out_layout == QMOE_OUT_TOKEN_SUM;
            if (!mbar_wait(&bar_tfull[acc], aph, abort, p.d_status)) break;
            tc_fence_after();
            const uint32_t t_base =
                tmem_base + (static_cast<uint32_t>(q * 32) << 16) + static_cast<uint32_t>(acc * kAccCols);
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
                    // even lane: column j at (n, n+1); odd lane: column j+1 at (n-1, n)
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
            // accumulator read out: hand it back to the MMA of CTA 0
            tc_fence_before();
            mbar_arrive_cluster(acc == 0 ? tempty0 : tempty1);
            ++tcount;
        }
    }

    // Both CTAs past their loops (the MMA thread after its drain): no arrival,
    // MMA operand read or accumulator write can reach either CTA after this.
    __syncwarp();
    tc_fence_before();
    cluster_sync_all();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc_pair(tmem_base, kTmemCols);
    }
}

template <int kAccBufs, int kKS>
qmoe_status_t launch_pair(const void* w, int64_t E, int64_t N, int64_t K, const GemmParams& p, int64_t max_padded,
                          int64_t a_rows, int64_t lda, cudaStream_t st) {
    using PC = PairCfg<kKS>;
    constexpr int kDynSmem = PC::kDynSmem;
    static std::mutex mu;
    static bool attr_set[64] = {false};
    static int max_clusters[64] = {0};
    auto kern = moe_gemm_pair_kernel<kAccBufs, kKS>;
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
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = kDynSmem;
    cfg.stream = st;
    cfg.attrs = attr;
    {
        std::lock_guard<std::mutex> g(mu);
        if (!attr_set[dev]) {
            if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kDynSmem) != cudaSuccess)
                return QMOE_ERR_CUDA;
            // clusters of two that fit on the device at once (one CTA per SM): a
            // persistent grid larger than that would run its last clusters after
            // the others instead of beside them
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
    if (!make_weight_map(&map, w, E, N, K, kBK, kRowsCta, true)) return QMOE_ERR_CUDA;
    if (!make_act_map(&amap, p.a, a_rows, K, lda, 1, kBoxRows)) return QMOE_ERR_CUDA;
    // (one more tile per expert: an expert's last pair may hold a single 128-slot block)
    const int64_t max_tiles = ((max_padded + kTileSlots - 1) / kTileSlots + E) * ((N + kTileRows - 1) / kTileRows);
    const int64_t clusters = max_tiles < max_clusters[dev] ? max_tiles : max_clusters[dev];
    if (clusters <= 0) return QMOE_OK;
    cfg.gridDim = dim3(static_cast<unsigned>(2 * clusters));
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, kern, map, amap, p) == cudaSuccess ? QMOE_OK : QMOE_ERR_CUDA;
}

}  // namespace pairtile

// Launch of the pair-tile GEMM (declared in gemm_kernel.cuh): FP8 e4m3
// weights and activations with per-row scales, activation rows contiguous per
// tile (GROUPED or PADDED layouts, loaded by TMA), any output layout.
qmoe_status_t launch_gemm_pair(const void* w, int64_t E, int64_t N, int64_t K, const GemmParams& p,
                               int64_t max_padded, int64_t a_rows, int64_t lda, cudaStream_t st) {
    return pairtile::launch_pair<2, 2>(w, E, N, K, p, max_padded, a_rows, lda, st);
}

}  // namespace qmoe
