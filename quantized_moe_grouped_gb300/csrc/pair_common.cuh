// pair_common.cuh -- helpers of the CTA-pair GEMM tiles (tcgen05 cta_group::2):
// cluster addressing, cross-CTA barrier arrivals and TMA completions, pair
// TMEM allocation, pair MMAs and commits, and the pair tile decoder.
#pragma once

#include "gemm_kernel.cuh"

namespace qmoe {
namespace pairtile {

constexpr int kTileSlots = 256;               // slots per pair tile (at most)
constexpr int kTileRows = 256;                // weight rows per pair tile (both CTAs)
constexpr int kRowsCta = 128;                 // weight rows per CTA (the MMA A operand's half)

// ------------------------------------------------------------ cluster PTX ---
// (cluster_ctarank, cluster_id_x, num_clusters_x and cluster_sync_all are in
// common.cuh)
// Address of the same shared-memory location in CTA `rank` of the cluster.
QMOE_DI uint32_t map_shared_rank(const void* p, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_u32(p)), "r"(rank));
    return r;
}
// Arrive on an mbarrier given by its cluster-window address (possibly in the
// partner CTA).  The waits on these barriers are ordinary CTA-scope waits: what
// the arrival hands over is shared or tensor memory that the tensor core reads
// or writes after a tcgen05 fence, not data the waiting thread loads itself.
QMOE_DI void mbar_arrive_cluster(uint32_t cluster_addr) {
    asm volatile("mbarrier.arrive.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr) : "memory");
}
// The same with release semantics at cluster scope: shared-memory stores this
// thread made (and fenced for the async proxy) are ordered before the arrival
// for the partner CTA too.
QMOE_DI void mbar_arrive_cluster_release(uint32_t cluster_addr) {
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr) : "memory");
}
// Tiled TMA loads into this CTA's shared memory that complete on an mbarrier
// in the pair's CTA 0 (cluster-window address of that barrier).
QMOE_DI void tma_load_3d_to_leader(const CUtensorMap* map, uint32_t bar_cluster, void* dst, int x, int y, int z) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.cta_group::2"
        " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(bar_cluster)
        : "memory");
}
QMOE_DI void tma_load_2d_to_leader(const CUtensorMap* map, uint32_t bar_cluster, void* dst, int x, int y) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.cta_group::2"
        " [%0], [%1, {%2, %3}], [%4];" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar_cluster)
        : "memory");
}
QMOE_DI void tma_prefetch_l2_3d_box(const CUtensorMap* map, int x, int y, int z) {
    asm volatile("cp.async.bulk.prefetch.tensor.3d.L2.global.tile [%0, {%1, %2, %3}];" ::"l"(
                     reinterpret_cast<uint64_t>(map)),
                 "r"(x), "r"(y), "r"(z)
                 : "memory");
}

// -------------------------------------------------- tcgen05, CTA pairs ---
QMOE_DI void tmem_alloc_pair(uint32_t* dst_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst_smem)),
                 "r"(ncols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}
QMOE_DI void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
// D[tmem of both CTAs] (+)= A[smem of both CTAs] * B[smem of both CTAs]^T, e4m3 -> f32.
QMOE_DI void mma_pair_f8f6f4(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                             uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}
// The same with bf16 operands (kind::f16).
QMOE_DI void mma_pair_f16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}
// Arrive once on the mbarrier at this shared-memory offset in every CTA of
// `cta_mask` when all MMAs issued so far by this thread have completed.
QMOE_DI void tc_commit_pair(uint64_t* bar, uint16_t cta_mask) {
    asm volatile(
        "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(
            smem_u32(bar)),
        "h"(cta_mask)
        : "memory");
}

// Tile t of the launch: expert e (binary search over the per-expert tile
// prefix), weight block nb (256 rows), first padded position s0 of its slots,
// valid slots nv (1..256) and MMA width nt = roundup(nv, 32).  Inside an
// expert the tiles run weight block major, slot pair fastest, so the slot
// pairs that share a weight tile run at the same time.
struct Tile {
    int e, nb, pr, s0, nv, nt;
};
QMOE_DI Tile decode_tile(int t, int E, int n_blocks, const int32_t* s_pre, const int32_t* s_poff,
                         const int32_t* expert_offsets) {
    int lo = 0, hi = E - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (s_pre[mid] * n_blocks <= t) lo = mid;
        else hi = mid - 1;
    }
    Tile x;
    x.e = lo;
    const int np = s_pre[lo + 1] - s_pre[lo];
    const int local = t - s_pre[lo] * n_blocks;
    x.nb = local / np;
    const int pr = local % np;
    x.pr = pr;
    x.s0 = s_poff[lo] + kTileSlots * pr;
    const int cnt = expert_offsets[lo + 1] - expert_offsets[lo];
    const int rows = min(kTileSlots, s_poff[lo + 1] - x.s0);
    x.nv = max(1, min(rows, cnt - kTileSlots * pr));
    x.nt = (x.nv + 31) & ~31;  // each CTA's half of the B operand: a multiple of 16 rows
    return x;
}

}  // namespace pairtile
}  // namespace qmoe
