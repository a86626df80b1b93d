// align_quant.cu -- moe_align_block_size, the per-row FP8/INT8 quantisers,
// SwiGLU + per-token / MXFP8 requantisation, and the element-level test hooks.
#include <cuda_runtime.h>
#include <stdint.h>

#include "common.cuh"
#include "host_util.h"
#include "qmoe.h"

namespace qmoe {

// ======================================================================
// moe_align_block_size: one CTA of 1024 threads; warp w owns the contiguous
// slot range [w * chunk, (w + 1) * chunk) (chunk a multiple of 32).
//   1. per-warp expert counts: the warp walks its range 32 slots at a time
//      (the ids of 8 steps loaded together, kept in registers for step 3 when
//      the range is at most 256 slots);
//      __match_any_sync groups equal ids, the group's first lane adds the
//      group size to the warp's own counter row (no atomics);
//   2. per expert, an exclusive scan over the 32 warps (the warp's first
//      position inside the expert's group) and the expert totals; then the
//      unpadded and padded prefix sums (one thread), sentinel fill and the
//      block -> expert map;
//   3. the warp walks its range again: a slot's position is its expert's
//      padded offset + the warp's running cursor for the expert + its rank
//      among the equal ids of lower lanes; the group's first lane advances
//      the cursor.  Ranges, steps and lanes are in ascending slot order, so
//      the placement is stable.
// ======================================================================
constexpr int kAlignThreads = 1024;
constexpr int kAlignMaxE = 256;
constexpr int kAlignBatch = 8;  // 32-slot steps whose ids a lane loads at once


__global__ void __launch_bounds__(kAlignThreads, 1)
    align_kernel(const int32_t* __restrict__ ids, int64_t T, int E, int BM, int32_t* __restrict__ sorted_ids,
                 int64_t sorted_cap, int32_t* __restrict__ expert_ids, int64_t blocks_cap,
                 int32_t* __restrict__ num_post_padded, int32_t* __restrict__ expert_offsets,
                 int32_t* __restrict__ padded_offsets, int32_t* d_status) {
    pdl_launch_dependents();
    pdl_wait();  // inputs from, and buffers shared with, the previous kernel
    __shared__ int s_cnt[kAlignMaxE];
    __shared__ int s_poff[kAlignMaxE + 1];
    __shared__ int s_wcnt[32 * kAlignMaxE];  // [warp][expert]: counts, then running positions
    __shared__ int s_bad;
    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    const int64_t chunk = ((T + 31) / 32 + 31) / 32 * 32;
    const int64_t w_begin = warp * chunk;
    const int64_t w_end = w_begin + chunk < T ? w_begin + chunk : T;

    for (int i = tid; i < 32 * E; i += blockDim.x) s_wcnt[i] = 0;
    if (tid == 0) s_bad = 0;
    __syncthreads();

    const unsigned lt_mask = (1u << lane) - 1u;
    int* wrow = s_wcnt + warp * E;
    // ids of kAlignBatch 32-slot steps per lane, loaded together (one memory latency per batch)
    int ev[kAlignBatch];
    auto load_batch = [&](int64_t base) {
#pragma unroll
        for (int i = 0; i < kAlignBatch; ++i) {
            const int64_t sl = base + i * 32 + lane;
            ev[i] = (sl < w_end) ? ids[sl] : -1;
        }
    };
    const bool one_batch = chunk <= 32 * kAlignBatch;  // the range's ids stay in registers for pass 3
    for (int64_t b0 = w_begin; b0 < w_end; b0 += 32 * kAlignBatch) {
        load_batch(b0);
#pragma unroll
        for (int i = 0; i < kAlignBatch; ++i) {
            const int e = ev[i];
            const bool valid = e >= 0 && e < E;
            if (b0 + i * 32 + lane < w_end && !valid) s_bad = 1;
            const unsigned peers = __match_any_sync(0xFFFFFFFFu, valid ? e : E);
            if (valid && (peers & lt_mask) == 0) wrow[e] += __popc(peers);
            __syncwarp();
        }
    }
    __syncthreads();

    for (int e = tid; e < E; e += blockDim.x) {
        int run = 0;
        for (int w = 0; w < 32; ++w) {
            const int c = s_wcnt[w * E + e];
            s_wcnt[w * E + e] = run;
            run += c;
        }
        s_cnt[e] = run;
    }
    __syncthreads();

    if (tid == 0) {
        int off = 0, poff = 0;
        for (int e = 0; e < E; ++e) {
            expert_offsets[e] = off;
            padded_offsets[e] = poff;
            s_poff[e] = poff;
            off += s_cnt[e];
            poff += (s_cnt[e] + BM - 1) / BM * BM;
        }
        expert_offsets[E] = off;
        padded_offsets[E] = poff;
        s_poff[E] = poff;
        *num_post_padded = poff;
        if (s_bad && d_status) atomicOr(reinterpret_cast<int*>(d_status), QMOE_DEV_INVALID_EXPERT);
    }
    __syncthreads();

    const int32_t sentinel = static_cast<int32_t>(T);
    for (int64_t p = tid; p < sorted_cap; p += blockDim.x) sorted_ids[p] = sentinel;
    for (int64_t b = tid; b < blocks_cap; b += blockDim.x) {
        const int64_t p = b * BM;
        int owner = -1;
        if (p < s_poff[E]) {
            int lo = 0, hi = E - 1;  // last e with s_poff[e] <= p
            while (lo < hi) {
                const int mid = (lo + hi + 1) >> 1;
                if (s_poff[mid] <= p) lo = mid;
                else hi = mid - 1;
            }
            owner = lo;
        }
        expert_ids[b] = owner;
    }
    __syncthreads();

    for (int64_t b0 = w_begin; b0 < w_end; b0 += 32 * kAlignBatch) {
        if (!one_batch) load_batch(b0);
#pragma unroll
        for (int i = 0; i < kAlignBatch; ++i) {
            const int64_t sl = b0 + i * 32 + lane;
            const int e = ev[i];
            const bool valid = e >= 0 && e < E;
            const unsigned peers = __match_any_sync(0xFFFFFFFFu, valid ? e : E);
            const int cur = valid ? wrow[e] : 0;
            __syncwarp();
            if (valid) {
                sorted_ids[s_poff[e] + cur + __popc(peers & lt_mask)] = static_cast<int32_t>(sl);
                if ((peers & lt_mask) == 0) wrow[e] = cur + __popc(peers);
            }
            __syncwarp();
        }
    }
}

// ======================================================================
// moe_align_block_size for many slots: a cluster of kAlignCtas CTAs (16 warps
// each).  Global warp g = rank * 16 + warp owns slots [g * chunk, (g+1) *
// chunk), so ranks, warps, steps and lanes run in ascending slot order.
//   1. per-warp expert counts, as in align_kernel;
//   2. per expert, an exclusive scan over the CTA's warps and the CTA's total;
//      cluster barrier; each CTA reads the other CTAs' totals through
//      distributed shared memory (its own offset inside every expert's group
//      and the expert totals); cluster barrier (no CTA leaves while another
//      may still read its shared memory);
//   3. every CTA computes the padded offsets; CTA 0 writes them; the CTAs
//      split the sentinel fill of the pad positions and the block -> expert
//      map; each warp places its slots.
// Pad positions and slot positions are disjoint, so the fill and the scatter
// need no ordering between CTAs.
// ======================================================================
constexpr int kAlignCtas = 8;
constexpr int kAlignCThreads = 512;
constexpr int64_t kAlignClusterMinSlots = 2048;
constexpr int kAlignCWarps = kAlignCThreads / 32;

// A 32-bit word of CTA `rank`'s shared memory at the offset of `p` in this CTA.
QMOE_DI int load_cluster_peer(const int* p, uint32_t rank) {
    uint32_t a;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(a) : "r"(smem_u32(p)), "r"(rank));
    int v;
    asm volatile("ld.shared::cluster.u32 %0, [%1];" : "=r"(v) : "r"(a));
    return v;
}

__global__ void __launch_bounds__(kAlignCThreads, 1)
    align_cluster_kernel(const int32_t* __restrict__ ids, int64_t T, int E, int BM, int32_t* __restrict__ sorted_ids,
                         int64_t sorted_cap, int32_t* __restrict__ expert_ids, int64_t blocks_cap,
                         int32_t* __restrict__ num_post_padded, int32_t* __restrict__ expert_offsets,
                         int32_t* __restrict__ padded_offsets, int32_t* d_status) {
    pdl_launch_dependents();
    pdl_wait();  // inputs from, and buffers shared with, the previous kernel
    __shared__ int s_wcnt[kAlignCWarps * kAlignMaxE];  // [warp][expert]: counts, then running positions
    __shared__ int s_ccnt[kAlignMaxE];                  // this CTA's count per expert (read by the others)
    __shared__ int s_coff[kAlignMaxE];                  // this CTA's first position inside each expert's group
    __shared__ int s_cnt[kAlignMaxE];
    __shared__ int s_poff[kAlignMaxE + 1];
    __shared__ int s_bad;
    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    const uint32_t rank = cluster_ctarank();
    const int64_t nwarps = static_cast<int64_t>(kAlignCtas) * kAlignCWarps;
    const int64_t chunk = ((T + nwarps - 1) / nwarps + 31) / 32 * 32;
    const int64_t gw = static_cast<int64_t>(rank) * kAlignCWarps + warp;
    const int64_t w_begin = gw * chunk < T ? gw * chunk : T;
    const int64_t w_end = w_begin + chunk < T ? w_begin + chunk : T;

    for (int i = tid; i < kAlignCWarps * E; i += blockDim.x) s_wcnt[i] = 0;
    if (tid == 0) s_bad = 0;
    __syncthreads();

    const unsigned lt_mask = (1u << lane) - 1u;
    int* wrow = s_wcnt + warp * E;
    int ev[kAlignBatch];
    auto load_batch = [&](int64_t base) {
#pragma unroll
        for (int i = 0; i < kAlignBatch; ++i) {
            const int64_t sl = base + i * 32 + lane;
            ev[i] = (sl < w_end) ? ids[sl] : -1;
        }
    };
    const bool one_batch = chunk <= 32 * kAlignBatch;
    for (int64_t b0 = w_begin; b0 < w_end; b0 += 32 * kAlignBatch) {
        load_batch(b0);
#pragma unroll
        for (int i = 0; i < kAlignBatch; ++i) {
            const int e = ev[i];
            const bool valid = e >= 0 && e < E;
            if (b0 + i * 32 + lane < w_end && !valid) s_bad = 1;
            const unsigned peers = __match_any_sync(0xFFFFFFFFu, valid ? e : E);
            if (valid && (peers & lt_mask) == 0) wrow[e] += __popc(peers);
            __syncwarp();
        }
    }
    __syncthreads();
    for (int e = tid; e < E; e += blockDim.x) {
        int run = 0;
        for (int w = 0; w < kAlignCWarps; ++w) {
            const int c = s_wcnt[w * E + e];
            s_wcnt[w * E + e] = run;
            run += c;
        }
        s_ccnt[e] = run;
    }
    cluster_sync_all();  // every CTA's totals are in its shared memory
    for (int e = tid; e < E; e += blockDim.x) {
        int v[kAlignCtas];  // all CTAs' counts, loaded together (one remote latency)
#pragma unroll
        for (int c = 0; c < kAlignCtas; ++c) v[c] = load_cluster_peer(&s_ccnt[e], static_cast<uint32_t>(c));
        int before = 0, total = 0;
#pragma unroll
        for (int c = 0; c < kAlignCtas; ++c) {
            if (c < static_cast<int>(rank)) before += v[c];
            total += v[c];
        }
        s_coff[e] = before;
        s_cnt[e] = total;
    }
    cluster_sync_all();  // no CTA reads another's shared memory after this point
    if (tid == 0) {
        int off = 0, poff = 0;
        for (int e = 0; e < E; ++e) {
            if (rank == 0) {
                expert_offsets[e] = off;
                padded_offsets[e] = poff;
            }
            s_poff[e] = poff;
            off += s_cnt[e];
            poff += (s_cnt[e] + BM - 1) / BM * BM;
        }
        s_poff[E] = poff;
        if (rank == 0) {
            expert_offsets[E] = off;
            padded_offsets[E] = poff;
            *num_post_padded = poff;
        }
        if (s_bad && d_status) atomicOr(reinterpret_cast<int*>(d_status), QMOE_DEV_INVALID_EXPERT);
    }
    __syncthreads();

    // the expert owning padded position p (last e with s_poff[e] <= p), or -1 past the groups
    auto owner_of = [&](int64_t p) {
        if (p >= s_poff[E]) return -1;
        int lo = 0, hi = E - 1;
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (s_poff[mid] <= p) lo = mid;
            else hi = mid - 1;
        }
        return lo;
    };
    const int32_t sentinel = static_cast<int32_t>(T);
    const int64_t stride = static_cast<int64_t>(kAlignCtas) * kAlignCThreads;
    for (int64_t p = static_cast<int64_t>(rank) * kAlignCThreads + tid; p < sorted_cap; p += stride) {
        const int e = owner_of(p);
        if (e < 0 || p - s_poff[e] >= s_cnt[e]) sorted_ids[p] = sentinel;
    }
    for (int64_t b = static_cast<int64_t>(rank) * kAlignCThreads + tid; b < blocks_cap; b += stride)
        expert_ids[b] = owner_of(b * BM);

    for (int64_t b0 = w_begin; b0 < w_end; b0 += 32 * kAlignBatch) {
        if (!one_batch) load_batch(b0);
#pragma unroll
        for (int i = 0; i < kAlignBatch; ++i) {
            const int64_t sl = b0 + i * 32 + lane;
            const int e = ev[i];
            const bool valid = e >= 0 && e < E;
            const unsigned peers = __match_any_sync(0xFFFFFFFFu, valid ? e : E);
            const int cur = valid ? wrow[e] : 0;
            __syncwarp();
            if (valid) {
                sorted_ids[s_poff[e] + s_coff[e] + cur + __popc(peers & lt_mask)] = static_cast<int32_t>(sl);
                if ((peers & lt_mask) == 0) wrow[e] = cur + __popc(peers);
            }
            __syncwarp();
        }
    }
}

// ======================================================================
// Per-row quantisers: one CTA per row.  Pass 1 takes the row's amax, pass 2
// re-reads the row (L1/L2) and writes the codes.  The vector path moves 8
// elements per step (16-byte bf16 or 2x16-byte fp32 loads, 8-byte stores).
// ======================================================================
constexpr int kRowThreads = 256;

QMOE_DI float block_max(float v, float* red) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xFFFFFFFFu, v, o));
    const int warp = threadIdx.x >> 5;
    if ((threadIdx.x & 31) == 0) red[warp] = v;
    __syncthreads();
    if (threadIdx.x < 32) {
        float x = (threadIdx.x < (blockDim.x >> 5)) ? red[threadIdx.x] : 0.0f;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) x = fmaxf(x, __shfl_xor_sync(0xFFFFFFFFu, x, o));
        if (threadIdx.x == 0) red[32] = x;
    }
    __syncthreads();
    return red[32];
}

QMOE_DI void unpack8(const uint4 w, float (&v)[8]) {
    v[0] = bf16_lo(w.x); v[1] = bf16_hi(w.x); v[2] = bf16_lo(w.y); v[3] = bf16_hi(w.y);
    v[4] = bf16_lo(w.z); v[5] = bf16_hi(w.z); v[6] = bf16_lo(w.w); v[7] = bf16_hi(w.w);
}
QMOE_DI void load8(const uint16_t* p, float (&v)[8]) {
    const uint4 w = *reinterpret_cast<const uint4*>(p);
    v[0] = bf16_lo(w.x); v[1] = bf16_hi(w.x); v[2] = bf16_lo(w.y); v[3] = bf16_hi(w.y);
    v[4] = bf16_lo(w.z); v[5] = bf16_hi(w.z); v[6] = bf16_lo(w.w); v[7] = bf16_hi(w.w);
}
QMOE_DI void load8(const float* p, float (&v)[8]) {
    const float4 a = *reinterpret_cast<const float4*>(p);
    const float4 b = *reinterpret_cast<const float4*>(p + 4);
    v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w; v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
}
QMOE_DI float load1(const uint16_t* p) { return __uint_as_float(static_cast<uint32_t>(*p) << 16); }
QMOE_DI float load1(const float* p) { return *p; }

// e4m3 codes of v[0..7] / s (correctly rounded quotients, see div_rn_by), 8 bytes.
QMOE_DI uint2 quant8(const float (&v)[8], float s, float rinv) {
    float q[8];
#pragma unroll
    for (int i = 0; i < 8; i += 2) div2_rn_by(v[i], v[i + 1], s, rinv, q[i], q[i + 1]);
    uint2 o;
    o.x = e4m3x4(q[0], q[1], q[2], q[3]);
    o.y = e4m3x4(q[4], q[5], q[6], q[7]);
    return o;
}

template <typename Tin, bool kVec>
__global__ void __launch_bounds__(kRowThreads)
    quant_rows_fp8_kernel(const Tin* __restrict__ x, int64_t cols, int64_t ldx, uint8_t* __restrict__ q,
                          float* __restrict__ scale) {
    __shared__ float red[33];
    const int64_t row = blockIdx.x;
    const Tin* xr = x + row * ldx;
    uint8_t* qr = q + row * cols;
    float amax = 0.0f;
    if (kVec) {
        for (int64_t c = static_cast<int64_t>(threadIdx.x) * 8; c < cols; c += kRowThreads * 8) {
            float v[8];
            load8(xr + c, v);
#pragma unroll
            for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fabsf(v[i]));
        }
    } else {
        for (int64_t c = threadIdx.x; c < cols; c += kRowThreads) amax = fmaxf(amax, fabsf(load1(xr + c)));
    }
    amax = block_max(amax, red);
    const float s = (amax == 0.0f) ? 1.0f : __fdiv_rn(amax, 448.0f);
    const float rinv = __frcp_rn(s);
    if (threadIdx.x == 0) scale[row] = s;
    if (kVec) {
        for (int64_t c = static_cast<int64_t>(threadIdx.x) * 8; c < cols; c += kRowThreads * 8) {
            float v[8];
            load8(xr + c, v);
            *reinterpret_cast<uint2*>(qr + c) = quant8(v, s, rinv);
        }
    } else {
        for (int64_t c = threadIdx.x; c < cols; c += kRowThreads)
            qr[c] = static_cast<uint8_t>(e4m3x2(div_rn_by(load1(xr + c), s, rinv), 0.0f) & 0xFFu);
    }
}

// Per-token FP8 quantisation written in padded sorted order: one warp per
// padded position (8 per CTA, grid-stride), so no block barrier sits between
// a row's loads and its stores.  Rows of up to kWarpVec * 8 * 32 values are
// read once into registers with all loads in flight; longer rows are read in
// batches of kWarpVec loads per lane, twice (amax, then codes; the second
// pass mostly hits L1/L2).  The amax is a warp shuffle reduction.  The token
// row is quantised again for each of its slots (the second read hits L2).
constexpr int kWarpVec = 4;
__global__ void __launch_bounds__(kRowThreads)
    quant_rows_fp8_sorted_kernel(const uint16_t* __restrict__ x, int64_t cols, int64_t ldx,
                                 const int32_t* __restrict__ sorted_ids, const int32_t* __restrict__ npp,
                                 int64_t T, int top_k, uint8_t* __restrict__ q, float* __restrict__ scale) {
    pdl_launch_dependents();
    pdl_wait();  // inputs from, and buffers shared with, the previous kernel
    const int lane = threadIdx.x & 31;
    const int64_t warps = static_cast<int64_t>(gridDim.x) * (kRowThreads / 32);
    const int64_t n = *npp;
    const bool in_regs = cols <= static_cast<int64_t>(kWarpVec) * 8 * 32;
    for (int64_t p = static_cast<int64_t>(blockIdx.x) * (kRowThreads / 32) + (threadIdx.x >> 5); p < n;
         p += warps) {
        const int s = sorted_ids[p];
        uint8_t* qr = q + p * cols;
        if (s < 0 || s >= T) {  // pad position
            for (int64_t c = static_cast<int64_t>(lane) * 16; c < cols; c += 32 * 16)
                *reinterpret_cast<uint4*>(qr + c) = make_uint4(0u, 0u, 0u, 0u);
            if (lane == 0) scale[p] = 0.0f;
            continue;
        }
        const uint16_t* xr = x + static_cast<int64_t>(s / top_k) * ldx;
        float amax = 0.0f;
        uint4 xv[kWarpVec];
        if (in_regs) {
#pragma unroll
            for (int j = 0; j < kWarpVec; ++j) {
                const int64_t c = (static_cast<int64_t>(j) * 32 + lane) * 8;
                xv[j] = (c < cols) ? *reinterpret_cast<const uint4*>(xr + c) : make_uint4(0u, 0u, 0u, 0u);
            }
#pragma unroll
            for (int j = 0; j < kWarpVec; ++j) {
                float v[8];
                unpack8(xv[j], v);
#pragma unroll
                for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fabsf(v[i]));
            }
        } else {
            for (int64_t c0 = 0; c0 < cols; c0 += static_cast<int64_t>(kWarpVec) * 32 * 8) {
#pragma unroll
                for (int j = 0; j < kWarpVec; ++j) {
                    const int64_t c = c0 + (static_cast<int64_t>(j) * 32 + lane) * 8;
                    xv[j] = (c < cols) ? *reinterpret_cast<const uint4*>(xr + c) : make_uint4(0u, 0u, 0u, 0u);
                }
#pragma unroll
                for (int j = 0; j < kWarpVec; ++j) {
                    float v[8];
                    unpack8(xv[j], v);
#pragma unroll
                    for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fabsf(v[i]));
                }
            }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, o));
        const float sc = (amax == 0.0f) ? 1.0f : __fdiv_rn(amax, 448.0f);
        const float rinv = __frcp_rn(sc);
        if (lane == 0) scale[p] = sc;
        if (in_regs) {
#pragma unroll
            for (int j = 0; j < kWarpVec; ++j) {
                const int64_t c = (static_cast<int64_t>(j) * 32 + lane) * 8;
                if (c >= cols) break;
                float v[8];
                unpack8(xv[j], v);
                *reinterpret_cast<uint2*>(qr + c) = quant8(v, sc, rinv);
            }
        } else {
            for (int64_t c0 = 0; c0 < cols; c0 += static_cast<int64_t>(kWarpVec) * 32 * 8) {
#pragma unroll
                for (int j = 0; j < kWarpVec; ++j) {
                    const int64_t c = c0 + (static_cast<int64_t>(j) * 32 + lane) * 8;
                    xv[j] = (c < cols) ? *reinterpret_cast<const uint4*>(xr + c) : make_uint4(0u, 0u, 0u, 0u);
                }
#pragma unroll
                for (int j = 0; j < kWarpVec; ++j) {
                    const int64_t c = c0 + (static_cast<int64_t>(j) * 32 + lane) * 8;
                    if (c >= cols) break;
                    float v[8];
                    unpack8(xv[j], v);
                    *reinterpret_cast<uint2*>(qr + c) = quant8(v, sc, rinv);
                }
            }
        }
    }
}

// The same codes and scales, one warp per TOKEN: the token row is read and
// quantised once and its codes and scale are written to every padded
// position of the token's top_k slots.  Each CTA (16 warps) first inverts
// sorted_ids into a slot -> position table in shared memory (T <=
// kTokMaxSlots, 16-byte loads); pad positions are zero-filled by the same
// grid.  Rows of up to kWarpVec * 8 * 32 values stay in registers; longer
// rows take an amax pass and a code pass over batches of kWarpVec vectors
// (the second read mostly hits L1/L2), which keeps the registers per thread,
// and so the warps in flight per SM, where the per-position kernel has them.
constexpr int kTokThreads = 512;
constexpr int kTokMaxSlots = 8192;
__global__ void __launch_bounds__(kTokThreads)
    quant_tokens_fp8_scatter_kernel(const uint16_t* __restrict__ x, int64_t cols, int64_t ldx,
                                    const int32_t* __restrict__ sorted_ids, const int32_t* __restrict__ npp,
                                    int64_t M, int top_k, uint8_t* __restrict__ q, float* __restrict__ scale) {
    __shared__ int32_t s_pos[kTokMaxSlots];
    pdl_launch_dependents();
    pdl_wait();  // inputs from, and buffers shared with, the previous kernel
    const int64_t T = M * top_k;
    const int64_t n = *npp;
    for (int64_t i = threadIdx.x; i < T; i += kTokThreads) s_pos[i] = -1;
    __syncthreads();
    {
        // sorted_ids (16-byte aligned, as every tensor the library takes) in 16-byte vectors
        const int64_t nv = n / 4;
        const int4* sv = reinterpret_cast<const int4*>(sorted_ids);
        for (int64_t v0 = threadIdx.x; v0 < nv; v0 += kTokThreads * 4) {
            int4 w[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int64_t v = v0 + i * kTokThreads;
                w[i] = v < nv ? sv[v] : make_int4(-1, -1, -1, -1);
            }
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int32_t p = static_cast<int32_t>(4 * (v0 + i * kTokThreads));
                if (w[i].x >= 0 && w[i].x < T) s_pos[w[i].x] = p;
                if (w[i].y >= 0 && w[i].y < T) s_pos[w[i].y] = p + 1;
                if (w[i].z >= 0 && w[i].z < T) s_pos[w[i].z] = p + 2;
                if (w[i].w >= 0 && w[i].w < T) s_pos[w[i].w] = p + 3;
            }
        }
        for (int64_t p = 4 * nv + threadIdx.x; p < n; p += kTokThreads) {
            const int sl = sorted_ids[p];
            if (sl >= 0 && sl < T) s_pos[sl] = static_cast<int32_t>(p);
        }
    }
    __syncthreads();
    const int lane = threadIdx.x & 31;
    const int64_t gw = static_cast<int64_t>(blockIdx.x) * (kTokThreads / 32) + (threadIdx.x >> 5);
    const int64_t nw = static_cast<int64_t>(gridDim.x) * (kTokThreads / 32);
    for (int64_t p0 = gw * 32; p0 < n; p0 += nw * 32) {  // pad positions, 32 checked per warp step
        const int64_t p = p0 + lane;
        const int sl = p < n ? sorted_ids[p] : 0;
        unsigned pads = __ballot_sync(0xFFFFFFFFu, p < n && (sl < 0 || sl >= T));
        while (pads) {
            const int64_t pp = p0 + __ffs(pads) - 1;
            pads &= pads - 1;
            uint8_t* qr = q + pp * cols;
            for (int64_t c = static_cast<int64_t>(lane) * 16; c < cols; c += 32 * 16)
                *reinterpret_cast<uint4*>(qr + c) = make_uint4(0u, 0u, 0u, 0u);
            if (lane == 0) scale[pp] = 0.0f;
        }
    }
    const bool in_regs = cols <= static_cast<int64_t>(kWarpVec) * 8 * 32;
    constexpr int64_t kBatch = static_cast<int64_t>(kWarpVec) * 32 * 8;  // values per batch of loads
    for (int64_t m = gw; m < M; m += nw) {
        const uint16_t* xr = x + m * ldx;
        const int32_t* tpos = s_pos + m * top_k;
        uint4 xv[kWarpVec];
        auto load_batch = [&](int64_t c0) {
#pragma unroll
            for (int j = 0; j < kWarpVec; ++j) {
                const int64_t c = c0 + (static_cast<int64_t>(j) * 32 + lane) * 8;
                xv[j] = (c < cols) ? *reinterpret_cast<const uint4*>(xr + c) : make_uint4(0u, 0u, 0u, 0u);
            }
        };
        float amax = 0.0f;
        for (int64_t c0 = 0; c0 < cols; c0 += kBatch) {
            load_batch(c0);
#pragma unroll
            for (int j = 0; j < kWarpVec; ++j) {
                float v[8];
                unpack8(xv[j], v);
#pragma unroll
                for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fabsf(v[i]));
            }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, o));
        const float sc = (amax == 0.0f) ? 1.0f : __fdiv_rn(amax, 448.0f);
        const float rinv = __frcp_rn(sc);
        if (lane < top_k && tpos[lane] >= 0) scale[tpos[lane]] = sc;
        for (int64_t c0 = 0; c0 < cols; c0 += kBatch) {
            if (!in_regs) load_batch(c0);
#pragma unroll
            for (int j = 0; j < kWarpVec; ++j) {
                const int64_t c = c0 + (static_cast<int64_t>(j) * 32 + lane) * 8;
                if (c >= cols) break;
                float v[8];
                unpack8(xv[j], v);
                const uint2 code = quant8(v, sc, rinv);
                for (int t = 0; t < top_k; ++t) {
                    const int32_t pt = tpos[t];
                    if (pt >= 0) *reinterpret_cast<uint2*>(q + static_cast<int64_t>(pt) * cols + c) = code;
                }
            }
        }
    }
}

// The same quantisation with every token row brought into shared memory by a
// bulk asynchronous copy (cp.async.bulk, completing on an mbarrier): a
// 128-thread CTA walks its padded positions (grid-stride) with nbuf rows in
// flight, so the bytes in flight per SM are bounded by shared memory rather
// than registers.  Pad positions arrive on their buffer's barrier without
// bytes, so every buffer's phases stay in step.  Codes and scales as above.
constexpr int kBulkRowThreads = 128;
constexpr int kBulkMaxBuf = 8;
constexpr int64_t kBulkRowsBytes = 32768;  // shared memory for the rows in flight, per CTA
__global__ void __launch_bounds__(kBulkRowThreads)
    quant_rows_fp8_sorted_bulk_kernel(const uint16_t* __restrict__ x, int64_t cols, int64_t ldx,
                                      const int32_t* __restrict__ sorted_ids, const int32_t* __restrict__ npp,
                                      int64_t T, int top_k, int nbuf, uint8_t* __restrict__ q,
                                      float* __restrict__ scale) {
    extern __shared__ __align__(128) uint8_t s_rows[];
    __shared__ uint64_t bars[kBulkMaxBuf];
    __shared__ float s_red[2][kBulkRowThreads / 32];
    __shared__ int s_abort;
    const int tid = threadIdx.x;
    const int lane = tid & 31;
    if (tid == 0) {
        for (int b = 0; b < nbuf; ++b) mbar_init(&bars[b], 1);
        s_abort = 0;
        fence_mbar_init();
    }
    __syncthreads();
    pdl_launch_dependents();
    pdl_wait();  // inputs from, and buffers shared with, the previous kernel
    const int64_t n = *npp;
    const uint32_t row_bytes = static_cast<uint32_t>(cols * 2);
    const int64_t chunks = cols / 8;
    // k-th position of this CTA: p = blockIdx.x + k * gridDim.x, in buffer k % nbuf
    auto issue = [&](int64_t k) {
        const int64_t p = blockIdx.x + k * static_cast<int64_t>(gridDim.x);
        if (p >= n) return;
        uint64_t* bar = &bars[k % nbuf];
        const int s = sorted_ids[p];
        if (s >= 0 && s < T) {
            mbar_arrive_expect_tx(bar, row_bytes);
            bulk_load(s_rows + (k % nbuf) * static_cast<int64_t>(row_bytes),
                      x + static_cast<int64_t>(s / top_k) * ldx, row_bytes, bar);
        } else {
            mbar_arrive(bar);
        }
    };
    if (tid == 0)
        for (int k = 0; k < nbuf; ++k) issue(k);
    int red = 0;
    for (int64_t k = 0;; ++k) {
        const int64_t p = blockIdx.x + k * static_cast<int64_t>(gridDim.x);
        if (p >= n) break;
        const int s = sorted_ids[p];
        uint8_t* qr = q + p * cols;
        if (s < 0 || s >= T) {  // pad position (uniform over the CTA)
            for (int64_t c = static_cast<int64_t>(tid) * 16; c < cols; c += kBulkRowThreads * 16)
                *reinterpret_cast<uint4*>(qr + c) = make_uint4(0u, 0u, 0u, 0u);
            if (tid == 0) scale[p] = 0.0f;
        } else {
            const bool landed = mbar_wait(&bars[k % nbuf], static_cast<uint32_t>(k / nbuf) & 1u, &s_abort, nullptr);
            if (!__syncthreads_and(landed)) break;  // (only after a copy that never completed)
            const uint4* xr = reinterpret_cast<const uint4*>(s_rows + (k % nbuf) * static_cast<int64_t>(row_bytes));
            float amax = 0.0f;
            for (int64_t c = tid; c < chunks; c += kBulkRowThreads) {
                float v[8];
                unpack8(xr[c], v);
#pragma unroll
                for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fabsf(v[i]));
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, o));
            if (lane == 0) s_red[red][tid >> 5] = amax;
            __syncthreads();
#pragma unroll
            for (int w = 0; w < kBulkRowThreads / 32; ++w) amax = fmaxf(amax, s_red[red][w]);
            red ^= 1;
            const float sc = (amax == 0.0f) ? 1.0f : __fdiv_rn(amax, 448.0f);
            const float rinv = __frcp_rn(sc);
            if (tid == 0) scale[p] = sc;
            for (int64_t c = tid; c < chunks; c += kBulkRowThreads) {
                float v[8];
                unpack8(xr[c], v);
                *reinterpret_cast<uint2*>(qr + c * 8) = quant8(v, sc, rinv);
            }
        }
        __syncthreads();  // every thread is done with this buffer before it is refilled
        if (tid == 0) issue(k + nbuf);
    }
}

// ======================================================================
// Router: softmax -> top-k -> renormalise.  The top-k of the softmax are the
// top-k logits and the renormalised weights are the softmax over the selected
// logits, so per token: the k largest logits, descending, ties to the lower
// id (one pass over the E logits, an insertion into a k-long register list
// ordered by (value desc, id asc)); p_j = exp_seq(l_j - l_1); S = sum of p_j
// in order; w_j = p_j / S.
// ======================================================================
constexpr int kRouterMaxE = 256;
constexpr int kRouterMaxK = 8;

QMOE_DI void route_token(const float* __restrict__ l, int E, int k, int* ids, float* w) {
    float tv[kRouterMaxK];
    int ti[kRouterMaxK];
#pragma unroll
    for (int j = 0; j < kRouterMaxK; ++j) {
        tv[j] = 0.0f;
        ti[j] = -1;
    }
    for (int e = 0; e < E; ++e) {
        float v = l[e];
        int id = e;
#pragma unroll
        for (int j = 0; j < kRouterMaxK; ++j) {
            if (j < k && (ti[j] < 0 || v > tv[j] || (v == tv[j] && id < ti[j]))) {
                const float t = tv[j];
                const int u = ti[j];
                tv[j] = v;
                ti[j] = id;
                v = t;
                id = u;
                if (id < 0) break;
            }
        }
    }
    float p[kRouterMaxK];
    float S = 0.0f;
#pragma unroll
    for (int j = 0; j < kRouterMaxK; ++j) {
        if (j < k) {
            p[j] = exp_seq(__fsub_rn(tv[j], tv[0]));
            S = __fadd_rn(S, p[j]);
        }
    }
#pragma unroll
    for (int j = 0; j < kRouterMaxK; ++j) {
        if (j < k) {
            ids[j] = ti[j];
            w[j] = __fdiv_rn(p[j], S);
        }
    }
}

__global__ void router_topk_kernel(const float* __restrict__ logits, int64_t M, int E, int k,
                                   int32_t* __restrict__ topk_ids, float* __restrict__ topk_w) {
    for (int64_t m = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; m < M;
         m += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        int ids[kRouterMaxK];
        float w[kRouterMaxK];
        route_token(logits + m * E, E, k, ids, w);
#pragma unroll
        for (int j = 0; j < kRouterMaxK; ++j) {
            if (j >= k) break;
            topk_ids[m * k + j] = ids[j];
            topk_w[m * k + j] = w[j];
        }
    }
}

// ======================================================================
// Fused align + sorted per-token quantisation for small slot counts (one
// launch).  CTAs 0..M-1: one token each -- histogram of all ids in shared
// memory, padded offsets, the padded position of each of the token's slots
// (its rank among the earlier slots of the same expert), one quantisation of
// the token row written to every such position, and sorted_ids at those
// positions.  CTA M: expert/padded offsets, num_post_padded, the block ->
// expert map and the sentinel at every pad position.  Pad rows of q are left
// unwritten (the grouped GEMM never stores their results).
// ======================================================================
constexpr int kFusedMaxT = 4096;
constexpr int kRouteFusedMaxM = 64;  // largest M routed inside the align + quantisation launch

// kRoute: the ids come from routing fp32 logits [M, E] in the same launch --
// every CTA routes all tokens (its histogram needs them) and CTA m writes
// token m's ids and weights.
template <bool kRoute>
__global__ void __launch_bounds__(kRowThreads)
    align_quant_fused_kernel(const uint16_t* __restrict__ x, int64_t M, int64_t cols, int64_t ldx,
                             const int32_t* __restrict__ ids, const float* __restrict__ logits,
                             int32_t* __restrict__ ids_out, float* __restrict__ w_out, int top_k, int E, int BM,
                             int32_t* __restrict__ sorted_ids, int64_t cap, int32_t* __restrict__ expert_ids,
                             int32_t* __restrict__ num_post_padded, int32_t* __restrict__ expert_offsets,
                             int32_t* __restrict__ padded_offsets, uint8_t* __restrict__ q,
                             float* __restrict__ scale, int32_t* d_status) {
    pdl_launch_dependents();
    pdl_wait();  // inputs from, and buffers shared with, the previous kernel
    __shared__ int s_ids[kFusedMaxT];
    __shared__ int s_cnt[kAlignMaxE];
    __shared__ int s_poff[kAlignMaxE + 1];
    __shared__ int s_rank[8];
    __shared__ int s_redc[kRowThreads / 32][8];
    __shared__ float s_reda[kRowThreads / 32];
    __shared__ float s_sc;
    const int T = static_cast<int>(M) * top_k;
    const int tid = threadIdx.x;
    // Token CTAs load their row first (rows of up to kRegVec * 8 * kRowThreads
    // values stay in registers), so the load latency overlaps the histogram
    // and the ranking instead of following them.
    constexpr int kRegVec = 4;
    const bool in_regs = cols <= static_cast<int64_t>(kRegVec) * 8 * kRowThreads;
    uint4 xv[kRegVec];
    if (blockIdx.x < M && in_regs) {
        const uint16_t* xr0 = x + static_cast<int64_t>(blockIdx.x) * ldx;
#pragma unroll
        for (int j = 0; j < kRegVec; ++j) {
            const int64_t c = (static_cast<int64_t>(j) * kRowThreads + tid) * 8;
            xv[j] = (c < cols) ? *reinterpret_cast<const uint4*>(xr0 + c) : make_uint4(0u, 0u, 0u, 0u);
        }
    }
    for (int e = tid; e < E; e += blockDim.x) s_cnt[e] = 0;
    __syncthreads();
    if constexpr (kRoute) {
        for (int m = tid; m < static_cast<int>(M); m += blockDim.x) {
            int rid[kRouterMaxK];
            float rw[kRouterMaxK];
            route_token(logits + static_cast<int64_t>(m) * E, E, top_k, rid, rw);
#pragma unroll
            for (int j = 0; j < kRouterMaxK; ++j) {
                if (j >= top_k) break;
                s_ids[m * top_k + j] = rid[j];
                atomicAdd(&s_cnt[rid[j]], 1);
                if (m == static_cast<int>(blockIdx.x)) {
                    ids_out[m * top_k + j] = rid[j];
                    w_out[m * top_k + j] = rw[j];
                }
            }
        }
    } else {
        for (int i = tid; i < T; i += blockDim.x) {
            const int e = ids[i];
            s_ids[i] = e;
            if (e >= 0 && e < E) atomicAdd(&s_cnt[e], 1);
        }
    }
    __syncthreads();
    if (tid == 0) {
        int poff = 0;
        for (int e = 0; e < E; ++e) {
            s_poff[e] = poff;
            poff += (s_cnt[e] + BM - 1) / BM * BM;
        }
        s_poff[E] = poff;
    }
    __syncthreads();
    const int64_t b = blockIdx.x;
    if (b == M) {
        // offsets, block map and pad sentinels
        if (tid == 0) {
            int off = 0;
            bool bad = false;
            for (int e = 0; e < E; ++e) {
                expert_offsets[e] = off;
                padded_offsets[e] = s_poff[e];
                off += s_cnt[e];
            }
            expert_offsets[E] = off;
            padded_offsets[E] = s_poff[E];
            *num_post_padded = s_poff[E];
            bad = off != T;
            if (bad && d_status) atomicOr(reinterpret_cast<int*>(d_status), QMOE_DEV_INVALID_EXPERT);
        }
        for (int64_t blk = tid; blk < cap / BM; blk += blockDim.x) {
            const int64_t p = blk * BM;
            int owner = -1;
            if (p < s_poff[E]) {
                int lo = 0, hi = E - 1;
                while (lo < hi) {
                    const int mid = (lo + hi + 1) >> 1;
                    if (s_poff[mid] <= p) lo = mid;
                    else hi = mid - 1;
                }
                owner = lo;
            }
            expert_ids[blk] = owner;
        }
        for (int64_t p = tid; p < cap; p += blockDim.x) {
            bool pad = p >= s_poff[E];
            if (!pad) {
                int lo = 0, hi = E - 1;
                while (lo < hi) {
                    const int mid = (lo + hi + 1) >> 1;
                    if (s_poff[mid] <= p) lo = mid;
                    else hi = mid - 1;
                }
                pad = p - s_poff[lo] >= s_cnt[lo];
            }
            if (pad) sorted_ids[p] = T;
        }
        return;
    }
    // token b: the rank of each of its top_k slots among the earlier slots of
    // the same expert, and the row amax, in one block reduction
    const int s0 = static_cast<int>(b) * top_k;
    int es[8], cnt[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        es[j] = (j < top_k) ? s_ids[s0 + j] : -1;
        cnt[j] = 0;
    }
    for (int i = tid; i < s0 + top_k; i += blockDim.x) {
        const int ei = s_ids[i];
#pragma unroll
        for (int j = 0; j < 8; ++j) cnt[j] += (j < top_k && i < s0 + j && ei == es[j]) ? 1 : 0;
    }
    const uint16_t* xr = x + b * ldx;
    float amax = 0.0f;
    if (in_regs) {
#pragma unroll
        for (int j = 0; j < kRegVec; ++j) {
            float v[8];
            unpack8(xv[j], v);
#pragma unroll
            for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fabsf(v[i]));
        }
    } else {
        for (int64_t c = static_cast<int64_t>(tid) * 8; c < cols; c += kRowThreads * 8) {
            float v[8];
            load8(xr + c, v);
#pragma unroll
            for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fabsf(v[i]));
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, o));
#pragma unroll
        for (int j = 0; j < 8; ++j) cnt[j] += __shfl_xor_sync(0xFFFFFFFFu, cnt[j], o);
    }
    const int warp = tid >> 5;
    if ((tid & 31) == 0) {
        s_reda[warp] = amax;
#pragma unroll
        for (int j = 0; j < 8; ++j) s_redc[warp][j] = cnt[j];
    }
    __syncthreads();
    if (tid < top_k) {
        int tot = 0;
        for (int w = 0; w < kRowThreads / 32; ++w) tot += s_redc[w][tid];
        const int e = s_ids[s0 + tid];
        const bool ok = e >= 0 && e < E;
        s_rank[tid] = ok ? s_poff[e] + tot : -1;
        if (ok) sorted_ids[s_poff[e] + tot] = s0 + tid;
    } else if (tid == 32) {
        float a = 0.0f;
        for (int w = 0; w < kRowThreads / 32; ++w) a = fmaxf(a, s_reda[w]);
        s_sc = (a == 0.0f) ? 1.0f : __fdiv_rn(a, 448.0f);
    }
    __syncthreads();
    const float sc = s_sc;
    const float rinv = __frcp_rn(sc);
    if (tid < top_k && s_rank[tid] >= 0) scale[s_rank[tid]] = sc;
    int rk[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) rk[j] = (j < top_k) ? s_rank[j] : -1;
    if (in_regs) {
#pragma unroll
        for (int j = 0; j < kRegVec; ++j) {
            const int64_t c = (static_cast<int64_t>(j) * kRowThreads + tid) * 8;
            if (c >= cols) break;
            float v[8];
            unpack8(xv[j], v);
            const uint2 o = quant8(v, sc, rinv);
#pragma unroll
            for (int t = 0; t < 8; ++t)
                if (rk[t] >= 0) *reinterpret_cast<uint2*>(q + static_cast<int64_t>(rk[t]) * cols + c) = o;
        }
    } else {
        for (int64_t c = static_cast<int64_t>(tid) * 8; c < cols; c += kRowThreads * 8) {
            float v[8];
            load8(xr + c, v);
            const uint2 o = quant8(v, sc, rinv);
#pragma unroll
            for (int t = 0; t < 8; ++t)
                if (rk[t] >= 0) *reinterpret_cast<uint2*>(q + static_cast<int64_t>(rk[t]) * cols + c) = o;
        }
    }
}

// bf16 token rows copied into padded sorted order (one CTA per padded
// position; pad rows zeroed, rows at or past num_post_padded untouched).
__global__ void __launch_bounds__(kRowThreads)
    gather_sorted_bf16_kernel(const uint16_t* __restrict__ x, int64_t cols, int64_t ldx,
                              const int32_t* __restrict__ sorted_ids, const int32_t* __restrict__ npp, int64_t T,
                              int top_k, uint16_t* __restrict__ out) {
    const int64_t p = blockIdx.x;
    if (p >= *npp) return;
    const int s = sorted_ids[p];
    uint4* dst = reinterpret_cast<uint4*>(out + p * cols);
    if (s < 0 || s >= T) {
        for (int64_t c = threadIdx.x; c < cols / 8; c += kRowThreads) dst[c] = make_uint4(0u, 0u, 0u, 0u);
        return;
    }
    const uint4* src = reinterpret_cast<const uint4*>(x + static_cast<int64_t>(s / top_k) * ldx);
    for (int64_t c = threadIdx.x; c < cols / 8; c += kRowThreads) dst[c] = src[c];
}

__global__ void __launch_bounds__(kRowThreads)
    quant_rows_int8_kernel(const float* __restrict__ x, int64_t cols, int8_t* __restrict__ q,
                           float* __restrict__ scale) {
    __shared__ float red[33];
    const int64_t row = blockIdx.x;
    const float* xr = x + row * cols;
    int8_t* qr = q + row * cols;
    float amax = 0.0f;
    for (int64_t c = threadIdx.x; c < cols; c += kRowThreads) amax = fmaxf(amax, fabsf(xr[c]));
    amax = block_max(amax, red);
    const float s = (amax == 0.0f) ? 1.0f : __fdiv_rn(amax, 127.0f);
    const float rinv = __frcp_rn(s);
    if (threadIdx.x == 0) scale[row] = s;
    for (int64_t c = threadIdx.x; c < cols; c += kRowThreads) {
        const float v = fminf(fmaxf(rintf(div_rn_by(xr[c], s, rinv)), -127.0f), 127.0f);
        qr[c] = static_cast<int8_t>(static_cast<int>(v));
    }
}

// ======================================================================
// SwiGLU + requantisation.
// Per-token: one CTA per row; h is kept in dynamic shared memory (I floats)
// between the amax pass and the quantisation pass.
// MX: one CTA per row, one thread per 1x32 block (h in registers); the CTA
// also zeroes its row's pad columns and a share of its expert's pad rows.
// ======================================================================
// h for 8 elements from raw gate / up words (already loaded).
QMOE_DI void silu8w(const uint4 gw, const uint4 uw, float (&h)[8]) {
    float gv[8], uv[8];
    unpack8(gw, gv);
    unpack8(uw, uv);
#pragma unroll
    for (int i = 0; i < 8; i += 2) silu_mul2(gv[i], gv[i + 1], uv[i], uv[i + 1], h[i], h[i + 1]);
}
constexpr int kSiluBatch = 4;  // 8-element chunks whose loads are issued before any arithmetic

// Activations of the requantisation kernels.  Gated: h = silu(gate) * up from
// a fused gate|up row; not gated: h = relu(x)^2 (SReLU; the fp32 square of a
// bf16 value is exact).
struct ActSwiGLU {
    static constexpr bool kGated = true;
    QMOE_DI static void apply8(const uint4 gw, const uint4 uw, float (&h)[8]) { silu8w(gw, uw, h); }
};
struct ActSReLU {
    static constexpr bool kGated = false;
    QMOE_DI static void apply8(const uint4 xw, const uint4, float (&h)[8]) {
        float v[8];
        unpack8(xw, v);
#pragma unroll
        for (int i = 0; i < 8; ++i) h[i] = (v[i] > 0.0f) ? __fmul_rn(v[i], v[i]) : 0.0f;
    }
};

// No activation: plain MXFP8 / per-token quantisation of bf16 rows.
struct ActIdentity {
    static constexpr bool kGated = false;
    QMOE_DI static void apply8(const uint4 xw, const uint4, float (&h)[8]) { unpack8(xw, h); }
};

// kT threads per row.  Long SwiGLU rows (ALU-bound) run 512: with the row's
// fp32 h in shared memory that keeps 32 warps resident per SM instead of 24;
// short rows keep 256 so that no thread idles.
template <class Act, int kT>
__global__ void __launch_bounds__(kT)
    act_quant_token_kernel(const uint16_t* __restrict__ y, int64_t I, int64_t ldy, uint8_t* __restrict__ q,
                           float* __restrict__ scale) {
    extern __shared__ float s_h[];
    __shared__ float red[33];
    const int64_t row = blockIdx.x;
    const uint16_t* yr = y + row * ldy;
    float amax = 0.0f;
    for (int64_t c0 = static_cast<int64_t>(threadIdx.x) * 8; c0 < I; c0 += kT * 8 * kSiluBatch) {
        uint4 gw[kSiluBatch], uw[kSiluBatch];
#pragma unroll
        for (int j = 0; j < kSiluBatch; ++j) {
            const int64_t c = c0 + static_cast<int64_t>(j) * kT * 8;
            if (c < I) {
                gw[j] = *reinterpret_cast<const uint4*>(yr + c);
                uw[j] = Act::kGated ? *reinterpret_cast<const uint4*>(yr + I + c) : make_uint4(0u, 0u, 0u, 0u);
            }
        }
#pragma unroll
        for (int j = 0; j < kSiluBatch; ++j) {
            const int64_t c = c0 + static_cast<int64_t>(j) * kT * 8;
            if (c < I) {
                float h[8];
                Act::apply8(gw[j], uw[j], h);
                *reinterpret_cast<float4*>(s_h + c) = make_float4(h[0], h[1], h[2], h[3]);
                *reinterpret_cast<float4*>(s_h + c + 4) = make_float4(h[4], h[5], h[6], h[7]);
#pragma unroll
                for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fabsf(h[i]));
            }
        }
    }
    amax = block_max(amax, red);  // (contains __syncthreads: s_h is complete)
    const float s = (amax == 0.0f) ? 1.0f : __fdiv_rn(amax, 448.0f);
    const float rinv = __frcp_rn(s);
    if (threadIdx.x == 0) scale[row] = s;
    uint8_t* qr = q + row * I;
    for (int64_t c = static_cast<int64_t>(threadIdx.x) * 8; c < I; c += kT * 8) {
        const float4 a = *reinterpret_cast<const float4*>(s_h + c);
        const float4 b = *reinterpret_cast<const float4*>(s_h + c + 4);
        const float h[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
        *reinterpret_cast<uint2*>(qr + c) = quant8(h, s, rinv);
    }
}

// Second pass of the per-token SwiGLU quantisation when h comes from the up
// GEMM's epilogue (qmoe_moe_gemm_w8a8_silu_fp8_token): rows of fp32 h whose
// amax |h| the epilogue has already reduced, scale = amax/448 (1 for an
// all-zero row), q = e4m3(h / scale) -- the same operations as the quantisation
// pass of act_quant_token_kernel.  One thread per 8 elements, flat grid.
__global__ void __launch_bounds__(256)
    quant_h_token_kernel(const float* __restrict__ h, const float* __restrict__ amax, int64_t rows, int64_t I,
                         uint8_t* __restrict__ q, float* __restrict__ scale) {
    pdl_launch_dependents();
    pdl_wait();
    const int64_t per_row = I / 8;
    for (int64_t g = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; g < rows * per_row;
         g += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int64_t r = g / per_row;
        const int64_t c = (g - r * per_row) * 8;
        const float a = amax[r];
        const float s = (a == 0.0f) ? 1.0f : __fdiv_rn(a, 448.0f);
        const float rinv = __frcp_rn(s);
        const float4 x0 = __ldcs(reinterpret_cast<const float4*>(h + r * I + c));
        const float4 x1 = __ldcs(reinterpret_cast<const float4*>(h + r * I + c + 4));
        const float v[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
        *reinterpret_cast<uint2*>(q + r * I + c) = quant8(v, s, rinv);
        if (c == 0) scale[r] = s;
    }
}

qmoe_status_t launch_quant_h_token(const float* h, const float* amax, int64_t rows, int64_t I, uint8_t* q,
                                   float* scale, cudaStream_t st) {
    if (rows <= 0) return QMOE_OK;
    const int64_t n = rows * (I / 8);
    const int sms = device_sm_count();
    int64_t blocks = (n + 255) / 256;
    const int64_t cap = static_cast<int64_t>(sms > 0 ? sms : 132) * 16;
    if (blocks > cap) blocks = cap;
    return launch_pdl(quant_h_token_kernel, dim3(static_cast<unsigned>(blocks)), dim3(256), 0, st, h, amax, rows, I,
                      q, scale);
}

constexpr int kMxThreads = 256;

// One thread per (row, 1x32 block) item over a flat grid, so short rows keep
// every thread busy.  The thread with b == 0 of a row also zeroes the row's pad
// columns and its share of the expert's pad rows.
template <class Act>
__global__ void __launch_bounds__(kMxThreads)
    act_quant_mx_kernel(const uint16_t* __restrict__ y, int64_t rows, int64_t I, int64_t ldy,
                        uint8_t* __restrict__ q, uint8_t* __restrict__ sf, int64_t sf_ld,
                        const int32_t* __restrict__ eoff, const int32_t* __restrict__ soff, int E,
                        int32_t* d_status) {
    const int64_t nblk = I / 32;
    const int64_t g = blockIdx.x * static_cast<int64_t>(kMxThreads) + threadIdx.x;
    if (g >= rows * nblk) return;
    const int64_t r = g / nblk;
    const int64_t b = g - r * nblk;
    if (r >= eoff[E]) return;  // row past the last expert's rows
    int lo = 0, hi = E - 1;    // last e with eoff[e] <= r
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (eoff[mid] <= r) lo = mid;
        else hi = mid - 1;
    }
    const int e = lo;
    const int64_t local = r - eoff[e];
    const int64_t cnt = eoff[e + 1] - eoff[e];
    const int64_t srow = soff[e] + local;
    const uint16_t* yr = y + r * ldy;
    uint8_t* qr = q + r * I;
    uint8_t* sfr = sf + srow * sf_ld;
    float h[32];
    uint4 gw[4], uw[4];
#pragma unroll
    for (int c = 0; c < 4; ++c) {
        gw[c] = *reinterpret_cast<const uint4*>(yr + b * 32 + c * 8);
        uw[c] = Act::kGated ? *reinterpret_cast<const uint4*>(yr + I + b * 32 + c * 8) : make_uint4(0u, 0u, 0u, 0u);
    }
#pragma unroll
    for (int c = 0; c < 4; ++c) {
        float t[8];
        Act::apply8(gw[c], uw[c], t);
#pragma unroll
        for (int i = 0; i < 8; ++i) h[c * 8 + i] = t[i];
    }
    float a = 0.0f;
#pragma unroll
    for (int i = 0; i < 32; ++i) a = fmaxf(a, fabsf(h[i]));
    const int ex = mx_block_exponent(a);
    const float mul = pow2_neg(ex);
    sfr[b] = static_cast<uint8_t>(ex + 127);
    uint32_t o[8];
#pragma unroll
    for (int i = 0; i < 8; ++i)
        o[i] = e4m3x4(__fmul_rn(h[4 * i], mul), __fmul_rn(h[4 * i + 1], mul), __fmul_rn(h[4 * i + 2], mul),
                      __fmul_rn(h[4 * i + 3], mul));
    *reinterpret_cast<uint4*>(qr + b * 32) = make_uint4(o[0], o[1], o[2], o[3]);
    *reinterpret_cast<uint4*>(qr + b * 32 + 16) = make_uint4(o[4], o[5], o[6], o[7]);
    if (b == 0) {
        for (int64_t c = nblk; c < sf_ld; ++c) sfr[c] = 0;  // pad columns
        // pad rows of expert e (soff[e]+cnt .. soff[e+1]-1), shared out over the expert's rows
        for (int64_t pr = soff[e] + cnt + local; pr < soff[e + 1]; pr += cnt) {
            uint8_t* pp = sf + pr * sf_ld;
            for (int64_t c = 0; c < sf_ld; ++c) pp[c] = 0;
        }
    }
    (void)d_status;
}

// ======================================================================
// element hooks for the exhaustive tests
// ======================================================================
__global__ void debug_e4m3_kernel(const float* __restrict__ x, uint8_t* __restrict__ q, int64_t n) {
    for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < n;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x)
        q[i] = static_cast<uint8_t>(e4m3x2(x[i], 0.0f) & 0xFFu);
}
__global__ void debug_i8_kernel(const uint32_t* __restrict__ x, uint2* __restrict__ y, int64_t nw) {
    for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < nw;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        uint32_t lo, hi;
        int8x4_to_bf16x4(x[i], lo, hi);
        y[i] = make_uint2(lo, hi);
    }
}
// Pairs go through the packed sequence the kernels use, an odd last element
// through the scalar one.
__global__ void debug_silu_kernel(const float* __restrict__ g, const float* __restrict__ u, float* __restrict__ h,
                                  int64_t n) {
    for (int64_t i = 2 * (blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x); i < n;
         i += 2 * static_cast<int64_t>(gridDim.x) * blockDim.x) {
        if (i + 1 < n) silu_mul2(g[i], g[i + 1], u[i], u[i + 1], h[i], h[i + 1]);
        else h[i] = silu_mul(g[i], u[i]);
    }
}
__global__ void debug_rcp_kernel(const float* __restrict__ d, float* __restrict__ y, int64_t n) {
    for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < n;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x)
        y[i] = rcp_rn_ge1(d[i]);
}
__global__ void debug_div_kernel(const float* __restrict__ x, float s, float* __restrict__ q, int64_t n) {
    const float rinv = __frcp_rn(s);
    for (int64_t i = 2 * (blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x); i < n;
         i += 2 * static_cast<int64_t>(gridDim.x) * blockDim.x) {
        if (i + 1 < n) div2_rn_by(x[i], x[i + 1], s, rinv, q[i], q[i + 1]);
        else q[i] = div_rn_by(x[i], s, rinv);
    }
}

// The quantisers' e4m3 codes of x[i] / s (quant8), eight values per thread
// (a short tail padded with zeros, its codes dropped).
__global__ void debug_quant_kernel(const float* __restrict__ x, float s, uint8_t* __restrict__ q, int64_t n) {
    const float rinv = __frcp_rn(s);
    for (int64_t i = 8 * (blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x); i < n;
         i += 8 * static_cast<int64_t>(gridDim.x) * blockDim.x) {
        float v[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) v[k] = i + k < n ? x[i + k] : 0.0f;
        const uint2 c = quant8(v, s, rinv);
#pragma unroll
        for (int k = 0; k < 8; ++k)
            if (i + k < n) q[i + k] = static_cast<uint8_t>(((k < 4 ? c.x : c.y) >> (8 * (k & 3))) & 0xFFu);
    }
}

// One thread waits on an mbarrier that nothing arrives at, through the same
// bounded wait the GEMM uses, with a short limit: it must give up, record
// QMOE_DEV_TIMEOUT and return.
__global__ void debug_wait_timeout_kernel(int32_t* d_status, uint64_t limit_ns) {
    __shared__ uint64_t bar;
    __shared__ int abort_flag;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        abort_flag = 0;
        fence_mbar_init();
        mbar_wait(&bar, 0, &abort_flag, d_status, limit_ns);
    }
}

static int grid_for(int64_t n, int threads) {
    const int64_t b = (n + threads - 1) / threads;
    const int64_t cap = static_cast<int64_t>(device_sm_count() > 0 ? device_sm_count() : 132) * 16;
    return static_cast<int>(b < cap ? (b > 0 ? b : 1) : cap);
}

template <class Act>
static qmoe_status_t run_act_quant(const uint16_t* y, int64_t rows, int64_t I, int64_t ldy, int32_t mode,
                                   uint8_t* q, float* scale, uint8_t* sf, int64_t sf_ld,
                                   const int32_t* expert_offsets, const int32_t* sf_padded_offsets, int32_t E,
                                   int32_t* d_status, qmoe_stream_t stream) {
    const int64_t width = Act::kGated ? 2 * I : I;
    if (rows < 0 || I < 8 || I % 8 != 0 || ldy < width || ldy % 8 != 0) return QMOE_ERR_INVALID_ARG;
    if (rows == 0) return QMOE_OK;
    if (!y || !q || !aligned16(y) || !aligned16(q) || rows > 0x7FFFFFFF) return QMOE_ERR_INVALID_ARG;
    if (mode == QMOE_SCALE_PER_TOKEN) {
        if (!scale) return QMOE_ERR_INVALID_ARG;
        const size_t smem = static_cast<size_t>(I) * sizeof(float);
        if (smem > 200 * 1024) return QMOE_ERR_UNSUPPORTED;
        const bool wide = Act::kGated && I >= 8192;
        if (smem > 48 * 1024) {
            if (cudaFuncSetAttribute(wide ? act_quant_token_kernel<Act, 512> : act_quant_token_kernel<Act, kRowThreads>,
                                     cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem)) != cudaSuccess)
                return QMOE_ERR_CUDA;
        }
        if (wide)
            act_quant_token_kernel<Act, 512><<<static_cast<unsigned>(rows), 512, smem, stream>>>(y, I, ldy, q, scale);
        else
            act_quant_token_kernel<Act, kRowThreads><<<static_cast<unsigned>(rows), kRowThreads, smem, stream>>>(
                y, I, ldy, q, scale);
        return launch_status();
    }
    if (mode == QMOE_SCALE_MX_1X32) {
        if (I % 32 != 0 || !sf || sf_ld < I / 32 || !expert_offsets || !sf_padded_offsets || E < 1 || E > 256)
            return QMOE_ERR_INVALID_ARG;
        const int64_t items = rows * (I / 32);
        const int64_t blocks = (items + kMxThreads - 1) / kMxThreads;
        if (blocks > 0x7FFFFFFF) return QMOE_ERR_UNSUPPORTED;
        act_quant_mx_kernel<Act><<<static_cast<unsigned>(blocks), kMxThreads, 0, stream>>>(
            y, rows, I, ldy, q, sf, sf_ld, expert_offsets, sf_padded_offsets, E, d_status);
        return launch_status();
    }
    return QMOE_ERR_INVALID_ARG;
}

}  // namespace qmoe

using namespace qmoe;

extern "C" {

int64_t qmoe_align_max_padded(int64_t T, int32_t E, int32_t BM) {
    if (T < 0 || E < 1 || BM < 1) return -1;
    const int64_t cap = T + static_cast<int64_t>(E) * (BM - 1);
    return (cap + BM - 1) / BM * BM;
}

qmoe_status_t qmoe_moe_align_block_size(const int32_t* topk_ids, int64_t T, int32_t E, int32_t BM,
                                        int32_t* sorted_ids, int32_t* expert_ids, int32_t* num_post_padded,
                                        int32_t* expert_offsets, int32_t* padded_offsets, int32_t* d_status,
                                        qmoe_stream_t stream) {
    if (T < 0 || E < 1 || E > kAlignMaxE || BM < 1 || BM > 1024) return QMOE_ERR_INVALID_ARG;
    const int64_t cap = qmoe_align_max_padded(T, E, BM);
    if (cap >= (int64_t(1) << 31)) return QMOE_ERR_UNSUPPORTED;
    if ((T > 0 && !topk_ids) || !sorted_ids || !expert_ids || !num_post_padded || !expert_offsets ||
        !padded_offsets)
        return QMOE_ERR_INVALID_ARG;
    if (T >= kAlignClusterMinSlots) {  // a cluster of CTAs: more SMs on the per-slot work
        cudaLaunchConfig_t cfg = {};
        cudaLaunchAttribute attr[2];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = kAlignCtas;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[1].val.programmaticStreamSerializationAllowed = 1;
        cfg.gridDim = dim3(kAlignCtas);
        cfg.blockDim = dim3(kAlignCThreads);
        cfg.stream = stream;
        cfg.attrs = attr;
        cfg.numAttrs = 2;
        return cudaLaunchKernelEx(&cfg, align_cluster_kernel, topk_ids, T, static_cast<int>(E), static_cast<int>(BM),
                                  sorted_ids, cap, expert_ids, cap / BM, num_post_padded, expert_offsets,
                                  padded_offsets, d_status) == cudaSuccess
                   ? QMOE_OK
                   : QMOE_ERR_CUDA;
    }
    return launch_pdl(align_kernel, dim3(1), dim3(kAlignThreads), 0, stream, topk_ids, T, E, BM, sorted_ids, cap,
                      expert_ids, cap / BM, num_post_padded, expert_offsets, padded_offsets, d_status);
}

qmoe_status_t qmoe_quant_act_fp8(const uint16_t* x, int64_t rows, int64_t cols, int64_t ldx, uint8_t* q,
                                 float* scale, qmoe_stream_t stream) {
    if (rows < 0 || cols < 1 || ldx < cols) return QMOE_ERR_INVALID_ARG;
    if (rows == 0) return QMOE_OK;
    if (!x || !q || !scale || rows > 0x7FFFFFFF) return QMOE_ERR_INVALID_ARG;
    const bool vec = (cols % 8 == 0) && (ldx % 8 == 0) && aligned16(x) && ((reinterpret_cast<uintptr_t>(q) & 7) == 0);
    if (vec)
        quant_rows_fp8_kernel<uint16_t, true><<<static_cast<unsigned>(rows), kRowThreads, 0, stream>>>(x, cols, ldx, q, scale);
    else
        quant_rows_fp8_kernel<uint16_t, false><<<static_cast<unsigned>(rows), kRowThreads, 0, stream>>>(x, cols, ldx, q, scale);
    return launch_status();
}

qmoe_status_t qmoe_quant_act_fp8_sorted(const uint16_t* x, int64_t M, int64_t cols, int64_t ldx,
                                        const int32_t* sorted_ids, const int32_t* num_post_padded, int32_t top_k,
                                        int64_t cap, uint8_t* q, float* scale, qmoe_stream_t stream) {
    if (M < 0 || cols < 16 || cols % 16 != 0 || ldx < cols || ldx % 8 != 0 || top_k < 1 || cap < 0)
        return QMOE_ERR_INVALID_ARG;
    if (cap == 0) return QMOE_OK;
    if (!x || !sorted_ids || !num_post_padded || !q || !scale || !aligned16(x) || !aligned16(q) ||
        cap > 0x7FFFFFFF)
        return QMOE_ERR_INVALID_ARG;
    const int64_t sms = device_sm_count() > 0 ? device_sm_count() : 132;
    // one warp per token (every row read and quantised once) while the slot -> position
    // table fits in shared memory and the row in registers
    const int64_t T = M * top_k;
    if (T <= kTokMaxSlots && M > 0 && aligned16(sorted_ids)) {
        static int per_sm_cache[64] = {0};
        int dev = 0;
        if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return QMOE_ERR_CUDA;
        if (per_sm_cache[dev] == 0) {
            int per_sm = 0;
            if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, quant_tokens_fp8_scatter_kernel, kTokThreads,
                                                              0) != cudaSuccess ||
                per_sm < 1)
                per_sm = 1;
            per_sm_cache[dev] = per_sm;
        }
        const int64_t want = (M + kTokThreads / 32 - 1) / (kTokThreads / 32);
        const int64_t most = sms * per_sm_cache[dev];
        const int64_t blocks = want < most ? want : most;
        return launch_pdl(quant_tokens_fp8_scatter_kernel, dim3(static_cast<unsigned>(blocks)), dim3(kTokThreads), 0,
                          stream, x, cols, ldx, sorted_ids, num_post_padded, M, top_k, q, scale);
    }
    // rows of 4097..8192 values: bulk copies, at least two in flight per CTA (measured at 6144 values: 37 us
    // against 43 for the warp kernel; at 4096 values the warp kernel is the faster, 31 against 33 us)
    if (cols > 4096 && cols * 2 <= kBulkRowsBytes / 2) {
        int64_t nbuf = kBulkRowsBytes / (cols * 2);
        if (nbuf > kBulkMaxBuf) nbuf = kBulkMaxBuf;
        // one wave of resident CTAs (shared memory bounds how many fit on an SM)
        int per_sm = 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, quant_rows_fp8_sorted_bulk_kernel, kBulkRowThreads,
                                                          static_cast<size_t>(nbuf * cols * 2)) != cudaSuccess ||
            per_sm < 1)
            per_sm = 1;
        const int64_t wave = sms * per_sm;
        const int64_t blocks = cap < wave ? cap : wave;
        return launch_pdl(quant_rows_fp8_sorted_bulk_kernel, dim3(static_cast<unsigned>(blocks)),
                          dim3(kBulkRowThreads), static_cast<size_t>(nbuf * cols * 2), stream, x, cols, ldx,
                          sorted_ids, num_post_padded, M * top_k, top_k, static_cast<int>(nbuf), q, scale);
    }
    // other rows: one warp per padded position, at most 8 CTAs per SM (grid-stride beyond)
    const int64_t want = (cap + kRowThreads / 32 - 1) / (kRowThreads / 32);
    const int64_t most = sms * 8;
    const int64_t blocks = want < most ? want : most;
    return launch_pdl(quant_rows_fp8_sorted_kernel, dim3(static_cast<unsigned>(blocks)), dim3(kRowThreads), 0, stream,
                      x, cols, ldx, sorted_ids, num_post_padded, M * top_k, top_k, q, scale);
}

qmoe_status_t qmoe_moe_align_quant_fp8(const uint16_t* x, int64_t M, int64_t cols, int64_t ldx,
                                       const int32_t* topk_ids, int32_t top_k, int32_t E, int32_t BM,
                                       int32_t* sorted_ids, int32_t* expert_ids, int32_t* num_post_padded,
                                       int32_t* expert_offsets, int32_t* padded_offsets, uint8_t* q, float* scale,
                                       int32_t* d_status, qmoe_stream_t stream) {
    if (M < 0 || top_k < 1 || top_k > 8 || E < 1 || E > kAlignMaxE || BM < 1 || BM > 1024) return QMOE_ERR_INVALID_ARG;
    if (cols < 16 || cols % 16 != 0 || ldx < cols || ldx % 8 != 0) return QMOE_ERR_INVALID_ARG;
    const int64_t T = M * top_k;
    const int64_t cap = qmoe_align_max_padded(T, E, BM);
    if (cap >= (int64_t(1) << 31)) return QMOE_ERR_UNSUPPORTED;
    if ((M > 0 && (!x || !topk_ids)) || !sorted_ids || !expert_ids || !num_post_padded || !expert_offsets ||
        !padded_offsets || !q || !scale || (M > 0 && !aligned16(x)) || !aligned16(q))
        return QMOE_ERR_INVALID_ARG;
    if (T > kFusedMaxT) {  // large batches: the two separate launches
        qmoe_status_t st = qmoe_moe_align_block_size(topk_ids, T, E, BM, sorted_ids, expert_ids, num_post_padded,
                                                     expert_offsets, padded_offsets, d_status, stream);
        if (st != QMOE_OK) return st;
        return qmoe_quant_act_fp8_sorted(x, M, cols, ldx, sorted_ids, num_post_padded, top_k, cap, q, scale, stream);
    }
    return launch_pdl(align_quant_fused_kernel<false>, dim3(static_cast<unsigned>(M + 1)), dim3(kRowThreads), 0, stream,
                      x, M, cols, ldx, topk_ids, static_cast<const float*>(nullptr), static_cast<int32_t*>(nullptr),
                      static_cast<float*>(nullptr), top_k, E, BM, sorted_ids, cap, expert_ids, num_post_padded,
                      expert_offsets, padded_offsets, q, scale, d_status);
}

qmoe_status_t qmoe_moe_router_topk(const float* logits, int64_t M, int32_t E, int32_t top_k, int32_t* topk_ids,
                                   float* topk_weights, qmoe_stream_t stream) {
    if (M < 0 || E < 1 || E > kRouterMaxE || top_k < 1 || top_k > 8 || top_k > E) return QMOE_ERR_INVALID_ARG;
    if (M == 0) return QMOE_OK;
    if (!logits || !topk_ids || !topk_weights) return QMOE_ERR_INVALID_ARG;
    router_topk_kernel<<<grid_for(M, 128), 128, 0, stream>>>(logits, M, E, top_k, topk_ids, topk_weights);
    return launch_status();
}

qmoe_status_t qmoe_moe_route_align_quant_fp8(const float* logits, const uint16_t* x, int64_t M, int64_t cols,
                                             int64_t ldx, int32_t E, int32_t top_k, int32_t BM, int32_t* topk_ids,
                                             float* topk_weights, int32_t* sorted_ids, int32_t* expert_ids,
                                             int32_t* num_post_padded, int32_t* expert_offsets,
                                             int32_t* padded_offsets, uint8_t* q, float* scale, int32_t* d_status,
                                             qmoe_stream_t stream) {
    if (M < 0 || top_k < 1 || top_k > 8 || top_k > E || E < 1 || E > kAlignMaxE || BM < 1 || BM > 1024)
        return QMOE_ERR_INVALID_ARG;
    if (cols < 16 || cols % 16 != 0 || ldx < cols || ldx % 8 != 0) return QMOE_ERR_INVALID_ARG;
    const int64_t T = M * top_k;
    const int64_t cap = qmoe_align_max_padded(T, E, BM);
    if (cap >= (int64_t(1) << 31)) return QMOE_ERR_UNSUPPORTED;
    if ((M > 0 && (!x || !logits)) || !topk_ids || !topk_weights || !sorted_ids || !expert_ids ||
        !num_post_padded || !expert_offsets || !padded_offsets || !q || !scale || (M > 0 && !aligned16(x)) ||
        !aligned16(q))
        return QMOE_ERR_INVALID_ARG;
    if (T > kFusedMaxT) {  // large batches: router, align and quantisation as three launches
        qmoe_status_t st = qmoe_moe_router_topk(logits, M, E, top_k, topk_ids, topk_weights, stream);
        if (st != QMOE_OK) return st;
        st = qmoe_moe_align_block_size(topk_ids, T, E, BM, sorted_ids, expert_ids, num_post_padded, expert_offsets,
                                       padded_offsets, d_status, stream);
        if (st != QMOE_OK) return st;
        return qmoe_quant_act_fp8_sorted(x, M, cols, ldx, sorted_ids, num_post_padded, top_k, cap, q, scale, stream);
    }
    if (M > kRouteFusedMaxM) {
        // every CTA of the one-launch form routes all M tokens (work ~ M^2):
        // past a few dozen tokens the router's own launch is cheaper
        // (measured at M=512: 14.3 us for router + align/quant against 22.5)
        const qmoe_status_t st = qmoe_moe_router_topk(logits, M, E, top_k, topk_ids, topk_weights, stream);
        if (st != QMOE_OK) return st;
        return qmoe_moe_align_quant_fp8(x, M, cols, ldx, topk_ids, top_k, E, BM, sorted_ids, expert_ids,
                                        num_post_padded, expert_offsets, padded_offsets, q, scale, d_status, stream);
    }
    return launch_pdl(align_quant_fused_kernel<true>, dim3(static_cast<unsigned>(M + 1)), dim3(kRowThreads), 0, stream,
                      x, M, cols, ldx, static_cast<const int32_t*>(nullptr), logits, topk_ids, topk_weights, top_k, E,
                      BM, sorted_ids, cap, expert_ids, num_post_padded, expert_offsets, padded_offsets, q, scale,
                      d_status);
}

qmoe_status_t qmoe_gather_sorted_bf16(const uint16_t* x, int64_t M, int64_t cols, int64_t ldx,
                                      const int32_t* sorted_ids, const int32_t* num_post_padded, int32_t top_k,
                                      int64_t cap, uint16_t* out, qmoe_stream_t stream) {
    if (M < 0 || cols < 8 || cols % 8 != 0 || ldx < cols || ldx % 8 != 0 || top_k < 1 || cap < 0)
        return QMOE_ERR_INVALID_ARG;
    if (cap == 0) return QMOE_OK;
    if (!x || !sorted_ids || !num_post_padded || !out || !aligned16(x) || !aligned16(out) || cap > 0x7FFFFFFF)
        return QMOE_ERR_INVALID_ARG;
    gather_sorted_bf16_kernel<<<static_cast<unsigned>(cap), kRowThreads, 0, stream>>>(
        x, cols, ldx, sorted_ids, num_post_padded, M * top_k, top_k, out);
    return launch_status();
}

qmoe_status_t qmoe_quant_weight_fp8(const float* w, int64_t rows, int64_t cols, uint8_t* q, float* scale,
                                    qmoe_stream_t stream) {
    if (rows < 0 || cols < 1) return QMOE_ERR_INVALID_ARG;
    if (rows == 0) return QMOE_OK;
    if (!w || !q || !scale || rows > 0x7FFFFFFF) return QMOE_ERR_INVALID_ARG;
    const bool vec = (cols % 8 == 0) && aligned16(w) && ((reinterpret_cast<uintptr_t>(q) & 7) == 0);
    if (vec)
        quant_rows_fp8_kernel<float, true><<<static_cast<unsigned>(rows), kRowThreads, 0, stream>>>(w, cols, cols, q, scale);
    else
        quant_rows_fp8_kernel<float, false><<<static_cast<unsigned>(rows), kRowThreads, 0, stream>>>(w, cols, cols, q, scale);
    return launch_status();
}

qmoe_status_t qmoe_quant_weight_int8(const float* w, int64_t rows, int64_t cols, int8_t* q, float* scale,
                                     qmoe_stream_t stream) {
    if (rows < 0 || cols < 1) return QMOE_ERR_INVALID_ARG;
    if (rows == 0) return QMOE_OK;
    if (!w || !q || !scale || rows > 0x7FFFFFFF) return QMOE_ERR_INVALID_ARG;
    quant_rows_int8_kernel<<<static_cast<unsigned>(rows), kRowThreads, 0, stream>>>(w, cols, q, scale);
    return launch_status();
}

qmoe_status_t qmoe_silu_mul_quant(const uint16_t* y, int64_t rows, int64_t I, int64_t ldy, int32_t mode,
                                  uint8_t* q, float* scale, uint8_t* sf, int64_t sf_ld,
                                  const int32_t* expert_offsets, const int32_t* sf_padded_offsets, int32_t E,
                                  int32_t* d_status, qmoe_stream_t stream) {
    return run_act_quant<ActSwiGLU>(y, rows, I, ldy, mode, q, scale, sf, sf_ld, expert_offsets, sf_padded_offsets,
                                    E, d_status, stream);
}

qmoe_status_t qmoe_srelu_quant(const uint16_t* y, int64_t rows, int64_t I, int64_t ldy, int32_t mode, uint8_t* q,
                               float* scale, uint8_t* sf, int64_t sf_ld, const int32_t* expert_offsets,
                               const int32_t* sf_padded_offsets, int32_t E, int32_t* d_status,
                               qmoe_stream_t stream) {
    return run_act_quant<ActSReLU>(y, rows, I, ldy, mode, q, scale, sf, sf_ld, expert_offsets, sf_padded_offsets,
                                   E, d_status, stream);
}

qmoe_status_t qmoe_quant_mxfp8(const uint16_t* x, int64_t rows, int64_t I, int64_t ldx, uint8_t* q, uint8_t* sf,
                               int64_t sf_ld, const int32_t* expert_offsets, const int32_t* sf_padded_offsets,
                               int32_t E, int32_t* d_status, qmoe_stream_t stream) {
    return run_act_quant<ActIdentity>(x, rows, I, ldx, QMOE_SCALE_MX_1X32, q, nullptr, sf, sf_ld, expert_offsets,
                                      sf_padded_offsets, E, d_status, stream);
}

qmoe_status_t qmoe_debug_e4m3_encode(const float* x, uint8_t* q, int64_t n, qmoe_stream_t stream) {
    if (n < 0 || (n > 0 && (!x || !q))) return QMOE_ERR_INVALID_ARG;
    if (n == 0) return QMOE_OK;
    debug_e4m3_kernel<<<grid_for(n, 256), 256, 0, stream>>>(x, q, n);
    return launch_status();
}

qmoe_status_t qmoe_debug_int8_to_bf16(const int8_t* x, uint16_t* y, int64_t n, qmoe_stream_t stream) {
    if (n < 0 || n % 4 != 0 || (n > 0 && (!x || !y || !aligned4(x) || (reinterpret_cast<uintptr_t>(y) & 7))))
        return QMOE_ERR_INVALID_ARG;
    if (n == 0) return QMOE_OK;
    debug_i8_kernel<<<grid_for(n / 4, 256), 256, 0, stream>>>(reinterpret_cast<const uint32_t*>(x),
                                                              reinterpret_cast<uint2*>(y), n / 4);
    return launch_status();
}

qmoe_status_t qmoe_debug_silu_mul(const float* g, const float* u, float* h, int64_t n, qmoe_stream_t stream) {
    if (n < 0 || (n > 0 && (!g || !u || !h))) return QMOE_ERR_INVALID_ARG;
    if (n == 0) return QMOE_OK;
    debug_silu_kernel<<<grid_for((n + 1) / 2, 256), 256, 0, stream>>>(g, u, h, n);
    return launch_status();
}

qmoe_status_t qmoe_debug_wait_timeout(int32_t* d_status, int64_t limit_ns, qmoe_stream_t stream) {
    if (!d_status || limit_ns < 0 || limit_ns > 1000000000) return QMOE_ERR_INVALID_ARG;
    debug_wait_timeout_kernel<<<1, 32, 0, stream>>>(d_status, static_cast<uint64_t>(limit_ns));
    return launch_status();
}

qmoe_status_t qmoe_debug_rcp_ge1(const float* d, float* y, int64_t n, qmoe_stream_t stream) {
    if (n < 0 || (n > 0 && (!d || !y))) return QMOE_ERR_INVALID_ARG;
    if (n == 0) return QMOE_OK;
    debug_rcp_kernel<<<grid_for(n, 256), 256, 0, stream>>>(d, y, n);
    return launch_status();
}

qmoe_status_t qmoe_debug_div_by_scale(const float* x, float s, float* q, int64_t n, qmoe_stream_t stream) {
    if (n < 0 || (n > 0 && (!x || !q))) return QMOE_ERR_INVALID_ARG;
    if (n == 0) return QMOE_OK;
    debug_div_kernel<<<grid_for((n + 1) / 2, 256), 256, 0, stream>>>(x, s, q, n);
    return launch_status();
}

qmoe_status_t qmoe_debug_quant_by_scale(const float* x, float s, uint8_t* q, int64_t n, qmoe_stream_t stream) {
    if (n < 0 || (n > 0 && (!x || !q))) return QMOE_ERR_INVALID_ARG;
    if (n == 0) return QMOE_OK;
    debug_quant_kernel<<<grid_for((n + 7) / 8, 256), 256, 0, stream>>>(x, s, q, n);
    return launch_status();
}

}  // extern "C"
