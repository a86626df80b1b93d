"""GPU parity of the grouped GEMMs' CTA-pair tiles (two SMs per 256 x 256
tile, tcgen05 cta_group::2; FP8 W8A8 and the INT8 / INT4 weight-only GEMMs)
against the CPU oracle, forced on every shape through qmoe_debug_moe_gemm_tile:
grouped and padded activation rows, every output layout, ragged N and K tails,
empty experts, skewed routing, top_k = 3, more tiles than CTA pairs, and
experts whose last slot pair holds a single or a partly filled 128-slot block;
and the regular entry points on shapes the library sends to the pair tiles.
Bound: |gpu - oracle| <= 8e-3 |oracle| + 1e-2 rms(oracle)."""
import numpy as np
import pytest
import torch

from quantized_moe_grouped_gb300 import inputs
from tests.gpu_util import bf16_to_np_f32, status, to_dev, to_dev_bf16

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def q():
    import quantized_moe_grouped_gb300 as q
    q.load_library()
    return q


def run_case(q, orc, M, K, N, E, top_k, BM, a_layout, out_layout, seed, zipf=None, weights=True, ids=None):
    a = inputs.activations_bf16(M, K, seed)
    w = inputs.expert_weights_f32(E, N, K, seed)
    if ids is None:
        ids, tw = inputs.routing(M, E, top_k, seed, zipf)
    else:
        tw = np.full(ids.shape, 1.0 / top_k, dtype=np.float32)
    wq, ws = q.quant_weight_fp8(to_dev(w))
    rwq, rws = orc.quant_rows_fp8_f32(w)
    raq, rsa = orc.quant_rows_fp8_bf16(a)
    T = M * top_k
    al = q.moe_align_block_size(to_dev(ids), E, BM)
    if a_layout == q.A_GROUPED:
        pos = orc.compact_row_of_slot(ids, E)
        order = np.empty(T, dtype=np.int64)
        order[pos] = np.arange(T)
        aq, sa = q.quant_act_fp8(to_dev_bf16(np.ascontiguousarray(a[order // top_k])))
        raq, rsa = raq[order // top_k], rsa[order // top_k]   # the oracle reads the same grouped rows
        ref_layout = "grouped"
    else:
        aq, sa = q.quant_act_fp8_sorted(to_dev_bf16(a), al, top_k)
        ref_layout = "token"
    twd = to_dev(tw) if weights else None
    st = status()
    out = q.moe_gemm_w8a8(aq, sa, wq, ws, al, twd, M=M, top_k=top_k, BM=BM, a_layout=a_layout,
                          out_layout=out_layout, d_status=st, tile=q.TILE_PAIR)
    torch.cuda.synchronize()
    assert int(st.item()) == 0, f"device status {int(st.item())}"
    ref = orc.moe_gemm(a_kind=orc.A_FP8_TOKEN, a=raq, a_scale=rsa, w_kind=orc.W_FP8, w=rwq, w_scale=rws,
                       topk_ids=ids, topk_w=tw if weights else None, E=E, a_layout=ref_layout,
                       out_layout={0: "slot", 1: "grouped", 2: "token_sum"}[out_layout])
    gpu = bf16_to_np_f32(out)
    assert np.all(np.isfinite(gpu))
    ok, ratio = orc.gemm_tolerance_ok(gpu, ref)
    assert ok, f"worst |err|/bound = {ratio:.3f}"


@pytest.mark.parametrize("a_layout,out_layout", [(1, 0), (1, 1), (1, 2), (2, 0), (2, 1), (2, 2)])
@pytest.mark.parametrize("M,K,N,E,top_k,BM,zipf", [
    (200, 256, 512, 8, 2, 128, None),      # one or two 128-slot blocks per expert
    (520, 384, 272, 8, 2, 128, 1.2),       # N % 256 = 16, skewed experts, odd block counts
    (90, 400, 528, 5, 3, 256, None),       # K % 128 = 16, top_k = 3, BM = 256
    (2048, 512, 2048, 8, 2, 128, None),    # more tiles than CTA pairs
])
def test_pair_tile_parity(q, orc, a_layout, out_layout, M, K, N, E, top_k, BM, zipf):
    run_case(q, orc, M, K, N, E, top_k, BM, a_layout, out_layout, seed=M + K + N + a_layout, zipf=zipf)


def test_pair_tile_without_routing_weights(q, orc):
    run_case(q, orc, 300, 256, 768, 8, 2, 128, 2, 0, seed=5, weights=False)


def test_pair_tile_empty_experts_and_single_slots(q, orc):
    """Experts 1 and 5 get no slot, expert 2 exactly one, expert 3 exactly 129
    (a second 128-block of one slot), the rest share the remainder."""
    M, E, top_k = 400, 8, 1
    ids = np.zeros((M, 1), dtype=np.int32)
    ids[0, 0] = 2
    ids[1:130, 0] = 3
    rest = np.array([0, 4, 6, 7], dtype=np.int32)
    ids[130:, 0] = rest[np.arange(M - 130) % 4]
    run_case(q, orc, M, 256, 512, E, top_k, 128, 1, 0, seed=9, ids=ids)


def test_pair_tile_rejects_unsupported_forms(q):
    import quantized_moe_grouped_gb300 as qq
    M, K, N, E = 64, 128, 256, 4
    ids, tw = inputs.routing(M, E, 2, seed=3)
    al = q.moe_align_block_size(to_dev(ids), E, 64)
    aq = torch.zeros(M, K, dtype=torch.uint8, device="cuda")
    sa = torch.ones(M, dtype=torch.float32, device="cuda")
    wq = torch.zeros(E, N, K, dtype=torch.uint8, device="cuda")
    ws = torch.ones(E, N, dtype=torch.float32, device="cuda")
    with pytest.raises(qq.QmoeError):  # token-gathered rows
        q.moe_gemm_w8a8(aq, sa, wq, ws, al, None, M=M, top_k=2, BM=64, tile=q.TILE_PAIR)


def test_regular_entry_point_takes_the_pair_tile_for_long_k(q, orc):
    """qmoe_moe_gemm_w8a8 itself (no forced tile) on a down-projection-like shape
    the library sends to the pair tile: K >= 8192, 256 slots per expert."""
    M, K, N, E, top_k = 1024, 8192, 256, 8, 2
    a = inputs.activations_bf16(M, K, 31)
    w = inputs.expert_weights_f32(E, N, K, 31)
    ids, tw = inputs.routing(M, E, top_k, 31)
    T = M * top_k
    pos = orc.compact_row_of_slot(ids, E)
    order = np.empty(T, dtype=np.int64)
    order[pos] = np.arange(T)
    ag = np.ascontiguousarray(a[order // top_k])
    wq, ws = q.quant_weight_fp8(to_dev(w))
    aq, sa = q.quant_act_fp8(to_dev_bf16(ag))
    al = q.moe_align_block_size(to_dev(ids), E, 128)
    st = status()
    out = q.moe_gemm_w8a8(aq, sa, wq, ws, al, to_dev(tw), M=M, top_k=top_k, BM=128, a_layout=q.A_GROUPED,
                          out_layout=q.OUT_TOKEN_SUM, d_status=st)
    forced = q.moe_gemm_w8a8(aq, sa, wq, ws, al, to_dev(tw), M=M, top_k=top_k, BM=128, a_layout=q.A_GROUPED,
                             out_layout=q.OUT_TOKEN_SUM, d_status=st, tile=q.TILE_PAIR)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    assert torch.equal(out, forced)
    raq, rsa = orc.quant_rows_fp8_bf16(ag)
    rwq, rws = orc.quant_rows_fp8_f32(w)
    ref = orc.moe_gemm(a_kind=orc.A_FP8_TOKEN, a=raq, a_scale=rsa, w_kind=orc.W_FP8, w=rwq, w_scale=rws,
                       topk_ids=ids, topk_w=tw, E=E, a_layout="grouped", out_layout="token_sum")
    ok, ratio = orc.gemm_tolerance_ok(bf16_to_np_f32(out), ref)
    assert ok, f"worst |err|/bound = {ratio:.3f}"


@pytest.mark.parametrize("kind", ["int8", "int4"])
@pytest.mark.parametrize("a_layout,out_layout", [(1, 0), (2, 1), (2, 2), (1, 2)])
@pytest.mark.parametrize("M,K,N,E,top_k,BM,zipf", [
    (64, 256, 512, 8, 2, 128, None),       # decode-like: about 16 slots per expert (32-slot tiles)
    (520, 384, 272, 8, 2, 128, 1.2),       # N % 256 = 16, skewed experts
    (90, 512, 528, 5, 3, 64, None),        # top_k = 3, BM = 64
    (1100, 256, 1024, 8, 2, 128, None),    # more tiles than CTA pairs, full 256-slot tiles
])
def test_pair_tile_a16_parity(q, orc, kind, a_layout, out_layout, M, K, N, E, top_k, BM, zipf):
    """The weight-only GEMMs (INT8 per-row scales, INT4 per-group scales) on the
    CTA-pair tile against the oracle's fp64 dequantisation."""
    a = inputs.activations_bf16(M, K, seed=M + N + a_layout)
    w = inputs.expert_weights_f32(E, N, K, seed=M + N)
    ids, tw = inputs.routing(M, E, top_k, seed=M + N, zipf_s=zipf)
    T = M * top_k
    al = q.moe_align_block_size(to_dev(ids), E, BM)
    if a_layout == q.A_GROUPED:
        pos = orc.compact_row_of_slot(ids, E)
        order = np.empty(T, dtype=np.int64)
        order[pos] = np.arange(T)
        a_in = np.ascontiguousarray(a[order // top_k])
        a_dev = to_dev_bf16(a_in)
        ref_layout = "grouped"
    else:
        a_dev = q.gather_sorted_bf16(to_dev_bf16(a), al, top_k)
        a_in, ref_layout = a, "token"
    if kind == "int8":
        wq, ws = q.quant_weight_int8(to_dev(w))
        rwq, rws = orc.quant_rows_int8_f32(w)
        gemm, w_kind = q.moe_gemm_w8a16, orc.W_INT8
    else:
        wq, ws = q.quant_weight_int4(to_dev(w))
        rwq, rws = orc.quant_rows_int4_f32(w)
        gemm, w_kind = q.moe_gemm_w4a16, orc.W_INT4
    assert np.array_equal(wq.cpu().numpy(), rwq)
    st = status()
    out = gemm(a_dev, wq, ws, al, to_dev(tw), M=M, top_k=top_k, BM=BM, a_layout=a_layout, out_layout=out_layout,
               d_status=st, tile=q.TILE_PAIR)
    torch.cuda.synchronize()
    assert int(st.item()) == 0, f"device status {int(st.item())}"
    ref = orc.moe_gemm(a_kind=orc.A_BF16, a=a_in, w_kind=w_kind, w=rwq, w_scale=rws, topk_ids=ids, topk_w=tw,
                       E=E, a_layout=ref_layout, out_layout={0: "slot", 1: "grouped", 2: "token_sum"}[out_layout])
    gpu = bf16_to_np_f32(out)
    assert np.all(np.isfinite(gpu))
    ok, ratio = orc.gemm_tolerance_ok(gpu, ref)
    assert ok, f"worst |err|/bound = {ratio:.3f}"


def test_regular_entry_point_takes_the_pair_tile_for_large_m_short_k(q, orc):
    """qmoe_moe_gemm_w8a8 itself at 512 slots per expert and K < 8192 (an up
    projection the library sends to the pair tile), padded rows, slot output."""
    M, K, N, E, top_k = 2048, 256, 512, 8, 2
    a = inputs.activations_bf16(M, K, 41)
    w = inputs.expert_weights_f32(E, N, K, 41)
    ids, tw = inputs.routing(M, E, top_k, 41)
    wq, ws = q.quant_weight_fp8(to_dev(w))
    al = q.moe_align_block_size(to_dev(ids), E, 128)
    aq, sa = q.quant_act_fp8_sorted(to_dev_bf16(a), al, top_k)
    st = status()
    out = q.moe_gemm_w8a8(aq, sa, wq, ws, al, to_dev(tw), M=M, top_k=top_k, BM=128, a_layout=q.A_PADDED,
                          d_status=st)
    forced = q.moe_gemm_w8a8(aq, sa, wq, ws, al, to_dev(tw), M=M, top_k=top_k, BM=128, a_layout=q.A_PADDED,
                             d_status=st, tile=q.TILE_PAIR)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    assert torch.equal(out, forced)
    raq, rsa = orc.quant_rows_fp8_bf16(a)
    rwq, rws = orc.quant_rows_fp8_f32(w)
    ref = orc.moe_gemm(a_kind=orc.A_FP8_TOKEN, a=raq, a_scale=rsa, w_kind=orc.W_FP8, w=rwq, w_scale=rws,
                       topk_ids=ids, topk_w=tw, E=E)
    ok, ratio = orc.gemm_tolerance_ok(bf16_to_np_f32(out), ref)
    assert ok, f"worst |err|/bound = {ratio:.3f}"


@pytest.mark.parametrize("kind", ["int8", "int4"])
def test_regular_a16_entry_points_take_the_pair_tile_at_large_m(q, orc, kind):
    """qmoe_moe_gemm_w8a16 / _w4a16 themselves at 1024 slots per expert (the
    library sends these to the pair tile), padded rows, routing weights."""
    M, K, N, E, top_k, BM = 4096, 256, 512, 8, 2, 128
    a = inputs.activations_bf16(M, K, 77)
    w = inputs.expert_weights_f32(E, N, K, 77)
    ids, tw = inputs.routing(M, E, top_k, 77)
    al = q.moe_align_block_size(to_dev(ids), E, BM)
    ap = q.gather_sorted_bf16(to_dev_bf16(a), al, top_k)
    if kind == "int8":
        wq, ws = q.quant_weight_int8(to_dev(w))
        rwq, rws = orc.quant_rows_int8_f32(w)
        gemm, w_kind = q.moe_gemm_w8a16, orc.W_INT8
    else:
        wq, ws = q.quant_weight_int4(to_dev(w))
        rwq, rws = orc.quant_rows_int4_f32(w)
        gemm, w_kind = q.moe_gemm_w4a16, orc.W_INT4
    st = status()
    out = gemm(ap, wq, ws, al, to_dev(tw), M=M, top_k=top_k, BM=BM, a_layout=q.A_PADDED, d_status=st)
    one = gemm(ap, wq, ws, al, to_dev(tw), M=M, top_k=top_k, BM=BM, a_layout=q.A_PADDED, d_status=st,
               tile=q.TILE_ONE_SM)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    assert torch.equal(out, one)   # both families give the same bytes on this shape
    ref = orc.moe_gemm(a_kind=orc.A_BF16, a=a, w_kind=w_kind, w=rwq, w_scale=rws, topk_ids=ids, topk_w=tw, E=E)
    ok, ratio = orc.gemm_tolerance_ok(bf16_to_np_f32(out), ref)
    assert ok, f"worst |err|/bound = {ratio:.3f}"
