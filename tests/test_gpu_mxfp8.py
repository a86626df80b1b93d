"""GPU parity of the MXFP8 operands ("[PyTorch] Let GroupedLinear accept MXFP8
input and gradient"): weight, plain-row and columnwise quantisers bit-exact
against the oracle, and the grouped GEMM with both operands block-scaled
within |gpu - oracle| <= 8e-3 |oracle| + 1e-2 rms(oracle)."""
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


@pytest.mark.parametrize("E,N,K", [(3, 40, 96), (8, 256, 512), (2, 16, 4096)])
def test_quant_weight_mxfp8_bitexact(q, orc, E, N, K):
    w = inputs.expert_weights_f32(E, N, K, seed=E + N + K)
    w[0, 0, :32] = 0.0
    w[-1, -1, -32:] *= 1e-30
    w[0, 1, 32:64] *= 1e6
    qq, sf = q.quant_weight_mxfp8(to_dev(w))
    torch.cuda.synchronize()
    rq, rsf = orc.quant_rows_mxfp8_f32(w)
    assert np.array_equal(qq.cpu().numpy(), rq)
    assert np.array_equal(sf.cpu().numpy(), rsf)


def test_quant_weight_mxfp8_block_exponent_edges(q, orc):
    """The E8M0 block exponent at its edges, codes and factors bit-exact: block
    maxima m * 2^x in every fp32 binade x = -126..127 with m = 1, the mantissas
    either side of 1.75 (448 = 1.75 * 2^8, where the exponent steps), 1.75
    itself, the largest mantissa and a random one; subnormal maxima (exponent
    clamped to -127) and the largest finite value.  Each maximum sits at a
    random position of its 32-block with a random sign and 31 smaller values."""
    rng = np.random.default_rng(17)
    f = np.float32
    ms = [f(1.0), np.nextafter(f(1.75), f(0)), f(1.75), np.nextafter(f(1.75), f(2)), np.nextafter(f(2.0), f(0))]
    amax = [np.ldexp(m, x).astype(np.float32) for x in range(-126, 128) for m in ms + [f(1 + rng.random())]]
    amax += [np.float32(v) for v in (np.array([1, 2, 3, 7, 1 << 20, (1 << 23) - 1], np.uint32).view(np.float32))]
    amax += [np.finfo(np.float32).max]
    amax = np.array(amax, dtype=np.float32)
    assert np.all(np.isfinite(amax)) and np.all(amax > 0)
    blocks = (rng.random((amax.size, 32)).astype(np.float32) * amax[:, None]).astype(np.float32)
    blocks *= np.where(rng.random(blocks.shape) < 0.5, f(-1), f(1))
    pos = rng.integers(0, 32, amax.size)
    blocks[np.arange(amax.size), pos] = amax * np.where(rng.random(amax.size) < 0.5, f(-1), f(1))
    per_row = 32
    rows = -(-amax.size // per_row)
    w = np.zeros((rows * per_row, 32), dtype=np.float32)
    w[:amax.size] = blocks
    w = w.reshape(rows, per_row * 32)
    qq, sf = q.quant_weight_mxfp8(to_dev(w))
    torch.cuda.synchronize()
    rq, rsf = orc.quant_rows_mxfp8_f32(w)
    assert np.array_equal(sf.cpu().numpy(), rsf)
    assert np.array_equal(qq.cpu().numpy(), rq)


@pytest.mark.parametrize("cnt,I", [([5, 0, 130, 1], 96), ([4000] * 8, 4096 // 8), ([64, 64], 128)])
def test_quant_mxfp8_rows_bitexact(q, orc, cnt, I):
    R = sum(cnt)
    x = inputs.activations_bf16(R, I, seed=R + I)
    eoff = np.array([0] + list(np.cumsum(cnt)), dtype=np.int32)
    soff = np.array([0] + list(np.cumsum([-(-c // 128) * 128 for c in cnt])), dtype=np.int32)
    st = status()
    qq, sf = q.quant_mxfp8(to_dev_bf16(x), expert_offsets=to_dev(eoff), sf_padded_offsets=to_dev(soff),
                           sf_rows=int(soff[-1]), d_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    rq, rsf = orc.quant_mxfp8_rows(x, eoff, soff)
    assert np.array_equal(qq.cpu().numpy(), rq)
    assert np.array_equal(sf.cpu().numpy(), rsf)


@pytest.mark.parametrize("R,C", [(64, 128), (128, 128), (70, 32), (4000, 1024), (33, 200)])
def test_quant_mxfp8_colwise_bitexact(q, orc, R, C):
    x = inputs.activations_bf16(R, C, seed=R * 3 + C)
    x[:32, 0] = 0
    qq, sf = q.quant_mxfp8_colwise(to_dev_bf16(x))
    torch.cuda.synchronize()
    rq, rsf = orc.quant_mxfp8_cols(x)
    assert tuple(sf.shape) == rsf.shape
    assert np.array_equal(qq.cpu().numpy(), rq)
    assert np.array_equal(sf.cpu().numpy(), rsf)


@pytest.mark.parametrize("E,N,K", [(2, 256, 128), (3, 300, 416), (8, 4096, 14336)])
def test_weight_sf_tiled_bitexact(q, orc, E, N, K):
    ld = (K // 32 + 3) // 4 * 4
    sf = np.random.default_rng(E + N + K).integers(0, 255, size=(E * N, ld), dtype=np.uint8)
    t = q.mx_weight_sf_tiled(to_dev(sf), E, N, K)
    torch.cuda.synchronize()
    assert np.array_equal(t.cpu().numpy(), orc.mx_weight_sf_tiled(sf, E, N, K))


def check(gpu, ref):
    import oracle
    ok, ratio = oracle.gemm_tolerance_ok(gpu, ref)
    assert ok, f"worst |err|/bound = {ratio:.3f}"
    assert np.all(np.isfinite(gpu))


@pytest.mark.parametrize("M,K,N,E,BM,zipf,out_layout,with_wscale", [
    (256, 256, 256, 8, 128, None, 2, False),
    (300, 384, 272, 8, 256, 1.2, 1, False),
    (150, 160, 384, 5, 128, None, 2, True),
    (1024, 256, 2560, 8, 128, 1.2, 2, False),
])
def test_gemm_mxfp8_both_operands(q, orc, M, K, N, E, BM, zipf, out_layout, with_wscale):
    """Grouped activations and weights both MXFP8 (block scales inside the MMA);
    the last case has more tiles than SMs."""
    top_k = 2
    T = M * top_k
    ids, tw = inputs.routing(M, E, top_k, seed=M + K, zipf_s=zipf)
    al = q.moe_align_block_size(to_dev(ids), E, BM)
    al128 = q.moe_align_block_size(to_dev(ids), E, 128)
    ref_al = orc.moe_align(ids, E, 128)
    eoff, poff = ref_al["expert_offsets"], ref_al["padded_offsets"]
    x = inputs.activations_bf16(T, K, seed=M + 2 * K)          # grouped rows
    aq, asf = q.quant_mxfp8(to_dev_bf16(x), expert_offsets=al128["expert_offsets"],
                            sf_padded_offsets=al128["padded_offsets"], sf_rows=q.align_max_padded(T, E, 128))
    raq, rasf = orc.quant_mxfp8_rows(x, eoff, poff)
    assert np.array_equal(aq.cpu().numpy(), raq)
    w = inputs.expert_weights_f32(E, N, K, seed=M + 3 * K)
    wq, wsf = q.quant_weight_mxfp8(to_dev(w))
    rwq, rwsf = orc.quant_rows_mxfp8_f32(w)
    assert np.array_equal(wq.cpu().numpy(), rwq) and np.array_equal(wsf.cpu().numpy(), rwsf)
    ws = (np.random.default_rng(M).random((E, N)) + 0.5).astype(np.float32) if with_wscale else None
    st = status()
    out = q.moe_gemm_w8a8(aq, None, wq, None if ws is None else to_dev(ws), al, to_dev(tw), M=M, top_k=top_k,
                          BM=BM, a_layout=q.A_GROUPED, out_layout=out_layout, a_scale_mode=q.SCALE_MX_1X32,
                          a_sf=asf, a_sf_padded_offsets=al128["padded_offsets"], w_scale_mode=q.SCALE_MX_1X32,
                          w_sf=q.mx_weight_sf_tiled(wsf.view(E * N, -1), E, N, K), d_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    sf_row = np.empty(T, dtype=np.int64)
    for e in range(E):
        sf_row[eoff[e]:eoff[e + 1]] = poff[e] + np.arange(eoff[e + 1] - eoff[e])
    ref = orc.moe_gemm(a_kind=orc.A_FP8_MX, a=raq, a_sf=rasf, a_sf_row=sf_row, w_kind=orc.W_MX, w=rwq,
                       w_scale=ws, w_sf=rwsf, topk_ids=ids, topk_w=tw, E=E, a_layout="grouped",
                       out_layout={1: "grouped", 2: "token_sum"}[out_layout])
    check(bf16_to_np_f32(out), ref)


def test_gemm_mx_weights_need_mx_activations(q, orc):
    import quantized_moe_grouped_gb300 as qq
    M, K, N, E = 16, 64, 32, 2
    ids, tw = inputs.routing(M, E, 2, seed=3)
    al = q.moe_align_block_size(to_dev(ids), E, 128)
    aq = torch.zeros(M, K, dtype=torch.uint8, device="cuda")
    sa = torch.ones(M, dtype=torch.float32, device="cuda")
    wq = torch.zeros(E, N, K, dtype=torch.uint8, device="cuda")
    wsf = torch.zeros(1024, dtype=torch.uint8, device="cuda")
    with pytest.raises(qq.QmoeError):
        q.moe_gemm_w8a8(aq, sa, wq, None, al, None, M=M, top_k=2, BM=128, w_scale_mode=q.SCALE_MX_1X32, w_sf=wsf)


@pytest.mark.parametrize("M,K,I,E,top_k,zipf,a_layout,routed,pad_cols", [
    (256, 256, 384, 8, 2, None, 2, False, 0),     # padded A, ragged expert counts
    (150, 160, 256, 5, 3, None, 0, True, 4),      # token-gather A, ragged K, routing weights, wider factor rows
    (300, 512, 1024, 16, 2, None, 1, False, 0),   # grouped A, five experts without slots
    (1024, 256, 2560, 8, 2, 1.2, 2, False, 0),    # Zipf skew, more tiles than SMs
])
def test_gemm_silu_mxfp8_epilogue_bitexact(q, orc, M, K, I, E, top_k, zipf, a_layout, routed, pad_cols):
    """FP8 [gate | up] projection with SwiGLU + MXFP8 in the GEMM epilogue: codes
    and E8M0 factors (incl. the zeroed pad rows and pad columns) identical to
    the oracle's SwiGLU + MXFP8 of the bf16 output the same GEMM stores without
    the fused epilogue; that output itself within the GEMM tolerance of the
    oracle's fp64 GEMM."""
    T, N = M * top_k, 2 * I
    seed = M + K + I
    if E == 16:
        ids, tw = inputs.routing(M, 11, top_k, seed)
        ids = np.where(ids < 5, ids, ids + 5).astype(np.int32)
    else:
        ids, tw = inputs.routing(M, E, top_k, seed, zipf)
    a = inputs.activations_bf16(M, K, seed)
    w = inputs.expert_weights_f32(E, N, K, seed)
    wq, ws = q.quant_weight_fp8(to_dev(w))
    aq, sa = q.quant_act_fp8(to_dev_bf16(a))
    rwq, rws = orc.quant_rows_fp8_f32(w)
    raq, rsa = orc.quant_rows_fp8_bf16(a)
    al = q.moe_align_block_size(to_dev(ids), E, 128)
    ref_al = orc.moe_align(ids, E, 128)
    eoff, poff = ref_al["expert_offsets"], ref_al["padded_offsets"]
    twd = to_dev(tw) if routed else None
    if a_layout == q.A_PADDED:
        a_in, s_in = q.quant_act_fp8_sorted(to_dev_bf16(a), al, top_k)
    elif a_layout == q.A_GROUPED:
        order = np.empty(T, dtype=np.int64)
        order[orc.compact_row_of_slot(ids, E)] = np.arange(T)
        src = to_dev(order // top_k)
        a_in, s_in = aq[src].contiguous(), sa[src].contiguous()
    else:
        a_in, s_in = aq, sa
    st = status()
    y = q.moe_gemm_w8a8(a_in, s_in, wq, ws, al, twd, M=M, top_k=top_k, BM=128, a_layout=a_layout,
                        out_layout=q.OUT_GROUPED, d_status=st)
    rows = q.align_max_padded(T, E, 128)
    ld = q.mx_sf_ld(I) + pad_cols
    sf = torch.full((rows, ld), 0xAB, dtype=torch.uint8, device=aq.device)
    hq, sf = q.moe_gemm_w8a8_silu_mxfp8(a_in, s_in, wq, ws, al, M=M, top_k=top_k, a_layout=a_layout,
                                         topk_weights=twd, sf=sf, d_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    ref_y = orc.moe_gemm(a_kind=orc.A_FP8_TOKEN, a=raq, a_scale=rsa, w_kind=orc.W_FP8, w=rwq, w_scale=rws,
                         topk_ids=ids, topk_w=tw if routed else None, E=E, out_layout="grouped")
    import oracle
    ok, ratio = oracle.gemm_tolerance_ok(bf16_to_np_f32(y), ref_y)
    assert ok, f"unfused GEMM: worst |err|/bound = {ratio:.3f}"
    y_bits = y.view(torch.int16).cpu().numpy().view(np.uint16)
    rq, rsf = orc.silu_mul_quant_mx(y_bits, eoff, poff)
    assert np.array_equal(hq.cpu().numpy(), rq)
    got_sf = sf.cpu().numpy()
    n = int(poff[-1])
    assert np.array_equal(got_sf[:n, :q.mx_sf_ld(I)], rsf)
    assert not got_sf[:n, q.mx_sf_ld(I):].any()                    # pad columns zeroed
    assert np.all(got_sf[n:] == 0xAB)                             # rows past the last expert untouched


def test_gemm_silu_mxfp8_rejects(q):
    """Host checks: BM must be 128, N a multiple of 256, FP8 per-token operands."""
    import quantized_moe_grouped_gb300 as qq
    M, K, E = 16, 64, 2
    ids, _ = inputs.routing(M, E, 2, seed=4)
    aq, sa = q.quant_act_fp8(to_dev_bf16(inputs.activations_bf16(M, K, 4)))
    wq, ws = q.quant_weight_fp8(to_dev(inputs.expert_weights_f32(E, 384, K, 4)))   # N = 384: not a multiple of 256
    al = q.moe_align_block_size(to_dev(ids), E, 128)
    with pytest.raises(qq.QmoeError):
        q.moe_gemm_w8a8_silu_mxfp8(aq, sa, wq, ws, al, M=M, top_k=2)
