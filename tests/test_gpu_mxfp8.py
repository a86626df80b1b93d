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
