"""GPU parity of the INT4 weight-only path (the "int4wo" recipe of "Enabling MOE
Quantization using linear decomposition", read as symmetric groups of 128
along K): the int4 quantiser bit-exact against the oracle, and the W4A16
grouped GEMM within |gpu - oracle| <= 8e-3 |oracle| + 1e-2 rms(oracle)."""
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


@pytest.mark.parametrize("E,N,K", [(2, 24, 384), (8, 256, 4096)])
def test_quant_weight_int4_bitexact(q, orc, E, N, K):
    w = inputs.expert_weights_f32(E, N, K, seed=E + N + K)
    w[0, 0, :128] = 0.0
    w[-1, -1, 128:256] *= 1e-20
    qq, s = q.quant_weight_int4(to_dev(w))
    torch.cuda.synchronize()
    rq, rs = orc.quant_rows_int4_f32(w)
    assert np.array_equal(qq.cpu().numpy(), rq)
    assert np.array_equal(s.cpu().numpy().view(np.uint32), rs.view(np.uint32))


def check(gpu, ref):
    import oracle
    ok, ratio = oracle.gemm_tolerance_ok(gpu, ref)
    assert ok, f"worst |err|/bound = {ratio:.3f}"
    assert np.all(np.isfinite(gpu))


@pytest.mark.parametrize("a_layout,out_layout", [(0, 0), (1, 2), (2, 1), (0, 2)])
@pytest.mark.parametrize("M,K,N,E,top_k,BM,zipf", [(64, 256, 272, 8, 2, 128, None), (520, 384, 256, 8, 2, 128, 1.2),
                                                   (90, 128, 528, 5, 3, 256, None), (1024, 256, 1024, 8, 2, 128, None),
                                                   (64, 256, 272, 8, 2, 64, None), (300, 384, 512, 6, 3, 64, 1.2)])
def test_w4a16_parity(q, orc, a_layout, out_layout, M, K, N, E, top_k, BM, zipf):
    a = inputs.activations_bf16(M, K, seed=M + N)
    w = inputs.expert_weights_f32(E, N, K, seed=M + N)
    ids, tw = inputs.routing(M, E, top_k, seed=M + N, zipf_s=zipf)
    wq, ws = q.quant_weight_int4(to_dev(w))
    rwq, rws = orc.quant_rows_int4_f32(w)
    assert np.array_equal(wq.cpu().numpy(), rwq)
    T = M * top_k
    al = q.moe_align_block_size(to_dev(ids), E, BM)
    if a_layout == q.A_GROUPED:
        pos = orc.compact_row_of_slot(ids, E)
        order = np.empty(T, dtype=np.int64)
        order[pos] = np.arange(T)
        a_in = np.ascontiguousarray(a[order // top_k])
        a_dev = to_dev_bf16(a_in)
        ref_layout = "grouped"
    elif a_layout == q.A_PADDED:
        a_dev = q.gather_sorted_bf16(to_dev_bf16(a), al, top_k)
        a_in, ref_layout = a, "token"          # the padded rows are copies of the token rows
    else:
        a_in, a_dev, ref_layout = a, to_dev_bf16(a), "token"
    st = status()
    out = q.moe_gemm_w4a16(a_dev, wq, ws, al, to_dev(tw), M=M, top_k=top_k, BM=BM, a_layout=a_layout,
                           out_layout=out_layout, d_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    ref = orc.moe_gemm(a_kind=orc.A_BF16, a=a_in, w_kind=orc.W_INT4, w=rwq, w_scale=rws, topk_ids=ids, topk_w=tw,
                       E=E, a_layout=ref_layout, out_layout={0: "slot", 1: "grouped", 2: "token_sum"}[out_layout])
    check(bf16_to_np_f32(out), ref)


def test_w4a16_rejects_small_tiles(q):
    import quantized_moe_grouped_gb300 as qq
    M, K, N, E = 16, 128, 32, 2
    ids, tw = inputs.routing(M, E, 2, seed=3)
    al = q.moe_align_block_size(to_dev(ids), E, 32)
    a = torch.zeros(M, K, dtype=torch.bfloat16, device="cuda")
    wq = torch.zeros(E, N, K // 2, dtype=torch.uint8, device="cuda")
    ws = torch.ones(E, N, K // 128, dtype=torch.float32, device="cuda")
    with pytest.raises(qq.QmoeError):
        q.moe_gemm_w4a16(a, wq, ws, al, None, M=M, top_k=2, BM=32)
