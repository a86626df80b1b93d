"""GPU parity at the workloads' full sizes, in the launch configurations
bench.py times, on every output row -- the decode FP8 sweep (K=4096,
N=14336, M=64..512), the INT8 W8A16 sweep (K=4096, N=7168 and 14336,
M=64..4096), the Mixtral-8x7B-shaped FP8 layer stage by stage and the
Mixtral-8x22B-shaped MXFP8 layer.  Bound:
|gpu - oracle| <= 8e-3 |oracle| + 1e-2 rms(oracle), rms over the whole output
of the call; quantised bytes bit-exact.  The oracle computes each whole output
on the host's cores (a few minutes for the file)."""
import numpy as np
import pytest
import torch

from quantized_moe_grouped_gb300 import inputs
from tests.gpu_util import bf16_to_np_f32, dev, status, to_dev, to_dev_bf16

pytestmark = pytest.mark.gpu

E, TOP_K = 8, 2


@pytest.fixture(scope="module")
def q():
    import quantized_moe_grouped_gb300 as q
    q.load_library()
    return q


def check_full(gpu: torch.Tensor, ref: np.ndarray, rows_per_chunk: int = 512):
    """Whole-output comparison, chunked over rows to bound host memory."""
    import oracle
    assert tuple(gpu.shape) == ref.shape
    rms = float(np.sqrt(np.mean(ref * ref)))
    worst = 0.0
    for r0 in range(0, ref.shape[0], rows_per_chunk):
        g = bf16_to_np_f32(gpu[r0:r0 + rows_per_chunk])
        assert np.all(np.isfinite(g)), f"non-finite output in rows {r0}.."
        ok, ratio = oracle.gemm_tolerance_ok(g, ref[r0:r0 + rows_per_chunk], rms=rms)
        worst = max(worst, ratio)
        assert ok, f"rows {r0}..: worst |err|/bound = {ratio:.3f}"
    return worst


def fp8_weights(q, orc, N, K, seed, weight_set=0):
    """Per expert: GPU quantisation (device copy) and oracle quantisation (host
    copy) of the same fp32 draws; the two must agree bit for bit."""
    wq = torch.empty(E, N, K, dtype=torch.uint8, device=dev())
    ws = torch.empty(E, N, dtype=torch.float32, device=dev())
    rwq = np.empty((E, N, K), dtype=np.uint8)
    rws = np.empty((E, N), dtype=np.float32)
    for e in range(E):
        we = inputs.expert_weight_f32(N, K, seed, e, weight_set)
        qe, se = q.quant_weight_fp8(to_dev(we))
        wq[e].copy_(qe)
        ws[e].copy_(se)
        rwq[e], rws[e] = orc.quant_rows_fp8_f32(we)
        assert np.array_equal(se.cpu().numpy(), rws[e])
    return wq, ws, rwq, rws


@pytest.fixture(scope="module")
def decode_weights(q, orc):
    return fp8_weights(q, orc, 14336, 4096, seed=1000)


@pytest.mark.parametrize("M", [64, 128, 256, 512])
def test_decode_sweep_full_size(q, orc, decode_weights, M):
    """bench.py's step for this M: moe_align_quant_fp8 then moe_gemm_w8a8 on the
    padded sorted rows with the bench's slot tile; every slot row."""
    import bench
    K, N = 4096, 14336
    BM = bench.slot_tile(M)
    wq, ws, rwq, rws = decode_weights
    a = inputs.activations_bf16(M, K, 1000 + M)
    ids, tw = inputs.routing(M, E, TOP_K, 1000 + M)
    st = status()
    al, aq, sa = q.moe_align_quant_fp8(to_dev_bf16(a), to_dev(ids), E, BM, d_status=st)
    out = q.moe_gemm_w8a8(aq, sa, wq, ws, al, to_dev(tw), M=M, top_k=TOP_K, BM=BM, a_layout=q.A_PADDED,
                          d_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    raq, rsa = orc.quant_rows_fp8_bf16(a)
    ref = orc.moe_gemm(a_kind=orc.A_FP8_TOKEN, a=raq, a_scale=rsa, w_kind=orc.W_FP8, w=rwq, w_scale=rws,
                       topk_ids=ids, topk_w=tw, E=E)
    check_full(out, ref)


_W8A16 = {}


def w8a16_weights(q, orc, N):
    """INT8 weights for K=4096 and this N (GPU and oracle quantisation of the
    same draws, scales bit-exact), kept for the module's other M."""
    if N not in _W8A16:
        _W8A16.clear()
        K = 4096
        wq = torch.empty(E, N, K, dtype=torch.int8, device=dev())
        ws = torch.empty(E, N, dtype=torch.float32, device=dev())
        rwq = np.empty((E, N, K), dtype=np.int8)
        rws = np.empty((E, N), dtype=np.float32)
        for e in range(E):
            we = inputs.expert_weight_f32(N, K, 2000 + N, e)
            qe, se = q.quant_weight_int8(to_dev(we))
            wq[e].copy_(qe)
            ws[e].copy_(se)
            rwq[e], rws[e] = orc.quant_rows_int8_f32(we)
            assert np.array_equal(se.cpu().numpy(), rws[e])
        assert np.array_equal(wq.cpu().numpy(), rwq)
        _W8A16[N] = (wq, ws, rwq, rws)
    return _W8A16[N]


@pytest.mark.parametrize("N", [7168, 14336])
@pytest.mark.parametrize("M", [64, 1024, 4096])
def test_w8a16_sweep_full_size(q, orc, M, N):
    """The W8A16 sweep's launch (BM=128, bf16 rows gathered into padded sorted
    order); every slot row."""
    K, BM = 4096, 128
    wq, ws, rwq, rws = w8a16_weights(q, orc, N)
    a = inputs.activations_bf16(M, K, 2000 + M)
    ids, tw = inputs.routing(M, E, TOP_K, 2000 + M)
    al = q.moe_align_block_size(to_dev(ids), E, BM)
    ap = q.gather_sorted_bf16(to_dev_bf16(a), al, TOP_K)
    st = status()
    out = q.moe_gemm_w8a16(ap, wq, ws, al, to_dev(tw), M=M, top_k=TOP_K, BM=BM, a_layout=q.A_PADDED, d_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    ref = orc.moe_gemm(a_kind=orc.A_BF16, a=a, w_kind=orc.W_INT8, w=rwq, w_scale=rws, topk_ids=ids, topk_w=tw,
                       E=E)
    check_full(out, ref)


def layer_up(q, orc, wl, fused=None):
    """The layer's first stages as bench.py launches them: moe_align_block_size
    (BM=128), quant_act_fp8_sorted into padded sorted rows, then the up GEMM
    (padded A -> grouped out).  Align, the quantised rows and the up
    projection are checked in full.  fused ("mx" or "token"):
    also the same projection with SwiGLU and that requantisation in its
    epilogue, whose (codes, factors or scales) are returned last."""
    M, K, I = wl.M, wl.K, wl.inter
    T, BM = M * TOP_K, 128
    ids, tw = inputs.routing(M, E, TOP_K, wl.seed, wl.zipf_s)
    a = inputs.activations_bf16(M, K, wl.seed)
    al = q.moe_align_block_size(to_dev(ids), E, BM)
    ref_al = orc.moe_align(ids, E, BM)
    npp = int(ref_al["num_post_padded"])
    assert int(al["num_post_padded"].item()) == npp
    srt = al["sorted_ids"].cpu().numpy()[:npp]
    assert np.array_equal(srt, ref_al["sorted_ids"][:npp])
    for key in ("expert_offsets", "padded_offsets"):
        assert np.array_equal(al[key].cpu().numpy(), ref_al[key])
    aq, sa = q.quant_act_fp8_sorted(to_dev_bf16(a), al, TOP_K)
    raq, rsa = orc.quant_rows_fp8_bf16(a)
    valid = np.nonzero(srt < T)[0]
    assert np.array_equal(aq.cpu().numpy()[valid], raq[srt[valid] // TOP_K])
    assert np.array_equal(sa.cpu().numpy()[valid], rsa[srt[valid] // TOP_K])
    w1q, w1s, r1q, r1s = fp8_weights(q, orc, 2 * I, K, wl.seed, weight_set=0)
    st = status()
    up = q.moe_gemm_w8a8(aq, sa, w1q, w1s, al, None, M=M, top_k=TOP_K, BM=BM, a_layout=q.A_PADDED,
                         out_layout=q.OUT_GROUPED, d_status=st)
    fused_out = None
    if fused == "mx":
        fused_out = q.moe_gemm_w8a8_silu_mxfp8(aq, sa, w1q, w1s, al, M=M, top_k=TOP_K, a_layout=q.A_PADDED,
                                               d_status=st)
    elif fused == "token":
        fused_out = q.moe_gemm_w8a8_silu_fp8_token(aq, sa, w1q, w1s, al, M=M, top_k=TOP_K, a_layout=q.A_PADDED,
                                                   d_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    del w1q, aq
    ref_up = orc.moe_gemm(a_kind=orc.A_FP8_TOKEN, a=raq, a_scale=rsa, w_kind=orc.W_FP8, w=r1q, w_scale=r1s,
                          topk_ids=ids, topk_w=None, E=E, out_layout="grouped")
    del r1q
    check_full(up, ref_up)
    del ref_up
    return (ids, tw, al, ref_al, up) + ((fused_out,) if fused else ())


def test_mixtral_8x7b_layer_full_size(q, orc):
    """M=4096, K=4096, I=14336, N=4096: align, sorted quant, up GEMM, then
    SwiGLU + per-token FP8 (bit-exact on every row; the up GEMM's fused SwiGLU
    epilogue and per-token pass give the same bytes), then the down GEMM
    (grouped A -> sum over top_k with routing weights) on every token.
    Each stage's oracle takes the GPU's previous-stage output."""
    wl = inputs.mixtral_8x7b_layer()
    M, I, Nd = wl.M, wl.inter, wl.N
    ids, tw, al, _, up, (fq, fs) = layer_up(q, orc, wl, fused="token")
    hq, hs = q.silu_mul_quant(up)
    rhq, rhs = orc.silu_mul_quant_token(up.view(torch.int16).cpu().numpy().view(np.uint16))
    del up
    assert np.array_equal(hq.cpu().numpy(), rhq) and np.array_equal(hs.cpu().numpy(), rhs)
    # the same intermediate from the up GEMM's SwiGLU epilogue + per-token pass
    assert torch.equal(fq, hq) and torch.equal(fs, hs)
    del fq, fs
    w2q, w2s, r2q, r2s = fp8_weights(q, orc, Nd, I, wl.seed, weight_set=1)
    st = status()
    down = q.moe_gemm_w8a8(hq, hs, w2q, w2s, al, to_dev(tw), M=M, top_k=TOP_K, BM=128, a_layout=q.A_GROUPED,
                           out_layout=q.OUT_TOKEN_SUM, d_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    ref = orc.moe_gemm(a_kind=orc.A_FP8_TOKEN, a=rhq, a_scale=rhs, w_kind=orc.W_FP8, w=r2q, w_scale=r2s,
                       topk_ids=ids, topk_w=tw, E=E, a_layout="grouped", out_layout="token_sum")
    check_full(down, ref)


def test_mixtral_8x22b_mx_layer_full_size(q, orc):
    """M=4096 with Zipf(1.2)-skewed routing, K=6144, I=16384, N=6144: align,
    sorted quant, up GEMM, then SwiGLU + MXFP8 over the grouped rows (codes and
    E8M0 factors bit-exact on every row; the up GEMM's fused SwiGLU + MXFP8
    epilogue gives the same bytes), then the block-scaled down GEMM with
    per-row FP8 weights and again with MXFP8 weights (tiled factors), each on
    every token."""
    wl = inputs.mixtral_8x22b_layer()
    M, I, Nd = wl.M, wl.inter, wl.N
    T = M * TOP_K
    ids, tw, al, ref_al, up, (fq, fsf) = layer_up(q, orc, wl, fused="mx")
    eoff, poff = ref_al["expert_offsets"], ref_al["padded_offsets"]
    hq, sf = q.silu_mul_quant(up, q.SCALE_MX_1X32, expert_offsets=al["expert_offsets"],
                              sf_padded_offsets=al["padded_offsets"], sf_rows=q.align_max_padded(T, E, 128))
    rq, rsf = orc.silu_mul_quant_mx(up.view(torch.int16).cpu().numpy().view(np.uint16), eoff, poff)
    del up
    assert np.array_equal(hq.cpu().numpy(), rq)
    assert np.array_equal(sf.cpu().numpy()[: poff[-1]], rsf)
    # the same intermediate from the up GEMM's SwiGLU + MXFP8 epilogue
    assert torch.equal(fq, hq) and torch.equal(fsf[: poff[-1]], sf[: poff[-1]])
    del fq, fsf
    sf_row = np.empty(T, dtype=np.int64)
    for e in range(E):
        sf_row[eoff[e]:eoff[e + 1]] = poff[e] + np.arange(eoff[e + 1] - eoff[e])
    twd = to_dev(tw)
    mx_a = dict(a_scale_mode=q.SCALE_MX_1X32, a_sf=sf, a_sf_padded_offsets=al["padded_offsets"])

    w2q, w2s, r2q, r2s = fp8_weights(q, orc, Nd, I, wl.seed, weight_set=1)
    st = status()
    down = q.moe_gemm_w8a8(hq, None, w2q, w2s, al, twd, M=M, top_k=TOP_K, BM=128, a_layout=q.A_GROUPED,
                           out_layout=q.OUT_TOKEN_SUM, d_status=st, **mx_a)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    del w2q
    ref = orc.moe_gemm(a_kind=orc.A_FP8_MX, a=rq, a_sf=rsf, a_sf_row=sf_row, w_kind=orc.W_FP8, w=r2q,
                       w_scale=r2s, topk_ids=ids, topk_w=tw, E=E, a_layout="grouped", out_layout="token_sum")
    check_full(down, ref)
    del r2q

    ld = q.mx_sf_ld(I)
    wmq = torch.empty(E, Nd, I, dtype=torch.uint8, device=dev())
    wmsf = torch.empty(E * Nd, ld, dtype=torch.uint8, device=dev())
    rwmq = np.empty((E, Nd, I), dtype=np.uint8)
    rwmsf = np.empty((E * Nd, ld), dtype=np.uint8)
    for e in range(E):
        we = inputs.expert_weight_f32(Nd, I, wl.seed, e, 2)
        q.quant_weight_mxfp8(to_dev(we), q=wmq[e], sf=wmsf[e * Nd:(e + 1) * Nd])
        rwmq[e], rwmsf[e * Nd:(e + 1) * Nd] = orc.quant_rows_mxfp8_f32(we)
    assert np.array_equal(wmsf.cpu().numpy(), rwmsf)
    tiled = q.mx_weight_sf_tiled(wmsf, E, Nd, I)
    assert np.array_equal(tiled.cpu().numpy(), orc.mx_weight_sf_tiled(rwmsf, E, Nd, I))
    down = q.moe_gemm_w8a8(hq, None, wmq, None, al, twd, M=M, top_k=TOP_K, BM=128, a_layout=q.A_GROUPED,
                           out_layout=q.OUT_TOKEN_SUM, d_status=st, w_scale_mode=q.SCALE_MX_1X32, w_sf=tiled, **mx_a)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    assert np.array_equal(wmq.cpu().numpy(), rwmq)
    ref = orc.moe_gemm(a_kind=orc.A_FP8_MX, a=rq, a_sf=rsf, a_sf_row=sf_row, w_kind=orc.W_MX, w=rwmq,
                       w_scale=None, w_sf=rwmsf, topk_ids=ids, topk_w=tw, E=E, a_layout="grouped",
                       out_layout="token_sum")
    check_full(down, ref)
