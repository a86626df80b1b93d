"""GPU parity of the grouped GEMMs against the CPU oracle:
|gpu - oracle| <= 8e-3 |oracle| + 1e-2 rms(oracle) elementwise, where the oracle
dequantises the same quantised bytes to fp64 and runs the dense per-token
expert loop.  Covers every layout, every tile size, ragged N/K tails, empty
experts, skewed routing, a whole FFN layer stage by stage, and the full
decode shape on sampled slots."""
import numpy as np
import pytest
import torch

from quantized_moe_grouped_gb300 import inputs
from tests.gpu_util import bf16_to_np_f32, dev, status, to_dev, to_dev_bf16

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def q():
    import quantized_moe_grouped_gb300 as q
    q.load_library()
    return q


def fp8_problem(q, orc, M, K, N, E, top_k, seed, zipf=None, ids=None, tw=None):
    a = inputs.activations_bf16(M, K, seed)
    w = inputs.expert_weights_f32(E, N, K, seed)
    if ids is None:
        ids, tw = inputs.routing(M, E, top_k, seed, zipf)
    wq, ws = q.quant_weight_fp8(to_dev(w))
    aq, sa = q.quant_act_fp8(to_dev_bf16(a))
    rwq, rws = orc.quant_rows_fp8_f32(w)
    raq, rsa = orc.quant_rows_fp8_bf16(a)
    # the two quantisers agree bit for bit (tested on their own elsewhere)
    assert np.array_equal(wq.cpu().numpy(), rwq) and np.array_equal(aq.cpu().numpy(), raq)
    return dict(a=a, ids=ids, tw=tw, wq=wq, ws=ws, aq=aq, sa=sa, rwq=rwq, rws=rws, raq=raq, rsa=rsa)


def check(gpu, ref):
    import oracle
    ok, ratio = oracle.gemm_tolerance_ok(gpu, ref)
    assert ok, f"worst |err|/bound = {ratio:.3f}"
    assert np.all(np.isfinite(gpu))
    return ratio


LAYOUTS = [(0, 0), (0, 1), (0, 2), (1, 0), (1, 2)]


@pytest.mark.parametrize("BM", [16, 32, 64, 128, 256])
def test_w8a8_tiny_all_tile_sizes(q, orc, BM):
    """M=64 K=128 N=256 E=8 top_k=2 (the tiny workload), SLOT output with routing weights."""
    M, K, N, E, top_k = 64, 128, 256, 8, 2
    p = fp8_problem(q, orc, M, K, N, E, top_k, seed=0)
    st = status()
    al = q.moe_align_block_size(to_dev(p["ids"]), E, BM)
    out = q.moe_gemm_w8a8(p["aq"], p["sa"], p["wq"], p["ws"], al, to_dev(p["tw"]), M=M, top_k=top_k, BM=BM,
                          d_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    ref = orc.moe_gemm(a_kind=orc.A_FP8_TOKEN, a=p["raq"], a_scale=p["rsa"], w_kind=orc.W_FP8, w=p["rwq"],
                       w_scale=p["rws"], topk_ids=p["ids"], topk_w=p["tw"], E=E)
    check(bf16_to_np_f32(out), ref)


@pytest.mark.parametrize("a_layout,out_layout", LAYOUTS)
@pytest.mark.parametrize("M,K,N,E,top_k,BM", [(200, 272, 208, 8, 2, 32), (37, 512, 384, 5, 3, 16),
                                              (300, 96, 128, 4, 1, 64), (150, 272, 400, 8, 2, 128),
                                              (90, 160, 272, 5, 3, 256), (700, 128, 528, 8, 2, 128)])
def test_w8a8_layouts_ragged(q, orc, a_layout, out_layout, M, K, N, E, top_k, BM):
    p = fp8_problem(q, orc, M, K, N, E, top_k, seed=M + K + N)
    T = M * top_k
    use_w = out_layout != 1 or a_layout == 1
    tw_d = to_dev(p["tw"]) if use_w else None
    ids_d = to_dev(p["ids"])
    al = q.moe_align_block_size(ids_d, E, BM)
    if a_layout == q.A_GROUPED:
        pos = orc.compact_row_of_slot(p["ids"], E)
        order = np.empty(T, dtype=np.int64)
        order[pos] = np.arange(T)
        a_rows = order // top_k                          # compact row -> token row
        aq_in = p["aq"][to_dev(a_rows)].contiguous()
        sa_in = p["sa"][to_dev(a_rows)].contiguous()
        raq_in, rsa_in = p["raq"][a_rows], p["rsa"][a_rows]
    else:
        aq_in, sa_in, raq_in, rsa_in = p["aq"], p["sa"], p["raq"], p["rsa"]
    st = status()
    out = q.moe_gemm_w8a8(aq_in, sa_in, p["wq"], p["ws"], al, tw_d, M=M, top_k=top_k, BM=BM,
                          a_layout=a_layout, out_layout=out_layout, d_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    ref = orc.moe_gemm(a_kind=orc.A_FP8_TOKEN, a=raq_in, a_scale=rsa_in, w_kind=orc.W_FP8, w=p["rwq"],
                       w_scale=p["rws"], topk_ids=p["ids"], topk_w=p["tw"] if use_w else None, E=E,
                       a_layout="grouped" if a_layout == 1 else "token",
                       out_layout={0: "slot", 1: "grouped", 2: "token_sum"}[out_layout])
    check(bf16_to_np_f32(out), ref)


@pytest.mark.parametrize("a_layout,out_layout", [(0, 0), (1, 2), (2, 1), (0, 2)])
@pytest.mark.parametrize("M,K,N,E,top_k", [(64, 256, 272, 8, 2), (150, 400, 528, 6, 3), (520, 128, 256, 8, 2)])
def test_w8a8_wide64_tile(q, orc, a_layout, out_layout, M, K, N, E, top_k):
    """The 64-slot wide FP8 tile (M = 64 MMAs over 256 weight rows, the BM = 64
    tile): every activation layout, ragged N and K, top_k = 3."""
    p = fp8_problem(q, orc, M, K, N, E, top_k, seed=M + K + N + 3)
    T = M * top_k
    BM = 64
    ids_d = to_dev(p["ids"])
    al = q.moe_align_block_size(ids_d, E, BM)
    if a_layout == q.A_GROUPED:
        pos = orc.compact_row_of_slot(p["ids"], E)
        order = np.empty(T, dtype=np.int64)
        order[pos] = np.arange(T)
        rows = order // top_k
        aq_in, sa_in = p["aq"][to_dev(rows)].contiguous(), p["sa"][to_dev(rows)].contiguous()
        ra, rs, ref_layout = p["raq"][rows], p["rsa"][rows], "grouped"
    elif a_layout == q.A_PADDED:
        a_bf = to_dev_bf16(p["a"])
        aq_in, sa_in = q.quant_act_fp8_sorted(a_bf, al, top_k)
        ra, rs, ref_layout = p["raq"], p["rsa"], "token"
    else:
        aq_in, sa_in, ra, rs, ref_layout = p["aq"], p["sa"], p["raq"], p["rsa"], "token"
    st = status()
    out = q.moe_gemm_w8a8(aq_in, sa_in, p["wq"], p["ws"], al, to_dev(p["tw"]), M=M, top_k=top_k, BM=BM,
                          a_layout=a_layout, out_layout=out_layout, d_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    ref = orc.moe_gemm(a_kind=orc.A_FP8_TOKEN, a=ra, a_scale=rs, w_kind=orc.W_FP8, w=p["rwq"], w_scale=p["rws"],
                       topk_ids=p["ids"], topk_w=p["tw"], E=E, a_layout=ref_layout,
                       out_layout={0: "slot", 1: "grouped", 2: "token_sum"}[out_layout])
    check(bf16_to_np_f32(out), ref)


def test_w8a8_token_sum_deterministic(q, orc):
    M, K, N, E, top_k, BM = 256, 256, 256, 8, 2, 32
    p = fp8_problem(q, orc, M, K, N, E, top_k, seed=5)
    al = q.moe_align_block_size(to_dev(p["ids"]), E, BM)
    outs = [q.moe_gemm_w8a8(p["aq"], p["sa"], p["wq"], p["ws"], al, to_dev(p["tw"]), M=M, top_k=top_k, BM=BM,
                            out_layout=q.OUT_TOKEN_SUM).clone() for _ in range(3)]
    assert all(torch.equal(outs[0], o) for o in outs[1:])


@pytest.mark.parametrize("BM,K", [(128, 256), (256, 8192)])
def test_w8a8_token_sum_deterministic_wide(q, orc, BM, K):
    """The wide tiles (one 128-slot block, and two of them sharing each weight
    stage at K >= 8192) add their slot results into the fp32 accumulator: for
    top_k = 2 the sum 0 + a + b does not depend on the order, so repeated
    launches agree bit for bit."""
    M, N, E, top_k = 300, 272, 8, 2
    p = fp8_problem(q, orc, M, K, N, E, top_k, seed=6)
    al = q.moe_align_block_size(to_dev(p["ids"]), E, BM)
    pos = orc.compact_row_of_slot(p["ids"], E)
    order = np.empty(M * top_k, dtype=np.int64)
    order[pos] = np.arange(M * top_k)
    rows = to_dev(order // top_k)
    aq_g, sa_g = p["aq"][rows].contiguous(), p["sa"][rows].contiguous()
    outs = [q.moe_gemm_w8a8(aq_g, sa_g, p["wq"], p["ws"], al, to_dev(p["tw"]), M=M, top_k=top_k, BM=BM,
                            a_layout=q.A_GROUPED, out_layout=q.OUT_TOKEN_SUM).clone() for _ in range(3)]
    assert all(torch.equal(outs[0], o) for o in outs[1:])
    ref = orc.moe_gemm(a_kind=orc.A_FP8_TOKEN, a=p["raq"][order // top_k], a_scale=p["rsa"][order // top_k],
                       w_kind=orc.W_FP8, w=p["rwq"], w_scale=p["rws"], topk_ids=p["ids"], topk_w=p["tw"], E=E,
                       a_layout="grouped", out_layout="token_sum")
    check(bf16_to_np_f32(outs[0]), ref)


@pytest.mark.parametrize("M,K,N,E,top_k,BM", [(96, 256, 400, 16, 8, 128), (130, 128, 528, 12, 5, 256),
                                              (64, 128, 256, 8, 1, 128)])
def test_w8a8_token_sum_large_top_k(q, orc, M, K, N, E, top_k, BM):
    """TOKEN_SUM with up to eight contributions per token and output segment."""
    p = fp8_problem(q, orc, M, K, N, E, top_k, seed=M + top_k)
    al = q.moe_align_block_size(to_dev(p["ids"]), E, BM)
    st = status()
    out = q.moe_gemm_w8a8(p["aq"], p["sa"], p["wq"], p["ws"], al, to_dev(p["tw"]), M=M, top_k=top_k, BM=BM,
                          out_layout=q.OUT_TOKEN_SUM, d_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    ref = orc.moe_gemm(a_kind=orc.A_FP8_TOKEN, a=p["raq"], a_scale=p["rsa"], w_kind=orc.W_FP8, w=p["rwq"],
                       w_scale=p["rws"], topk_ids=p["ids"], topk_w=p["tw"], E=E, out_layout="token_sum")
    check(bf16_to_np_f32(out), ref)


@pytest.mark.parametrize("BM,K,a_layout", [(128, 256, 0), (64, 256, 0), (256, 8192, 1)])
def test_w8a8_token_sum_dropped_slots(q, orc, BM, K, a_layout):
    """Slots routed outside [0, E) are dropped by the align; their tokens then
    have fewer than top_k contributions (some none at all): TOKEN_SUM gives
    every token's sum over its valid slots, 0 for a token without any."""
    M, N, E, top_k = 160, 272, 8, 2
    p = fp8_problem(q, orc, M, K, N, E, top_k, seed=21)
    ids = p["ids"].copy()
    rng = np.random.default_rng(21)
    drop = rng.random(ids.shape) < 0.15
    ids[drop] = np.where(rng.random(ids.shape) < 0.5, -1, E + 3)[drop]
    ids[:5] = -1                                             # tokens without any valid slot
    valid = ((ids >= 0) & (ids < E)).ravel()
    T = M * top_k
    al = q.moe_align_block_size(to_dev(ids), E, BM)
    slots = np.nonzero(valid)[0]
    if a_layout == q.A_GROUPED:
        pos = orc.compact_row_of_slot(ids, E)
        order = np.empty(slots.size, dtype=np.int64)
        order[pos[slots]] = slots
        a_rows = order // top_k                              # compact row -> token row
        aq_in, sa_in = p["aq"][to_dev(a_rows)].contiguous(), p["sa"][to_dev(a_rows)].contiguous()
        ra, rs = p["raq"][a_rows], p["rsa"][a_rows]
        a_row_of_slot = np.zeros(T, dtype=np.int64)
        a_row_of_slot[slots] = pos[slots]
    else:
        aq_in, sa_in, ra, rs = p["aq"], p["sa"], p["raq"], p["rsa"]
        a_row_of_slot = np.arange(T, dtype=np.int64) // top_k
    st = status()
    out = q.moe_gemm_w8a8(aq_in, sa_in, p["wq"], p["ws"], al, to_dev(p["tw"]), M=M, top_k=top_k, BM=BM,
                          a_layout=a_layout, out_layout=q.OUT_TOKEN_SUM, d_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    per_slot = orc.moe_gemm_slots(a_kind=orc.A_FP8_TOKEN, a=ra, a_scale=rs, w_kind=orc.W_FP8, w=p["rwq"],
                                  w_scale=p["rws"], topk_ids=np.where(valid.reshape(ids.shape), ids, 0),
                                  topk_w=p["tw"], a_row=a_row_of_slot, slots=slots, N=N, K=K)
    ref = np.zeros((M, N))
    np.add.at(ref, slots // top_k, per_slot)
    got = bf16_to_np_f32(out)
    check(got, ref)
    assert np.all(got[:5] == 0.0)


def test_w8a8_skewed_and_empty_experts(q, orc):
    M, K, N, E, top_k, BM = 512, 256, 128, 8, 2, 64
    ids = np.zeros((M, top_k), dtype=np.int32)
    ids[:, 0] = 0
    ids[:, 1] = np.where(np.arange(M) % 5 == 0, 3, 1)     # experts 2, 4..7 get nothing
    tw = np.full((M, top_k), 0.5, dtype=np.float32)
    p = fp8_problem(q, orc, M, K, N, E, top_k, seed=8, ids=ids, tw=tw)
    al = q.moe_align_block_size(to_dev(ids), E, BM)
    out = q.moe_gemm_w8a8(p["aq"], p["sa"], p["wq"], p["ws"], al, to_dev(tw), M=M, top_k=top_k, BM=BM,
                          out_layout=q.OUT_TOKEN_SUM)
    ref = orc.moe_gemm(a_kind=orc.A_FP8_TOKEN, a=p["raq"], a_scale=p["rsa"], w_kind=orc.W_FP8, w=p["rwq"],
                       w_scale=p["rws"], topk_ids=ids, topk_w=tw, E=E, out_layout="token_sum")
    check(bf16_to_np_f32(out), ref)


def test_w8a8_single_row(q, orc):
    p = fp8_problem(q, orc, 1, 64, 32, 4, 2, seed=11)
    al = q.moe_align_block_size(to_dev(p["ids"]), 4, 16)
    out = q.moe_gemm_w8a8(p["aq"], p["sa"], p["wq"], p["ws"], al, to_dev(p["tw"]), M=1, top_k=2, BM=16)
    ref = orc.moe_gemm(a_kind=orc.A_FP8_TOKEN, a=p["raq"], a_scale=p["rsa"], w_kind=orc.W_FP8, w=p["rwq"],
                       w_scale=p["rws"], topk_ids=p["ids"], topk_w=p["tw"], E=4)
    check(bf16_to_np_f32(out), ref)


@pytest.mark.parametrize("a_layout,out_layout", [(0, 0), (1, 2), (0, 1)])
@pytest.mark.parametrize("M,K,N,E,top_k,BM", [(64, 128, 256, 8, 2, 16), (150, 336, 144, 6, 2, 64),
                                              (520, 256, 256, 8, 2, 128), (70, 64, 512, 3, 3, 256)])
def test_w8a16_parity(q, orc, a_layout, out_layout, M, K, N, E, top_k, BM):
    a = inputs.activations_bf16(M, K, seed=M + N)
    w = inputs.expert_weights_f32(E, N, K, seed=M + N)
    ids, tw = inputs.routing(M, E, top_k, seed=M + N)
    wq, ws = q.quant_weight_int8(to_dev(w))
    rwq, rws = orc.quant_rows_int8_f32(w)
    assert np.array_equal(wq.cpu().numpy(), rwq)
    T = M * top_k
    if a_layout == q.A_GROUPED:
        pos = orc.compact_row_of_slot(ids, E)
        order = np.empty(T, dtype=np.int64)
        order[pos] = np.arange(T)
        a_in = np.ascontiguousarray(a[order // top_k])
    else:
        a_in = a
    al = q.moe_align_block_size(to_dev(ids), E, BM)
    st = status()
    out = q.moe_gemm_w8a16(to_dev_bf16(a_in), wq, ws, al, to_dev(tw), M=M, top_k=top_k, BM=BM,
                           a_layout=a_layout, out_layout=out_layout, d_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    ref = orc.moe_gemm(a_kind=orc.A_BF16, a=a_in, w_kind=orc.W_INT8, w=rwq, w_scale=rws, topk_ids=ids, topk_w=tw,
                       E=E, a_layout="grouped" if a_layout == 1 else "token",
                       out_layout={0: "slot", 1: "grouped", 2: "token_sum"}[out_layout])
    check(bf16_to_np_f32(out), ref)


@pytest.mark.parametrize("BM", [64, 128])
def test_fp8_layer_stagewise(q, orc, BM):
    """One FFN layer (reduced Mixtral shape): up GEMM (token gather -> grouped
    rows) -> SwiGLU + per-token FP8 -> down GEMM (grouped rows -> sum over
    top_k with routing weights).  Each stage's oracle takes the GPU's
    previous-stage output, so quantised bytes must match exactly."""
    M, K, I, Nd, E, top_k = 256, 256, 384, 256, 8, 2
    a = inputs.activations_bf16(M, K, 31)
    w1 = inputs.expert_weights_f32(E, 2 * I, K, 31, weight_set=0)
    w2 = inputs.expert_weights_f32(E, Nd, I, 31, weight_set=1)
    ids, tw = inputs.routing(M, E, top_k, 31)
    w1q, w1s = q.quant_weight_fp8(to_dev(w1))
    w2q, w2s = q.quant_weight_fp8(to_dev(w2))
    r1q, r1s = orc.quant_rows_fp8_f32(w1)
    r2q, r2s = orc.quant_rows_fp8_f32(w2)
    al = q.moe_align_block_size(to_dev(ids), E, BM)
    aq, sa = q.quant_act_fp8(to_dev_bf16(a))
    up = q.moe_gemm_w8a8(aq, sa, w1q, w1s, al, None, M=M, top_k=top_k, BM=BM, out_layout=q.OUT_GROUPED)
    raq, rsa = orc.quant_rows_fp8_bf16(a)
    ref_up = orc.moe_gemm(a_kind=orc.A_FP8_TOKEN, a=raq, a_scale=rsa, w_kind=orc.W_FP8, w=r1q, w_scale=r1s,
                          topk_ids=ids, topk_w=None, E=E, out_layout="grouped")
    check(bf16_to_np_f32(up), ref_up)
    hq, hs = q.silu_mul_quant(up)
    up_bits = up.view(torch.int16).cpu().numpy().view(np.uint16)
    rhq, rhs = orc.silu_mul_quant_token(up_bits)
    assert np.array_equal(hq.cpu().numpy(), rhq) and np.array_equal(hs.cpu().numpy(), rhs)
    down = q.moe_gemm_w8a8(hq, hs, w2q, w2s, al, to_dev(tw), M=M, top_k=top_k, BM=BM, a_layout=q.A_GROUPED,
                           out_layout=q.OUT_TOKEN_SUM)
    ref_down = orc.moe_gemm(a_kind=orc.A_FP8_TOKEN, a=rhq, a_scale=rhs, w_kind=orc.W_FP8, w=r2q, w_scale=r2s,
                            topk_ids=ids, topk_w=tw, E=E, a_layout="grouped", out_layout="token_sum")
    check(bf16_to_np_f32(down), ref_down)


def test_w8a8_decode_full_size_sampled(q, orc):
    """M=64 K=4096 N=14336 E=8 top_k=2 with BM=32 (the launch the benchmark
    times): 16 sampled slots, every output channel, against the oracle."""
    M, K, N, E, top_k, BM = 64, 4096, 14336, 8, 2, 32
    seed = 1000
    a = inputs.activations_bf16(M, K, seed)
    ids, tw = inputs.routing(M, E, top_k, seed)
    wq = torch.empty(E, N, K, dtype=torch.uint8, device=dev())
    ws = torch.empty(E, N, dtype=torch.float32, device=dev())
    rwq = np.empty((E, N, K), dtype=np.uint8)
    rws = np.empty((E, N), dtype=np.float32)
    for e in range(E):
        we = inputs.expert_weight_f32(N, K, seed, e)
        qe, se = q.quant_weight_fp8(to_dev(we))
        wq[e].copy_(qe)
        ws[e].copy_(se)
        rwq[e], rws[e] = orc.quant_rows_fp8_f32(we)
    assert np.array_equal(ws.cpu().numpy(), rws)
    al = q.moe_align_block_size(to_dev(ids), E, BM)
    aq, sa = q.quant_act_fp8(to_dev_bf16(a))
    out = q.moe_gemm_w8a8(aq, sa, wq, ws, al, to_dev(tw), M=M, top_k=top_k, BM=BM)
    raq, rsa = orc.quant_rows_fp8_bf16(a)
    slots = np.random.default_rng(0).choice(M * top_k, 16, replace=False)
    ref = orc.moe_gemm(a_kind=orc.A_FP8_TOKEN, a=raq, a_scale=rsa, w_kind=orc.W_FP8, w=rwq, w_scale=rws,
                       topk_ids=ids, topk_w=tw, E=E, slots=slots)
    full = bf16_to_np_f32(out)
    rms = float(np.sqrt(np.mean(ref * ref)))
    import oracle
    ok, ratio = oracle.gemm_tolerance_ok(full[slots], ref, rms=rms)
    assert ok, ratio
    assert np.all(np.isfinite(full))


@pytest.mark.parametrize("M,K,N,E,top_k,BM,out_layout", [(64, 128, 256, 8, 2, 32, 0), (200, 272, 208, 8, 2, 64, 2),
                                                         (333, 512, 400, 8, 2, 128, 0), (90, 160, 272, 5, 3, 256, 2),
                                                         (300, 6144, 128, 8, 2, 128, 2), (64, 8320, 128, 8, 2, 128, 0)])
def test_w8a8_padded_sorted_activations(q, orc, M, K, N, E, top_k, BM, out_layout):
    """quant_act_fp8_sorted (bit-exact against the oracle's per-token codes placed
    at the padded sorted positions) feeding the GEMM's PADDED activation layout."""
    p = fp8_problem(q, orc, M, K, N, E, top_k, seed=M * 3 + BM)
    al = q.moe_align_block_size(to_dev(p["ids"]), E, BM)
    aq_p, sa_p = q.quant_act_fp8_sorted(to_dev_bf16(p["a"]), al, top_k)
    ref_al = orc.moe_align(p["ids"], E, BM)
    n = ref_al["num_post_padded"]
    srt = ref_al["sorted_ids"][:n]
    valid = srt < M * top_k
    exp_q = np.zeros((n, K), dtype=np.uint8)
    exp_s = np.zeros(n, dtype=np.float32)
    exp_q[valid] = p["raq"][srt[valid] // top_k]
    exp_s[valid] = p["rsa"][srt[valid] // top_k]
    assert np.array_equal(aq_p.cpu().numpy()[:n], exp_q)
    assert np.array_equal(sa_p.cpu().numpy()[:n], exp_s)
    out = q.moe_gemm_w8a8(aq_p, sa_p, p["wq"], p["ws"], al, to_dev(p["tw"]), M=M, top_k=top_k, BM=BM,
                          a_layout=q.A_PADDED, out_layout=out_layout)
    cap = aq_p.shape[0]
    a_full = np.zeros((cap, K), dtype=np.uint8)
    s_full = np.zeros(cap, dtype=np.float32)
    a_full[:n], s_full[:n] = exp_q, exp_s
    ref = orc.moe_gemm(a_kind=orc.A_FP8_TOKEN, a=a_full, a_scale=s_full, w_kind=orc.W_FP8, w=p["rwq"],
                       w_scale=p["rws"], topk_ids=p["ids"], topk_w=p["tw"], E=E, a_layout="padded", BM=BM,
                       out_layout={0: "slot", 2: "token_sum"}[out_layout])
    check(bf16_to_np_f32(out), ref)


@pytest.mark.parametrize("M,I,N,E,BM,zipf,out_layout", [(256, 256, 256, 8, 128, None, 2), (300, 384, 272, 8, 256, 1.2, 2),
                                                        (150, 160, 384, 5, 128, None, 1),
                                                        (1024, 256, 2560, 8, 128, 1.2, 2)])
def test_w8a8_mx_activations(q, orc, M, I, N, E, BM, zipf, out_layout):
    """Down GEMM on MXFP8 activations: SwiGLU + MX 1x32 requantisation (bit-exact
    against the oracle), then the block-scaled FP8 GEMM over the grouped rows,
    against the oracle's fp64 dequantisation with the E8M0 block scales.  The
    last case has more tiles than the GPU has SMs, so CTAs reuse their single
    accumulator."""
    top_k = 2
    T = M * top_k
    ids, tw = inputs.routing(M, E, top_k, seed=M + I, zipf_s=zipf)
    y = inputs.activations_bf16(T, 2 * I, seed=M + I)
    al = q.moe_align_block_size(to_dev(ids), E, BM)
    al128 = q.moe_align_block_size(to_dev(ids), E, 128)
    hq, sf = q.silu_mul_quant(to_dev_bf16(y), q.SCALE_MX_1X32, expert_offsets=al128["expert_offsets"],
                              sf_padded_offsets=al128["padded_offsets"], sf_rows=q.align_max_padded(T, E, 128))
    ref_al = orc.moe_align(ids, E, 128)
    rq, rsf = orc.silu_mul_quant_mx(y, ref_al["expert_offsets"], ref_al["padded_offsets"])
    assert np.array_equal(hq.cpu().numpy(), rq)
    nsf = ref_al["padded_offsets"][-1]
    assert np.array_equal(sf.cpu().numpy()[:nsf], rsf)
    w = inputs.expert_weights_f32(E, N, I, seed=M + I, weight_set=1)
    wq, ws = q.quant_weight_fp8(to_dev(w))
    rwq, rws = orc.quant_rows_fp8_f32(w)
    st = status()
    out = q.moe_gemm_w8a8(hq, None, wq, ws, al, to_dev(tw), M=M, top_k=top_k, BM=BM, a_layout=q.A_GROUPED,
                          out_layout=out_layout, a_scale_mode=q.SCALE_MX_1X32, a_sf=sf,
                          a_sf_padded_offsets=al128["padded_offsets"], d_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    eoff, poff = ref_al["expert_offsets"], ref_al["padded_offsets"]
    sf_row = np.empty(T, dtype=np.int64)
    for e in range(E):
        sf_row[eoff[e]:eoff[e + 1]] = poff[e] + np.arange(eoff[e + 1] - eoff[e])
    ref = orc.moe_gemm(a_kind=orc.A_FP8_MX, a=rq, a_sf=rsf, a_sf_row=sf_row, w_kind=orc.W_FP8, w=rwq, w_scale=rws,
                       topk_ids=ids, topk_w=tw, E=E, a_layout="grouped",
                       out_layout={1: "grouped", 2: "token_sum"}[out_layout])
    check(bf16_to_np_f32(out), ref)


@pytest.mark.parametrize("a_layout,out_layout", [(2, 0), (2, 2), (1, 1), (1, 2)])
@pytest.mark.parametrize("M,K,N,E,top_k,zipf,BM,rows", [
    (700, 8288, 272, 8, 2, None, 128, None),     # ~175 slots per expert: pairs with both halves; ragged K and N
    (300, 8192, 256, 4, 1, None, 256, None),     # ~75 slots per expert: every second half empty
    (1000, 8192, 3072, 8, 2, 1.2, 128, 24),      # Zipf skew, more tiles than SMs: 24 sampled tokens
    (150, 8192, 272, 16, 2, None, 128, None),    # five experts that receive nothing
])
def test_w8a8_two_half_tile(q, orc, a_layout, out_layout, M, K, N, E, top_k, zipf, BM, rows):
    """K >= 8192 with activation rows loaded by TMA (PADDED from
    quant_act_fp8_sorted, or GROUPED) runs the two-half tile: one weight pass
    serves two consecutive 128-slot blocks of an expert, one accumulator each,
    and the second is skipped when it lies outside the expert's region or holds
    only padding.  Whole outputs, or the rows of sampled tokens."""
    T = M * top_k
    seed = M + 13 * N
    ids = tw = None
    if E == 16:
        ids, tw = inputs.routing(M, 11, top_k, seed)
        ids = np.where(ids < 5, ids, ids + 5).astype(np.int32)   # experts 5..9 empty
    p = fp8_problem(q, orc, M, K, N, E, top_k, seed=seed, zipf=zipf, ids=ids, tw=tw)
    al = q.moe_align_block_size(to_dev(p["ids"]), E, BM)
    if a_layout == q.A_PADDED:
        a_in, s_in = q.quant_act_fp8_sorted(to_dev_bf16(p["a"]), al, top_k)
        ref_al = orc.moe_align(p["ids"], E, BM)
        n = ref_al["num_post_padded"]
        srt = ref_al["sorted_ids"][:n]
        valid = srt < T
        ra = np.zeros((a_in.shape[0], K), dtype=np.uint8)
        rs = np.zeros(a_in.shape[0], dtype=np.float32)
        ra[:n][valid] = p["raq"][srt[valid] // top_k]
        rs[:n][valid] = p["rsa"][srt[valid] // top_k]
        assert np.array_equal(a_in.cpu().numpy()[:n][valid], ra[:n][valid])
        ref_layout = "padded"
    else:
        order = np.empty(T, dtype=np.int64)
        order[orc.compact_row_of_slot(p["ids"], E)] = np.arange(T)
        src = order // top_k                               # compact row -> token row
        a_in, s_in = p["aq"][to_dev(src)].contiguous(), p["sa"][to_dev(src)].contiguous()
        ra, rs = p["raq"][src], p["rsa"][src]
        ref_layout = "grouped"
    st = status()
    out = q.moe_gemm_w8a8(a_in, s_in, p["wq"], p["ws"], al, to_dev(p["tw"]), M=M, top_k=top_k, BM=BM,
                          a_layout=a_layout, out_layout=out_layout, d_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    got = bf16_to_np_f32(out)
    args = dict(a_kind=orc.A_FP8_TOKEN, a=ra, a_scale=rs, w_kind=orc.W_FP8, w=p["rwq"], w_scale=p["rws"],
                topk_ids=p["ids"], topk_w=p["tw"], E=E, a_layout=ref_layout, BM=BM)
    if rows is None:
        ref = orc.moe_gemm(out_layout={0: "slot", 1: "grouped", 2: "token_sum"}[out_layout], **args)
        check(got, ref)
        return
    toks = np.random.default_rng(seed).choice(M, rows, replace=False)
    slots = (toks[:, None] * top_k + np.arange(top_k)[None, :]).ravel()
    per_slot = orc.moe_gemm(slots=slots, **args)
    if out_layout == q.OUT_TOKEN_SUM:
        check(got[toks], per_slot.reshape(rows, top_k, N).sum(axis=1))
    elif out_layout == q.OUT_GROUPED:
        check(got[orc.compact_row_of_slot(p["ids"], E)[slots]], per_slot)
    else:
        check(got[slots], per_slot)


@pytest.mark.parametrize("M,K,N,E,top_k,BM,out_layout", [(64, 4096, 256, 8, 2, 32, 0), (200, 272, 208, 8, 2, 64, 2),
                                                         (520, 256, 400, 8, 2, 128, 0), (90, 160, 272, 5, 3, 256, 2),
                                                         (33, 512, 128, 4, 2, 16, 0)])
def test_w8a16_padded_sorted_activations(q, orc, M, K, N, E, top_k, BM, out_layout):
    """gather_sorted_bf16 (exact copy of token rows to padded sorted positions)
    feeding the W8A16 GEMM's PADDED layout, with the decoupled int8 ring."""
    a = inputs.activations_bf16(M, K, seed=M + N + 7)
    w = inputs.expert_weights_f32(E, N, K, seed=M + N + 7)
    ids, tw = inputs.routing(M, E, top_k, seed=M + N + 7)
    wq, ws = q.quant_weight_int8(to_dev(w))
    rwq, rws = orc.quant_rows_int8_f32(w)
    al = q.moe_align_block_size(to_dev(ids), E, BM)
    ap = q.gather_sorted_bf16(to_dev_bf16(a), al, top_k)
    ref_al = orc.moe_align(ids, E, BM)
    n = ref_al["num_post_padded"]
    srt = ref_al["sorted_ids"][:n]
    valid = srt < M * top_k
    exp = np.zeros((n, K), dtype=np.uint16)
    exp[valid] = a[srt[valid] // top_k]
    got = ap.view(torch.int16).cpu().numpy().view(np.uint16)[:n]
    assert np.array_equal(got, exp)
    out = q.moe_gemm_w8a16(ap, wq, ws, al, to_dev(tw), M=M, top_k=top_k, BM=BM, a_layout=q.A_PADDED,
                           out_layout=out_layout)
    a_full = np.zeros((ap.shape[0], K), dtype=np.uint16)
    a_full[:n] = exp
    ref = orc.moe_gemm(a_kind=orc.A_BF16, a=a_full, w_kind=orc.W_INT8, w=rwq, w_scale=rws, topk_ids=ids, topk_w=tw,
                       E=E, a_layout="padded", BM=BM, out_layout={0: "slot", 2: "token_sum"}[out_layout])
    check(bf16_to_np_f32(out), ref)


@pytest.mark.parametrize("M,K,I,E,top_k,zipf,a_layout,routed", [
    (256, 256, 384, 8, 2, None, 2, False),     # padded A, ragged expert counts
    (150, 160, 256, 5, 3, None, 0, True),      # token-gather A, ragged K, routing weights
    (300, 512, 1024, 16, 2, None, 1, False),   # grouped A, five experts without slots
    (1024, 256, 2560, 8, 2, 1.2, 2, False),    # Zipf skew, more tiles than SMs
])
def test_gemm_silu_fp8_token_epilogue_bitexact(q, orc, M, K, I, E, top_k, zipf, a_layout, routed):
    """FP8 [gate | up] projection with SwiGLU in the GEMM epilogue (fp32 h and
    row maxima) and the per-token requantisation pass: codes and scales
    identical to the oracle's per-token SwiGLU quantisation of the bf16 output
    the same GEMM stores without the fused epilogue."""
    T, N = M * top_k, 2 * I
    seed = 7 * M + K + I
    if E == 16:
        ids, tw = inputs.routing(M, 11, top_k, seed)
        ids = np.where(ids < 5, ids, ids + 5).astype(np.int32)
        p = fp8_problem(q, orc, M, K, N, E, top_k, seed=seed, ids=ids, tw=tw)
    else:
        p = fp8_problem(q, orc, M, K, N, E, top_k, seed=seed, zipf=zipf)
    al = q.moe_align_block_size(to_dev(p["ids"]), E, 128)
    twd = to_dev(p["tw"]) if routed else None
    if a_layout == q.A_PADDED:
        a_in, s_in = q.quant_act_fp8_sorted(to_dev_bf16(p["a"]), al, top_k)
    elif a_layout == q.A_GROUPED:
        order = np.empty(T, dtype=np.int64)
        order[orc.compact_row_of_slot(p["ids"], E)] = np.arange(T)
        src = to_dev(order // top_k)
        a_in, s_in = p["aq"][src].contiguous(), p["sa"][src].contiguous()
    else:
        a_in, s_in = p["aq"], p["sa"]
    st = status()
    y = q.moe_gemm_w8a8(a_in, s_in, p["wq"], p["ws"], al, twd, M=M, top_k=top_k, BM=128, a_layout=a_layout,
                        out_layout=q.OUT_GROUPED, d_status=st)
    hq, hs = q.moe_gemm_w8a8_silu_fp8_token(a_in, s_in, p["wq"], p["ws"], al, M=M, top_k=top_k, a_layout=a_layout,
                                            topk_weights=twd, d_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    rq, rs = orc.silu_mul_quant_token(y.view(torch.int16).cpu().numpy().view(np.uint16))
    assert np.array_equal(hs.cpu().numpy(), rs)
    assert np.array_equal(hq.cpu().numpy(), rq)


def test_gemm_silu_fp8_token_rejects_before_launch(q, orc):
    """A host-side argument error (K % 16 != 0) returns before anything is
    launched: the scratch keeps its contents."""
    import quantized_moe_grouped_gb300 as qq
    M, K, N, E = 32, 40, 256, 2
    p = fp8_problem(q, orc, M, K, N, E, 2, seed=12)
    al = q.moe_align_block_size(to_dev(p["ids"]), E, 128)
    scratch = torch.full((M * 2 * (N // 2) + M * 2,), 3.0, device=dev())
    with pytest.raises(qq.QmoeError):
        q.moe_gemm_w8a8_silu_fp8_token(p["aq"], p["sa"], p["wq"], p["ws"], al, M=M, top_k=2, h_scratch=scratch)
    torch.cuda.synchronize()
    assert bool((scratch == 3.0).all())


@pytest.mark.parametrize("M,K,N,E,top_k,BM", [(40, 64, 48, 256, 8, 16), (40, 64, 48, 256, 8, 128),
                                              (3, 16, 16, 2, 1, 16), (5, 16, 32, 2, 2, 256)])
@pytest.mark.parametrize("a_layout,out_layout", [(0, 0), (1, 1), (0, 2)])
def test_w8a8_extreme_shapes(q, orc, M, K, N, E, top_k, BM, a_layout, out_layout):
    """The largest expert count (E = 256) with top_k = 8 (most experts get no
    slot or one), and the smallest N and K (16) the tiles accept."""
    p = fp8_problem(q, orc, M, K, N, E, top_k, seed=M * 31 + E + N)
    T = M * top_k
    al = q.moe_align_block_size(to_dev(p["ids"]), E, BM)
    if a_layout == q.A_GROUPED:
        order = np.empty(T, dtype=np.int64)
        order[orc.compact_row_of_slot(p["ids"], E)] = np.arange(T)
        src = order // top_k
        a_in, s_in = p["aq"][to_dev(src)].contiguous(), p["sa"][to_dev(src)].contiguous()
        ra, rs = p["raq"][src], p["rsa"][src]
    else:
        a_in, s_in, ra, rs = p["aq"], p["sa"], p["raq"], p["rsa"]
    st = status()
    out = q.moe_gemm_w8a8(a_in, s_in, p["wq"], p["ws"], al, to_dev(p["tw"]), M=M, top_k=top_k, BM=BM,
                          a_layout=a_layout, out_layout=out_layout, d_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    ref = orc.moe_gemm(a_kind=orc.A_FP8_TOKEN, a=ra, a_scale=rs, w_kind=orc.W_FP8, w=p["rwq"], w_scale=p["rws"],
                       topk_ids=p["ids"], topk_w=p["tw"], E=E, a_layout="grouped" if a_layout == 1 else "token",
                       out_layout={0: "slot", 1: "grouped", 2: "token_sum"}[out_layout])
    check(bf16_to_np_f32(out), ref)


def test_w8a16_extreme_shapes(q, orc):
    """W8A16 with E = 256 and top_k = 8."""
    M, K, N, E, top_k, BM = 40, 64, 48, 256, 8, 128
    a = inputs.activations_bf16(M, K, seed=77)
    w = inputs.expert_weights_f32(E, N, K, seed=77)
    ids, tw = inputs.routing(M, E, top_k, seed=77)
    wq, ws = q.quant_weight_int8(to_dev(w))
    rwq, rws = orc.quant_rows_int8_f32(w)
    al = q.moe_align_block_size(to_dev(ids), E, BM)
    st = status()
    out = q.moe_gemm_w8a16(to_dev_bf16(a), wq, ws, al, to_dev(tw), M=M, top_k=top_k, BM=BM, d_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    ref = orc.moe_gemm(a_kind=orc.A_BF16, a=a, w_kind=orc.W_INT8, w=rwq, w_scale=rws, topk_ids=ids, topk_w=tw, E=E)
    check(bf16_to_np_f32(out), ref)


def test_gemms_with_no_tokens(q, orc):
    """M = 0 (T = 0): every GEMM entry point returns OK and writes nothing."""
    K, N, E, top_k = 128, 256, 4, 2
    ids = np.zeros((0, top_k), dtype=np.int32)
    al = q.moe_align_block_size(to_dev(ids), E, 128)
    assert int(al["num_post_padded"].item()) == 0
    w = inputs.expert_weights_f32(E, N, K, seed=3)
    wq, ws = q.quant_weight_fp8(to_dev(w))
    wq8, ws8 = q.quant_weight_int8(to_dev(w))
    aq = torch.zeros(1, K, dtype=torch.uint8, device=dev())
    sa = torch.ones(1, dtype=torch.float32, device=dev())
    abf = torch.zeros(1, K, dtype=torch.bfloat16, device=dev())
    tw = torch.zeros(1, top_k, dtype=torch.float32, device=dev())
    sentinel = torch.full((4, N), 7.0, dtype=torch.bfloat16, device=dev())
    for layout in (q.OUT_SLOT, q.OUT_GROUPED, q.OUT_TOKEN_SUM):
        out = sentinel.clone()
        q.moe_gemm_w8a8(aq, sa, wq, ws, al, tw, M=0, top_k=top_k, BM=128, out_layout=layout, out=out)
        q.moe_gemm_w8a16(abf, wq8, ws8, al, tw, M=0, top_k=top_k, BM=128, out_layout=layout, out=out)
        torch.cuda.synchronize()
        assert torch.equal(out, sentinel)
    hq, hs = q.moe_gemm_w8a8_silu_fp8_token(aq, sa, wq, ws, al, M=0, top_k=top_k)
    fq, fsf = q.moe_gemm_w8a8_silu_mxfp8(aq, sa, wq, ws, al, M=0, top_k=top_k)
    torch.cuda.synchronize()
    assert hq.numel() == 0 and hs.numel() == 0 and fq.numel() == 0


@pytest.mark.parametrize("BM", [16, 128])
def test_w8a8_token_gather_single_token_deep_k(q, orc, BM):
    """One token (M=1, top_k=2) over several k-blocks with token-gathered
    activation rows: every gathered row is row 0."""
    M, K, N, E, top_k = 1, 512, 256, 4, 2
    p = fp8_problem(q, orc, M, K, N, E, top_k, seed=21)
    al = q.moe_align_block_size(to_dev(p["ids"]), E, BM)
    st = status()
    out = q.moe_gemm_w8a8(p["aq"], p["sa"], p["wq"], p["ws"], al, to_dev(p["tw"]), M=M, top_k=top_k, BM=BM,
                          d_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    ref = orc.moe_gemm(a_kind=orc.A_FP8_TOKEN, a=p["raq"], a_scale=p["rsa"], w_kind=orc.W_FP8, w=p["rwq"],
                       w_scale=p["rws"], topk_ids=p["ids"], topk_w=p["tw"], E=E)
    check(bf16_to_np_f32(out), ref)
