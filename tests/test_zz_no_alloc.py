"""The no-allocation FP8 TOKEN_SUM entry point (kept in its own file so that it
is collected last).

Some callers cannot call cudaMalloc -- runtimes whose memory pool forbids it on
the hot path, or plugins that are handed only their inputs and outputs -- so
they cannot pass the fp32 accumulation buffer the sum over top_k needs.
qmoe_moe_gemm_w8a8_token_sum_noalloc uses a fixed array inside the library
instead.  These tests call it through the C ABI, several times in a row on
different inputs (the array keeps the previous call's sums, so every later
call checks that it is cleared), and compare each result with the regular
entry point's and with the CPU oracle, within the GEMM tolerance used
everywhere else.  The calls cover token-gathered and grouped activation rows,
with and without routing weights, and the two-half tile of long-K problems."""
import ctypes

import numpy as np
import pytest
import torch

from quantized_moe_grouped_gb300 import inputs
from tests.gpu_util import dev, to_dev, to_dev_bf16

pytestmark = pytest.mark.gpu


def _problem(q, orc, M, K, N, E, top_k, BM, seed, grouped, weights):
    a = inputs.activations_bf16(M, K, seed)
    w = inputs.expert_weights_f32(E, N, K, seed)
    ids, tw = inputs.routing(M, E, top_k, seed)
    wq, ws = q.quant_weight_fp8(to_dev(w))
    aq, sa = q.quant_act_fp8(to_dev_bf16(a))
    if grouped:  # activation rows in expert-grouped compact order, one per slot
        pos = orc.compact_row_of_slot(ids, E)
        order = np.empty(M * top_k, dtype=np.int64)
        order[pos] = np.arange(M * top_k)
        rows = torch.from_numpy(order // top_k).to(dev())
        aq, sa = aq[rows].contiguous(), sa[rows].contiguous()
    al = q.moe_align_block_size(to_dev(ids), E, BM)
    return dict(aq=aq, sa=sa, wq=wq, ws=ws, al=al, ids=ids, tw=tw if weights else None,
                tw_dev=to_dev(tw) if weights else None, M=M, N=N, K=K, E=E, top_k=top_k, BM=BM,
                a_layout=q.A_GROUPED if grouped else q.A_TOKEN_GATHER)


def _args(q, p, out):
    args = q.GemmArgs()
    args.struct_size = ctypes.sizeof(q.GemmArgs)
    args.a, args.lda, args.a_scale = p["aq"].data_ptr(), p["K"], p["sa"].data_ptr()
    args.a_scale_mode, args.a_layout = q.SCALE_PER_TOKEN, p["a_layout"]
    args.w, args.w_scale = p["wq"].data_ptr(), p["ws"].data_ptr()
    al = p["al"]
    args.sorted_ids, args.expert_ids = al["sorted_ids"].data_ptr(), al["expert_ids"].data_ptr()
    args.num_post_padded = al["num_post_padded"].data_ptr()
    args.expert_offsets, args.padded_offsets = al["expert_offsets"].data_ptr(), al["padded_offsets"].data_ptr()
    args.topk_weights = p["tw_dev"].data_ptr() if p["tw_dev"] is not None else None
    args.out, args.out_layout = out.data_ptr(), q.OUT_TOKEN_SUM
    args.M, args.N, args.K, args.E, args.top_k, args.BM = p["M"], p["N"], p["K"], p["E"], p["top_k"], p["BM"]
    args.accum = None
    return args


# (M, K, N, E, top_k, BM, seed, grouped activation rows, routing weights)
CALLS = [
    (300, 256, 512, 8, 2, 64, 71, False, True),
    (150, 384, 640, 6, 3, 128, 72, False, True),
    (200, 512, 384, 8, 2, 128, 74, True, False),     # grouped rows, no routing weights
    (260, 8192, 256, 4, 2, 128, 75, True, True),     # K >= 8192: the two-half (256-slot) tile
]


def test_noalloc_token_sum_matches_regular_entry_point_and_oracle():
    import oracle
    import quantized_moe_grouped_gb300 as q
    lib = q.load_library()
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    for call, (M, K, N, E, top_k, BM, seed, grouped, weights) in enumerate(CALLS):
        p = _problem(q, oracle, M, K, N, E, top_k, BM, seed, grouped, weights)
        ref = q.moe_gemm_w8a8(p["aq"], p["sa"], p["wq"], p["ws"], p["al"], p["tw_dev"], M=M, top_k=top_k, BM=BM,
                              a_layout=p["a_layout"], out_layout=q.OUT_TOKEN_SUM)
        out = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device=dev())
        st = lib.qmoe_moe_gemm_w8a8_token_sum_noalloc(ctypes.byref(_args(q, p, out)), stream)
        assert st == q.QMOE_OK, f"call {call}: status {st}"
        torch.cuda.synchronize()
        got = out.float().cpu().numpy()
        want = ref.float().cpu().numpy().astype(np.float64)
        ok, ratio = oracle.gemm_tolerance_ok(got, want)
        assert ok, f"call {call}: against the regular entry point, worst |err|/bound = {ratio:.3f}"
        orc_ref = oracle.moe_gemm(a_kind=oracle.A_FP8_TOKEN, a=p["aq"].cpu().numpy(), a_scale=p["sa"].cpu().numpy(),
                                  w_kind=oracle.W_FP8, w=p["wq"].cpu().numpy(), w_scale=p["ws"].cpu().numpy(),
                                  topk_ids=p["ids"], topk_w=p["tw"], E=E,
                                  a_layout="grouped" if grouped else "token", out_layout="token_sum")
        ok, ratio = oracle.gemm_tolerance_ok(got, orc_ref)
        assert ok, f"call {call}: against the oracle, worst |err|/bound = {ratio:.3f}"


def test_noalloc_rejects_sizes_beyond_its_scratch():
    import oracle
    import quantized_moe_grouped_gb300 as q
    lib = q.load_library()
    p = _problem(q, oracle, 64, 128, 256, 8, 2, 32, 73, False, True)
    out = torch.empty(64, 256, dtype=torch.bfloat16, device=dev())
    args = _args(q, p, out)
    args.M = q.NOALLOC_ACCUM_MAX_ELEMS // 256 + 1                   # M*N one row past the scratch
    assert lib.qmoe_moe_gemm_w8a8_token_sum_noalloc(ctypes.byref(args), None) == q.QMOE_ERR_UNSUPPORTED
    big = (1 << 63) - 1
    for M, N in [(big, 256), (64, big), (big, big), (1 << 32, 1 << 32)]:  # products that overflow int64
        args.M, args.N = M, N
        assert lib.qmoe_moe_gemm_w8a8_token_sum_noalloc(ctypes.byref(args), None) == q.QMOE_ERR_UNSUPPORTED
    args.M, args.N, args.out_layout = 64, 256, q.OUT_SLOT              # only the TOKEN_SUM layout
    assert lib.qmoe_moe_gemm_w8a8_token_sum_noalloc(ctypes.byref(args), None) == q.QMOE_ERR_INVALID_ARG
