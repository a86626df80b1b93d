"""The C-ABI library builds, loads and exports every entry point that
include/qmoe.h declares (no compute calls: no GPU needed), and rejects
invalid arguments on the host before launching anything."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions():
    src = open(os.path.join(ROOT, "include", "qmoe.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(qmoe_[a-z0-9_]+)\s*\(", src)))


@pytest.fixture(scope="module")
def lib():
    from quantized_moe_grouped_gb300 import build
    build.build()
    import quantized_moe_grouped_gb300 as q
    return q.load_library()


def test_every_declared_symbol_is_exported(lib):
    names = declared_functions()
    assert len(names) >= 10
    for n in names:
        assert hasattr(lib, n), n
    import quantized_moe_grouped_gb300 as q
    assert sorted(q.EXPORTED) == names


def test_status_strings_and_sizes(lib):
    assert lib.qmoe_status_string(0) == b"ok"
    assert lib.qmoe_version() >= 1
    assert lib.qmoe_align_max_padded(128, 8, 16) == 128 + 8 * 15 + (16 - (128 + 8 * 15) % 16) % 16
    assert lib.qmoe_align_max_padded(0, 8, 128) == 8 * 127 + 1 - 1 + (128 - (8 * 127) % 128) % 128
    assert lib.qmoe_align_max_padded(-1, 8, 16) == -1


def test_host_validation_rejects_before_launch(lib):
    import quantized_moe_grouped_gb300 as q
    vp = ctypes.c_void_p
    # E out of range, BM out of range: invalid argument, nothing launched
    assert lib.qmoe_moe_align_block_size(vp(16), 4, 0, 16, vp(16), vp(16), vp(16), vp(16), vp(16), None, None) == 1
    assert lib.qmoe_moe_align_block_size(vp(16), 4, 8, 0, vp(16), vp(16), vp(16), vp(16), vp(16), None, None) == 1
    # GEMM: bad struct size, N not a multiple of 16, unsupported BM, MX scales
    args = q.GemmArgs()
    args.struct_size = 8
    assert lib.qmoe_moe_gemm_w8a8(ctypes.byref(args), None) == 1
    args.struct_size = ctypes.sizeof(q.GemmArgs)
    args.M, args.N, args.K, args.E, args.top_k, args.BM, args.lda = 4, 24, 64, 8, 2, 16, 64
    assert lib.qmoe_moe_gemm_w8a8(ctypes.byref(args), None) == 1
    args.N, args.BM = 32, 48
    assert lib.qmoe_moe_gemm_w8a8(ctypes.byref(args), None) == 2
    args.BM, args.a_scale_mode = 16, 1
    assert lib.qmoe_moe_gemm_w8a8(ctypes.byref(args), None) == 2
    # SwiGLU quant: I not a multiple of 8
    assert lib.qmoe_silu_mul_quant(vp(16), 4, 12, 24, 0, vp(16), vp(16), None, 0, None, None, 1, None, None) == 1
    # nothing to do is fine
    assert lib.qmoe_quant_act_fp8(None, 0, 64, 64, None, None, None) == 0


# Calls that each break one documented rule (the same calls with that one field
# valid pass every host check); every one must come back with the listed status
# from the host checks, before any CUDA call, so they are safe with or without
# a GPU.
_P = 1 << 20          # a 16-byte-aligned dummy address (never dereferenced on the host)
_U = (1 << 20) + 8    # 8-byte aligned only


def _gemm_args(q, **kw):
    a = q.GemmArgs()
    a.struct_size = ctypes.sizeof(q.GemmArgs)
    base = dict(a=_P, lda=256, a_scale=_P, a_scale_mode=0, a_layout=0, w=_P, w_scale=_P, sorted_ids=_P,
                expert_ids=_P, num_post_padded=_P, expert_offsets=_P, padded_offsets=_P, topk_weights=None,
                out=_P, out_layout=0, M=4, N=256, K=256, E=8, top_k=2, BM=128, d_status=None, accum=None,
                w_scale_mode=0, w_sf=None)
    base.update(kw)
    for k, v in base.items():
        setattr(a, k, v)
    return ctypes.byref(a)


_CASES = {
    "w8a8: weights not 16-byte aligned": (1, lambda L, q: L.qmoe_moe_gemm_w8a8(_gemm_args(q, w=_U), None)),
    "w8a8: no sorted_ids": (1, lambda L, q: L.qmoe_moe_gemm_w8a8(_gemm_args(q, sorted_ids=None), None)),
    "w8a8: top_k > E": (1, lambda L, q: L.qmoe_moe_gemm_w8a8(_gemm_args(q, top_k=9), None)),
    "w8a8: E > 256": (1, lambda L, q: L.qmoe_moe_gemm_w8a8(_gemm_args(q, E=257), None)),
    "w8a8: unknown out layout": (1, lambda L, q: L.qmoe_moe_gemm_w8a8(_gemm_args(q, out_layout=7), None)),
    "w8a8: token sum without accum": (1, lambda L, q: L.qmoe_moe_gemm_w8a8(_gemm_args(q, out_layout=2), None)),
    "w8a16: MX activation scales": (2, lambda L, q: L.qmoe_moe_gemm_w8a16(
        _gemm_args(q, a_scale=None, a_scale_mode=1), None)),
    "w8a16: lda < K": (1, lambda L, q: L.qmoe_moe_gemm_w8a16(_gemm_args(q, a_scale=None, lda=128), None)),
    "w8a16: activations not 16-byte aligned": (1, lambda L, q: L.qmoe_moe_gemm_w8a16(
        _gemm_args(q, a_scale=None, a=_U), None)),
    "w4a16: BM below 64": (2, lambda L, q: L.qmoe_moe_gemm_w4a16(_gemm_args(q, a_scale=None, BM=32), None)),
    "w4a16: K not a multiple of 128": (1, lambda L, q: L.qmoe_moe_gemm_w4a16(
        _gemm_args(q, a_scale=None, K=192, lda=192), None)),
    "fused per-token SwiGLU: K % 16 != 0": (1, lambda L, q: L.qmoe_moe_gemm_w8a8_silu_fp8_token(
        _gemm_args(q, K=40, lda=48, out=None, out_layout=1), ctypes.c_void_p(_P), ctypes.c_void_p(_P),
        ctypes.c_void_p(_P), None)),
    "fused per-token SwiGLU: slot output layout": (1, lambda L, q: L.qmoe_moe_gemm_w8a8_silu_fp8_token(
        _gemm_args(q, out=None, out_layout=0), ctypes.c_void_p(_P), ctypes.c_void_p(_P), ctypes.c_void_p(_P),
        None)),
    "fused MX SwiGLU: gate|up width not a multiple of 256": (1, lambda L, q: L.qmoe_moe_gemm_w8a8_silu_mxfp8(
        _gemm_args(q, N=272, out=None, out_layout=1), ctypes.c_void_p(_P), ctypes.c_void_p(_P), 16,
        ctypes.c_void_p(_P), None)),
    "router: top_k > E": (1, lambda L, q: L.qmoe_moe_router_topk(_P, 4, 8, 9, _P, _P, None)),
    "router: no experts": (1, lambda L, q: L.qmoe_moe_router_topk(_P, 4, 0, 1, _P, _P, None)),
    "align: BM above 1024": (1, lambda L, q: L.qmoe_moe_align_block_size(_P, 8, 8, 2048, _P, _P, _P, _P, _P,
                                                                          None, None)),
    "int4 weights: K not a multiple of 128": (1, lambda L, q: L.qmoe_quant_weight_int4(_P, 4, 192, _P, _P, None)),
    "int8 weights: no columns": (1, lambda L, q: L.qmoe_quant_weight_int8(_P, 4, 0, _P, _P, None)),
    "MXFP8 weights: K not a multiple of 32": (1, lambda L, q: L.qmoe_quant_weight_mxfp8(_P, 4, 48, _P, _P, 4,
                                                                                       None)),
    "MXFP8 rows: width not a multiple of 32": (1, lambda L, q: L.qmoe_quant_mxfp8(
        _P, 4, 48, 48, _P, _P, 4, _P, _P, 1, None, None)),
    "gather_sorted_bf16: lda < K": (1, lambda L, q: L.qmoe_gather_sorted_bf16(_P, 4, 256, 128, _P, _P, 2, 256,
                                                                              _P, None)),
    "quant_act_fp8: ldx < cols": (1, lambda L, q: L.qmoe_quant_act_fp8(_P, 4, 256, 128, _P, _P, None)),
    "silu_mul_quant: unknown mode": (1, lambda L, q: L.qmoe_silu_mul_quant(_P, 4, 64, 128, 5, _P, _P, None, 0,
                                                                           None, None, 1, None, None)),
    "srelu_quant: unknown mode": (1, lambda L, q: L.qmoe_srelu_quant(_P, 4, 64, 64, 5, _P, _P, None, 0, None,
                                                                     None, 1, None, None)),
}


@pytest.mark.parametrize("case", sorted(_CASES))
def test_host_validation_table(lib, case):
    import quantized_moe_grouped_gb300 as q
    want, call = _CASES[case]
    assert call(lib, q) == want
