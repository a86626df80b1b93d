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
