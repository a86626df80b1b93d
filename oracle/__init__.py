"""CPU oracle for the quantized MoE grouped GEMM path (test infrastructure).

Only the tests, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline
leg may import this package.  The library path never does: it shares no code
with it, and it fails loudly when its CUDA extension is missing rather than
route through anything here.

The arithmetic lives in ``qmoe_oracle.c`` (plain C, fp64 accumulation, fp32
where the quantisation decision is taken, contraction off).  This module builds
it with gcc and wraps it with ctypes + numpy; the only arithmetic done here is
placing rows of the per-slot GEMM result into the requested output layout and
summing the top_k slot rows of one token (a plain fp64 reduction).

Pins (tests/test_oracle_*.py): every function is checked against something
other than itself -- torch's e4m3/bf16 casts, a brute-force dense MoE and a
per-expert decomposition written independently in numpy, closed forms,
invariants, fp64 ``math.exp`` bounds and the worked scale-factor padding
example of the TransformerEngine MXFP8 GroupedLinear page.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "qmoe_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "liboracle.so")
_lock = threading.Lock()
_lib = None

A_FP8_TOKEN, A_FP8_MX, A_BF16 = 0, 1, 2
W_FP8, W_INT8, W_MX, W_INT4 = 0, 1, 2, 3


def build(force: bool = False) -> str:
    """Compile the oracle into oracle/_build/liboracle.so (gcc, OpenMP)."""
    os.makedirs(_BUILD, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=gnu11", "-ffp-contract=off", "-fno-fast-math", "-fopenmp",
           "-shared", "-fPIC", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _p(a):
    return a.ctypes.data_as(ctypes.c_void_p) if a is not None else None


def lib():
    global _lib
    with _lock:
        if _lib is None:
            path = build()
            L = ctypes.CDLL(path)
            i64, i32, vp = ctypes.c_int64, ctypes.c_int32, ctypes.c_void_p
            L.orc_num_threads.restype = ctypes.c_int
            L.orc_set_num_threads.argtypes = [ctypes.c_int]
            L.orc_bf16_from_f32.argtypes = [ctypes.c_float]
            L.orc_bf16_from_f32.restype = ctypes.c_uint16
            L.orc_bf16_to_f32.argtypes = [ctypes.c_uint16]
            L.orc_bf16_to_f32.restype = ctypes.c_float
            L.orc_e4m3_to_f64.argtypes = [ctypes.c_uint8]
            L.orc_e4m3_to_f64.restype = ctypes.c_double
            L.orc_e4m3_from_f32.argtypes = [ctypes.c_float]
            L.orc_e4m3_from_f32.restype = ctypes.c_uint8
            L.orc_e8m0_to_f64.argtypes = [ctypes.c_uint8]
            L.orc_e8m0_to_f64.restype = ctypes.c_double
            L.orc_mx_scale_exponent.argtypes = [ctypes.c_float]
            L.orc_mx_scale_exponent.restype = ctypes.c_int
            L.orc_mx_scale_exponent_array.argtypes = [vp, i64, vp]
            L.orc_bf16_from_f32_array.argtypes = [vp, i64, vp]
            L.orc_exp_f32.argtypes = [ctypes.c_float]
            L.orc_exp_f32.restype = ctypes.c_float
            L.orc_silu_mul_f32.argtypes = [ctypes.c_float, ctypes.c_float]
            L.orc_silu_mul_f32.restype = ctypes.c_float
            L.orc_moe_align.argtypes = [vp, i64, i32, i32, vp, i64, vp, i64, vp, vp, vp]
            L.orc_moe_align.restype = ctypes.c_int
            L.orc_quant_rows_fp8_f32.argtypes = [vp, i64, i64, i64, vp, vp]
            L.orc_quant_rows_fp8_bf16.argtypes = [vp, i64, i64, i64, vp, vp]
            L.orc_quant_rows_int8_f32.argtypes = [vp, i64, i64, i64, vp, vp]
            L.orc_silu_mul_quant_token.argtypes = [vp, i64, i64, i64, vp, vp]
            L.orc_silu_mul_quant_mx.argtypes = [vp, i64, i64, i64, vp, vp, i32, vp, vp, i64]
            L.orc_srelu_quant_token.argtypes = [vp, i64, i64, i64, vp, vp]
            L.orc_srelu_quant_mx.argtypes = [vp, i64, i64, i64, vp, vp, i32, vp, vp, i64]
            L.orc_quant_mxfp8_rows.argtypes = [vp, i64, i64, i64, vp, vp, i32, vp, vp, i64]
            L.orc_quant_mxfp8_cols_bf16.argtypes = [vp, i64, i64, i64, vp, vp, i64, i64]
            L.orc_quant_rows_mxfp8_f32.argtypes = [vp, i64, i64, vp, vp, i64]
            L.orc_mx_weight_sf_tiled.argtypes = [vp, i64, i64, i64, i64, vp]
            L.orc_quant_rows_int4_f32.argtypes = [vp, i64, i64, vp, vp]
            L.orc_router_topk.argtypes = [vp, i64, i32, i32, vp, vp]
            L.orc_srelu_f32.argtypes = [ctypes.c_float]
            L.orc_srelu_f32.restype = ctypes.c_float
            L.orc_e4m3_from_f32_array.argtypes = [vp, i64, vp]
            L.orc_exp_f32_array.argtypes = [vp, i64, vp]
            L.orc_silu_mul_f32_array.argtypes = [vp, vp, i64, vp]
            L.orc_moe_gemm.argtypes = [ctypes.c_int, vp, i64, vp, vp, i64, vp,
                                       ctypes.c_int, vp, vp, vp, i64, vp, vp, vp, i64, vp, i64, i64, vp]
            _lib = L
    return _lib


def num_threads() -> int:
    return int(lib().orc_num_threads())


def set_num_threads(n: int) -> None:
    lib().orc_set_num_threads(int(n))


# ---------------------------------------------------------------- formats ---
def bf16_from_f32(x) -> np.ndarray:
    f = lib().orc_bf16_from_f32
    x = np.asarray(x, dtype=np.float32).ravel()
    return np.array([f(float(v)) for v in x], dtype=np.uint16)


def bf16_from_f32_array(x: np.ndarray) -> np.ndarray:
    x = np.ascontiguousarray(x, dtype=np.float32)
    h = np.empty(x.shape, dtype=np.uint16)
    lib().orc_bf16_from_f32_array(_p(x), x.size, _p(h))
    return h


def bf16_to_f32(b) -> np.ndarray:
    f = lib().orc_bf16_to_f32
    b = np.asarray(b, dtype=np.uint16).ravel()
    return np.array([f(int(v)) for v in b], dtype=np.float32)


def e4m3_to_f64(b) -> np.ndarray:
    f = lib().orc_e4m3_to_f64
    return np.array([f(int(v)) for v in np.asarray(b, dtype=np.uint8).ravel()], dtype=np.float64)


def e4m3_from_f32(x) -> np.ndarray:
    f = lib().orc_e4m3_from_f32
    return np.array([f(float(v)) for v in np.asarray(x, dtype=np.float32).ravel()], dtype=np.uint8)


def e4m3_from_f32_array(x: np.ndarray) -> np.ndarray:
    x = np.ascontiguousarray(x, dtype=np.float32)
    q = np.empty(x.shape, dtype=np.uint8)
    lib().orc_e4m3_from_f32_array(_p(x), x.size, _p(q))
    return q


def exp_f32_array(x: np.ndarray) -> np.ndarray:
    x = np.ascontiguousarray(x, dtype=np.float32)
    y = np.empty(x.shape, dtype=np.float32)
    lib().orc_exp_f32_array(_p(x), x.size, _p(y))
    return y


def silu_mul_f32_array(g: np.ndarray, u: np.ndarray) -> np.ndarray:
    g = np.ascontiguousarray(g, dtype=np.float32)
    u = np.ascontiguousarray(u, dtype=np.float32)
    h = np.empty(g.shape, dtype=np.float32)
    lib().orc_silu_mul_f32_array(_p(g), _p(u), g.size, _p(h))
    return h


def e8m0_to_f64(b) -> np.ndarray:
    f = lib().orc_e8m0_to_f64
    return np.array([f(int(v)) for v in np.asarray(b, dtype=np.uint8).ravel()], dtype=np.float64)


def mx_scale_exponent(a: float) -> int:
    return int(lib().orc_mx_scale_exponent(float(a)))


def mx_scale_exponent_array(a: np.ndarray) -> np.ndarray:
    a = np.ascontiguousarray(a, dtype=np.float32)
    e = np.empty(a.shape, dtype=np.int32)
    lib().orc_mx_scale_exponent_array(_p(a), a.size, _p(e))
    return e


def exp_f32(x) -> np.ndarray:
    f = lib().orc_exp_f32
    return np.array([f(float(v)) for v in np.asarray(x, dtype=np.float32).ravel()], dtype=np.float32)


def silu_mul_f32(g, u) -> np.ndarray:
    f = lib().orc_silu_mul_f32
    g = np.asarray(g, dtype=np.float32).ravel()
    u = np.asarray(u, dtype=np.float32).ravel()
    return np.array([f(float(a), float(b)) for a, b in zip(g, u)], dtype=np.float32)


# ------------------------------------------------------------------ align ---
def align_max_padded(T: int, E: int, BM: int) -> int:
    return int(T) + int(E) * (int(BM) - 1)


def moe_align(topk_ids: np.ndarray, E: int, BM: int):
    ids = np.ascontiguousarray(topk_ids, dtype=np.int32).ravel()
    T = ids.size
    cap = align_max_padded(T, E, BM)
    cap = (cap + BM - 1) // BM * BM
    sorted_ids = np.empty(cap, dtype=np.int32)
    expert_ids = np.empty(cap // BM, dtype=np.int32)
    npp = np.zeros(1, dtype=np.int32)
    eoff = np.zeros(E + 1, dtype=np.int32)
    poff = np.zeros(E + 1, dtype=np.int32)
    bad = lib().orc_moe_align(_p(ids), T, E, BM, _p(sorted_ids), cap, _p(expert_ids), cap // BM,
                              _p(npp), _p(eoff), _p(poff))
    return dict(sorted_ids=sorted_ids, expert_ids=expert_ids, num_post_padded=int(npp[0]),
                expert_offsets=eoff, padded_offsets=poff, invalid=bool(bad))


# ------------------------------------------------------------- quantisers ---
def quant_rows_fp8_bf16(x_bits: np.ndarray):
    x = np.ascontiguousarray(x_bits, dtype=np.uint16)
    R, C = x.shape
    q = np.empty((R, C), dtype=np.uint8)
    s = np.empty(R, dtype=np.float32)
    lib().orc_quant_rows_fp8_bf16(_p(x), R, C, C, _p(q), _p(s))
    return q, s


def quant_rows_fp8_f32(x: np.ndarray):
    x = np.ascontiguousarray(x, dtype=np.float32)
    shp = x.shape
    x2 = x.reshape(-1, shp[-1])
    R, C = x2.shape
    q = np.empty((R, C), dtype=np.uint8)
    s = np.empty(R, dtype=np.float32)
    lib().orc_quant_rows_fp8_f32(_p(x2), R, C, C, _p(q), _p(s))
    return q.reshape(shp), s.reshape(shp[:-1])


def quant_rows_int8_f32(x: np.ndarray):
    x = np.ascontiguousarray(x, dtype=np.float32)
    shp = x.shape
    x2 = x.reshape(-1, shp[-1])
    R, C = x2.shape
    q = np.empty((R, C), dtype=np.int8)
    s = np.empty(R, dtype=np.float32)
    lib().orc_quant_rows_int8_f32(_p(x2), R, C, C, _p(q), _p(s))
    return q.reshape(shp), s.reshape(shp[:-1])


def silu_mul_quant_token(y_bits: np.ndarray):
    y = np.ascontiguousarray(y_bits, dtype=np.uint16)
    R, C2 = y.shape
    I = C2 // 2
    q = np.empty((R, I), dtype=np.uint8)
    s = np.empty(R, dtype=np.float32)
    lib().orc_silu_mul_quant_token(_p(y), R, I, C2, _p(q), _p(s))
    return q, s


def mx_sf_ld(I: int) -> int:
    """Row length of the rowwise MX scale matrix: I/32 rounded up to 4."""
    return (I // 32 + 3) // 4 * 4


def silu_mul_quant_mx(y_bits: np.ndarray, expert_offsets: np.ndarray, sf_padded_offsets: np.ndarray):
    y = np.ascontiguousarray(y_bits, dtype=np.uint16)
    R, C2 = y.shape
    I = C2 // 2
    E = len(expert_offsets) - 1
    eoff = np.ascontiguousarray(expert_offsets, dtype=np.int32)
    soff = np.ascontiguousarray(sf_padded_offsets, dtype=np.int32)
    ld = mx_sf_ld(I)
    q = np.zeros((R, I), dtype=np.uint8)
    sf = np.zeros((int(soff[E]), ld), dtype=np.uint8)
    lib().orc_silu_mul_quant_mx(_p(y), R, I, C2, _p(eoff), _p(soff), E, _p(q), _p(sf), ld)
    return q, sf


def srelu_f32(x) -> np.ndarray:
    f = lib().orc_srelu_f32
    return np.array([f(float(v)) for v in np.asarray(x, dtype=np.float32).ravel()], dtype=np.float32)


def srelu_quant_token(y_bits: np.ndarray):
    y = np.ascontiguousarray(y_bits, dtype=np.uint16)
    R, I = y.shape
    q = np.empty((R, I), dtype=np.uint8)
    s = np.empty(R, dtype=np.float32)
    lib().orc_srelu_quant_token(_p(y), R, I, I, _p(q), _p(s))
    return q, s


def srelu_quant_mx(y_bits: np.ndarray, expert_offsets: np.ndarray, sf_padded_offsets: np.ndarray):
    y = np.ascontiguousarray(y_bits, dtype=np.uint16)
    R, I = y.shape
    E = len(expert_offsets) - 1
    eoff = np.ascontiguousarray(expert_offsets, dtype=np.int32)
    soff = np.ascontiguousarray(sf_padded_offsets, dtype=np.int32)
    ld = mx_sf_ld(I)
    q = np.zeros((R, I), dtype=np.uint8)
    sf = np.zeros((int(soff[E]), ld), dtype=np.uint8)
    lib().orc_srelu_quant_mx(_p(y), R, I, I, _p(eoff), _p(soff), E, _p(q), _p(sf), ld)
    return q, sf


def quant_mxfp8_rows(y_bits: np.ndarray, expert_offsets: np.ndarray, sf_padded_offsets: np.ndarray):
    """bf16 rows [R, I] -> e4m3 [R, I] + E8M0 rowwise factors padded per expert (no activation)."""
    y = np.ascontiguousarray(y_bits, dtype=np.uint16)
    R, I = y.shape
    E = len(expert_offsets) - 1
    eoff = np.ascontiguousarray(expert_offsets, dtype=np.int32)
    soff = np.ascontiguousarray(sf_padded_offsets, dtype=np.int32)
    ld = mx_sf_ld(I)
    q = np.zeros((R, I), dtype=np.uint8)
    sf = np.zeros((int(soff[E]), ld), dtype=np.uint8)
    lib().orc_quant_mxfp8_rows(_p(y), R, I, I, _p(eoff), _p(soff), E, _p(q), _p(sf), ld)
    return q, sf


def mx_colwise_sf_shape(R: int, C: int):
    """Columnwise factor shape: ceil(R/32) blocks padded to a multiple of 4, C padded to 128."""
    return ((R + 31) // 32 + 3) // 4 * 4, (C + 127) // 128 * 128


def quant_mxfp8_cols(x_bits: np.ndarray):
    """bf16 [R, C] -> e4m3 [R, C] quantised in 32x1 column blocks + E8M0 factors."""
    x = np.ascontiguousarray(x_bits, dtype=np.uint16)
    R, C = x.shape
    sr, sc = mx_colwise_sf_shape(R, C)
    q = np.zeros((R, C), dtype=np.uint8)
    sf = np.zeros((sr, sc), dtype=np.uint8)
    lib().orc_quant_mxfp8_cols_bf16(_p(x), R, C, C, _p(q), _p(sf), sr, sc)
    return q, sf


def quant_rows_mxfp8_f32(w: np.ndarray):
    """fp32 [..., C] rows -> e4m3 codes (same shape) + E8M0 [rows, mx_sf_ld(C)]."""
    w = np.ascontiguousarray(w, dtype=np.float32)
    C = w.shape[-1]
    R = w.size // C
    ld = mx_sf_ld(C)
    q = np.zeros(w.shape, dtype=np.uint8)
    sf = np.zeros((R, ld), dtype=np.uint8)
    lib().orc_quant_rows_mxfp8_f32(_p(w), R, C, _p(q), _p(sf), ld)
    return q, sf


def quant_rows_int4_f32(w: np.ndarray):
    """fp32 [..., K] rows -> (packed int4 uint8 [..., K/2], fp32 group scales [..., K/128])."""
    w = np.ascontiguousarray(w, dtype=np.float32)
    K = w.shape[-1]
    R = w.size // K
    q = np.zeros(w.shape[:-1] + (K // 2,), dtype=np.uint8)
    s = np.zeros(w.shape[:-1] + (K // 128,), dtype=np.float32)
    lib().orc_quant_rows_int4_f32(_p(w), R, K, _p(q), _p(s))
    return q, s


def mx_weight_sf_tiled(sf: np.ndarray, E: int, N: int, K: int):
    """E8M0 weight factors [E*N, ld] -> the GEMM's tiled blocks (uint8, flat)."""
    sf = np.ascontiguousarray(sf, dtype=np.uint8)
    nb, kb = (N + 255) // 256, (K + 127) // 128
    out = np.zeros(E * nb * kb * 1024, dtype=np.uint8)
    lib().orc_mx_weight_sf_tiled(_p(sf), E, N, K, sf.shape[-1], _p(out))
    return out


def router_topk(logits: np.ndarray, k: int):
    """fp32 logits [M, E] -> (topk_ids int32 [M, k], topk_weights fp32 [M, k])."""
    l = np.ascontiguousarray(logits, dtype=np.float32)
    M, E = l.shape
    ids = np.empty((M, k), dtype=np.int32)
    w = np.empty((M, k), dtype=np.float32)
    lib().orc_router_topk(_p(l), M, E, k, _p(ids), _p(w))
    return ids, w


# ------------------------------------------------------------------- GEMM ---
def moe_gemm_slots(*, a_kind, a, a_scale=None, a_sf=None, a_sf_row=None, w_kind, w, w_scale,
                   topk_ids, topk_w, a_row, slots, N, K, w_sf=None):
    """Per-slot result [len(slots), N] in fp64 (see orc_moe_gemm)."""
    a = np.ascontiguousarray(a)
    lda = a.shape[-1]
    ids = np.ascontiguousarray(topk_ids, dtype=np.int32).ravel()
    tw = None if topk_w is None else np.ascontiguousarray(topk_w, dtype=np.float32).ravel()
    slots = np.ascontiguousarray(slots, dtype=np.int64)
    a_row = np.ascontiguousarray(a_row, dtype=np.int64)
    a_scale = None if a_scale is None else np.ascontiguousarray(a_scale, dtype=np.float32)
    a_sf = None if a_sf is None else np.ascontiguousarray(a_sf, dtype=np.uint8)
    a_sf_ld = 0 if a_sf is None else a_sf.shape[-1]
    a_sf_row = None if a_sf_row is None else np.ascontiguousarray(a_sf_row, dtype=np.int64)
    w = np.ascontiguousarray(w)
    w_scale = None if w_scale is None else np.ascontiguousarray(w_scale, dtype=np.float32)
    w_sf = None if w_sf is None else np.ascontiguousarray(w_sf, dtype=np.uint8)
    w_sf_ld = 0 if w_sf is None else w_sf.shape[-1]
    out = np.empty((slots.size, N), dtype=np.float64)
    lib().orc_moe_gemm(int(a_kind), _p(a), lda, _p(a_scale), _p(a_sf), a_sf_ld, _p(a_sf_row),
                       int(w_kind), _p(w), _p(w_scale), _p(w_sf), w_sf_ld, _p(ids), _p(tw),
                       _p(slots), slots.size, _p(a_row), int(N), int(K), _p(out))
    return out


def compact_row_of_slot(topk_ids: np.ndarray, E: int) -> np.ndarray:
    """Position of every slot in the expert-grouped compact order (from the
    oracle's own align with BM = 1, which is the stable sort by expert)."""
    ids = np.asarray(topk_ids, dtype=np.int32).ravel()
    al = moe_align(ids, E, 1)
    pos = np.empty(ids.size, dtype=np.int64)
    n = al["num_post_padded"]
    pos[al["sorted_ids"][:n]] = np.arange(n, dtype=np.int64)
    return pos


def padded_row_of_slot(topk_ids: np.ndarray, E: int, BM: int) -> np.ndarray:
    """Padded sorted position of every slot (the oracle's own align with BM)."""
    ids = np.asarray(topk_ids, dtype=np.int32).ravel()
    al = moe_align(ids, E, BM)
    pos = np.empty(ids.size, dtype=np.int64)
    srt = al["sorted_ids"][: al["num_post_padded"]]
    valid = srt < ids.size
    pos[srt[valid]] = np.nonzero(valid)[0]
    return pos


def moe_gemm(*, a_kind, a, a_scale=None, a_sf=None, a_sf_row=None, w_kind, w, w_scale,
             topk_ids, topk_w, E, a_layout="token", out_layout="slot", slots=None, BM=None, w_sf=None):
    """Whole grouped GEMM in fp64 with the requested layouts.

    a_layout "token": A row of slot s is s // top_k; "grouped": A row of slot
    s is its compact grouped position; "padded": A row of slot s is its padded
    sorted position for tile size BM.  out_layout "slot": [T, N] indexed by
    s; "grouped": [T, N] indexed by compact position; "token_sum": [M, N], the
    sum over j of slot rows m*top_k + j.  With ``slots`` given, only those
    slots are computed and the per-slot rows [len(slots), N] are returned.
    """
    ids = np.asarray(topk_ids, dtype=np.int32)
    M, top_k = ids.shape
    T = M * top_k
    N = w.shape[1]
    K = w.shape[2] * (2 if w_kind == W_INT4 else 1)   # packed int4: two values per byte
    pos = compact_row_of_slot(ids, E)
    if a_layout == "token":
        a_row = np.arange(T, dtype=np.int64) // top_k
    elif a_layout == "padded":
        a_row = padded_row_of_slot(ids, E, BM)
    else:
        a_row = pos
    sl = np.arange(T, dtype=np.int64) if slots is None else np.asarray(slots, dtype=np.int64)
    res = moe_gemm_slots(a_kind=a_kind, a=a, a_scale=a_scale, a_sf=a_sf, a_sf_row=a_sf_row,
                         w_kind=w_kind, w=w, w_scale=w_scale, topk_ids=ids, topk_w=topk_w,
                         a_row=a_row, slots=sl, N=N, K=K, w_sf=w_sf)
    if slots is not None:
        return res
    if out_layout == "slot":
        return res
    if out_layout == "grouped":
        out = np.empty_like(res)
        out[pos] = res
        return out
    if out_layout == "token_sum":
        return res.reshape(M, top_k, N).sum(axis=1)
    raise ValueError(out_layout)


def gemm_tolerance_ok(gpu: np.ndarray, ref: np.ndarray, rms: float | None = None,
                      rel: float = 8e-3, abs_rms: float = 1e-2):
    """|gpu - ref| <= rel*|ref| + abs_rms*rms(ref) elementwise; returns (ok, worst ratio)."""
    ref = np.asarray(ref, dtype=np.float64)
    gpu = np.asarray(gpu, dtype=np.float64)
    if ref.size == 0:
        return True, 0.0
    if rms is None:
        rms = float(np.sqrt(np.mean(ref * ref)))
    bound = rel * np.abs(ref) + abs_rms * rms
    err = np.abs(gpu - ref)
    ratio = float(np.max(err / np.maximum(bound, 1e-300)))
    return bool(np.all(err <= bound)), ratio
