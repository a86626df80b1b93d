"""Python binding of libqmoe.so (the quantized MoE grouped GEMM path on GB300).

Argument marshalling only: every function here takes torch CUDA tensors,
checks dtypes/devices, passes raw device pointers and the current CUDA stream
to the C ABI declared in include/qmoe.h and raises on a non-OK status.  All
arithmetic runs in the library's kernels; there is no CPU or PyTorch fallback,
and a missing library is an ImportError-like failure at first use.

Names follow the C entry points (without the ``qmoe_`` prefix).
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libqmoe.so")
_lib = None
_lock = threading.Lock()

QMOE_OK, QMOE_ERR_INVALID_ARG, QMOE_ERR_UNSUPPORTED, QMOE_ERR_CUDA = 0, 1, 2, 3
DEV_INVALID_EXPERT, DEV_TIMEOUT = 1, 2
SCALE_PER_TOKEN, SCALE_MX_1X32 = 0, 1
A_TOKEN_GATHER, A_GROUPED, A_PADDED = 0, 1, 2
OUT_SLOT, OUT_GROUPED, OUT_TOKEN_SUM = 0, 1, 2

EXPORTED = (
    "qmoe_status_string", "qmoe_version", "qmoe_align_max_padded", "qmoe_moe_align_block_size",
    "qmoe_quant_act_fp8", "qmoe_quant_act_fp8_sorted", "qmoe_moe_align_quant_fp8", "qmoe_moe_router_topk", "qmoe_moe_route_align_quant_fp8", "qmoe_gather_sorted_bf16", "qmoe_quant_weight_fp8", "qmoe_quant_weight_int8", "qmoe_moe_gemm_w8a8",
    "qmoe_moe_gemm_w8a16", "qmoe_silu_mul_quant", "qmoe_srelu_quant", "qmoe_debug_e4m3_encode", "qmoe_debug_int8_to_bf16",
    "qmoe_debug_silu_mul", "qmoe_debug_div_by_scale", "qmoe_debug_quant_by_scale", "qmoe_debug_wait_timeout",
    "qmoe_moe_gemm_w8a8_token_sum_noalloc", "qmoe_quant_weight_mxfp8", "qmoe_quant_mxfp8", "qmoe_quant_mxfp8_colwise",
    "qmoe_mx_weight_sf_tiled_bytes", "qmoe_mx_weight_sf_tiled", "qmoe_quant_weight_int4", "qmoe_moe_gemm_w4a16",
    "qmoe_moe_gemm_w8a8_silu_mxfp8", "qmoe_moe_gemm_w8a8_silu_fp8_token", "qmoe_debug_rcp_ge1",
    "qmoe_debug_moe_gemm_tile",
)
TILE_AUTO, TILE_ONE_SM, TILE_PAIR = 0, 1, 2
NOALLOC_ACCUM_MAX_ELEMS = 4 << 20


class QmoeError(RuntimeError):
    pass


class GemmArgs(ctypes.Structure):
    _fields_ = [
        ("struct_size", ctypes.c_size_t),
        ("a", ctypes.c_void_p), ("lda", ctypes.c_int64), ("a_scale", ctypes.c_void_p),
        ("a_scale_mode", ctypes.c_int32), ("a_sf", ctypes.c_void_p), ("a_sf_ld", ctypes.c_int64),
        ("a_sf_padded_offsets", ctypes.c_void_p), ("a_layout", ctypes.c_int32),
        ("w", ctypes.c_void_p), ("w_scale", ctypes.c_void_p),
        ("sorted_ids", ctypes.c_void_p), ("expert_ids", ctypes.c_void_p), ("num_post_padded", ctypes.c_void_p),
        ("expert_offsets", ctypes.c_void_p), ("padded_offsets", ctypes.c_void_p),
        ("topk_weights", ctypes.c_void_p),
        ("out", ctypes.c_void_p), ("out_layout", ctypes.c_int32),
        ("M", ctypes.c_int64), ("N", ctypes.c_int64), ("K", ctypes.c_int64),
        ("E", ctypes.c_int32), ("top_k", ctypes.c_int32), ("BM", ctypes.c_int32),
        ("d_status", ctypes.c_void_p),
        ("accum", ctypes.c_void_p),
        ("w_scale_mode", ctypes.c_int32), ("w_sf", ctypes.c_void_p),
    ]


def load_library(path: str | None = None):
    """Load libqmoe.so (built in-tree by quantized_moe_grouped_gb300.build)."""
    global _lib
    with _lock:
        if _lib is None:
            p = path or LIB_PATH
            if not os.path.exists(p):
                raise QmoeError(f"libqmoe.so not found at {p}; run `python -m quantized_moe_grouped_gb300.build`")
            L = ctypes.CDLL(p)
            vp, i64, i32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32
            st = ctypes.c_int
            L.qmoe_status_string.argtypes = [st]
            L.qmoe_status_string.restype = ctypes.c_char_p
            L.qmoe_version.restype = ctypes.c_int
            L.qmoe_align_max_padded.argtypes = [i64, i32, i32]
            L.qmoe_align_max_padded.restype = i64
            L.qmoe_moe_align_block_size.argtypes = [vp, i64, i32, i32, vp, vp, vp, vp, vp, vp, vp]
            L.qmoe_quant_act_fp8.argtypes = [vp, i64, i64, i64, vp, vp, vp]
            L.qmoe_quant_act_fp8_sorted.argtypes = [vp, i64, i64, i64, vp, vp, i32, i64, vp, vp, vp]
            L.qmoe_moe_align_quant_fp8.argtypes = [vp, i64, i64, i64, vp, i32, i32, i32, vp, vp, vp, vp, vp, vp,
                                                   vp, vp, vp]
            L.qmoe_moe_router_topk.argtypes = [vp, i64, i32, i32, vp, vp, vp]
            L.qmoe_quant_weight_mxfp8.argtypes = [vp, i64, i64, vp, vp, i64, vp]
            L.qmoe_quant_mxfp8.argtypes = [vp, i64, i64, i64, vp, vp, i64, vp, vp, i32, vp, vp]
            L.qmoe_quant_mxfp8_colwise.argtypes = [vp, i64, i64, i64, vp, vp, i64, i64, vp]
            L.qmoe_mx_weight_sf_tiled_bytes.argtypes = [i64, i64, i64]
            L.qmoe_mx_weight_sf_tiled_bytes.restype = i64
            L.qmoe_mx_weight_sf_tiled.argtypes = [vp, i64, i64, i64, i64, vp, vp]
            L.qmoe_quant_weight_int4.argtypes = [vp, i64, i64, vp, vp, vp]
            L.qmoe_moe_route_align_quant_fp8.argtypes = [vp, vp, i64, i64, i64, i32, i32, i32, vp, vp, vp, vp, vp,
                                                         vp, vp, vp, vp, vp, vp]
            L.qmoe_gather_sorted_bf16.argtypes = [vp, i64, i64, i64, vp, vp, i32, i64, vp, vp]
            L.qmoe_quant_weight_fp8.argtypes = [vp, i64, i64, vp, vp, vp]
            L.qmoe_quant_weight_int8.argtypes = [vp, i64, i64, vp, vp, vp]
            L.qmoe_moe_gemm_w8a8.argtypes = [ctypes.POINTER(GemmArgs), vp]
            L.qmoe_moe_gemm_w8a16.argtypes = [ctypes.POINTER(GemmArgs), vp]
            L.qmoe_moe_gemm_w8a8_token_sum_noalloc.argtypes = [ctypes.POINTER(GemmArgs), vp]
            L.qmoe_moe_gemm_w8a8_silu_mxfp8.argtypes = [ctypes.POINTER(GemmArgs), vp, vp, i64, vp, vp]
            L.qmoe_moe_gemm_w8a8_silu_fp8_token.argtypes = [ctypes.POINTER(GemmArgs), vp, vp, vp, vp]
            L.qmoe_silu_mul_quant.argtypes = [vp, i64, i64, i64, i32, vp, vp, vp, i64, vp, vp, i32, vp, vp]
            L.qmoe_srelu_quant.argtypes = [vp, i64, i64, i64, i32, vp, vp, vp, i64, vp, vp, i32, vp, vp]
            L.qmoe_debug_e4m3_encode.argtypes = [vp, vp, i64, vp]
            L.qmoe_debug_int8_to_bf16.argtypes = [vp, vp, i64, vp]
            L.qmoe_debug_silu_mul.argtypes = [vp, vp, vp, i64, vp]
            L.qmoe_debug_div_by_scale.argtypes = [vp, ctypes.c_float, vp, i64, vp]
            L.qmoe_debug_quant_by_scale.argtypes = [vp, ctypes.c_float, vp, i64, vp]
            L.qmoe_debug_rcp_ge1.argtypes = [vp, vp, i64, vp]
            L.qmoe_debug_wait_timeout.argtypes = [vp, i64, vp]
            L.qmoe_debug_moe_gemm_tile.argtypes = [ctypes.POINTER(GemmArgs), i32, i32, vp]
            for name in EXPORTED:
                if name not in ("qmoe_status_string", "qmoe_version", "qmoe_align_max_padded"):
                    getattr(L, name).restype = st
            _lib = L
    return _lib


def _check(status: int, what: str) -> None:
    if status != QMOE_OK:
        msg = load_library().qmoe_status_string(status).decode()
        raise QmoeError(f"{what}: {msg} (status {status})")


def _ptr(t: torch.Tensor | None):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream: torch.cuda.Stream | None = None):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _empty(*size, dtype, device) -> torch.Tensor:
    """Every output and scratch tensor the binding allocates comes from here
    (uninitialised device memory, like torch.empty)."""
    return torch.empty(*size, dtype=dtype, device=device)


def _need(t: torch.Tensor, dtype, name: str):
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise QmoeError(f"{name} must be a CUDA tensor")
    if dtype is not None and t.dtype != dtype:
        raise QmoeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise QmoeError(f"{name} must be contiguous")


# ----------------------------------------------------------------- align ---
def align_max_padded(T: int, E: int, BM: int) -> int:
    """Capacity of sorted_ids for T slots, E experts and tile BM (qmoe_align_max_padded):
    T + E*(BM-1) rounded up to a multiple of BM."""
    return int(load_library().qmoe_align_max_padded(int(T), int(E), int(BM)))


def alloc_align_outputs(T: int, E: int, BM: int, device="cuda") -> dict:
    """Empty device buffers for moe_align_block_size: sorted_ids, expert_ids,
    num_post_padded, expert_offsets, padded_offsets."""
    cap = align_max_padded(T, E, BM)
    i32 = torch.int32
    return dict(sorted_ids=_empty(cap, dtype=i32, device=device),
                expert_ids=_empty(cap // BM, dtype=i32, device=device),
                num_post_padded=_empty(1, dtype=i32, device=device),
                expert_offsets=_empty(E + 1, dtype=i32, device=device),
                padded_offsets=_empty(E + 1, dtype=i32, device=device))


def moe_align_block_size(topk_ids: torch.Tensor, E: int, BM: int, out: dict | None = None,
                         d_status: torch.Tensor | None = None, stream=None) -> dict:
    """Sort token-slots by expert and pad every expert to a multiple of BM (qmoe_moe_align_block_size).

    topk_ids int32 [M, top_k] on the device.  Returns the dict of alloc_align_outputs,
    filled on the stream: slots in ascending order within an expert, pads = T."""
    _need(topk_ids, torch.int32, "topk_ids")
    T = topk_ids.numel()
    o = out if out is not None else alloc_align_outputs(T, E, BM, topk_ids.device)
    st = load_library().qmoe_moe_align_block_size(
        _ptr(topk_ids), T, E, BM, _ptr(o["sorted_ids"]), _ptr(o["expert_ids"]), _ptr(o["num_post_padded"]),
        _ptr(o["expert_offsets"]), _ptr(o["padded_offsets"]), _ptr(d_status), _stream(stream))
    _check(st, "moe_align_block_size")
    return o


# ------------------------------------------------------------ quantisers ---
def quant_act_fp8(x: torch.Tensor, q: torch.Tensor | None = None, scale: torch.Tensor | None = None, stream=None):
    """bf16 [rows, cols] -> (e4m3 bytes uint8 [rows, cols], fp32 scale [rows])."""
    if not x.is_cuda or x.dtype != torch.bfloat16 or x.dim() != 2 or x.stride(1) != 1:
        raise QmoeError("x must be a 2-D CUDA bf16 tensor with unit column stride")
    rows, cols = x.shape
    q = q if q is not None else _empty(rows, cols, dtype=torch.uint8, device=x.device)
    scale = scale if scale is not None else _empty(rows, dtype=torch.float32, device=x.device)
    st = load_library().qmoe_quant_act_fp8(_ptr(x), rows, cols, x.stride(0), _ptr(q), _ptr(scale), _stream(stream))
    _check(st, "quant_act_fp8")
    return q, scale


def quant_act_fp8_sorted(x: torch.Tensor, align: dict, top_k: int, q: torch.Tensor | None = None,
                         scale: torch.Tensor | None = None, stream=None):
    """bf16 token rows [M, K] -> e4m3 rows in padded sorted order [cap, K] + fp32 scales [cap]
    (cap = len(align["sorted_ids"])), the A operand of the QMOE_A_PADDED layout."""
    if not x.is_cuda or x.dtype != torch.bfloat16 or x.dim() != 2 or x.stride(1) != 1:
        raise QmoeError("x must be a 2-D CUDA bf16 tensor with unit column stride")
    M, cols = x.shape
    cap = align["sorted_ids"].numel()
    q = q if q is not None else _empty(cap, cols, dtype=torch.uint8, device=x.device)
    scale = scale if scale is not None else _empty(cap, dtype=torch.float32, device=x.device)
    st = load_library().qmoe_quant_act_fp8_sorted(_ptr(x), M, cols, x.stride(0), _ptr(align["sorted_ids"]),
                                                  _ptr(align["num_post_padded"]), top_k, cap, _ptr(q), _ptr(scale),
                                                  _stream(stream))
    _check(st, "quant_act_fp8_sorted")
    return q, scale


def moe_align_quant_fp8(x: torch.Tensor, topk_ids: torch.Tensor, E: int, BM: int, align: dict | None = None,
                        q: torch.Tensor | None = None, scale: torch.Tensor | None = None,
                        d_status: torch.Tensor | None = None, stream=None):
    """moe_align_block_size + quant_act_fp8_sorted in one launch (small batches).
    Returns (align dict, q [cap, K] uint8, scale [cap] fp32); pad rows unwritten."""
    if not x.is_cuda or x.dtype != torch.bfloat16 or x.dim() != 2 or x.stride(1) != 1:
        raise QmoeError("x must be a 2-D CUDA bf16 tensor with unit column stride")
    _need(topk_ids, torch.int32, "topk_ids")
    M, cols = x.shape
    top_k = topk_ids.numel() // max(M, 1) if M > 0 else 1
    T = topk_ids.numel()
    o = align if align is not None else alloc_align_outputs(T, E, BM, x.device)
    cap = o["sorted_ids"].numel()
    q = q if q is not None else _empty(cap, cols, dtype=torch.uint8, device=x.device)
    scale = scale if scale is not None else _empty(cap, dtype=torch.float32, device=x.device)
    st = load_library().qmoe_moe_align_quant_fp8(
        _ptr(x), M, cols, x.stride(0), _ptr(topk_ids), top_k, E, BM, _ptr(o["sorted_ids"]), _ptr(o["expert_ids"]),
        _ptr(o["num_post_padded"]), _ptr(o["expert_offsets"]), _ptr(o["padded_offsets"]), _ptr(q), _ptr(scale),
        _ptr(d_status), _stream(stream))
    _check(st, "moe_align_quant_fp8")
    return o, q, scale


def moe_router_topk(logits: torch.Tensor, top_k: int, topk_ids=None, topk_weights=None, stream=None):
    """fp32 logits [M, E] -> (topk_ids int32 [M, top_k], topk_weights fp32 [M, top_k])."""
    _need(logits, torch.float32, "logits")
    M, E = logits.shape
    ids = topk_ids if topk_ids is not None else _empty(M, top_k, dtype=torch.int32, device=logits.device)
    w = topk_weights if topk_weights is not None else _empty(M, top_k, dtype=torch.float32, device=logits.device)
    _check(load_library().qmoe_moe_router_topk(_ptr(logits), M, E, top_k, _ptr(ids), _ptr(w), _stream(stream)),
           "moe_router_topk")
    return ids, w


def moe_route_align_quant_fp8(logits: torch.Tensor, x: torch.Tensor, top_k: int, BM: int, align: dict | None = None,
                              topk_ids=None, topk_weights=None, q=None, scale=None, d_status=None, stream=None):
    """Router + align + per-token e4m3 rows in padded sorted order (one launch for small batches).
    Returns (topk_ids, topk_weights, align dict, q [cap, K], scale [cap])."""
    _need(logits, torch.float32, "logits")
    if not x.is_cuda or x.dtype != torch.bfloat16 or x.dim() != 2 or x.stride(1) != 1:
        raise QmoeError("x must be a 2-D CUDA bf16 tensor with unit column stride")
    M, E = logits.shape
    cols = x.shape[1]
    T = M * top_k
    o = align if align is not None else alloc_align_outputs(T, E, BM, x.device)
    ids = topk_ids if topk_ids is not None else _empty(M, top_k, dtype=torch.int32, device=x.device)
    w = topk_weights if topk_weights is not None else _empty(M, top_k, dtype=torch.float32, device=x.device)
    cap = o["sorted_ids"].numel()
    q = q if q is not None else _empty(cap, cols, dtype=torch.uint8, device=x.device)
    scale = scale if scale is not None else _empty(cap, dtype=torch.float32, device=x.device)
    st = load_library().qmoe_moe_route_align_quant_fp8(
        _ptr(logits), _ptr(x), M, cols, x.stride(0), E, top_k, BM, _ptr(ids), _ptr(w), _ptr(o["sorted_ids"]),
        _ptr(o["expert_ids"]), _ptr(o["num_post_padded"]), _ptr(o["expert_offsets"]), _ptr(o["padded_offsets"]),
        _ptr(q), _ptr(scale), _ptr(d_status), _stream(stream))
    _check(st, "moe_route_align_quant_fp8")
    return ids, w, o, q, scale


def gather_sorted_bf16(x: torch.Tensor, align: dict, top_k: int, out: torch.Tensor | None = None, stream=None):
    """bf16 token rows [M, K] -> rows in padded sorted order [cap, K] (the PADDED
    activation operand of moe_gemm_w8a16); pad rows zero."""
    if not x.is_cuda or x.dtype != torch.bfloat16 or x.dim() != 2 or x.stride(1) != 1:
        raise QmoeError("x must be a 2-D CUDA bf16 tensor with unit column stride")
    M, cols = x.shape
    cap = align["sorted_ids"].numel()
    out = out if out is not None else _empty(cap, cols, dtype=torch.bfloat16, device=x.device)
    st = load_library().qmoe_gather_sorted_bf16(_ptr(x), M, cols, x.stride(0), _ptr(align["sorted_ids"]),
                                                _ptr(align["num_post_padded"]), top_k, cap, _ptr(out),
                                                _stream(stream))
    _check(st, "gather_sorted_bf16")
    return out


def quant_weight_fp8(w: torch.Tensor, stream=None):
    """fp32 [..., K] -> (e4m3 uint8 [..., K], fp32 scale [...]) per row (output channel)."""
    _need(w, torch.float32, "w")
    K = w.shape[-1]
    rows = w.numel() // K
    q = _empty(w.shape, dtype=torch.uint8, device=w.device)
    s = _empty(w.shape[:-1], dtype=torch.float32, device=w.device)
    _check(load_library().qmoe_quant_weight_fp8(_ptr(w), rows, K, _ptr(q), _ptr(s), _stream(stream)),
           "quant_weight_fp8")
    return q, s


def quant_weight_int8(w: torch.Tensor, stream=None):
    """fp32 [..., K] weight rows -> (int8 codes, fp32 per-row scale amax/127), qmoe_quant_weight_int8."""
    _need(w, torch.float32, "w")
    K = w.shape[-1]
    rows = w.numel() // K
    q = _empty(w.shape, dtype=torch.int8, device=w.device)
    s = _empty(w.shape[:-1], dtype=torch.float32, device=w.device)
    _check(load_library().qmoe_quant_weight_int8(_ptr(w), rows, K, _ptr(q), _ptr(s), _stream(stream)),
           "quant_weight_int8")
    return q, s


def quant_weight_int4(w: torch.Tensor, q=None, scale=None, stream=None):
    """fp32 [..., K] rows (K % 128 == 0) -> (packed int4 uint8 [..., K/2], fp32 group scales [..., K/128])."""
    _need(w, torch.float32, "w")
    K = w.shape[-1]
    rows = w.numel() // K
    q = q if q is not None else _empty(w.shape[:-1] + (K // 2,), dtype=torch.uint8, device=w.device)
    scale = scale if scale is not None else _empty(w.shape[:-1] + (K // 128,), dtype=torch.float32,
                                                        device=w.device)
    _check(load_library().qmoe_quant_weight_int4(_ptr(w), rows, K, _ptr(q), _ptr(scale), _stream(stream)),
           "quant_weight_int4")
    return q, scale


def quant_weight_mxfp8(w: torch.Tensor, q=None, sf=None, stream=None):
    """fp32 [..., K] weight rows -> (e4m3 codes uint8 same shape, E8M0 [rows, roundup(K/32, 4)])."""
    _need(w, torch.float32, "w")
    K = w.shape[-1]
    rows = w.numel() // K
    q = q if q is not None else _empty(w.shape, dtype=torch.uint8, device=w.device)
    sf = sf if sf is not None else _empty(rows, mx_sf_ld(K), dtype=torch.uint8, device=w.device)
    _check(load_library().qmoe_quant_weight_mxfp8(_ptr(w), rows, K, _ptr(q), _ptr(sf), sf.stride(0),
                                                  _stream(stream)), "quant_weight_mxfp8")
    return q, sf


def quant_mxfp8(x: torch.Tensor, *, expert_offsets, sf_padded_offsets, sf_rows: int | None = None, q=None, sf=None,
                d_status=None, stream=None):
    """bf16 [rows, I] -> (e4m3 [rows, I], E8M0 rowwise factors padded per expert), no activation."""
    if not x.is_cuda or x.dtype != torch.bfloat16 or x.dim() != 2 or x.stride(1) != 1:
        raise QmoeError("x must be a 2-D CUDA bf16 tensor with unit column stride")
    _need(expert_offsets, torch.int32, "expert_offsets")
    _need(sf_padded_offsets, torch.int32, "sf_padded_offsets")
    rows, I = x.shape
    q = q if q is not None else _empty(rows, I, dtype=torch.uint8, device=x.device)
    if sf is None:
        if sf_rows is None:
            raise QmoeError("sf_rows (capacity of the scale-factor matrix) is required when sf is not given")
        sf = _empty(sf_rows, mx_sf_ld(I), dtype=torch.uint8, device=x.device)
    st = load_library().qmoe_quant_mxfp8(_ptr(x), rows, I, x.stride(0), _ptr(q), _ptr(sf), sf.stride(0),
                                         _ptr(expert_offsets), _ptr(sf_padded_offsets), expert_offsets.numel() - 1,
                                         _ptr(d_status), _stream(stream))
    _check(st, "quant_mxfp8")
    return q, sf


def mx_weight_sf_tiled(sf: torch.Tensor, E: int, N: int, K: int, out=None, stream=None):
    """E8M0 weight factors [E*N, ld] -> the flat uint8 tiled blocks moe_gemm_w8a8 streams."""
    _need(sf, torch.uint8, "sf")
    L = load_library()
    nbytes = int(L.qmoe_mx_weight_sf_tiled_bytes(E, N, K))
    out = out if out is not None else _empty(nbytes, dtype=torch.uint8, device=sf.device)
    _check(L.qmoe_mx_weight_sf_tiled(_ptr(sf), E, N, K, sf.stride(0), _ptr(out), _stream(stream)),
           "mx_weight_sf_tiled")
    return out


def mx_colwise_sf_shape(rows: int, cols: int):
    """ceil(rows/32) blocks padded to a multiple of 4 rows, columns padded to 128."""
    return ((rows + 31) // 32 + 3) // 4 * 4, (cols + 127) // 128 * 128


def quant_mxfp8_colwise(x: torch.Tensor, q=None, sf=None, stream=None):
    """bf16 [rows, cols] -> (e4m3 [rows, cols] in 32x1 column blocks, E8M0 [mx_colwise_sf_shape])."""
    if not x.is_cuda or x.dtype != torch.bfloat16 or x.dim() != 2 or x.stride(1) != 1:
        raise QmoeError("x must be a 2-D CUDA bf16 tensor with unit column stride")
    rows, cols = x.shape
    q = q if q is not None else _empty(rows, cols, dtype=torch.uint8, device=x.device)
    if sf is None:
        sr, sc = mx_colwise_sf_shape(rows, cols)
        sf = _empty(sr, sc, dtype=torch.uint8, device=x.device)
    st = load_library().qmoe_quant_mxfp8_colwise(_ptr(x), rows, cols, x.stride(0), _ptr(q), _ptr(sf), sf.shape[0],
                                                 sf.stride(0), _stream(stream))
    _check(st, "quant_mxfp8_colwise")
    return q, sf


# ------------------------------------------------------------------ GEMM ---
def _gemm(fn_name, *, a, a_scale, w, w_scale, align, topk_weights, out, M, top_k, BM, a_layout, out_layout,
          a_scale_mode=SCALE_PER_TOKEN, a_sf=None, a_sf_padded_offsets=None, d_status=None, accum=None,
          stream=None, w_scale_mode=0, w_sf=None, K=None, extra=()):
    E, N, Kw = w.shape
    K = Kw if K is None else K
    if out_layout == OUT_TOKEN_SUM and accum is None:
        accum = _empty(M, N, dtype=torch.float32, device=out.device)
    args = GemmArgs()
    args.struct_size = ctypes.sizeof(GemmArgs)
    args.a = a.data_ptr()
    args.lda = a.stride(0)
    args.a_scale = None if a_scale is None else a_scale.data_ptr()
    args.a_scale_mode = a_scale_mode
    args.a_sf = None if a_sf is None else a_sf.data_ptr()
    args.a_sf_ld = 0 if a_sf is None else a_sf.stride(0)
    args.a_sf_padded_offsets = None if a_sf_padded_offsets is None else a_sf_padded_offsets.data_ptr()
    args.a_layout = a_layout
    args.w = w.data_ptr()
    args.w_scale = None if w_scale is None else w_scale.data_ptr()
    args.w_scale_mode = w_scale_mode
    args.w_sf = None if w_sf is None else w_sf.data_ptr()
    args.sorted_ids = align["sorted_ids"].data_ptr()
    args.expert_ids = align["expert_ids"].data_ptr()
    args.num_post_padded = align["num_post_padded"].data_ptr()
    args.expert_offsets = align["expert_offsets"].data_ptr()
    args.padded_offsets = align["padded_offsets"].data_ptr()
    args.topk_weights = None if topk_weights is None else topk_weights.data_ptr()
    args.out = None if out is None else out.data_ptr()
    args.out_layout = out_layout
    args.M, args.N, args.K = M, N, K
    args.E, args.top_k, args.BM = E, top_k, BM
    args.d_status = None if d_status is None else d_status.data_ptr()
    args.accum = None if accum is None else accum.data_ptr()
    st = getattr(load_library(), fn_name)(ctypes.byref(args), *extra, _stream(stream))
    _check(st, fn_name)
    return out


def _out_for(out, out_layout, M, top_k, N, device):
    if out is not None:
        return out
    rows = M if out_layout == OUT_TOKEN_SUM else M * top_k
    return _empty(rows, N, dtype=torch.bfloat16, device=device)


def moe_gemm_w8a8(a_q: torch.Tensor, a_scale: torch.Tensor | None, w_q: torch.Tensor, w_scale: torch.Tensor,
                  align: dict, topk_weights: torch.Tensor | None, *, M: int, top_k: int, BM: int,
                  a_layout: int = A_TOKEN_GATHER, out_layout: int = OUT_SLOT, out: torch.Tensor | None = None,
                  d_status: torch.Tensor | None = None, accum: torch.Tensor | None = None,
                  a_scale_mode: int = SCALE_PER_TOKEN, a_sf: torch.Tensor | None = None,
                  a_sf_padded_offsets: torch.Tensor | None = None, w_scale_mode: int = SCALE_PER_TOKEN,
                  w_sf: torch.Tensor | None = None, stream=None, tile: int | None = None) -> torch.Tensor:
    """FP8 W8A8 grouped GEMM.  a_q uint8 e4m3 [rows, K] (token rows for TOKEN_GATHER,
    compact grouped rows for GROUPED), a_scale fp32 [rows], w_q uint8 e4m3 [E, N, K],
    w_scale fp32 [E, N], align = moe_align_block_size(..., BM), topk_weights fp32 [M, top_k]
    or None.  Returns bf16 [T, N] (SLOT/GROUPED) or [M, N] (TOKEN_SUM; accum is the
    fp32 [M, N] scratch the sum needs, allocated here when not given).  MXFP8 weights:
    w_scale_mode=SCALE_MX_1X32 with w_sf = mx_weight_sf_tiled(factors of quant_weight_mxfp8),
    w_scale then optional; needs MX activations.  tile (tests and timing only): TILE_ONE_SM
    or TILE_PAIR forces that tile family (qmoe_debug_moe_gemm_tile)."""
    _need(a_q, torch.uint8, "a_q")
    _need(w_q, torch.uint8, "w_q")
    if a_scale_mode == SCALE_PER_TOKEN:
        _need(a_scale, torch.float32, "a_scale")
    else:
        _need(a_sf, torch.uint8, "a_sf")
        _need(a_sf_padded_offsets, torch.int32, "a_sf_padded_offsets")
    if w_scale_mode == SCALE_MX_1X32:
        _need(w_sf, torch.uint8, "w_sf")
        if w_scale is not None:
            _need(w_scale, torch.float32, "w_scale")
    else:
        _need(w_scale, torch.float32, "w_scale")
    if topk_weights is not None:
        _need(topk_weights, torch.float32, "topk_weights")
    out = _out_for(out, out_layout, M, top_k, w_q.shape[1], a_q.device)
    return _gemm("qmoe_moe_gemm_w8a8" if tile is None else "qmoe_debug_moe_gemm_tile", a=a_q, a_scale=a_scale,
                 w=w_q, w_scale=w_scale, align=align, topk_weights=topk_weights, out=out, M=M, top_k=top_k, BM=BM,
                 a_layout=a_layout, out_layout=out_layout, d_status=d_status, accum=accum,
                 a_scale_mode=a_scale_mode, a_sf=a_sf, a_sf_padded_offsets=a_sf_padded_offsets, stream=stream,
                 w_scale_mode=w_scale_mode, w_sf=w_sf,
                 extra=() if tile is None else (ctypes.c_int32(0), ctypes.c_int32(tile)))


def moe_gemm_w8a8_silu_mxfp8(a_q: torch.Tensor, a_scale: torch.Tensor, w_q: torch.Tensor, w_scale: torch.Tensor,
                             align: dict, *, M: int, top_k: int, a_layout: int = A_TOKEN_GATHER,
                             topk_weights: torch.Tensor | None = None, q: torch.Tensor | None = None,
                             sf: torch.Tensor | None = None, sf_rows: int | None = None,
                             d_status: torch.Tensor | None = None, stream=None):
    """FP8 [gate | up] projection (w_q [E, 2I, K], gate rows first) with SwiGLU +
    MXFP8 in the GEMM epilogue; align from moe_align_block_size(..., 128).
    Returns (q [T, I] uint8 e4m3 codes in compact grouped rows, sf [sf_rows,
    mx_sf_ld(I)] uint8 E8M0), the bytes silu_mul_quant(SCALE_MX_1X32) writes for
    the bf16 output of moe_gemm_w8a8(..., out_layout=OUT_GROUPED)."""
    _need(a_q, torch.uint8, "a_q")
    _need(a_scale, torch.float32, "a_scale")
    _need(w_q, torch.uint8, "w_q")
    _need(w_scale, torch.float32, "w_scale")
    if topk_weights is not None:
        _need(topk_weights, torch.float32, "topk_weights")
    E, N, _ = w_q.shape
    I, T = N // 2, M * top_k
    q = q if q is not None else _empty(T, I, dtype=torch.uint8, device=a_q.device)
    if sf is None:
        rows = sf_rows if sf_rows is not None else align_max_padded(T, E, 128)
        sf = _empty(rows, mx_sf_ld(I), dtype=torch.uint8, device=a_q.device)
    _gemm("qmoe_moe_gemm_w8a8_silu_mxfp8", a=a_q, a_scale=a_scale, w=w_q, w_scale=w_scale, align=align,
          topk_weights=topk_weights, out=None, M=M, top_k=top_k, BM=128, a_layout=a_layout, out_layout=OUT_GROUPED,
          d_status=d_status, stream=stream,
          extra=(_ptr(q), _ptr(sf), sf.stride(0), _ptr(align["padded_offsets"])))
    return q, sf


def moe_gemm_w8a8_silu_fp8_token(a_q: torch.Tensor, a_scale: torch.Tensor, w_q: torch.Tensor,
                                 w_scale: torch.Tensor, align: dict, *, M: int, top_k: int,
                                 a_layout: int = A_TOKEN_GATHER, topk_weights: torch.Tensor | None = None,
                                 q: torch.Tensor | None = None, scale: torch.Tensor | None = None,
                                 h_scratch: torch.Tensor | None = None, d_status: torch.Tensor | None = None,
                                 stream=None):
    """FP8 [gate | up] projection (w_q [E, 2I, K]) with SwiGLU in the GEMM
    epilogue and per-token FP8 requantisation; align from
    moe_align_block_size(..., 128).  Returns (q [T, I] uint8, scale [T] fp32),
    the bytes silu_mul_quant(SCALE_PER_TOKEN) writes for the bf16 output of
    moe_gemm_w8a8(..., out_layout=OUT_GROUPED).  h_scratch: fp32, at least
    T*I + T elements (allocated here when not given)."""
    _need(a_q, torch.uint8, "a_q")
    _need(a_scale, torch.float32, "a_scale")
    _need(w_q, torch.uint8, "w_q")
    _need(w_scale, torch.float32, "w_scale")
    if topk_weights is not None:
        _need(topk_weights, torch.float32, "topk_weights")
    E, N, _ = w_q.shape
    I, T = N // 2, M * top_k
    q = q if q is not None else _empty(T, I, dtype=torch.uint8, device=a_q.device)
    scale = scale if scale is not None else _empty(T, dtype=torch.float32, device=a_q.device)
    if h_scratch is None:
        h_scratch = _empty(T * I + T, dtype=torch.float32, device=a_q.device)
    elif h_scratch.dtype != torch.float32 or h_scratch.numel() < T * I + T:
        raise QmoeError("h_scratch must be fp32 with at least T*I + T elements")
    _gemm("qmoe_moe_gemm_w8a8_silu_fp8_token", a=a_q, a_scale=a_scale, w=w_q, w_scale=w_scale, align=align,
          topk_weights=topk_weights, out=None, M=M, top_k=top_k, BM=128, a_layout=a_layout, out_layout=OUT_GROUPED,
          d_status=d_status, stream=stream, extra=(_ptr(q), _ptr(scale), _ptr(h_scratch)))
    return q, scale


def moe_gemm_w8a8_token_sum_noalloc(a_q: torch.Tensor, a_scale: torch.Tensor, w_q: torch.Tensor,
                                    w_scale: torch.Tensor, align: dict, topk_weights: torch.Tensor | None, *,
                                    M: int, top_k: int, BM: int, a_layout: int = A_TOKEN_GATHER,
                                    out: torch.Tensor | None = None, d_status: torch.Tensor | None = None,
                                    stream=None) -> torch.Tensor:
    """Sum over top_k of the FP8 grouped GEMM (bf16 [M, N]) using the library's
    built-in fp32 scratch instead of a caller buffer, for callers that cannot
    allocate device memory (M*N <= NOALLOC_ACCUM_MAX_ELEMS; calls that overlap
    on the GPU share the scratch and must not run concurrently)."""
    _need(a_q, torch.uint8, "a_q")
    _need(w_q, torch.uint8, "w_q")
    _need(a_scale, torch.float32, "a_scale")
    _need(w_scale, torch.float32, "w_scale")
    if M * w_q.shape[1] > NOALLOC_ACCUM_MAX_ELEMS:
        raise QmoeError(f"M*N = {M * w_q.shape[1]} exceeds the built-in scratch ({NOALLOC_ACCUM_MAX_ELEMS} floats)")
    out = _out_for(out, OUT_TOKEN_SUM, M, top_k, w_q.shape[1], a_q.device)
    E, N, K = w_q.shape
    args = GemmArgs()
    args.struct_size = ctypes.sizeof(GemmArgs)
    args.a, args.lda, args.a_scale = a_q.data_ptr(), a_q.stride(0), a_scale.data_ptr()
    args.a_scale_mode, args.a_layout = SCALE_PER_TOKEN, a_layout
    args.w, args.w_scale = w_q.data_ptr(), w_scale.data_ptr()
    args.sorted_ids, args.expert_ids = align["sorted_ids"].data_ptr(), align["expert_ids"].data_ptr()
    args.num_post_padded = align["num_post_padded"].data_ptr()
    args.expert_offsets, args.padded_offsets = align["expert_offsets"].data_ptr(), align["padded_offsets"].data_ptr()
    args.topk_weights = None if topk_weights is None else topk_weights.data_ptr()
    args.out, args.out_layout = out.data_ptr(), OUT_TOKEN_SUM
    args.M, args.N, args.K, args.E, args.top_k, args.BM = M, N, K, E, top_k, BM
    args.d_status = None if d_status is None else d_status.data_ptr()
    st = load_library().qmoe_moe_gemm_w8a8_token_sum_noalloc(ctypes.byref(args), _stream(stream))
    _check(st, "moe_gemm_w8a8_token_sum_noalloc")
    return out


def moe_gemm_w8a16(a: torch.Tensor, w_q: torch.Tensor, w_scale: torch.Tensor, align: dict,
                   topk_weights: torch.Tensor | None, *, M: int, top_k: int, BM: int,
                   a_layout: int = A_TOKEN_GATHER, out_layout: int = OUT_SLOT, out: torch.Tensor | None = None,
                   d_status: torch.Tensor | None = None, accum: torch.Tensor | None = None,
                   stream=None, tile: int | None = None) -> torch.Tensor:
    """INT8 W8A16 grouped GEMM: a bf16 [rows, K], w_q int8 [E, N, K], w_scale fp32 [E, N].
    tile (tests and timing only): TILE_ONE_SM or TILE_PAIR forces that tile family."""
    _need(a, torch.bfloat16, "a")
    _need(w_q, torch.int8, "w_q")
    _need(w_scale, torch.float32, "w_scale")
    if topk_weights is not None:
        _need(topk_weights, torch.float32, "topk_weights")
    out = _out_for(out, out_layout, M, top_k, w_q.shape[1], a.device)
    return _gemm("qmoe_moe_gemm_w8a16" if tile is None else "qmoe_debug_moe_gemm_tile", a=a, a_scale=None, w=w_q,
                 w_scale=w_scale, align=align, topk_weights=topk_weights, out=out, M=M, top_k=top_k, BM=BM,
                 a_layout=a_layout, out_layout=out_layout, d_status=d_status, accum=accum, stream=stream,
                 extra=() if tile is None else (ctypes.c_int32(1), ctypes.c_int32(tile)))


def moe_gemm_w4a16(a: torch.Tensor, w_q: torch.Tensor, w_scale: torch.Tensor, align: dict,
                   topk_weights: torch.Tensor | None, *, M: int, top_k: int, BM: int,
                   a_layout: int = A_TOKEN_GATHER, out_layout: int = OUT_SLOT, out: torch.Tensor | None = None,
                   d_status: torch.Tensor | None = None, accum: torch.Tensor | None = None,
                   stream=None, tile: int | None = None) -> torch.Tensor:
    """INT4 W4A16 grouped GEMM: a bf16 [rows, K], w_q packed int4 uint8 [E, N, K/2],
    w_scale fp32 group scales [E, N, K/128] (quant_weight_int4); BM 64, 128 or 256.
    tile (tests and timing only): TILE_ONE_SM or TILE_PAIR forces that tile family."""
    _need(a, torch.bfloat16, "a")
    _need(w_q, torch.uint8, "w_q")
    _need(w_scale, torch.float32, "w_scale")
    if topk_weights is not None:
        _need(topk_weights, torch.float32, "topk_weights")
    out = _out_for(out, out_layout, M, top_k, w_q.shape[1], a.device)
    return _gemm("qmoe_moe_gemm_w4a16" if tile is None else "qmoe_debug_moe_gemm_tile", a=a, a_scale=None, w=w_q,
                 w_scale=w_scale, align=align, topk_weights=topk_weights, out=out, M=M, top_k=top_k, BM=BM,
                 a_layout=a_layout, out_layout=out_layout, d_status=d_status, accum=accum, stream=stream,
                 K=2 * w_q.shape[2], extra=() if tile is None else (ctypes.c_int32(2), ctypes.c_int32(tile)))


# ------------------------------------------------------ SwiGLU + quant ---
def mx_sf_ld(I: int) -> int:
    """Row stride (bytes) of rowwise E8M0 factors for I columns: I/32 rounded up to a multiple of 4."""
    return (I // 32 + 3) // 4 * 4


def srelu_quant(y: torch.Tensor, mode: int = SCALE_PER_TOKEN, *, expert_offsets=None, sf_padded_offsets=None,
                sf_rows: int | None = None, q=None, scale=None, sf=None, d_status=None, stream=None):
    """y bf16 [rows, I] -> relu(y)^2 requantised like silu_mul_quant (per-token or MX)."""
    return _act_quant("qmoe_srelu_quant", False, y, mode, expert_offsets, sf_padded_offsets, sf_rows, q, scale, sf,
                      d_status, stream)


def silu_mul_quant(y: torch.Tensor, mode: int = SCALE_PER_TOKEN, *, expert_offsets=None, sf_padded_offsets=None,
                   sf_rows: int | None = None, q=None, scale=None, sf=None, d_status=None, stream=None):
    """y bf16 [rows, 2I] (gate | up) -> per-token: (q [rows, I] uint8, scale [rows] fp32);
    MX: (q, sf [sf_rows, roundup(I/32, 4)] uint8).  For MX, sf_rows must be at
    least sf_padded_offsets[E] (e.g. align_max_padded(T, E, 128))."""
    return _act_quant("qmoe_silu_mul_quant", True, y, mode, expert_offsets, sf_padded_offsets, sf_rows, q, scale, sf,
                      d_status, stream)


def _act_quant(fn_name, gated, y, mode, expert_offsets, sf_padded_offsets, sf_rows, q, scale, sf, d_status, stream):
    if not y.is_cuda or y.dtype != torch.bfloat16 or y.dim() != 2 or y.stride(1) != 1:
        raise QmoeError("y must be a 2-D CUDA bf16 tensor with unit column stride")
    rows, width = y.shape
    I = width // 2 if gated else width
    q = q if q is not None else _empty(rows, I, dtype=torch.uint8, device=y.device)
    fn = getattr(load_library(), fn_name)
    if mode == SCALE_PER_TOKEN:
        scale = scale if scale is not None else _empty(rows, dtype=torch.float32, device=y.device)
        st = fn(_ptr(y), rows, I, y.stride(0), mode, _ptr(q), _ptr(scale), None, 0, None, None, 1, _ptr(d_status),
                _stream(stream))
        _check(st, fn_name)
        return q, scale
    _need(expert_offsets, torch.int32, "expert_offsets")
    _need(sf_padded_offsets, torch.int32, "sf_padded_offsets")
    E = expert_offsets.numel() - 1
    ld = mx_sf_ld(I)
    if sf is None:
        if sf_rows is None:
            raise QmoeError("sf_rows (capacity of the scale-factor matrix) is required when sf is not given")
        sf = _empty(sf_rows, ld, dtype=torch.uint8, device=y.device)
    st = fn(_ptr(y), rows, I, y.stride(0), mode, _ptr(q), None, _ptr(sf), sf.stride(0), _ptr(expert_offsets),
            _ptr(sf_padded_offsets), E, _ptr(d_status), _stream(stream))
    _check(st, fn_name)
    return q, sf


# --------------------------------------------------------- element hooks ---
def debug_e4m3_encode(x: torch.Tensor, stream=None) -> torch.Tensor:
    """Test hook: the kernels' fp32 -> e4m3 conversion (RNE, satfinite) applied elementwise."""
    _need(x, torch.float32, "x")
    q = _empty(x.shape, dtype=torch.uint8, device=x.device)
    _check(load_library().qmoe_debug_e4m3_encode(_ptr(x), _ptr(q), x.numel(), _stream(stream)), "debug_e4m3_encode")
    return q


def debug_int8_to_bf16(x: torch.Tensor, stream=None) -> torch.Tensor:
    """Test hook: the W8A16 converters' int8 -> bf16 conversion applied elementwise."""
    _need(x, torch.int8, "x")
    y = _empty(x.shape, dtype=torch.bfloat16, device=x.device)
    _check(load_library().qmoe_debug_int8_to_bf16(_ptr(x), _ptr(y), x.numel(), _stream(stream)),
           "debug_int8_to_bf16")
    return y


def debug_silu_mul(g: torch.Tensor, u: torch.Tensor, stream=None) -> torch.Tensor:
    """Test hook: h = silu(g) * u by the kernels' packed fp32 sequence, elementwise."""
    _need(g, torch.float32, "g")
    _need(u, torch.float32, "u")
    h = _empty(g.shape, dtype=g.dtype, device=g.device)
    _check(load_library().qmoe_debug_silu_mul(_ptr(g), _ptr(u), _ptr(h), g.numel(), _stream(stream)),
           "debug_silu_mul")
    return h


def debug_rcp_ge1(d: torch.Tensor, stream=None) -> torch.Tensor:
    """Test hook: the SiLU's reciprocal 1/d for d >= 1, elementwise."""
    _need(d, torch.float32, "d")
    y = _empty(d.shape, dtype=d.dtype, device=d.device)
    _check(load_library().qmoe_debug_rcp_ge1(_ptr(d), _ptr(y), d.numel(), _stream(stream)), "debug_rcp_ge1")
    return y


def debug_quant_by_scale(x: torch.Tensor, s: float, stream=None) -> torch.Tensor:
    """Test hook: the e4m3 codes the quantisers write for x / s (row scale s), elementwise."""
    _need(x, torch.float32, "x")
    q = _empty(x.shape, dtype=torch.uint8, device=x.device)
    _check(load_library().qmoe_debug_quant_by_scale(_ptr(x), float(s), _ptr(q), x.numel(), _stream(stream)),
           "debug_quant_by_scale")
    return q


def debug_div_by_scale(x: torch.Tensor, s: float, stream=None) -> torch.Tensor:
    """Test hook: the correctly rounded division x / s by a row scale (packed pairs;
    the int8 weight quantiser's), elementwise."""
    _need(x, torch.float32, "x")
    q = _empty(x.shape, dtype=x.dtype, device=x.device)
    _check(load_library().qmoe_debug_div_by_scale(_ptr(x), float(s), _ptr(q), x.numel(), _stream(stream)),
           "debug_div_by_scale")
    return q


def debug_wait_timeout(d_status: torch.Tensor, limit_ns: int, stream=None) -> None:
    """Test hook: one bounded mbarrier wait that nothing completes; sets QMOE_DEV_TIMEOUT in d_status."""
    _need(d_status, torch.int32, "d_status")
    _check(load_library().qmoe_debug_wait_timeout(_ptr(d_status), int(limit_ns), _stream(stream)),
           "debug_wait_timeout")
