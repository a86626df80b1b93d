"""Seeded synthetic inputs for the quantized MoE grouped GEMM path.

This module only draws random numbers and lays them out; it holds none of the
quantisation, sorting or GEMM arithmetic of the path.  Both the CUDA path and
the CPU oracle consume what it returns, so the two sides always see the same
bytes.

Distributions (one seed per tensor, ``numpy.random.default_rng([seed, id])``):

* activations A[M, K]: N(0, 1), rounded to bf16 (round-to-nearest-even, done
  by torch's dtype cast);
* expert weights W[E, N, K]: N(0, 1/K) in fp32, drawn per expert so the host
  never holds more than one expert at a time when streaming;
* router logits [M, E]: N(0, 1), optionally plus ln p_e with a Zipf(s)
  expert prior p_e ~ (e+1)^-s, which makes the first expert take a large share
  of the slots (s = 1.2 gives about 40 % at E = 8).

The router (softmax -> top-k -> renormalise) is not part of the grouped GEMM
path, whose first step consumes ``topk_ids``/``topk_weights``; it is treated
as input synthesis here and done in fp64 with a stable sort (ties go to the
lower expert id), then cast to fp32.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

# tensor ids inside one seed
_ID_A = 1
_ID_LOGITS = 2
_ID_W_BASE = 100          # + 1000 * weight_set + expert
_ID_PERM = 7


def rng(seed: int, tensor_id: int) -> np.random.Generator:
    return np.random.default_rng([int(seed), int(tensor_id)])


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """fp32 -> bf16 bit patterns (uint16) via torch's RNE dtype cast."""
    import torch
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32))
    return t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16).copy()


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    """bf16 bit patterns -> fp32 values (exact widening)."""
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def activations_bf16(M: int, K: int, seed: int) -> np.ndarray:
    x = rng(seed, _ID_A).standard_normal((M, K), dtype=np.float32)
    return f32_to_bf16_bits(x)


def expert_weight_f32(N: int, K: int, seed: int, expert: int, weight_set: int = 0) -> np.ndarray:
    g = rng(seed, _ID_W_BASE + 1000 * weight_set + expert)
    return (g.standard_normal((N, K), dtype=np.float32) * np.float32(1.0 / np.sqrt(K))).astype(np.float32)


def expert_weights_f32(E: int, N: int, K: int, seed: int, weight_set: int = 0) -> np.ndarray:
    out = np.empty((E, N, K), dtype=np.float32)
    for e in range(E):
        out[e] = expert_weight_f32(N, K, seed, e, weight_set)
    return out


def router_logits(M: int, E: int, seed: int, zipf_s: float | None = None) -> np.ndarray:
    logits = rng(seed, _ID_LOGITS).standard_normal((M, E))
    if zipf_s is not None:
        p = (np.arange(1, E + 1, dtype=np.float64)) ** (-float(zipf_s))
        p /= p.sum()
        logits = logits + np.log(p)[None, :]
    return logits


def route_topk(logits: np.ndarray, top_k: int) -> tuple[np.ndarray, np.ndarray]:
    """softmax (fp64) -> top-k by stable descending sort -> renormalise -> fp32."""
    z = logits - logits.max(axis=1, keepdims=True)
    p = np.exp(z)
    p /= p.sum(axis=1, keepdims=True)
    order = np.argsort(-p, axis=1, kind="stable")[:, :top_k]
    w = np.take_along_axis(p, order, axis=1)
    w = w / w.sum(axis=1, keepdims=True)
    return order.astype(np.int32), w.astype(np.float32)


def routing(M: int, E: int, top_k: int, seed: int, zipf_s: float | None = None):
    return route_topk(router_logits(M, E, seed, zipf_s), top_k)


def token_permutation(M: int, seed: int) -> np.ndarray:
    return rng(seed, _ID_PERM).permutation(M).astype(np.int64)


@dataclass(frozen=True)
class Workload:
    """One shape of one named workload (sizes only; no arithmetic)."""
    name: str
    M: int
    K: int
    N: int
    E: int = 8
    top_k: int = 2
    seed: int = 0
    precision: str = "fp8"          # "fp8" (W8A8) or "int8" (W8A16)
    inter: int = 0                  # FFN intermediate size I for a full layer (up N = 2*I)
    act_scale: str = "token"        # "token" or "mx" for the layer intermediate
    zipf_s: float | None = None
    extra: dict = field(default_factory=dict, compare=False)


def tiny_fp8() -> Workload:
    return Workload("tiny fp8 w8a8 M=64 K=128 N=256 E=8 top2", 64, 128, 256, seed=0)


def decode_fp8_sweep() -> list[Workload]:
    return [Workload(f"decode fp8 w8a8 M={m} K=4096 N=14336 E=8 top2", m, 4096, 14336,
                     seed=1000 + i) for i, m in enumerate((64, 128, 256, 512))]


def int8_w8a16_sweep() -> list[Workload]:
    out = []
    i = 0
    for n in (7168, 14336):
        for m in (64, 1024, 4096):
            out.append(Workload(f"int8 w8a16 M={m} K=4096 N={n} E=8 top2", m, 4096, n,
                                seed=2000 + i, precision="int8"))
            i += 1
    return out


def mixtral_8x7b_layer() -> Workload:
    return Workload("mixtral-8x7b-shaped fp8 layer M=4096 K=4096 I=14336 E=8 top2",
                    4096, 4096, 4096, seed=3000, inter=14336)


def mixtral_8x22b_layer() -> Workload:
    return Workload("mixtral-8x22b-shaped fp8 layer M=4096 K=6144 I=16384 E=8 top2 mxfp8 zipf1.2",
                    4096, 6144, 6144, seed=4000, inter=16384, act_scale="mx", zipf_s=1.2)
