"""Pins for the oracle's grouped GEMM.

* brute-force dense MoE written independently in numpy: every token times
  every expert in fp64 (dequantised with torch's e4m3 decode), masked by the
  routing, for all three output layouts and all A/W kinds;
* the per-expert decomposition of "Enabling MOE Quantization using linear
  decomposition" (pytorch/ao PR 2043, Summary): gather each expert's rows and
  run one dense matmul per expert;
* invariants: a token permutation permutes the output; top_k = E with uniform
  weights equals the mean over all experts; E = 1, top_k = 1, w = 1 is a plain
  GEMM (numpy matmul).
"""
import numpy as np
import pytest
import torch

from quantized_moe_grouped_gb300 import inputs


def dq_e4m3(q):
    return torch.from_numpy(np.ascontiguousarray(q)).view(torch.float8_e4m3fn).to(torch.float64).numpy()


def make_fp8_case(orc, M, K, N, E, top_k, seed):
    a = inputs.activations_bf16(M, K, seed)
    w = inputs.expert_weights_f32(E, N, K, seed)
    ids, tw = inputs.routing(M, E, top_k, seed)
    qa, sa = orc.quant_rows_fp8_bf16(a)
    qw, sw = orc.quant_rows_fp8_f32(w)
    return dict(a=a, w=w, ids=ids, tw=tw, qa=qa, sa=sa, qw=qw, sw=sw)


def dense_moe(A, W, ids, tw):
    """A [M,K] fp64, W [E,N,K] fp64 -> [M, top_k, N]: every token through every
    expert, then pick the routed ones."""
    allx = np.einsum("mk,enk->men", A, W)               # [M, E, N]
    M, top_k = ids.shape
    out = np.empty((M, top_k, W.shape[1]))
    for j in range(top_k):
        out[:, j, :] = allx[np.arange(M), ids[:, j], :] * (tw[:, j][:, None] if tw is not None else 1.0)
    return out


@pytest.mark.parametrize("M,K,N,E,top_k", [(13, 64, 48, 4, 2), (31, 96, 32, 3, 1), (8, 32, 16, 5, 3)])
def test_fp8_vs_bruteforce_all_layouts(orc, M, K, N, E, top_k):
    c = make_fp8_case(orc, M, K, N, E, top_k, seed=M * 7 + K)
    A = dq_e4m3(c["qa"]) * c["sa"][:, None].astype(np.float64)
    W = dq_e4m3(c["qw"]) * c["sw"][..., None].astype(np.float64)
    ref = dense_moe(A, W, c["ids"], c["tw"])
    kw = dict(a_kind=orc.A_FP8_TOKEN, a=c["qa"], a_scale=c["sa"], w_kind=orc.W_FP8, w=c["qw"], w_scale=c["sw"],
              topk_ids=c["ids"], topk_w=c["tw"], E=E)
    slot = orc.moe_gemm(**kw, out_layout="slot")
    assert np.allclose(slot, ref.reshape(M * top_k, N), rtol=1e-12, atol=1e-12)
    tsum = orc.moe_gemm(**kw, out_layout="token_sum")
    assert np.allclose(tsum, ref.sum(axis=1), rtol=1e-12, atol=1e-12)
    grouped = orc.moe_gemm(**kw, out_layout="grouped")
    order = np.argsort(c["ids"].ravel(), kind="stable")
    assert np.allclose(grouped, ref.reshape(M * top_k, N)[order], rtol=1e-12, atol=1e-12)
    # grouped A layout: A rows pre-gathered into compact expert order
    Ag = c["qa"][order // top_k]
    sag = c["sa"][order // top_k]
    g2 = orc.moe_gemm(a_kind=orc.A_FP8_TOKEN, a=Ag, a_scale=sag, w_kind=orc.W_FP8, w=c["qw"], w_scale=c["sw"],
                      topk_ids=c["ids"], topk_w=c["tw"], E=E, a_layout="grouped", out_layout="slot")
    assert np.allclose(g2, ref.reshape(M * top_k, N), rtol=1e-12, atol=1e-12)


def test_int8_w8a16_vs_bruteforce(orc):
    M, K, N, E, top_k = 17, 80, 40, 4, 2
    a = inputs.activations_bf16(M, K, 3)
    w = inputs.expert_weights_f32(E, N, K, 3)
    ids, tw = inputs.routing(M, E, top_k, 3)
    qw, sw = orc.quant_rows_int8_f32(w)
    A = inputs.bf16_bits_to_f32(a).astype(np.float64)
    W = qw.astype(np.float64) * sw[..., None].astype(np.float64)
    ref = dense_moe(A, W, ids, tw)
    out = orc.moe_gemm(a_kind=orc.A_BF16, a=a, w_kind=orc.W_INT8, w=qw, w_scale=sw, topk_ids=ids, topk_w=tw, E=E)
    assert np.allclose(out, ref.reshape(M * top_k, N), rtol=1e-12, atol=1e-12)


def test_mx_a_vs_bruteforce(orc):
    M, I, N, E, top_k = 12, 64, 24, 3, 2
    ids, tw = inputs.routing(M, E, top_k, 4)
    T = M * top_k
    al = orc.moe_align(ids, E, 128)
    y = inputs.activations_bf16(T, 2 * I, 4)
    q, sf = orc.silu_mul_quant_mx(y, al["expert_offsets"], al["padded_offsets"])
    eoff, poff = al["expert_offsets"], al["padded_offsets"]
    sf_row = np.empty(T, dtype=np.int64)
    for e in range(E):
        for r in range(eoff[e], eoff[e + 1]):
            sf_row[r] = poff[e] + (r - eoff[e])
    w = inputs.expert_weights_f32(E, N, I, 4)
    qw, sw = orc.quant_rows_fp8_f32(w)
    # independent dequant of the grouped A rows
    scales = 2.0 ** (sf[sf_row][:, : I // 32].astype(np.float64) - 127)
    Ag = dq_e4m3(q) * np.repeat(scales, 32, axis=1)
    order = np.argsort(ids.ravel(), kind="stable")
    A_slot = np.empty_like(Ag)
    A_slot[order] = Ag                                     # row of slot s
    W = dq_e4m3(qw) * sw[..., None].astype(np.float64)
    ref = np.einsum("sk,snk->sn", A_slot, W[ids.ravel()]) * tw.ravel()[:, None]
    out = orc.moe_gemm(a_kind=orc.A_FP8_MX, a=q, a_sf=sf, a_sf_row=sf_row, w_kind=orc.W_FP8, w=qw, w_scale=sw,
                       topk_ids=ids, topk_w=tw, E=E, a_layout="grouped", out_layout="token_sum")
    assert np.allclose(out, ref.reshape(M, top_k, N).sum(axis=1), rtol=1e-12, atol=1e-12)


def test_per_expert_decomposition(orc):
    M, K, N, E, top_k = 40, 64, 32, 4, 2
    c = make_fp8_case(orc, M, K, N, E, top_k, seed=77)
    A = dq_e4m3(c["qa"]) * c["sa"][:, None].astype(np.float64)
    W = dq_e4m3(c["qw"]) * c["sw"][..., None].astype(np.float64)
    ref = np.zeros((M, N))
    for e in range(E):                                       # one unbalanced linear per expert
        m_idx, j_idx = np.nonzero(c["ids"] == e)
        if m_idx.size:
            ref[m_idx] += (A[m_idx] @ W[e].T) * c["tw"][m_idx, j_idx][:, None]
    out = orc.moe_gemm(a_kind=orc.A_FP8_TOKEN, a=c["qa"], a_scale=c["sa"], w_kind=orc.W_FP8, w=c["qw"],
                       w_scale=c["sw"], topk_ids=c["ids"], topk_w=c["tw"], E=E, out_layout="token_sum")
    assert np.allclose(out, ref, rtol=1e-12, atol=1e-12)


def test_permutation_invariance(orc):
    M, K, N, E, top_k = 23, 64, 16, 4, 2
    c = make_fp8_case(orc, M, K, N, E, top_k, seed=5)
    p = inputs.token_permutation(M, 5)
    kw = dict(a_kind=orc.A_FP8_TOKEN, w_kind=orc.W_FP8, w=c["qw"], w_scale=c["sw"], E=E)
    base = orc.moe_gemm(**kw, a=c["qa"], a_scale=c["sa"], topk_ids=c["ids"], topk_w=c["tw"]).reshape(M, top_k, N)
    perm = orc.moe_gemm(**kw, a=c["qa"][p], a_scale=c["sa"][p], topk_ids=c["ids"][p],
                        topk_w=c["tw"][p]).reshape(M, top_k, N)
    assert np.array_equal(perm, base[p])


def test_topk_all_experts_uniform_is_mean(orc):
    M, K, N, E = 9, 32, 16, 4
    c = make_fp8_case(orc, M, K, N, E, 2, seed=6)
    ids = np.tile(np.arange(E, dtype=np.int32), (M, 1))
    tw = np.full((M, E), 1.0 / E, dtype=np.float32)
    out = orc.moe_gemm(a_kind=orc.A_FP8_TOKEN, a=c["qa"], a_scale=c["sa"], w_kind=orc.W_FP8, w=c["qw"],
                       w_scale=c["sw"], topk_ids=ids, topk_w=tw, E=E, out_layout="token_sum")
    A = dq_e4m3(c["qa"]) * c["sa"][:, None].astype(np.float64)
    W = dq_e4m3(c["qw"]) * c["sw"][..., None].astype(np.float64)
    ref = sum(A @ W[e].T for e in range(E)) / E
    assert np.allclose(out, ref, rtol=1e-12, atol=1e-12)


def test_single_expert_is_plain_gemm(orc):
    M, K, N = 11, 48, 24
    c = make_fp8_case(orc, M, K, N, 1, 1, seed=7)
    out = orc.moe_gemm(a_kind=orc.A_FP8_TOKEN, a=c["qa"], a_scale=c["sa"], w_kind=orc.W_FP8, w=c["qw"],
                       w_scale=c["sw"], topk_ids=np.zeros((M, 1), np.int32), topk_w=None, E=1)
    A = dq_e4m3(c["qa"]) * c["sa"][:, None].astype(np.float64)
    W = dq_e4m3(c["qw"][0]) * c["sw"][0][:, None].astype(np.float64)
    assert np.allclose(out, np.matmul(A, W.T), rtol=1e-12, atol=1e-12)


def test_tolerance_helper_rejects_planted_error(orc):
    ref = np.random.default_rng(0).standard_normal((8, 8))
    ok, _ = orc.gemm_tolerance_ok(ref * (1 + 4e-3), ref)
    assert ok
    bad = ref.copy()
    bad[3, 3] += 0.5
    ok, ratio = orc.gemm_tolerance_ok(bad, ref)
    assert not ok and ratio > 1


def _ceil_5_significant_bits(x: np.ndarray) -> np.ndarray:
    """Smallest float with at most 5 significant bits that is >= x (x > 0, fp32),
    found with exact float64 arithmetic: 2^(e-4) * ceil(x / 2^(e-4)) where
    2^e <= x < 2^(e+1)."""
    x = x.astype(np.float64)
    e = np.floor(np.log2(x))
    e = np.where(2.0 ** e > x, e - 1, e)
    e = np.where(2.0 ** (e + 1) <= x, e + 1, e)
    ulp = 2.0 ** (e - 4)
    return (np.ceil(x / ulp) * ulp).astype(np.float32)


def test_int4_quant_rule_and_packing(orc):
    """Symmetric groups of 128: scale = amax/7 rounded up to 5 significant bits,
    codes rint(w/scale) clamped to [-7, 7], nibbles packed low-first;
    reconstruction within half a step; every q * scale a bf16 number."""
    w = inputs.expert_weights_f32(2, 24, 384, seed=41)
    w[0, 0, :128] = 0.0
    w[1, 3, 128:256] *= 1e-20
    q, s = orc.quant_rows_int4_f32(w)
    assert q.shape == (2, 24, 192) and s.shape == (2, 24, 3)
    lo = (q & 0xF).astype(np.int16)
    hi = (q >> 4).astype(np.int16)
    v = np.empty(w.shape, dtype=np.int16)
    v[..., 0::2] = np.where(lo >= 8, lo - 16, lo)
    v[..., 1::2] = np.where(hi >= 8, hi - 16, hi)
    assert v.min() >= -7 and v.max() <= 7
    g = w.reshape(2, 24, 3, 128)
    amax = np.abs(g).max(axis=-1)
    s0 = np.where(amax == 0, np.float32(1), (amax / np.float32(7)).astype(np.float32))
    exp_s = np.where(amax == 0, np.float32(1), _ceil_5_significant_bits(s0))
    assert np.array_equal(s, exp_s)
    # at most 5 significant bits, never below amax/7, less than 2^-4 relative above it
    assert np.all((s.view(np.uint32) & 0x7FFFF) == 0)
    assert np.all(s >= s0) and np.all(s.astype(np.float64) < s0.astype(np.float64) * (1 + 2.0 ** -4))
    ref = np.clip(np.rint((g / s[..., None]).astype(np.float32)), -7, 7).reshape(w.shape)
    assert np.array_equal(v, ref.astype(np.int16))
    rec = v.reshape(2, 24, 3, 128) * s[..., None].astype(np.float64)
    assert np.all(np.abs(rec - g) <= 0.5 * s[..., None] * (1 + 1e-6))
    assert np.all(v[0, 0, :128] == 0) and s[0, 0, 0] == 1.0
    # the dequantised weights are exact bf16 numbers (torch's bf16 cast leaves them unchanged)
    exact = (v.reshape(2, 24, 3, 128) * s[..., None].astype(np.float64)).astype(np.float32)
    assert np.array_equal(torch.from_numpy(exact).to(torch.bfloat16).float().numpy(), exact)


def test_int4_w4a16_vs_bruteforce(orc):
    M, K, N, E, top_k = 9, 256, 20, 3, 2
    a = inputs.activations_bf16(M, K, 42)
    w = inputs.expert_weights_f32(E, N, K, 42)
    ids, tw = inputs.routing(M, E, top_k, 42)
    q, s = orc.quant_rows_int4_f32(w)
    lo = (q & 0xF).astype(np.int16)
    hi = (q >> 4).astype(np.int16)
    v = np.empty((E, N, K), dtype=np.float64)
    v[..., 0::2] = np.where(lo >= 8, lo - 16, lo)
    v[..., 1::2] = np.where(hi >= 8, hi - 16, hi)
    # dequantised in fp64: q * scale
    W = v * np.repeat(s, 128, axis=-1).astype(np.float64)
    A = inputs.bf16_bits_to_f32(a).astype(np.float64)
    ref = dense_moe(A, W, ids, tw)
    out = orc.moe_gemm(a_kind=orc.A_BF16, a=a, w_kind=orc.W_INT4, w=q, w_scale=s, topk_ids=ids, topk_w=tw, E=E)
    assert np.allclose(out, ref.reshape(M * top_k, N), rtol=1e-12, atol=1e-12)
