"""Pins for the oracle's quantisers: closed forms, bounds implied by the
definitions, torch's e4m3 cast on the scaled values, and the worked MXFP8
scale-factor padding example of the TransformerEngine GroupedLinear page."""
import json
import math
import os

import numpy as np
import pytest
import torch

from quantized_moe_grouped_gb300 import inputs

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def e4m3_decode_torch(q):
    return torch.from_numpy(np.ascontiguousarray(q)).view(torch.float8_e4m3fn).to(torch.float64).numpy()


def test_quant_constant_row_closed_form(orc):
    for c in (1.0, -3.5, 0.0078125, 200.0):
        x = inputs.f32_to_bf16_bits(np.full((1, 64), c, dtype=np.float32))
        q, s = orc.quant_rows_fp8_bf16(x)
        assert s[0] == np.float32(abs(c)) / np.float32(448.0)
        assert np.all(q == (0x7E if c > 0 else 0xFE))


def test_quant_zero_row(orc):
    x = np.zeros((2, 32), dtype=np.uint16)
    x[1, ::2] = 0x8000                                         # -0.0
    q, s = orc.quant_rows_fp8_bf16(x)
    assert np.all(s == 1.0)
    assert np.all(q[0] == 0) and np.all(q[1, ::2] == 0x80) and np.all(q[1, 1::2] == 0)


def test_quant_rows_vs_torch_cast_and_bounds(orc):
    x = inputs.activations_bf16(37, 300, seed=5)
    q, s = orc.quant_rows_fp8_bf16(x)
    xf = inputs.bf16_bits_to_f32(x)
    amax = np.abs(xf).max(axis=1)
    assert np.array_equal(s, (amax / np.float32(448.0)).astype(np.float32))
    # the code of every element is torch's e4m3 cast of x/scale computed in fp32
    ref = torch.from_numpy((xf / s[:, None]).astype(np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(q, ref)
    # the amax element maps to +-448 (up to the rounding of the scale)
    d = e4m3_decode_torch(q)
    assert np.all(np.abs(d).max(axis=1) >= 416.0)
    # reconstruction error within half an e4m3 step (relative 2^-4) plus the subnormal floor
    err = np.abs(d * s[:, None] - xf)
    assert np.all(err <= np.abs(xf) * 2.0 ** -4 + s[:, None] * 2.0 ** -10 + 1e-30)


def test_quant_weights_fp8_per_channel(orc):
    w = inputs.expert_weights_f32(3, 40, 96, seed=1)
    q, s = orc.quant_rows_fp8_f32(w)
    assert q.shape == (3, 40, 96) and s.shape == (3, 40)
    ref = torch.from_numpy((w / s[..., None]).astype(np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(q, ref)


def test_quant_int8_properties(orc):
    w = inputs.expert_weights_f32(2, 50, 128, seed=2)
    q, s = orc.quant_rows_int8_f32(w)
    amax = np.abs(w).max(axis=-1)
    assert np.array_equal(s, (amax / np.float32(127.0)).astype(np.float32))
    assert np.all(np.abs(q.astype(np.int32)).max(axis=-1) == 127)
    assert np.all(q >= -127)
    err = np.abs(q.astype(np.float64) * s[..., None] - w)
    assert np.all(err <= s[..., None] * (0.5 + 1e-5))
    assert np.all(np.sign(q) * np.sign(w) >= 0)


def test_silu_quant_token_consistency(orc):
    y = inputs.activations_bf16(9, 2 * 96, seed=8)
    q, s = orc.silu_mul_quant_token(y)
    yf = inputs.bf16_bits_to_f32(y)
    h = orc.silu_mul_f32(yf[:, :96].ravel(), yf[:, 96:].ravel()).reshape(9, 96)
    amax = np.abs(h).max(axis=1)
    assert np.array_equal(s, (amax / np.float32(448.0)).astype(np.float32))
    ref = torch.from_numpy((h / s[:, None]).astype(np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(q, ref)
    g64, u64 = yf[:, :96].astype(np.float64), yf[:, 96:].astype(np.float64)
    h64 = g64 / (1.0 + np.exp(-g64)) * u64
    assert np.allclose(h, h64, rtol=1e-6, atol=1e-30)


def _mx_reference(h, block=32):
    """Exact restatement of the block rule: e = smallest integer with
    448*2^e >= amax (searched), codes = torch e4m3 cast of h*2^-e."""
    from fractions import Fraction
    R, I = h.shape
    sf = np.zeros((R, I // block), dtype=np.uint8)
    q = np.zeros((R, I), dtype=np.uint8)
    for r in range(R):
        for b in range(I // block):
            blk = h[r, b * block:(b + 1) * block]
            a = float(np.abs(blk).max())
            if a == 0:
                e = 0
            else:
                e = math.floor(math.log2(a)) - 10
                while Fraction(448) * Fraction(2) ** e < Fraction(a):
                    e += 1
                e = max(-127, min(127, e))
            sf[r, b] = e + 127
            q[r, b * block:(b + 1) * block] = torch.from_numpy(
                (blk * np.float32(2.0 ** -e)).astype(np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    return q, sf


def test_silu_quant_mx_two_expert_example(orc):
    spec = json.load(open(os.path.join(GOLDEN, "mxfp8_rowwise_sf_padding_two_experts.json")))
    E, rows, cols, pad = spec["experts"], spec["rows_per_expert"], spec["cols"], spec["sf_row_padding"]
    y = inputs.activations_bf16(E * rows, 2 * cols, seed=21)
    eoff = np.array([0, rows, 2 * rows], dtype=np.int32)
    soff = np.array([0, pad, 2 * pad], dtype=np.int32)
    q, sf = orc.silu_mul_quant_mx(y, eoff, soff)
    assert list(q.shape) == spec["whole_data_shape"]
    assert sf.shape == (E * pad, cols // spec["block"])
    blocks = [sf[e * pad:(e + 1) * pad] for e in range(E)]
    for blk in blocks:
        assert list(blk.shape) == spec["per_expert_rowwise_sf_padded_shape"]
        assert np.all(blk[rows:] == 0)                                     # padded rows
    # quantising each expert on its own gives identical data and padded sf
    for e in range(E):
        q1, sf1 = orc.silu_mul_quant_mx(y[e * rows:(e + 1) * rows], np.array([0, rows], np.int32),
                                        np.array([0, pad], np.int32))
        assert np.array_equal(q1, q[e * rows:(e + 1) * rows])
        assert np.array_equal(sf1, blocks[e])
    # and matches the exact block rule
    yf = inputs.bf16_bits_to_f32(y)
    h = orc.silu_mul_f32(yf[:, :cols].ravel(), yf[:, cols:].ravel()).reshape(E * rows, cols)
    qr, sfr = _mx_reference(h)
    assert np.array_equal(q, qr)
    for e in range(E):
        assert np.array_equal(blocks[e][:rows, : cols // 32], sfr[e * rows:(e + 1) * rows])


def test_silu_quant_mx_ragged_experts_and_pad_columns(orc):
    cnt = [5, 0, 130, 1]
    I = 96                                                                 # I/32 = 3 -> 4 sf columns
    R = sum(cnt)
    y = inputs.activations_bf16(R, 2 * I, seed=22)
    eoff = np.array([0] + list(np.cumsum(cnt)), dtype=np.int32)
    soff = np.array([0] + list(np.cumsum([-(-c // 128) * 128 for c in cnt])), dtype=np.int32)
    q, sf = orc.silu_mul_quant_mx(y, eoff, soff)
    assert sf.shape == (soff[-1], 4) and np.all(sf[:, 3] == 0)
    yf = inputs.bf16_bits_to_f32(y)
    h = orc.silu_mul_f32(yf[:, :I].ravel(), yf[:, I:].ravel()).reshape(R, I)
    qr, sfr = _mx_reference(h)
    assert np.array_equal(q, qr)
    for e in range(4):
        blk = sf[soff[e]:soff[e + 1]]
        assert np.array_equal(blk[: cnt[e], :3], sfr[eoff[e]:eoff[e + 1]])
        assert np.all(blk[cnt[e]:] == 0)


def test_srelu_exact_square(orc):
    x = inputs.f32_to_bf16_bits(np.concatenate([np.random.default_rng(4).standard_normal(2000) * 30,
                                               [0.0, -0.0, 1e-30, -1e-30, 3e38]]).astype(np.float32))
    xf = inputs.bf16_bits_to_f32(x)
    h = orc.srelu_f32(xf)
    with np.errstate(over="ignore"):
        ref = np.where(xf > 0, xf.astype(np.float64) ** 2, 0.0).astype(np.float32)   # exact, or overflow to inf
    assert np.array_equal(h, ref)
    assert np.all(h[xf <= 0] == 0) and not np.any(np.signbit(h))


def test_srelu_quant_token_and_mx(orc):
    y = inputs.activations_bf16(10, 96, seed=31)
    yf = inputs.bf16_bits_to_f32(y)
    h = np.where(yf > 0, yf * yf, np.float32(0)).astype(np.float32)
    q, s = orc.srelu_quant_token(y)
    assert np.array_equal(s, (np.abs(h).max(axis=1) / np.float32(448)).astype(np.float32))
    ref = torch.from_numpy((h / s[:, None]).astype(np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(q, ref)
    cnt = [3, 0, 7]
    y2 = inputs.activations_bf16(sum(cnt), 64, seed=32)
    eoff = np.array([0] + list(np.cumsum(cnt)), np.int32)
    soff = np.array([0] + list(np.cumsum([-(-c // 128) * 128 for c in cnt])), np.int32)
    q2, sf2 = orc.srelu_quant_mx(y2, eoff, soff)
    y2f = inputs.bf16_bits_to_f32(y2)
    h2 = np.where(y2f > 0, y2f * y2f, np.float32(0)).astype(np.float32)
    qr, sfr = _mx_reference(h2)
    assert np.array_equal(q2, qr)
    for e in range(3):
        assert np.array_equal(sf2[soff[e]:soff[e] + cnt[e], :2], sfr[eoff[e]:eoff[e + 1]])
        assert np.all(sf2[soff[e] + cnt[e]:soff[e + 1]] == 0)
