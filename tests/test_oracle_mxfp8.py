"""Pins of the oracle's MXFP8 quantisers and of the grouped GEMM on MXFP8
weights ("[PyTorch] Let GroupedLinear accept MXFP8 input and gradient",
Description and the two-expert example): the exact 1x32 block rule (searched),
columnwise blocks equal rowwise blocks of the transpose, the page's colwise
factor shapes, plain rows equal to the weight quantiser's rows, per-expert
padding, and a brute-force dense MoE on block-scaled operands."""
import json
import os

import numpy as np
import pytest
import torch

from quantized_moe_grouped_gb300 import inputs
from tests.test_oracle_quant import _mx_reference

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def dq_e4m3(q):
    return torch.from_numpy(np.ascontiguousarray(q)).view(torch.float8_e4m3fn).to(torch.float64).numpy()


def test_weight_rows_exact_block_rule(orc):
    w = inputs.expert_weights_f32(3, 40, 96, seed=31)
    w[0, 0, :32] = 0.0                                   # an all-zero block -> byte 127, zero codes
    w[1, 2, 32:64] *= 1e-30                              # tiny block
    w[2, 5, 64:] *= 1e6                                  # large block
    q, sf = orc.quant_rows_mxfp8_f32(w)
    assert q.shape == w.shape and sf.shape == (3 * 40, 4) and np.all(sf[:, 3] == 0)
    qr, sfr = _mx_reference(w.reshape(-1, 96))
    assert np.array_equal(q.reshape(-1, 96), qr)
    assert np.array_equal(sf[:, :3], sfr)
    assert sf[0, 0] == 127 and np.all(q[0, 0, :32] == 0)


def test_plain_rows_equal_weight_rows_and_expert_padding(orc):
    cnt = [37, 0, 64, 3]
    R, I = sum(cnt), 128
    y = inputs.activations_bf16(R, I, seed=32)
    eoff = np.array([0] + list(np.cumsum(cnt)), dtype=np.int32)
    soff = np.array([0] + list(np.cumsum([-(-c // 128) * 128 for c in cnt])), dtype=np.int32)
    q, sf = orc.quant_mxfp8_rows(y, eoff, soff)
    qw, sfw = orc.quant_rows_mxfp8_f32(inputs.bf16_bits_to_f32(y))
    assert np.array_equal(q, qw)
    for e in range(4):
        blk = sf[soff[e]:soff[e + 1]]
        assert np.array_equal(blk[: cnt[e]], sfw[eoff[e]:eoff[e + 1]])
        assert np.all(blk[cnt[e]:] == 0)


@pytest.mark.parametrize("R,C", [(64, 128), (128, 96), (256, 160)])
def test_colwise_is_rowwise_of_transpose(orc, R, C):
    x = inputs.activations_bf16(R, C, seed=R + C)
    x[5:37, 7] = 0                                        # one all-zero column block
    q, sf = orc.quant_mxfp8_cols(x)
    xt = np.ascontiguousarray(inputs.bf16_bits_to_f32(x).T)  # [C, R]
    qt, sft = orc.quant_rows_mxfp8_f32(xt)
    assert np.array_equal(q, qt.T)
    nrb = R // 32
    assert np.array_equal(sf[:nrb, :C], sft[:, :nrb].T)
    assert np.all(sf[nrb:] == 0) and np.all(sf[:, C:] == 0)


def test_colwise_ragged_last_block(orc):
    R, C = 70, 32                                        # blocks of 32, 32 and 6 rows
    x = inputs.activations_bf16(R, C, seed=33)
    q, sf = orc.quant_mxfp8_cols(x)
    xf = inputs.bf16_bits_to_f32(x)
    for rb, (r0, r1) in enumerate([(0, 32), (32, 64), (64, 70)]):
        blk = np.ascontiguousarray(xf[r0:r1].T)          # [C, rows of the block]
        pad = np.zeros((C, 32), dtype=np.float32)
        pad[:, : r1 - r0] = blk                          # zeros do not change the amax
        qr, sfr = _mx_reference(pad)
        assert np.array_equal(sf[rb, :C], sfr[:, 0])
        assert np.array_equal(q[r0:r1], qr[:, : r1 - r0].T)


def test_colwise_sf_shapes_of_the_page(orc):
    spec = json.load(open(os.path.join(GOLDEN, "mxfp8_colwise_sf_shapes.json")))
    for case in spec["cases"]:
        R, C = case["input_shape"]
        x = inputs.activations_bf16(R, C, seed=R)
        q, sf = orc.quant_mxfp8_cols(x)
        assert list(sf.shape) == case["colwise_sf_shape"]
        nrb = R // spec["block_rows"]
        assert np.all(sf[:nrb] != 0) and np.all(sf[nrb:] == 0)
    # two [64, 128] experts quantised one by one == the concatenation quantised as a whole
    x = inputs.activations_bf16(128, 128, seed=34)
    q, sf = orc.quant_mxfp8_cols(x)
    for e in range(2):
        q1, sf1 = orc.quant_mxfp8_cols(x[64 * e:64 * (e + 1)])
        assert np.array_equal(q1, q[64 * e:64 * (e + 1)])
        assert np.array_equal(sf1[:2], sf[2 * e:2 * e + 2])


def test_gemm_mx_weights_vs_bruteforce(orc):
    """Both operands block-scaled: A MX rows (grouped), W MX rows along K."""
    M, K, N, E, top_k = 10, 96, 40, 3, 2
    ids, tw = inputs.routing(M, E, top_k, 35)
    T = M * top_k
    al = orc.moe_align(ids, E, 128)
    eoff, poff = al["expert_offsets"], al["padded_offsets"]
    y = inputs.activations_bf16(T, K, 35)
    qa, sfa = orc.quant_mxfp8_rows(y, eoff, poff)
    sf_row = np.empty(T, dtype=np.int64)
    for e in range(E):
        sf_row[eoff[e]:eoff[e + 1]] = poff[e] + np.arange(eoff[e + 1] - eoff[e])
    w = inputs.expert_weights_f32(E, N, K, 35)
    qw, sfw = orc.quant_rows_mxfp8_f32(w)
    A = dq_e4m3(qa) * np.repeat(2.0 ** (sfa[sf_row][:, : K // 32].astype(np.float64) - 127), 32, axis=1)
    W = dq_e4m3(qw) * np.repeat(2.0 ** (sfw[:, : K // 32].astype(np.float64) - 127), 32, axis=1).reshape(E, N, K)
    order = np.argsort(ids.ravel(), kind="stable")
    A_slot = np.empty_like(A)
    A_slot[order] = A
    ref = np.einsum("sk,snk->sn", A_slot, W[ids.ravel()]) * tw.ravel()[:, None]
    out = orc.moe_gemm(a_kind=orc.A_FP8_MX, a=qa, a_sf=sfa, a_sf_row=sf_row, w_kind=orc.W_MX, w=qw, w_scale=None,
                       w_sf=sfw, topk_ids=ids, topk_w=tw, E=E, a_layout="grouped", out_layout="token_sum")
    assert np.allclose(out, ref.reshape(M, top_k, N).sum(axis=1), rtol=1e-12, atol=1e-12)
    # and the reconstruction error of the MX weights is within e4m3's half-ulp bound per block
    assert np.all(np.abs(W - w.astype(np.float64)) <= np.abs(w) * 2.0 ** -4 + 2.0 ** -9 * np.abs(W).max())


@pytest.mark.parametrize("E,N,K", [(2, 256, 128), (3, 300, 416), (1, 16, 32)])
def test_weight_sf_tiling_is_a_permutation_with_2pow0_padding(orc, E, N, K):
    """Undo the tiling with array reshapes (blocks [E][NB][KB][h][i][c][b]) and
    recover the natural factors; rows past N hold 127 (2^0)."""
    ld = (K // 32 + 3) // 4 * 4
    sf = np.random.default_rng(E * N + K).integers(0, 255, size=(E * N, ld), dtype=np.uint8)
    t = orc.mx_weight_sf_tiled(sf, E, N, K)
    NB, KB = -(-N // 256), -(-K // 128)
    v = t.reshape(E, NB, KB, 2, 32, 4, 4).transpose(0, 1, 3, 5, 4, 2, 6)   # e nb h c i kb b
    nat = v.reshape(E, NB * 256, KB * 4)
    assert np.array_equal(nat[:, :N, :], sf.reshape(E, N, ld)[:, :, : KB * 4])
    assert np.all(nat[:, N:, :] == 127)
