"""Exact read-out of the dequantised weights through each grouped GEMM.

Every activation row m is one-hot: a single 1.0 at column k = m.  The fp32
accumulator of output (m, n) then holds the one product 1.0 * w[e, n, m]
(e = the token's expert), and the epilogue's remaining factors (activation
scale, routing weight) are 1.  So output (m, n) must equal bf16 of the
dequantised weight: the code's value times its scale in fp32, cast to bf16,
both by torch on the host (library routines).  A wrong operand layout,
swizzle, nibble order, expert or scale index, or a rounding step that differs
from the per-weight dequantisation, moves or changes values.  Values are
compared, not bits: an exact zero takes its sign from the sum of the other
positions' zero products.
"""
import numpy as np
import pytest
import torch

from tests.gpu_util import dev, status, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def q():
    import quantized_moe_grouped_gb300 as q
    q.load_library()
    return q


def scales(rng, shape):
    """fp32 scales of either sign with exponents in [-60, 60] and random mantissas."""
    bits = ((rng.integers(0, 2, shape, dtype=np.uint32) << np.uint32(31)) |
            (rng.integers(127 - 60, 127 + 61, shape, dtype=np.uint32) << np.uint32(23)) |
            rng.integers(0, 1 << 23, shape, dtype=np.uint32))
    return bits.view(np.float32)


def one_hot_rows(M, K):
    a = torch.zeros(M, K, dtype=torch.float32)
    a[torch.arange(M), torch.arange(M)] = 1.0
    return a


def routing(M, E):
    ids = (np.arange(M, dtype=np.int32) % E).reshape(M, 1)  # token m -> expert m mod E
    return ids


def expected_rows(wdq, ids):
    """Output row m = dequantised weights of expert ids[m] at column k = m, as bf16."""
    M = ids.shape[0]
    return torch.stack([wdq[int(ids[m, 0]), :, m] for m in range(M)]).to(torch.bfloat16)


def run_align(q, ids, E, BM):
    return q.moe_align_block_size(to_dev(ids), E, BM)


@pytest.mark.parametrize("BM", [16, 32, 64, 128, 256])
def test_w8a8_readout(q, BM):
    E, N, K = 3, 400, 272
    M = K
    rng = np.random.default_rng(BM)
    codes = rng.integers(0, 256, (E, N, K), dtype=np.uint8)
    codes[(codes & 0x7F) == 0x7F] = 0x3C  # no NaN codes
    ws = scales(rng, (E, N))
    wdq = torch.from_numpy(codes).view(torch.float8_e4m3fn).float() * torch.from_numpy(ws)[:, :, None]
    ids = routing(M, E)
    a = one_hot_rows(M, K).to(torch.float8_e4m3fn).view(torch.uint8).to(dev())
    st = status()
    out = q.moe_gemm_w8a8(a, torch.ones(M, dtype=torch.float32, device=dev()), to_dev(codes), to_dev(ws),
                          run_align(q, ids, E, BM), None, M=M, top_k=1, BM=BM, d_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    got, exp = out.cpu().float(), expected_rows(wdq, ids).float()
    bad = torch.nonzero(got != exp)
    assert bad.numel() == 0, (bad[:4].tolist(), got[tuple(bad[0])].item(), exp[tuple(bad[0])].item())


@pytest.mark.parametrize("BM", [16, 32, 64, 128, 256])
def test_w8a16_readout(q, BM):
    E, N, K = 3, 400, 272
    M = K
    rng = np.random.default_rng(100 + BM)
    codes = rng.integers(-128, 128, (E, N, K), dtype=np.int8)
    ws = scales(rng, (E, N))
    wdq = torch.from_numpy(codes).float() * torch.from_numpy(ws)[:, :, None]
    ids = routing(M, E)
    a = one_hot_rows(M, K).to(torch.bfloat16).to(dev())
    st = status()
    out = q.moe_gemm_w8a16(a, to_dev(codes), to_dev(ws), run_align(q, ids, E, BM), None, M=M, top_k=1, BM=BM,
                           d_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    got, exp = out.cpu().float(), expected_rows(wdq, ids).float()
    bad = torch.nonzero(got != exp)
    assert bad.numel() == 0, (bad[:4].tolist(), got[tuple(bad[0])].item(), exp[tuple(bad[0])].item())


@pytest.mark.parametrize("BM", [64, 128, 256])
def test_w4a16_readout(q, BM):
    """Packed int4 (element 2j in the low nibble of byte j) times its group's
    scale (groups of 128 along K): every code in every nibble position."""
    E, N, K = 3, 400, 256
    M = K
    rng = np.random.default_rng(200 + BM)
    v = rng.integers(-8, 8, (E, N, K), dtype=np.int8)
    nib = (v & 0xF).astype(np.uint8)
    packed = nib[..., 0::2] | (nib[..., 1::2] << np.uint8(4))
    ws = scales(rng, (E, N, K // 128))
    wdq = torch.from_numpy(v).float() * torch.from_numpy(ws).repeat_interleave(128, dim=-1)
    ids = routing(M, E)
    a = one_hot_rows(M, K).to(torch.bfloat16).to(dev())
    st = status()
    out = q.moe_gemm_w4a16(a, to_dev(packed), to_dev(ws), run_align(q, ids, E, BM), None, M=M, top_k=1, BM=BM,
                           d_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    got, exp = out.cpu().float(), expected_rows(wdq, ids).float()
    bad = torch.nonzero(got != exp)
    assert bad.numel() == 0, (bad[:4].tolist(), got[tuple(bad[0])].item(), exp[tuple(bad[0])].item())
