"""GPU parity of the integer and quantisation kernels against the CPU oracle:
bit-exact sorting/padding, e4m3/int8 codes, scales, SwiGLU h and MX scale bytes."""
import numpy as np
import pytest
import torch

from quantized_moe_grouped_gb300 import inputs
from tests.gpu_util import bf16_to_np_f32, dev, status, to_dev, to_dev_bf16

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def q():
    import quantized_moe_grouped_gb300 as q
    q.load_library()
    return q


def test_e4m3_conversion_exhaustive(q, orc):
    """All 2^32 fp32 bit patterns except NaNs: hardware conversion == oracle encoder."""
    chunk = 1 << 26
    for c in range((1 << 32) // chunk):
        bits = np.arange(chunk, dtype=np.uint32) + np.uint32(c * chunk)
        x = bits.view(np.float32)
        keep = ~np.isnan(x)
        x = x[keep]
        got = q.debug_e4m3_encode(to_dev(x)).cpu().numpy()
        ref = orc.e4m3_from_f32_array(x)
        bad = np.nonzero(got != ref)[0]
        assert bad.size == 0, (c, x[bad[:4]], got[bad[:4]], ref[bad[:4]])


def test_int8_to_bf16_exhaustive(q):
    x = np.arange(-128, 128, dtype=np.int8)
    y = q.debug_int8_to_bf16(to_dev(x)).float().cpu().numpy()
    assert np.array_equal(y, x.astype(np.float32))


def test_silu_sequence_bitexact(q, orc):
    g = np.random.default_rng(1)
    gs = np.concatenate([
        (g.random(1 << 22, dtype=np.float32) * 220 - 110),
        g.standard_normal(1 << 21).astype(np.float32) * 3,
        np.array([0.0, -0.0, 89.0, -89.0, 104.0, -104.0, 1e-30, -1e-30, 3e38, -3e38], np.float32),
        # -g * log2 e rounds to a half-integer (41.5, 45.5, 53.5, 67.5): n = rint of the
        # rounded product, not of the exact one
        np.array([3253084151, 3254537786, 3256112480, 3258656341], np.uint32).view(np.float32)])
    us = g.standard_normal(gs.size).astype(np.float32)
    got = q.debug_silu_mul(to_dev(gs), to_dev(us)).cpu().numpy()
    ref = orc.silu_mul_f32_array(gs, us)
    assert np.array_equal(got.view(np.uint32), ref.view(np.uint32))


def test_silu_sequence_exhaustive(q, orc):
    """h = silu(g) * u on the GPU equals the oracle's op sequence bit for bit
    for every fp32 g in [-104, 89] (the range the exp reduction does not
    clamp; both signs of zero included), each g paired with a multiplier u in
    [1, 2) whose mantissa is taken from g's bit pattern (so the final product
    rounds too)."""
    chunk = 1 << 26
    spans = [(0, int(np.float32(89.0).view(np.uint32)) + 1),
             (0x80000000, int(np.float32(-104.0).view(np.uint32)) + 1)]
    for lo, hi in spans:
        for start in range(lo, hi, chunk):
            n = min(chunk, hi - start)
            b = torch.arange(start, start + n, dtype=torch.int64, device=dev())
            ub = 0x3F800000 | ((b ^ (b >> 9)) & 0x7FFFFF)
            g = torch.where(b >= (1 << 31), b - (1 << 32), b).to(torch.int32).view(torch.float32)
            u = ub.to(torch.int32).view(torch.float32)
            got = q.debug_silu_mul(g, u).cpu().numpy().view(np.uint32)
            del b, ub, g, u
            bits = np.arange(start, start + n, dtype=np.uint64).astype(np.uint32)
            un = (np.uint32(0x3F800000) | ((bits ^ (bits >> np.uint32(9))) & np.uint32(0x7FFFFF))).view(np.float32)
            ref = orc.silu_mul_f32_array(bits.view(np.float32), un).view(np.uint32)
            bad = np.nonzero(got != ref)[0]
            assert bad.size == 0, (hex(start), bits[bad[:4]], got[bad[:4]], ref[bad[:4]])


@pytest.mark.parametrize("M,E,BM", [(64, 8, 16), (64, 8, 32), (200, 8, 64), (4096, 8, 128), (4096, 8, 256),
                                    (17, 3, 16), (1, 1, 16), (3000, 64, 32), (512, 256, 16),
                                    (1024, 256, 16), (1023, 8, 64), (20000, 8, 128)])
def test_align_bitexact(q, orc, M, E, BM):
    """Single-CTA kernel below 2048 slots, the cluster kernel from 2048 on (one
    id batch per lane up to 32768 slots, several beyond)."""
    ids, _ = inputs.routing(M, E, 2 if E > 1 else 1, seed=M + E)
    st = status()
    al = q.moe_align_block_size(to_dev(ids), E, BM, d_status=st)
    ref = orc.moe_align(ids, E, BM)
    cap = q.align_max_padded(ids.size, E, BM)
    assert int(st.item()) == 0
    assert int(al["num_post_padded"].item()) == ref["num_post_padded"]
    assert np.array_equal(al["sorted_ids"].cpu().numpy(), ref["sorted_ids"][:cap])
    assert np.array_equal(al["expert_ids"].cpu().numpy(), ref["expert_ids"][: cap // BM])
    assert np.array_equal(al["expert_offsets"].cpu().numpy(), ref["expert_offsets"])
    assert np.array_equal(al["padded_offsets"].cpu().numpy(), ref["padded_offsets"])


def test_align_skewed_empty_and_invalid(q, orc):
    ids, _ = inputs.routing(4096, 8, 2, seed=4000, zipf_s=1.2)
    al = q.moe_align_block_size(to_dev(ids), 8, 128)
    ref = orc.moe_align(ids, 8, 128)
    assert np.array_equal(al["sorted_ids"].cpu().numpy(), ref["sorted_ids"])
    # empty input
    al0 = q.moe_align_block_size(to_dev(np.zeros(0, np.int32)), 8, 16)
    assert int(al0["num_post_padded"].item()) == 0
    assert np.all(al0["sorted_ids"].cpu().numpy() == 0)     # sentinel T == 0
    assert np.all(al0["expert_ids"].cpu().numpy() == -1)
    # ids outside [0, E) are dropped and flagged
    bad = np.array([0, 1, 9, -1, 1, 2], dtype=np.int32)
    st = status()
    alb = q.moe_align_block_size(to_dev(bad), 3, 16, d_status=st)
    refb = orc.moe_align(bad, 3, 16)
    assert int(st.item()) == q.DEV_INVALID_EXPERT and refb["invalid"]
    assert np.array_equal(alb["sorted_ids"].cpu().numpy(), refb["sorted_ids"])
    # the same on the cluster kernel (several thousand slots, a few invalid ids in two CTAs' ranges)
    big, _ = inputs.routing(3000, 8, 2, seed=4001)
    big = big.ravel().copy()
    big[[5, 4100, 5999]] = [8, -3, 100]
    st = status()
    alc = q.moe_align_block_size(to_dev(big), 8, 64, d_status=st)
    refc = orc.moe_align(big, 8, 64)
    assert int(st.item()) == q.DEV_INVALID_EXPERT and refc["invalid"]
    assert np.array_equal(alc["sorted_ids"].cpu().numpy(), refc["sorted_ids"])
    assert np.array_equal(alc["expert_ids"].cpu().numpy(), refc["expert_ids"][: alc["expert_ids"].numel()])


@pytest.mark.parametrize("rows,cols", [(64, 128), (64, 4096), (333, 6144), (5, 100), (7, 24), (1, 8)])
def test_quant_act_bitexact(q, orc, rows, cols):
    x = inputs.activations_bf16(rows, cols, seed=rows + cols)
    x[0, :] = 0                                   # zero row -> scale 1
    if rows > 2:
        x[1, ::3] = 0x8000                        # negative zeros
        x[2, :] = x[2, 0]                         # constant row
    qa, sa = q.quant_act_fp8(to_dev_bf16(x))
    ref_q, ref_s = orc.quant_rows_fp8_bf16(x)
    assert np.array_equal(qa.cpu().numpy(), ref_q)
    assert np.array_equal(sa.cpu().numpy().view(np.uint32), ref_s.view(np.uint32))


def test_quant_act_strided_rows(q, orc):
    x = inputs.activations_bf16(40, 256, seed=3)
    xd = to_dev_bf16(x)[:, :200]                  # ldx = 256, cols = 200
    qa, sa = q.quant_act_fp8(xd)
    ref_q, ref_s = orc.quant_rows_fp8_bf16(np.ascontiguousarray(x[:, :200]))
    assert np.array_equal(qa.cpu().numpy(), ref_q) and np.array_equal(sa.cpu().numpy(), ref_s)


@pytest.mark.parametrize("E,N,K", [(8, 256, 128), (3, 40, 100), (2, 64, 4096)])
def test_quant_weights_bitexact(q, orc, E, N, K):
    w = inputs.expert_weights_f32(E, N, K, seed=E * N)
    w[0, 0, :] = 0
    wq, ws = q.quant_weight_fp8(to_dev(w))
    rq, rs = orc.quant_rows_fp8_f32(w)
    assert np.array_equal(wq.cpu().numpy(), rq) and np.array_equal(ws.cpu().numpy(), rs)
    wq8, ws8 = q.quant_weight_int8(to_dev(w))
    rq8, rs8 = orc.quant_rows_int8_f32(w)
    assert np.array_equal(wq8.cpu().numpy(), rq8) and np.array_equal(ws8.cpu().numpy(), rs8)


@pytest.mark.parametrize("R,I", [(64, 256), (300, 1024), (8, 14336), (3, 40), (5, 8200)])
def test_silu_quant_token_bitexact(q, orc, R, I):
    y = inputs.activations_bf16(R, 2 * I, seed=R + I)
    y[0, :] = 0
    qq, ss = q.silu_mul_quant(to_dev_bf16(y))
    rq, rs = orc.silu_mul_quant_token(y)
    assert np.array_equal(qq.cpu().numpy(), rq)
    assert np.array_equal(ss.cpu().numpy().view(np.uint32), rs.view(np.uint32))


@pytest.mark.parametrize("cnt,I", [([64, 64], 128), ([5, 0, 130, 1, 300, 0, 7, 9], 96),
                                   ([1000, 40, 0, 513], 1024), ([3], 16384)])
def test_silu_quant_mx_bitexact(q, orc, cnt, I):
    R = sum(cnt)
    E = len(cnt)
    y = inputs.activations_bf16(R, 2 * I, seed=R + I + E)
    y[0, :64] = 0                                             # an all-zero 1x32 block
    eoff = np.array([0] + list(np.cumsum(cnt)), dtype=np.int32)
    soff = np.array([0] + list(np.cumsum([-(-c // 128) * 128 for c in cnt])), dtype=np.int32)
    ld = q.mx_sf_ld(I)
    sf = torch.full((int(soff[-1]) + 5, ld), 0xAB, dtype=torch.uint8, device=dev())   # poison, incl. 5 spare rows
    qq, sfo = q.silu_mul_quant(to_dev_bf16(y), q.SCALE_MX_1X32, expert_offsets=to_dev(eoff),
                               sf_padded_offsets=to_dev(soff), sf=sf)
    rq, rsf = orc.silu_mul_quant_mx(y, eoff, soff)
    assert np.array_equal(qq.cpu().numpy(), rq)
    got = sfo.cpu().numpy()
    assert np.array_equal(got[: soff[-1]], rsf)
    assert np.all(got[soff[-1]:] == 0xAB)                     # nothing written past the padded rows


def test_silu_quant_mx_whole_equals_per_expert(q):
    """Quantising the concatenated expert rows as a whole equals quantising
    each expert's rows on its own: identical data, identical padded scale
    factors (the two-expert example of the TransformerEngine MXFP8 page)."""
    cnt, I = [64, 64], 128
    y = inputs.activations_bf16(128, 2 * I, seed=99)
    yd = to_dev_bf16(y)
    eoff = to_dev(np.array([0, 64, 128], np.int32))
    soff = to_dev(np.array([0, 128, 256], np.int32))
    qw, sfw = q.silu_mul_quant(yd, q.SCALE_MX_1X32, expert_offsets=eoff, sf_padded_offsets=soff, sf_rows=256)
    for e in range(2):
        qe, sfe = q.silu_mul_quant(yd[e * 64:(e + 1) * 64], q.SCALE_MX_1X32,
                                   expert_offsets=to_dev(np.array([0, 64], np.int32)),
                                   sf_padded_offsets=to_dev(np.array([0, 128], np.int32)), sf_rows=128)
        assert torch.equal(qe, qw[e * 64:(e + 1) * 64])
        assert torch.equal(sfe, sfw[e * 128:(e + 1) * 128])
        assert sfe.shape == (128, 4)


@pytest.mark.parametrize("M,K,E,top_k,BM", [(64, 4096, 8, 2, 32), (1, 128, 8, 2, 16), (333, 256, 8, 2, 64),
                                            (512, 4096, 8, 2, 128), (100, 64, 5, 3, 16), (2100, 128, 8, 2, 128)])
def test_fused_align_quant_bitexact(q, orc, M, K, E, top_k, BM):
    """One-launch align + sorted quantisation == the oracle's align and per-token
    codes placed at every valid padded position (the last case exceeds the
    one-launch limit and takes the two-launch path)."""
    x = inputs.activations_bf16(M, K, seed=M + K)
    ids, _ = inputs.routing(M, E, top_k, seed=M + K)
    st = status()
    al, qq, ss = q.moe_align_quant_fp8(to_dev_bf16(x), to_dev(ids), E, BM, d_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    ref = orc.moe_align(ids, E, BM)
    cap = al["sorted_ids"].numel()
    assert np.array_equal(al["sorted_ids"].cpu().numpy(), ref["sorted_ids"][:cap])
    assert np.array_equal(al["expert_ids"].cpu().numpy(), ref["expert_ids"][: cap // BM])
    assert np.array_equal(al["expert_offsets"].cpu().numpy(), ref["expert_offsets"])
    assert np.array_equal(al["padded_offsets"].cpu().numpy(), ref["padded_offsets"])
    assert int(al["num_post_padded"].item()) == ref["num_post_padded"]
    rq, rs = orc.quant_rows_fp8_bf16(x)
    srt = ref["sorted_ids"][: ref["num_post_padded"]]
    valid = np.nonzero(srt < M * top_k)[0]
    assert np.array_equal(qq.cpu().numpy()[valid], rq[srt[valid] // top_k])
    assert np.array_equal(ss.cpu().numpy()[valid], rs[srt[valid] // top_k])


@pytest.mark.parametrize("M,K,E,top_k,BM,misaligned", [
    (300, 512, 6, 3, 64, False),     # one warp per token (slot table in shared memory), top_k = 3
    (300, 512, 6, 3, 64, True),      # sorted_ids only 4-byte aligned: one warp per padded position
    (5000, 256, 8, 2, 128, False),   # T = 10000 > 8192 slots: one warp per padded position
    (4200, 6144, 8, 2, 128, False),  # T = 8400 > 8192, rows of 6144 values: bulk row copies
])
def test_quant_act_fp8_sorted_bitexact(q, orc, M, K, E, top_k, BM, misaligned):
    """Every kernel behind quant_act_fp8_sorted: valid padded positions hold the
    oracle's per-token codes and scale of the slot's token, pad positions zero
    codes and scale 0; a slot with an invalid expert id is not placed."""
    x = inputs.activations_bf16(M, K, seed=M + K)
    ids, _ = inputs.routing(M, E, top_k, seed=M + K)
    ids[3, 0] = E + 5
    st = status()
    al = q.moe_align_block_size(to_dev(ids), E, BM, d_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == q.DEV_INVALID_EXPERT
    if misaligned:
        buf = torch.empty(al["sorted_ids"].numel() + 1, dtype=torch.int32, device=dev())
        buf[1:].copy_(al["sorted_ids"])
        al = dict(al, sorted_ids=buf[1:])
    qq, ss = q.quant_act_fp8_sorted(to_dev_bf16(x), al, top_k)
    torch.cuda.synchronize()
    ref = orc.moe_align(ids, E, BM)
    rq, rs = orc.quant_rows_fp8_bf16(x)
    srt = ref["sorted_ids"][: ref["num_post_padded"]]
    T = M * top_k
    valid = np.nonzero(srt < T)[0]
    pads = np.nonzero(srt >= T)[0]
    qn, sn = qq.cpu().numpy(), ss.cpu().numpy()
    assert np.array_equal(qn[valid], rq[srt[valid] // top_k])
    assert np.array_equal(sn[valid], rs[srt[valid] // top_k])
    assert not np.any(qn[pads]) and not np.any(sn[pads])
    assert 3 * top_k not in set(srt[valid].tolist())


def test_silu_reciprocal_exhaustive(q):
    """The reciprocal in the SiLU, 1/d with d = 1 + exp(-g) >= 1, equals IEEE
    fp32 division (numpy) bit for bit for every fp32 d in [1, 2^126), and for
    the largest values and +inf (which take the IEEE reciprocal)."""
    lo = int(np.float32(1.0).view(np.uint32))
    hi = int(np.float32(2.0 ** 126).view(np.uint32))
    chunk = 1 << 26
    one = np.float32(1.0)
    for start in range(lo, hi, chunk):
        n = min(chunk, hi - start)
        d = torch.arange(start, start + n, dtype=torch.int64, device=dev()).to(torch.int32).view(torch.float32)
        got = q.debug_rcp_ge1(d).cpu().numpy()
        dn = d.cpu().numpy()
        ref = one / dn
        bad = np.nonzero(got.view(np.uint32) != ref.view(np.uint32))[0]
        assert bad.size == 0, (dn[bad[:4]], got[bad[:4]], ref[bad[:4]])
    edge = np.array([2.0 ** 126, 1.5 * 2.0 ** 126, 2.0 ** 127, 3.0e38, np.finfo(np.float32).max, np.inf],
                    dtype=np.float32)
    got = q.debug_rcp_ge1(to_dev(edge)).cpu().numpy()
    assert np.array_equal(got.view(np.uint32), (one / edge).view(np.uint32))


@pytest.mark.parametrize("s", [np.float32(1.0), np.float32(1.0 / 448.0), np.float32(3.0), np.float32(0.0123456),
                               np.nextafter(np.float32(2.0), np.float32(0)), np.float32(7.0e-3) / np.float32(448.0),
                               # a huge scale (Markstein path from |x| >= 2^-99 s > 1) and a subnormal
                               # one (every dividend below the threshold: IEEE path throughout)
                               np.float32(1.37 * 2.0 ** 100), np.float32(1.5 * 2.0 ** -130)])
def test_division_by_row_scale_exhaustive(q, s):
    """The kernels' division by a row scale s equals IEEE fp32 division (numpy)
    bit for bit for every fp32 dividend the kernels can pass, |x| <= 512 s
    (they divide values bounded by amax = 448 s)."""
    chunk = 1 << 26
    sd = np.float32(s)
    lim = np.float32(512.0) * sd
    for c in range((1 << 32) // chunk):
        bits = np.arange(chunk, dtype=np.uint32) + np.uint32(c * chunk)
        x = bits.view(np.float32)
        x = x[np.isfinite(x) & (np.abs(x) <= lim)]
        if x.size == 0:
            continue
        got = q.debug_div_by_scale(to_dev(x), float(sd)).cpu().numpy()
        ref = (x / sd).astype(np.float32)
        bad = np.nonzero(got.view(np.uint32) != ref.view(np.uint32))[0]
        assert bad.size == 0, (float(sd), x[bad[:4]], got[bad[:4]], ref[bad[:4]])


# Every quantiser's code for x / s (row scale s): the correction of the reciprocal
# product above its guard (2^-99 max(1, s)), the IEEE division below it.  The whole
# range |x| <= 512 s for the typical activation scale and the tiny ones; for the
# others every dividend within a factor 4 of the guard (the switch between the two
# paths) and every 509th bit pattern elsewhere.
QUANT_SCALES = [(np.float32(1.0 / 448.0), True), (np.float32(1.0), False), (np.float32(1.37 * 2.0 ** 100), False),
                (np.float32(3.0), False), (np.float32(0.0123456), False),
                (np.float32(7.0e-3) / np.float32(448.0), False),
                # tiny scales: every dividend lies below the guard (the IEEE path), whole range
                (np.float32(1.5 * 2.0 ** -130), True),     # subnormal: RN(1/s) overflows
                (np.float32(2.0 ** -127), True), (np.float32(0.75 * 2.0 ** -120), True),
                (np.nextafter(np.float32(1.0), np.float32(0)), False)]


def _dividend_bits(lim, guard, full):
    """Positive fp32 bit patterns to check, in chunks: all up to lim (full), or
    all in [guard / 4, 4 guard) and every 509th one elsewhere up to lim."""
    f32_bits = lambda v: int(np.float32(v).view(np.uint32))
    top = min(f32_bits(lim) + 1, f32_bits(np.finfo(np.float32).max) + 1)
    lo, hi = (0, top) if full else (min(top, f32_bits(guard / 4)), min(top, f32_bits(4 * guard)))
    chunk = 1 << 26
    for b in range(0, lo, chunk * 509):
        yield np.arange(b, min(lo, b + chunk * 509), 509, dtype=np.uint32)
    for b in range(lo, hi, chunk):
        yield np.arange(b, min(hi, b + chunk), dtype=np.uint32)
    for b in range(hi, top, chunk * 509):
        yield np.arange(b, min(top, b + chunk * 509), 509, dtype=np.uint32)


@pytest.mark.parametrize("s,full", QUANT_SCALES)
def test_quant_codes_by_row_scale_exhaustive(q, orc, s, full):
    """The e4m3 code every quantiser writes for x / s equals the oracle's e4m3
    conversion of the IEEE fp32 quotient (numpy), for dividends of both signs
    up to |x| <= 512 s (the quantisers divide values bounded by amax = 448 s)."""
    sd = np.float32(s)
    lim = np.float32(512.0) * sd
    guard = np.float32(2.0 ** -99) * max(np.float32(1.0), sd)
    for bits in _dividend_bits(lim, guard, full):
        x = np.concatenate([bits.view(np.float32), (bits | np.uint32(0x80000000)).view(np.float32)])
        got = q.debug_quant_by_scale(to_dev(x), float(sd)).cpu().numpy()
        with np.errstate(under="ignore", over="ignore"):
            ref = orc.e4m3_from_f32_array((x / sd).astype(np.float32))
        bad = np.nonzero(got != ref)[0]
        assert bad.size == 0, (float(sd), x[bad[:4]], got[bad[:4]], ref[bad[:4]])


def test_bounded_wait_reports_timeout_and_context_survives(q, orc):
    """A wait on an mbarrier that nothing arrives at gives up after its limit,
    records QMOE_DEV_TIMEOUT in d_status and returns; the context keeps
    working (a quantisation launched afterwards is still bit-exact)."""
    import time
    st = status()
    t0 = time.perf_counter()
    q.debug_wait_timeout(st, 20_000_000)          # 20 ms
    torch.cuda.synchronize()
    dt = time.perf_counter() - t0
    assert int(st.item()) == q.DEV_TIMEOUT
    assert 0.015 < dt < 5.0
    x = inputs.activations_bf16(8, 64, seed=1)
    qa, sa = q.quant_act_fp8(to_dev_bf16(x))
    rq, rs = orc.quant_rows_fp8_bf16(x)
    assert np.array_equal(qa.cpu().numpy(), rq)


@pytest.mark.parametrize("R,I", [(64, 256), (300, 1024), (3, 40), (8, 16384)])
def test_srelu_quant_token_bitexact(q, orc, R, I):
    y = inputs.activations_bf16(R, I, seed=R + I + 5)
    y[0, :] = 0
    qq, ss = q.srelu_quant(to_dev_bf16(y))
    rq, rs = orc.srelu_quant_token(y)
    assert np.array_equal(qq.cpu().numpy(), rq)
    assert np.array_equal(ss.cpu().numpy().view(np.uint32), rs.view(np.uint32))


@pytest.mark.parametrize("cnt,I", [([64, 64], 128), ([5, 0, 130, 1, 300, 0, 7, 9], 96), ([4000, 4000], 256)])
def test_srelu_quant_mx_bitexact(q, orc, cnt, I):
    R = sum(cnt)
    y = inputs.activations_bf16(R, I, seed=R + I + 6)
    eoff = np.array([0] + list(np.cumsum(cnt)), dtype=np.int32)
    soff = np.array([0] + list(np.cumsum([-(-c // 128) * 128 for c in cnt])), dtype=np.int32)
    ld = q.mx_sf_ld(I)
    sf = torch.full((int(soff[-1]), ld), 0xAB, dtype=torch.uint8, device=dev())
    qq, sfo = q.srelu_quant(to_dev_bf16(y), q.SCALE_MX_1X32, expert_offsets=to_dev(eoff),
                            sf_padded_offsets=to_dev(soff), sf=sf)
    rq, rsf = orc.srelu_quant_mx(y, eoff, soff)
    assert np.array_equal(qq.cpu().numpy(), rq)
    assert np.array_equal(sfo.cpu().numpy(), rsf)


@pytest.mark.parametrize("M,E,k", [(1, 8, 2), (777, 8, 2), (300, 64, 6), (129, 256, 8), (64, 5, 5), (5000, 16, 1)])
def test_router_topk_bitexact(q, orc, M, E, k):
    """Router kernel == the oracle's fixed fp32 sequence: ids and weight bits."""
    l = inputs.router_logits(M, E, seed=M + E, zipf_s=1.0).astype(np.float32)
    l[0, :] = 0.0  # an all-tie row
    ids, w = q.moe_router_topk(to_dev(l), k)
    torch.cuda.synchronize()
    rid, rw = orc.router_topk(l, k)
    assert np.array_equal(ids.cpu().numpy(), rid)
    assert np.array_equal(w.cpu().numpy().view(np.uint32), rw.view(np.uint32))


@pytest.mark.parametrize("M,K,E,top_k,BM", [(64, 4096, 8, 2, 32), (1, 128, 8, 2, 16), (333, 256, 64, 6, 64),
                                            (512, 4096, 8, 2, 128), (2100, 128, 8, 2, 128)])
def test_fused_route_align_quant_bitexact(q, orc, M, K, E, top_k, BM):
    """Router + align + sorted quantisation in one launch == the oracle's router,
    align and per-token codes (the last case exceeds the one-launch limit)."""
    x = inputs.activations_bf16(M, K, seed=M + K + 1)
    l = inputs.router_logits(M, E, seed=M + 3, zipf_s=1.1).astype(np.float32)
    st = status()
    ids, w, al, qq, ss = q.moe_route_align_quant_fp8(to_dev(l), to_dev_bf16(x), top_k, BM, d_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    rid, rw = orc.router_topk(l, top_k)
    assert np.array_equal(ids.cpu().numpy(), rid)
    assert np.array_equal(w.cpu().numpy().view(np.uint32), rw.view(np.uint32))
    ref = orc.moe_align(rid, E, BM)
    cap = al["sorted_ids"].numel()
    assert np.array_equal(al["sorted_ids"].cpu().numpy(), ref["sorted_ids"][:cap])
    assert np.array_equal(al["expert_ids"].cpu().numpy(), ref["expert_ids"][: cap // BM])
    assert np.array_equal(al["expert_offsets"].cpu().numpy(), ref["expert_offsets"])
    assert np.array_equal(al["padded_offsets"].cpu().numpy(), ref["padded_offsets"])
    assert int(al["num_post_padded"].item()) == ref["num_post_padded"]
    rq, rs = orc.quant_rows_fp8_bf16(x)
    srt = ref["sorted_ids"][: ref["num_post_padded"]]
    valid = np.nonzero(srt < M * top_k)[0]
    assert np.array_equal(qq.cpu().numpy()[valid], rq[srt[valid] // top_k])
    assert np.array_equal(ss.cpu().numpy()[valid], rs[srt[valid] // top_k])
