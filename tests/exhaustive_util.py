"""Workers for the exhaustive CPU checks: module-level functions, so that a
spawned process pool can run them by name."""
import numpy as np


def exp_chunk_worst_ulp(span):
    """Over the fp32 bit patterns [lo, hi): the largest |orc_exp(x) - exp(x)|
    in units of the fp32 ulp of exp(x)'s binade, exp(x) taken in fp64 (numpy),
    and the x where it occurs.  Valid where exp(x) is a normal fp32."""
    import oracle
    lo, hi = span
    x = np.arange(lo, hi, dtype=np.uint32).view(np.float32)
    y = oracle.exp_f32_array(x)
    ref = np.exp(x.astype(np.float64))
    e = (ref.view(np.uint64) >> np.uint64(52)) & np.uint64(0x7FF)
    inv_ulp = ((np.uint64(2046 + 23) - e) << np.uint64(52)).view(np.float64)  # 2^(23 - unbiased exponent)
    d = np.abs(y - ref) * inv_ulp
    i = int(np.argmax(d))
    return float(d[i]), float(x[i])


def e4m3_chunk_mismatches(span):
    """Over the fp32 bit patterns [lo, hi) (NaNs skipped): the patterns where
    the oracle's e4m3 code differs from torch's float8_e4m3fn cast (where the
    cast is finite), or where the cast overflows to NaN and the oracle does not
    give the saturated +-448 (0x7E / 0xFE) or |x| is below 464.  At most 4."""
    import oracle
    import torch
    torch.set_num_threads(1)
    lo, hi = span
    bits = np.arange(lo, hi, dtype=np.uint32)
    x = bits.view(np.float32)
    keep = ~np.isnan(x)
    bits, x = bits[keep], x[keep]
    o = oracle.e4m3_from_f32_array(x)
    t = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    fin = (t & 0x7F) != 0x7F
    bad = fin & (o != t)
    sat = np.where(x < 0, 0xFE, 0x7E).astype(np.uint8)
    bad |= ~fin & ((o != sat) | (np.abs(x) < 464.0))
    return [int(b) for b in bits[bad][:4]]


def mx_exponent_chunk_mismatches(span):
    """Over the fp32 bit patterns [lo, hi) of non-negative finite values: the
    patterns where the oracle's MX block exponent differs from the smallest
    integer e with 448 * 2^e >= a (exact float64 comparisons against
    ldexp(448, e)), clamped to [-127, 127], and 0 for a = 0.  At most 4."""
    import oracle
    lo, hi = span
    bits = np.arange(lo, hi, dtype=np.uint32)
    a = bits.view(np.float32)
    got = oracle.mx_scale_exponent_array(a)
    a64 = a.astype(np.float64)
    pos = a64 > 0
    est = np.zeros(a.shape, dtype=np.int32)
    est[pos] = np.ceil(np.log2(a64[pos]) - np.log2(448.0)).astype(np.int32)
    for _ in range(2):  # the estimate is within one of the answer; settle it exactly
        est[pos & (np.ldexp(448.0, est) < a64)] += 1
        est[pos & (np.ldexp(448.0, est - 1) >= a64)] -= 1
    ref = np.clip(est, -127, 127)
    ref[~pos] = 0
    return [int(b) for b in bits[got != ref][:4]]


def silu_chunk_worst(span):
    """Over the fp32 bit patterns [lo, hi) of g: the largest error of the
    oracle's silu(g) (u = 1) against fp64 g / (1 + exp(-g)), in ulps of the
    fp64 value's binade where that value is a normal fp32, and in units of
    2^-149 where it is subnormal; each with the g where it occurs."""
    import oracle
    lo, hi = span
    x = np.arange(lo, hi, dtype=np.uint32).view(np.float32)
    h = oracle.silu_mul_f32_array(x, np.ones_like(x)).astype(np.float64)
    g = x.astype(np.float64)
    ref = g / (1.0 + np.exp(-g))
    normal = np.abs(ref) >= 2.0 ** -126
    e = (ref.view(np.uint64) >> np.uint64(52)) & np.uint64(0x7FF)
    inv_ulp = ((np.uint64(2046 + 23) - e) << np.uint64(52)).view(np.float64)
    d = np.abs(h - ref)
    dn = np.where(normal, d * inv_ulp, 0.0)
    ds = np.where(normal, 0.0, d * 2.0 ** 149)
    i, j = int(np.argmax(dn)), int(np.argmax(ds))
    return (float(dn[i]), float(x[i])), (float(ds[j]), float(x[j]))


def bf16_chunk_mismatches(span):
    """Over the fp32 bit patterns [lo, hi) (NaNs skipped): the patterns where
    the oracle's bf16 encoding differs from torch's bfloat16 cast.  At most 4."""
    import oracle
    import torch
    torch.set_num_threads(1)
    lo, hi = span
    bits = np.arange(lo, hi, dtype=np.uint32)
    x = bits.view(np.float32)
    keep = ~np.isnan(x)
    bits, x = bits[keep], x[keep]
    got = oracle.bf16_from_f32_array(x)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    return [int(b) for b in bits[got != ref][:4]]
