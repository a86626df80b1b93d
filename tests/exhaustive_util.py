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
