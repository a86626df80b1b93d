"""Guard bands for the GPU tests: the binding's allocation helper is replaced by
one that places every tensor between two margins of GUARD_BYTES filled with a
sentinel byte; check() reads every margin back and fails on any changed byte."""
import contextlib
import math

import numpy as np
import torch

GUARD_BYTES = 4096
SENTINEL = 0xA7


def _size(size):
    if len(size) == 1 and isinstance(size[0], (tuple, list, torch.Size)):
        return tuple(size[0])
    return tuple(size)


@contextlib.contextmanager
def guarded_allocations():
    import quantized_moe_grouped_gb300 as q
    bufs = []
    original = q._empty

    def empty(*size, dtype, device):
        shape = _size(size)
        nbytes = math.prod(shape) * torch.empty(0, dtype=dtype).element_size()
        buf = torch.empty(nbytes + 2 * GUARD_BYTES, dtype=torch.uint8, device=device)
        buf[:GUARD_BYTES].fill_(SENTINEL)
        buf[GUARD_BYTES + nbytes:].fill_(SENTINEL)
        bufs.append((buf, nbytes))
        return buf[GUARD_BYTES:GUARD_BYTES + nbytes].view(dtype).view(shape)

    def check():
        if torch.cuda.is_available():
            torch.cuda.synchronize()
        for i, (buf, nbytes) in enumerate(bufs):
            lo = buf[:GUARD_BYTES].cpu().numpy()
            hi = buf[GUARD_BYTES + nbytes:].cpu().numpy()
            bad_lo = np.nonzero(lo != SENTINEL)[0]
            bad_hi = np.nonzero(hi != SENTINEL)[0]
            assert bad_lo.size == 0, (f"allocation {i} ({nbytes} bytes): {bad_lo.size} bytes written before it, "
                                      f"nearest at offset {int(bad_lo.max()) - GUARD_BYTES}")
            assert bad_hi.size == 0, (f"allocation {i} ({nbytes} bytes): {bad_hi.size} bytes written past its end, "
                                      f"first at offset +{int(bad_hi.min())}")
        bufs.clear()

    q._empty = empty
    try:
        yield check
    finally:
        q._empty = original
        bufs.clear()
