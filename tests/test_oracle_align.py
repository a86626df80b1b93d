"""Pins for the oracle's moe_align_block_size: a brute-force restatement on
tiny inputs plus the invariants that define a sorted, padded slot layout."""
import itertools

import numpy as np
import pytest

from quantized_moe_grouped_gb300 import inputs


def brute_align(ids, E, BM):
    """Independent restatement: group slot indices by expert with a Python
    sort (stable), pad each group with the sentinel to a multiple of BM."""
    T = len(ids)
    groups = {e: [s for s, x in sorted(enumerate(ids), key=lambda t: (t[1], t[0])) if x == e] for e in range(E)}
    out, blocks = [], []
    for e in range(E):
        g = groups[e]
        padded = -(-len(g) // BM) * BM
        out += g + [T] * (padded - len(g))
        blocks += [e] * (padded // BM)
    return out, blocks


@pytest.mark.parametrize("BM", [1, 2, 4, 16])
def test_align_bruteforce_tiny(orc, BM):
    g = np.random.default_rng(BM)
    for trial in range(60):
        E = int(g.integers(1, 5))
        T = int(g.integers(0, 35))
        ids = g.integers(0, E, T).astype(np.int32)
        r = orc.moe_align(ids, E, BM)
        ref_sorted, ref_blocks = brute_align(list(ids), E, BM)
        n = r["num_post_padded"]
        assert n == len(ref_sorted)
        assert list(r["sorted_ids"][:n]) == ref_sorted
        assert np.all(r["sorted_ids"][n:] == T)
        assert list(r["expert_ids"][: n // BM]) == ref_blocks
        assert np.all(r["expert_ids"][n // BM:] == -1)
        cnt = np.bincount(ids, minlength=E)
        assert list(r["expert_offsets"]) == [0] + list(np.cumsum(cnt))
        assert list(r["padded_offsets"]) == [0] + list(np.cumsum(-(-cnt // BM) * BM))
        assert not r["invalid"]


def test_align_invariants_routing(orc):
    for M, E, BM in [(64, 8, 16), (257, 8, 64), (1000, 8, 128), (33, 3, 256)]:
        ids, _ = inputs.routing(M, E, 2, seed=M)
        r = orc.moe_align(ids, E, BM)
        T = ids.size
        n = r["num_post_padded"]
        s = r["sorted_ids"][:n]
        real = s[s < T]
        assert sorted(real.tolist()) == list(range(T))           # every slot exactly once
        flat = ids.ravel()
        for b in range(n // BM):
            blk = s[b * BM:(b + 1) * BM]
            blk = blk[blk < T]
            assert np.all(flat[blk] == r["expert_ids"][b])        # blocks never mix experts
            assert np.all(np.diff(blk) > 0)                       # ascending (stable) order
        assert n % BM == 0 and n <= orc.align_max_padded(T, E, BM)


def test_align_flags_invalid_ids(orc):
    ids = np.array([0, 1, 5, -1, 1], dtype=np.int32)
    r = orc.moe_align(ids, 2, 4)
    assert r["invalid"]
    assert r["expert_offsets"][-1] == 3                            # bad slots dropped


def test_align_empty(orc):
    r = orc.moe_align(np.zeros(0, dtype=np.int32), 8, 16)
    assert r["num_post_padded"] == 0 and np.all(r["expert_offsets"] == 0)
