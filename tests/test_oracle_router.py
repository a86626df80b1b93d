"""Pins of the oracle's router (softmax -> top-k -> renormalise over fp32
logits) against what the mathematics fixes: the fp64 definition, exact ties,
exact special cases and shift invariance on exactly representable logits."""
import numpy as np
import pytest

from quantized_moe_grouped_gb300 import inputs


def _fp64_reference(l: np.ndarray, k: int):
    """fp64 softmax over all E logits, its top-k (stable sort: ties to the lower
    id), renormalised."""
    l = l.astype(np.float64)
    p = np.exp(l - l.max(axis=1, keepdims=True))
    p /= p.sum(axis=1, keepdims=True)
    order = np.argsort(-p, axis=1, kind="stable")
    ids = order[:, :k]
    sel = np.take_along_axis(p, ids, axis=1)
    return ids, sel / sel.sum(axis=1, keepdims=True), order


@pytest.mark.parametrize("M,E,k,zipf", [(400, 8, 2, None), (200, 64, 6, 1.2), (64, 256, 8, None),
                                        (100, 5, 3, None), (50, 8, 8, None), (80, 16, 1, 0.8)])
def test_router_matches_fp64_definition(orc, M, E, k, zipf):
    l = inputs.router_logits(M, E, seed=E * 7 + k, zipf_s=zipf).astype(np.float32)
    ids, w = orc.router_topk(l, k)
    rid, rw, _ = _fp64_reference(l, k)
    assert np.array_equal(ids, rid)  # exact comparisons of the fp32 logits
    # a few fp32 ulp: k exps (~1 ulp each), a k-term sum, one division
    assert np.allclose(w, rw, rtol=2e-6, atol=0)
    assert np.allclose(w.sum(axis=1), 1.0, rtol=0, atol=4e-7 * k)
    assert np.all(np.diff(w, axis=1) <= 0)  # selection order is descending


def test_router_ties_go_to_the_lower_id(orc):
    l = np.zeros((3, 8), dtype=np.float32)
    l[1, [3, 5]] = 1.0
    l[2, [6, 2, 7]] = -1.0
    ids, w = orc.router_topk(l, 2)
    assert ids.tolist() == [[0, 1], [3, 5], [0, 1]]
    # E = 8 equal logits: every s_e = 1/8 exactly, so w = 1/2 exactly
    assert w[0].tolist() == [0.5, 0.5] and w[1].tolist() == [0.5, 0.5]
    ids4, w4 = orc.router_topk(np.zeros((1, 8), dtype=np.float32), 4)
    assert ids4.tolist() == [[0, 1, 2, 3]] and w4.tolist() == [[0.25] * 4]


def test_router_single_expert_weight_is_one(orc):
    l = inputs.router_logits(300, 32, seed=5).astype(np.float32)
    ids, w = orc.router_topk(l, 1)
    assert np.array_equal(ids[:, 0], np.argmax(l, axis=1))
    assert np.all(w == 1.0)


def test_router_shift_invariance_on_exact_logits(orc):
    """Logits on a 1/8 grid in [-4, 4]: l - max is exact before and after a
    shift by 16, so the results are bit-identical."""
    g = inputs.rng(11, 901)
    l = (g.integers(-32, 33, size=(500, 16)) / 8.0).astype(np.float32)
    a = orc.router_topk(l, 4)
    b = orc.router_topk(l + np.float32(16.0), 4)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1].view(np.uint32), b[1].view(np.uint32))


def test_router_underflow_keeps_only_the_dominant_expert(orc):
    """exp of a difference of -200 underflows to zero: the dominant expert gets
    weight one, the others weight zero, no NaN."""
    l = np.full((2, 8), -100.0, dtype=np.float32)
    l[0, 6] = 100.0
    l[1, 1] = 100.0
    ids, w = orc.router_topk(l, 3)
    assert ids[:, 0].tolist() == [6, 1]
    assert ids[0, 1:].tolist() == [0, 1] and ids[1, 1:].tolist() == [0, 2]
    assert np.all(w[:, 0] == 1.0) and np.all(w[:, 1:] == 0.0)
