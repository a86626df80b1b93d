"""The guard-band helper the GPU tests use, exercised on host tensors: intact
margins pass, a planted store one element past the end or before the start of
an allocation fails, and the binding's allocation helper is restored."""
import pytest
import torch

from tests import guard


def test_intact_margins_pass():
    import quantized_moe_grouped_gb300 as q
    original = q._empty
    with guard.guarded_allocations() as check:
        t = q._empty(3, 5, dtype=torch.float32, device="cpu")
        t.fill_(1.0)
        z = q._empty((0, 7), dtype=torch.bfloat16, device="cpu")
        assert z.shape == (0, 7) and t.shape == (3, 5) and t.is_contiguous()
        check()
    assert q._empty is original


@pytest.mark.parametrize("offset", [-1, 15])
def test_planted_store_outside_is_caught(offset):
    import quantized_moe_grouped_gb300 as q
    with guard.guarded_allocations() as check:
        t = q._empty(15, dtype=torch.int32, device="cpu")
        # a store one element before the start or one past the end of t
        wide = torch.as_strided(t, (17,), (1,), t.storage_offset() - 1)
        wide[offset + 1] = 12345
        with pytest.raises(AssertionError):
            check()
