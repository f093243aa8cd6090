"""The float64 oracle against the facts the pages and the mathematics fix."""
import pytest

import oracle
from tests.oracle_pins import ALL_PINS


@pytest.mark.parametrize("pin", ALL_PINS, ids=[p.__name__ for p in ALL_PINS])
def test_pin(pin):
    pin(oracle)


def test_bf16_inputs_upcast_exactly():
    # The oracle consumes the same bf16 tensors as the GPU path; upcasting
    # bf16 -> float64 is exact, so bf16 and pre-upcast inputs agree bit for bit.
    import torch
    from exact_attention_forward_04_gb300.inputs import make_qkv
    q, k, v = make_qkv(1, 2, 40, 16, seed=5)
    O1, L1 = oracle.attention_ref(q, k, v, 0.25, True)
    O2, L2 = oracle.attention_ref(q.double(), k.double(), v.double(), 0.25, True)
    assert torch.equal(O1, O2) and torch.equal(L1, L2)
