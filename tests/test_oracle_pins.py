"""The CPU oracle against library routines, closed forms and invariants."""
import pytest

import oracle.attention_fp64 as orc
import oracle_pins


@pytest.mark.parametrize("pin", oracle_pins.ALL_PINS, ids=lambda f: f.__name__)
def test_pin(pin):
    pin(orc)


def test_round_to_bf16_matches_torch():
    import numpy as np
    import torch
    x = torch.randn(100000, dtype=torch.float64, generator=torch.Generator().manual_seed(3)) * 10
    x = torch.cat([x, torch.tensor([0.0, -0.0, 1e-40, 3.0e38, 1 + 2**-8, 1 + 3 * 2**-8])])
    ref = x.to(torch.float32).to(torch.bfloat16).to(torch.float64).numpy()
    got = orc.round_to_bf16(x.numpy())
    assert np.array_equal(ref, got)
