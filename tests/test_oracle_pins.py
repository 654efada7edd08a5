"""The CPU oracle against its pins (no GPU)."""

import numpy as np
import pytest

import oracle.sel_attn as S
from _pins import PINS


@pytest.mark.parametrize("pin", PINS, ids=[p.__name__ for p in PINS])
def test_pin(pin):
    pin(S)


def test_kernel_rounding_emulation_uses_little_tolerance():
    """Rounding P to fp16 and summing in fp32 moves O/LSE far less than the
    parity tolerance (2e-3 abs + 2e-3 rel for O, 1e-3 abs for LSE)."""
    from nsa_block_selection_gb300 import inputs as gen

    w = gen.Workload("t", 1, 256, 256, 16, 2, 64, 32, 4, 1.5, "local")
    Q, K, V = gen.make_qkv(w, 7)
    idx = gen.make_block_indices(w, 7)
    rows = [(0, m, g) for m in range(0, 256, 5) for g in range(2)]
    O1, L1 = S.sel_attn_rows(Q, K, V, idx, rows, w.block_size)
    O2, L2 = S.sel_attn_rows(Q, K, V, idx, rows, w.block_size, route="online",
                             emulate_kernel_rounding=True)
    err_o = np.abs(O1 - O2) / (2e-3 + 2e-3 * np.abs(O1))
    assert err_o.max() < 0.25, err_o.max()
    assert np.abs(L1 - L2).max() < 1e-4
