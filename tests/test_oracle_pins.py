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


def test_round_bf16_matches_torch():
    """The oracle's bfloat16 rounding (used by the bf16 emulation) agrees bit
    for bit with torch's float32 -> bfloat16 conversion, ties included."""
    torch = __import__("pytest").importorskip("torch")
    rng = np.random.default_rng(5)
    x = np.concatenate([
        rng.standard_normal(20000).astype(np.float32) * np.float32(300.0),
        rng.random(20000).astype(np.float32),
        np.ldexp(rng.random(2000), rng.integers(-120, 120, 2000)).astype(np.float32),
    ])
    # exact ties: low 16 bits 0x8000, kept part even and odd
    hi = rng.integers(0x3000, 0x4F00, 4000).astype(np.uint32) << 16
    ties = (hi | 0x8000).view(np.float32)
    x = np.concatenate([x, ties, -ties, np.float32([0.0, 1.0, 255.99, 256.0])])
    want = torch.from_numpy(x).bfloat16().float().numpy()
    got = S.round_bf16(x)
    np.testing.assert_array_equal(got.view(np.uint32), want.view(np.uint32))
    assert (S.round_bf16(ties[:2]) != ties[:2]).all()


def test_bf16_rounding_emulation_within_derived_bound():
    """Rounding P to bfloat16 (8 significant bits, relative error <= 2^-8)
    moves O by at most 2^-8 * sum_n p_n |V[n]| per dimension, which the
    oracle gives exactly as its O for |V| (p does not depend on V); the row
    sums stay fp32, so LSE barely moves."""
    from nsa_block_selection_gb300 import inputs as gen

    w = gen.Workload("t", 1, 256, 256, 16, 2, 64, 32, 4, 1.0, "local")
    Q, K, V = gen.make_qkv(w, 7, "bf16")
    idx = gen.make_block_indices(w, 7)
    rows = [(0, m, g) for m in range(0, 256, 3) for g in range(2)]
    O1, L1 = S.sel_attn_rows(Q, K, V, idx, rows, w.block_size)
    A, _ = S.sel_attn_rows(Q, K, np.abs(V), idx, rows, w.block_size)
    O2, L2 = S.sel_attn_rows(Q, K, V, idx, rows, w.block_size, route="online",
                             emulate_kernel_rounding="bf16")
    ratio = np.abs(O2 - O1) / (2.0 ** -8 * A + 1e-6)
    assert ratio.max() <= 1.0, ratio.max()
    assert ratio.max() > 0.05  # the rounding does act: the bound is not vacuous
    assert np.abs(L1 - L2).max() < 1e-4
    O3, _ = S.sel_attn_rows(Q, K, V, idx, rows, w.block_size, route="online",
                            emulate_kernel_rounding="f16")
    assert np.abs(O3 - O1).max() < np.abs(O2 - O1).max()  # fp16 P is the finer one
