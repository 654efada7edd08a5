"""The oracle's backward against its pins, and planted mistakes (no GPU)."""

import numpy as np
import pytest

import oracle.sel_attn as S
from _pins_bwd import BPINS


@pytest.mark.parametrize("pin", BPINS, ids=[p.__name__ for p in BPINS])
def test_bwd_pin(pin):
    pin(S)


_orig_terms = S.softmax_grad_terms


def _no_delta(s, lse, v, do):
    p = np.exp(s - lse[:, None])
    return p, p * (do @ v.T)


def _delta_sign(s, lse, v, do):
    p = np.exp(s - lse[:, None])
    dp = do @ v.T
    return p, p * (dp + (p * dp).sum(axis=1)[:, None])


def _p_unnormalised(s, lse, v, do):
    p, ds = _orig_terms(s, lse, v, do)
    return np.exp(s), ds


def _dp_transposed_values(s, lse, v, do):
    return _orig_terms(s, lse, v[::-1], do)


def _ds_missing_p(s, lse, v, do):
    p = np.exp(s - lse[:, None])
    dp = do @ v.T
    return p, dp - (p * dp).sum(axis=1)[:, None]


def _mag_without_delta(s, lse, v, do):
    p = np.exp(s - lse[:, None])
    return p, p * (np.abs(do) @ np.abs(v).T)


def _mag_signed(s, lse, v, do):
    p = np.exp(s - lse[:, None])
    dp = do @ v.T
    return p, p * (dp + (p * dp).sum(axis=1)[:, None])


BMUTANTS = {
    "magnitude_without_delta": ("softmax_grad_magnitudes", _mag_without_delta),
    "magnitude_signed": ("softmax_grad_magnitudes", _mag_signed),
    "delta_dropped": ("softmax_grad_terms", _no_delta),
    "delta_sign": ("softmax_grad_terms", _delta_sign),
    "p_unnormalised": ("softmax_grad_terms", _p_unnormalised),
    "dp_values_misaligned": ("softmax_grad_terms", _dp_transposed_values),
    "ds_without_p": ("softmax_grad_terms", _ds_missing_p),
    "causal_strict": ("causal_visible", lambda n, m: n < m),
    "scale_dropped": ("scores", lambda q, k, scale: q @ k.T),
    "group_is_h_mod_G": ("head_group", lambda h, H, G: h % G),
}


@pytest.mark.parametrize("name", sorted(BMUTANTS))
def test_bwd_mutant_is_caught(name, monkeypatch):
    attr, fn = BMUTANTS[name]
    monkeypatch.setattr(S, attr, fn)
    failed = []
    for pin in BPINS:
        try:
            pin(S)
        except (AssertionError, ValueError, IndexError, FloatingPointError):
            failed.append(pin.__name__)
    assert failed, f"backward mutant {name} passed every pin"


def test_bwd_rounding_emulation_is_close():
    """fp16 operands (dO, P, dS) move the exact gradients by at most about
    one fp16 unit roundoff (2^-11) times each element's magnitude -- well
    inside the GPU tolerance of four units per element."""
    from nsa_block_selection_gb300 import inputs as gen

    w = gen.Workload("t", 1, 96, 96, 8, 1, 32, 16, 4, 1.0, "first_two_local")
    q, k, v, idx = gen.make_inputs(w, 3)
    dO = np.random.default_rng(4).standard_normal(q.shape)
    exact = S.sel_attn_bwd(q, k, v, idx, dO, 16)
    emul = S.sel_attn_bwd(q, k, v, idx, dO, 16, emulate_kernel_rounding=True)
    mags = S.sel_attn_bwd(q, k, v, idx, dO, 16, magnitudes=True)
    u16 = 2.0 ** -11
    for a, b, mg in zip(exact, emul, mags):
        assert np.abs(a - b).max() <= 5e-3 * np.abs(a).max()
        assert np.all(np.abs(a - b) <= 2 * u16 * mg + 1e-15)


def test_bwd_restricted_helpers_agree_with_full():
    """dQ of chosen rows and dK/dV of one block equal the full backward."""
    from nsa_block_selection_gb300 import inputs as gen

    w = gen.Workload("t", 2, 80, 80, 8, 2, 16, 8, 5, 1.0, "first_two_local")
    q, k, v, idx = gen.make_inputs(w, 5)
    dO = np.random.default_rng(6).standard_normal(q.shape)
    dQ, dK, dV = S.sel_attn_bwd(q, k, v, idx, dO, 8)
    rows = [(1, 79, 0), (0, 3, 1), (1, 40, 1)]
    got = S.sel_attn_bwd_dq_rows(q, k, v, idx, dO, rows, 8)
    for r, (b, m, g) in enumerate(rows):
        np.testing.assert_allclose(got[r], dQ[b, m, 4 * g:4 * g + 4], atol=1e-12)
    bk, bv = S.sel_attn_bwd_block(q, k, v, idx, dO, 1, 1, 3, 8)
    np.testing.assert_allclose(bk, dK[1, 24:32, 1], atol=1e-12)
    np.testing.assert_allclose(bv, dV[1, 24:32, 1], atol=1e-12)
