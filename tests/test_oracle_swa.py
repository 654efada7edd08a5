"""The sliding-window attention oracle against its pins, and planted
mistakes (one at a time, in the oracle module, on the CPU) that some pin
must catch."""

import math

import numpy as np
import pytest

import oracle.swa as W
from _pins_swa import PINS


@pytest.mark.parametrize("pin", PINS, ids=[p.__name__ for p in PINS])
def test_pin(pin):
    pin(W)


_orig_keys = W.window_keys
_orig_row = W.swa_row


def _keys_left_exclusive(i, N, left, right):
    return _orig_keys(i, N, left - 1 if left > 0 else left, right)


def _keys_right_exclusive(i, N, left, right):
    n = _orig_keys(i, N, left, right)
    return n[:-1] if right >= 0 and n.size and n[-1] == i + right else n


def _keys_swapped(i, N, left, right):
    return _orig_keys(i, N, right, left)


def _keys_off_by_one_top(i, N, left, right):
    # one key too many past the query when the right side is bounded
    n = _orig_keys(i, N, left, right)
    return n if right < 0 or i + right + 1 >= N else np.append(n, i + right + 1)


def _row_wrong_group(Q, K, V, b, i, g, left, right, scale=None):
    Hkv = K.shape[2]
    return _orig_row(Q, K, V, b, i, (g + 1) % Hkv, left, right, scale)


def _row_no_scale(Q, K, V, b, i, g, left, right, scale=None):
    return _orig_row(Q, K, V, b, i, g, left, right, 1.0)


def _row_lse_log2(Q, K, V, b, i, g, left, right, scale=None):
    o, lse = _orig_row(Q, K, V, b, i, g, left, right, scale)
    return o, lse / math.log(2)


def _row_heads_interleaved(Q, K, V, b, i, g, left, right, scale=None):
    # query heads g, g + H_kv, ... instead of a contiguous run
    H, Hkv = Q.shape[2], K.shape[2]
    Qp = Q.copy()
    hpg = H // Hkv
    perm = [(h % hpg) * Hkv + h // hpg for h in range(H)]
    Qp[:, :, :] = Q[:, :, perm]
    return _orig_row(Qp, K, V, b, i, g, left, right, scale)


MUTANTS = [
    ("window_keys", _keys_left_exclusive),
    ("window_keys", _keys_right_exclusive),
    ("window_keys", _keys_swapped),
    ("window_keys", _keys_off_by_one_top),
    ("swa_row", _row_wrong_group),
    ("swa_row", _row_no_scale),
    ("swa_row", _row_lse_log2),
    ("swa_row", _row_heads_interleaved),
]


@pytest.mark.parametrize("name,fn", MUTANTS, ids=[f.__name__ for _, f in MUTANTS])
def test_mutant_is_caught(monkeypatch, name, fn):
    monkeypatch.setattr(W, name, fn)
    failed = []
    for pin in PINS:
        try:
            pin(W)
        except (AssertionError, IndexError, ValueError):
            failed.append(pin.__name__)
    assert failed, f"no pin catches the planted mistake {fn.__name__}"
