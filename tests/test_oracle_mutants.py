"""Plant one plausible mistake at a time in the CPU oracle; some pin must fail.

Each mutant swaps one step of ``oracle.sel_attn`` for a wrong variant (a
dropped term, a wrong sign or index, a transposed operand, an off-by-one in
the gather range or the causal mask, the wrong head -> group map). The
mistake lives only in the oracle module, on the CPU, for one test.
"""

import math

import numpy as np
import pytest

import oracle.sel_attn as S
from _pins import PINS

_orig = {name: getattr(S, name) for name in
         ("head_group", "num_blocks", "block_keys", "causal_visible", "scores",
          "logsumexp_rows", "attend", "selected_blocks")}


def _block_keys_inclusive(t, bs, N):
    return np.arange(t * bs, min((t + 1) * bs + 1, N), dtype=np.int64)


def _block_keys_shifted(t, bs, N):
    return np.arange(t * bs + 1, min((t + 1) * bs + 1, N), dtype=np.int64)


def _block_keys_unclipped_stride(t, bs, N):
    return np.arange(t * (bs - 1), min(t * (bs - 1) + bs, N), dtype=np.int64)


def _selected_blocks_drop_zero(row, N, bs):
    return [t for t in _orig["selected_blocks"](row, N, bs) if t != 0]


def _selected_blocks_first_only(row, N, bs):
    return _orig["selected_blocks"](row, N, bs)[:1]


def _scores_no_scale(q, k, scale):
    return q @ k.T


def _scores_scale_twice(q, k, scale):
    return scale * scale * (q @ k.T)


def _scores_heads_reversed(q, k, scale):
    return scale * (q[::-1] @ k.T)


def _scores_sqrt_scale(q, k, scale):
    return math.sqrt(scale) * (q @ k.T)


def _lse_base2(s):
    if s.shape[1] == 0:
        return np.full(s.shape[0], -np.inf)
    mu = s.max(axis=1)
    return mu + np.log2(np.exp(s - mu[:, None]).sum(axis=1))


def _lse_without_max(s):
    if s.shape[1] == 0:
        return np.full(s.shape[0], -np.inf)
    mu = s.max(axis=1)
    return np.log(np.exp(s - mu[:, None]).sum(axis=1))


def _lse_plain_max(s):
    if s.shape[1] == 0:
        return np.full(s.shape[0], -np.inf)
    return s.max(axis=1)


def _attend_values_reversed(s, lse, v):
    if s.shape[1] == 0:
        return np.zeros((s.shape[0], v.shape[1]))
    return np.exp(s - lse[:, None]) @ v[::-1]


def _attend_unnormalised(s, lse, v):
    if s.shape[1] == 0:
        return np.zeros((s.shape[0], v.shape[1]))
    return np.exp(s) @ v


def _attend_sign(s, lse, v):
    if s.shape[1] == 0:
        return np.zeros((s.shape[0], v.shape[1]))
    return np.exp(lse[:, None] - s) @ v / s.shape[1] ** 2


MUTANTS = {
    "group_is_h_mod_G": ("head_group", lambda h, H, G: h % G),
    "num_blocks_floor": ("num_blocks", lambda N, bs: N // bs),
    "block_range_inclusive": ("block_keys", _block_keys_inclusive),
    "block_range_shifted": ("block_keys", _block_keys_shifted),
    "block_stride_wrong": ("block_keys", _block_keys_unclipped_stride),
    "causal_strict": ("causal_visible", lambda n, m: n < m),
    "causal_missing": ("causal_visible", lambda n, m: np.ones_like(n, dtype=bool)),
    "causal_reversed": ("causal_visible", lambda n, m: n >= m),
    "block_zero_dropped": ("selected_blocks", _selected_blocks_drop_zero),
    "only_first_block": ("selected_blocks", _selected_blocks_first_only),
    "scale_dropped": ("scores", _scores_no_scale),
    "scale_twice": ("scores", _scores_scale_twice),
    "scale_sqrt": ("scores", _scores_sqrt_scale),
    "heads_transposed": ("scores", _scores_heads_reversed),
    "lse_base2": ("logsumexp_rows", _lse_base2),
    "lse_max_term_dropped": ("logsumexp_rows", _lse_without_max),
    "lse_is_max": ("logsumexp_rows", _lse_plain_max),
    "values_misaligned": ("attend", _attend_values_reversed),
    "softmax_unnormalised": ("attend", _attend_unnormalised),
    "softmax_sign": ("attend", _attend_sign),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, monkeypatch):
    attr, fn = MUTANTS[name]
    monkeypatch.setattr(S, attr, fn)
    failed = []
    for pin in PINS:
        try:
            pin(S)
        except (AssertionError, ValueError, IndexError, FloatingPointError):
            failed.append(pin.__name__)
    assert failed, f"mutant {name} passed every pin"
