"""The top-k block selection oracle against its pins, and planted mistakes
(one at a time, in the oracle module, on the CPU) that some pin must catch."""

import numpy as np
import pytest

import oracle.topk as K
from _pins_topk import PINS


@pytest.mark.parametrize("pin", PINS, ids=[p.__name__ for p in PINS])
def test_pin(pin):
    pin(K)


_orig = {n: getattr(K, n) for n in ("last_candidate", "forced_blocks", "rank_order")}


def _rank_ties_high(scores, blocks):
    blocks = list(blocks)
    return sorted(blocks, key=lambda t: (np.isnan(scores[t]),
                                         -float(np.nan_to_num(scores[t])), -t))


def _rank_ascending(scores, blocks):
    return list(reversed(_orig["rank_order"](scores, blocks)))


def _rank_nan_first(scores, blocks):
    r = _orig["rank_order"](scores, blocks)
    nan = [t for t in r if np.isnan(scores[t])]
    return nan + [t for t in r if not np.isnan(scores[t])]


def _rank_signed_zero(scores, blocks):
    # ranks -0.0 below +0.0 (a bitwise order)
    blocks = list(blocks)
    return sorted(blocks, key=lambda t: (np.isnan(scores[t]), -float(scores[t]),
                                         bool(np.signbit(scores[t])), t))


def _last_unclipped(m, N, bs):
    return -1 if N <= 0 else m // bs


def _last_off_by_one(m, N, bs):
    return -1 if N <= 0 else max(0, min(m, N - 1) // bs - (1 if m % bs == 0 else 0))


def _forced_local_short(c, n_init, n_local):
    return {t for t in range(c + 1) if t < n_init or t > c - n_local + 1}


def _forced_none(c, n_init, n_local):
    return set()


def _forced_init_shifted(c, n_init, n_local):
    return {t for t in range(c + 1) if (1 <= t <= n_init) or t > c - n_local}


MUTANTS = [
    ("rank_order", _rank_ties_high),
    ("rank_order", _rank_ascending),
    ("rank_order", _rank_nan_first),
    ("rank_order", _rank_signed_zero),
    ("last_candidate", _last_unclipped),
    ("last_candidate", _last_off_by_one),
    ("forced_blocks", _forced_local_short),
    ("forced_blocks", _forced_none),
    ("forced_blocks", _forced_init_shifted),
]


@pytest.mark.parametrize("name,fn", MUTANTS, ids=[f.__name__ for _, f in MUTANTS])
def test_mutant_is_caught(monkeypatch, name, fn):
    monkeypatch.setattr(K, name, fn)
    failed = []
    for pin in PINS:
        try:
            pin(K)
        except (AssertionError, IndexError, ValueError):
            failed.append(pin.__name__)
    assert failed, f"no pin catches the planted mistake {fn.__name__}"
