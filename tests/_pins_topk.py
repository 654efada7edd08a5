"""Pins of the top-k block selection oracle, as functions of the module under
test (so planted mistakes can be run against them).

Each pin checks the oracle against something other than its own code: the
candidate set counted from the causal visibility of keys, the top-k set
characterised pairwise (every chosen block beats every block left out),
brute force over all subsets on tiny rows, closed forms for monotone, equal
and NaN scores, and the law of the choice under i.i.d. scores.
"""

from __future__ import annotations

import itertools
import math

import numpy as np


def _candidates(m, N, bs):
    """Blocks holding a key visible to query m, by looking at every key."""
    return sorted({n // bs for n in range(N) if n <= m})


def _better(s, a, b):
    """Block a ranks before block b: larger score, NaN below every number,
    equal scores (or two NaNs) to the lower index."""
    sa, sb = float(s[a]), float(s[b])
    na, nb = math.isnan(sa), math.isnan(sb)
    if na != nb:
        return nb
    if not na and sa != sb:
        return sa > sb
    return a < b


def _check_row(K, s, m, N, bs, T, n_init, n_local):
    out = [int(x) for x in K.topk_row(s, m, N, bs, T, n_init, n_local)]
    assert len(out) == T
    sel = [x for x in out if x >= 0]
    assert out == sel + [-1] * (T - len(sel)), "padding only at the end"
    assert all(a < b for a, b in zip(sel, sel[1:])), "ascending and distinct"
    cand = _candidates(m, N, bs)
    assert set(sel) <= set(cand)
    assert len(sel) == min(T, len(cand))
    if len(cand) <= T:
        return out
    forced = set(cand[:n_init]) | set(cand[len(cand) - n_local:])
    assert forced <= set(sel)
    free_sel = [a for a in sel if a not in forced]
    left = [b for b in cand if b not in sel]
    for a in free_sel:
        for b in left:
            assert _better(s, a, b), (m, a, b, s[a], s[b])
    return out


def _random_scores(rng, n, kind):
    if kind == "normal":
        return rng.standard_normal(n).astype(np.float32)
    if kind == "ties":
        return rng.integers(0, 4, n).astype(np.float32)
    if kind == "special":
        pool = np.float32([0.0, -0.0, 1.0, -1.0, np.inf, -np.inf, np.nan, 1e-45, -1e-45])
        return pool[rng.integers(0, pool.size, n)]
    raise ValueError(kind)


def pin_property_random_rows(K):
    rng = np.random.default_rng(1)
    for kind in ("normal", "ties", "special"):
        for _ in range(60):
            bs = int(rng.choice([1, 4, 32, 64]))
            N = int(rng.integers(1, 40 * bs))
            m = int(rng.integers(0, N + 3 * bs))
            T = int(rng.integers(1, 12))
            n_init = int(rng.integers(0, T + 1))
            n_local = int(rng.integers(0, T - n_init + 1))
            s = _random_scores(rng, -(-N // bs), kind)
            _check_row(K, s, m, N, bs, T, n_init, n_local)


def pin_brute_force_subsets(K):
    rng = np.random.default_rng(2)
    for _ in range(150):
        bs = int(rng.choice([1, 2, 3]))
        nblk = int(rng.integers(1, 10))
        N = nblk * bs - int(rng.integers(0, bs))
        m = int(rng.integers(0, N + 2))
        T = int(rng.integers(1, 7))
        n_init = int(rng.integers(0, T + 1))
        n_local = int(rng.integers(0, T - n_init + 1))
        s = _random_scores(rng, -(-N // bs), ["ties", "special"][int(rng.integers(2))])
        cand = _candidates(m, N, bs)
        k = min(T, len(cand))
        forced = set(cand[:n_init]) | set(cand[len(cand) - n_local:]) if len(cand) > T \
            else set(cand)
        valid = []
        for sub in itertools.combinations(cand, k):
            if not forced <= set(sub):
                continue
            free = [a for a in sub if a not in forced]
            left = [b for b in cand if b not in sub]
            if all(_better(s, a, b) for a in free for b in left):
                valid.append(list(sub))
        assert len(valid) == 1, "the top-k set is unique"
        want = valid[0] + [-1] * (T - k)
        got = [int(x) for x in K.topk_row(s, m, N, bs, T, n_init, n_local)]
        assert got == want, (got, want)


def pin_closed_forms(K):
    bs, N, T = 16, 16 * 50, 10
    m = N - 1  # candidates 0..49
    c = 49
    for n_init, n_local in ((0, 0), (1, 2), (3, 0), (0, 4), (5, 5)):
        free = T - n_init - n_local
        head = list(range(n_init))
        tail = list(range(c - n_local + 1, c + 1))
        low = sorted(set(head) | set(range(n_init, n_init + free)) | set(tail))
        high = sorted(set(head) | set(range(c - n_local - free + 1, c + 1)))
        dec = -np.arange(50, dtype=np.float32)
        args = (m, N, bs, T, n_init, n_local)
        assert list(K.topk_row(dec, *args)) == low
        assert list(K.topk_row(-dec, *args)) == high
        assert list(K.topk_row(np.zeros(50, np.float32), *args)) == low
        assert list(K.topk_row(np.full(50, np.nan, np.float32), *args)) == low
        zeros = np.where(np.arange(50) % 2 == 0, np.float32(0.0), np.float32(-0.0))
        assert list(K.topk_row(zeros, *args)) == low  # -0.0 ties with +0.0
        if free > 0:
            one = np.full(50, np.nan, np.float32)
            one[30] = -np.inf  # any number beats NaN
            got = list(K.topk_row(one, *args))
            assert 30 in got or 30 in tail
            spike = dec.copy()
            spike[20] = np.inf
            assert 20 in K.topk_row(spike, *args)


def pin_few_candidates_and_edges(K):
    bs = 64
    for m in (0, 1, 63, 64, 200, 64 * 7 - 1):
        got = [int(x) for x in K.topk_row(np.zeros(100, np.float32), m, 6400, bs, 8, 1, 2)]
        c = m // bs
        assert got == list(range(c + 1)) + [-1] * (8 - c - 1)
    # no keys: nothing to choose
    assert list(K.topk_row(np.zeros(0, np.float32), 5, 0, bs, 4, 1, 1)) == [-1] * 4
    # queries past the keys see every key
    got = K.topk_row(-np.arange(3, dtype=np.float32), 1000, 130, bs, 2, 0, 0)
    assert list(got) == [0, 1]
    assert K.topk_row(np.zeros(3, np.float32), 100, 130, bs, 0, 0, 0).shape == (0,)
    # whole-tensor entry point: row (b, m, g) uses scores[b, m, g]
    rng = np.random.default_rng(3)
    sc = rng.standard_normal((2, 300, 3, 10)).astype(np.float32)
    full = K.topk_blocks(sc, 300, 32, 4, 1, 1)
    for b, m, g in ((0, 0, 0), (1, 299, 2), (0, 150, 1), (1, 40, 0)):
        assert list(full[b, m, g]) == list(K.topk_row(sc[b, m, g], m, 300, 32, 4, 1, 1))


def pin_uniform_law(K):
    """i.i.d. scores: the free picks are a uniform subset of the free
    candidates (the workloads' index rule as a top-k)."""
    rng = np.random.default_rng(4)
    bs, T = 64, 8
    m = 64 * 40 - 1  # candidates 0..39; forced 0, 38, 39; 5 free picks from 1..37
    counts = np.zeros(40, np.int64)
    rows = 3000
    for _ in range(rows):
        s = rng.random(40).astype(np.float32)
        got = K.topk_row(s, m, 64 * 40, bs, T, 1, 2)
        assert {0, 38, 39} <= set(got.tolist())
        counts[got] += 1
    free = counts[1:38]
    assert free.sum() == rows * 5
    e = free.sum() / 37
    assert ((free - e) ** 2 / e).sum() < 68  # chi-square, 36 dof, 99.9 %


PINS = [pin_property_random_rows, pin_brute_force_subsets, pin_closed_forms,
        pin_few_candidates_and_edges, pin_uniform_law]
