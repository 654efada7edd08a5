"""The seeded input generator: index rows follow the stated rules."""

import numpy as np
import pytest

from nsa_block_selection_gb300 import inputs as gen


def _check_rows(w, idx):
    B, M, G, T = idx.shape
    assert (B, M, G, T) == (w.B, w.M, w.G, w.T) and idx.dtype == np.int32
    c = (np.arange(M) // w.block_size)[None, :, None]
    valid = idx >= 0
    # padding only at the end, valid entries strictly increasing and causal
    assert not (valid[..., 1:] & ~valid[..., :-1]).any()
    d = np.diff(idx.astype(np.int64), axis=-1)
    assert (d[valid[..., 1:]] > 0).all()
    assert (idx <= np.broadcast_to(c[..., None], idx.shape)).all()
    n = valid.sum(-1)
    # rows list min(T, c+1) blocks; the fixed blocks are always present
    assert (n == np.minimum(T, c + 1)).all()
    has = lambda blk: (idx == blk[..., None]).any(-1)  # noqa: E731
    cc = np.broadcast_to(c, n.shape)
    assert has(cc).all()
    if w.rule in ("first_local", "first_two_local", "all_causal"):
        assert has(np.zeros_like(cc)).all()
    if w.rule in ("first_two_local", "all_causal"):
        assert has(np.maximum(cc - 1, 0)).all()


@pytest.mark.parametrize("name", ["tiny_bs32", "m8k_bs64"])
def test_index_rules(name):
    w = gen.workload(name)
    _check_rows(w, gen.make_block_indices(w, gen.default_seed(name)))


@pytest.mark.parametrize("rule", ["local", "first_local", "first_two_local"])
def test_index_rules_small(rule):
    w = gen.Workload("t", 2, 3000, 3000, 16, 2, 64, 32, 7, 1.0, rule)
    _check_rows(w, gen.make_block_indices(w, 5))


def test_dense_rows():
    w = gen.workload("dense_m16k").replace(M=2048, N=2048, T=32)
    idx = gen.make_block_indices(w, 1)
    _check_rows(w, idx)
    np.testing.assert_array_equal(idx, gen.dense_causal_indices(1, 2048, 8, 32, 64))
    torch = pytest.importorskip("torch")
    t = gen.dense_causal_indices_torch(1, 2048, 8, 32, 64, "cpu").numpy()
    np.testing.assert_array_equal(idx, t)


def test_random_picks_are_uniform():
    """The random part of a row is a uniform subset of its pool."""
    w = gen.Workload("t", 1, 64 * 40, 64 * 40, 8, 1, 64, 64, 8, 1.0, "first_two_local")
    idx = gen.make_block_indices(w, 3)
    rows = idx[0, w.M - 64:, 0]  # c = 39: fixed {0, 38, 39}, 5 picks from [1, 38)
    picks = rows[(rows > 0) & (rows < 38)]
    counts = np.bincount(picks, minlength=38)[1:38]
    assert counts.sum() == 64 * 5
    # chi-square with 36 degrees of freedom; 99.9% quantile ~ 68
    e = counts.sum() / 37
    assert ((counts - e) ** 2 / e).sum() < 68


def test_deterministic_and_seed_sensitive():
    w = gen.workload("tiny_bs32")
    a = gen.make_inputs(w, 11)
    b = gen.make_inputs(w, 11)
    c = gen.make_inputs(w, 12)
    for x, y in zip(a, b):
        np.testing.assert_array_equal(x, y)
    assert not np.array_equal(a[0], c[0]) and not np.array_equal(a[3], c[3])


def test_value_distribution():
    w = gen.workload("m32k_bs32").replace(B=1, M=4096, N=4096)
    q, k, v = gen.make_qkv(w, 9)
    assert q.dtype == np.float16 and q.shape == (1, 4096, 32, 128)
    s = k.astype(np.float32).std()
    assert abs(s - 1.5) < 0.01  # sigma 1.5 read as the standard deviation
