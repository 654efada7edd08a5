"""Backward (dQ, dK, dV) on the GPU vs the fp64 oracle.

Tolerance, per element: |GPU - exact| <= 4 u |terms|, with u = 2^-11 the
fp16 unit roundoff and |terms| the oracle's magnitude of that element (the
sum of the absolute values of the terms that make it up, with |dS| bounded
by p (|dO|.|v| + |dO|.(sum p |v|))). The kernels round dO, P and dS to fp16
once each (at most u of a term's magnitude per rounded operand, two per
product) and accumulate in fp32; the forward's O enters delta with the error
of its own fp16 P, which the delta part of the dS bound covers. That sums to
about 2 u |terms|; four units leave a factor of two for fp32 accumulation.
An element no visible key reaches has |terms| = 0 and must be exactly 0.
"""

import numpy as np
import pytest

import oracle.sel_attn as oracle
from _parity import poisoned, small_inputs, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _need_gpu(cuda_lib):
    import torch

    assert torch.cuda.is_available()


def _run(q, k, v, idx, dO, bs, scale=None):
    import torch

    from nsa_block_selection_gb300 import sel_attn_fwd
    from nsa_block_selection_gb300._lib import sel_attn_bwd

    tq, tk, tv, ti, tdo = to_dev(q, k, v, idx, dO)
    B, M, H, D = tq.shape
    f32 = torch.float32
    O, L = sel_attn_fwd(tq, tk, tv, ti, bs, scale, out=poisoned((B, M, H, D), f32),
                        lse=poisoned((B, H, M), f32))
    grads = sel_attn_bwd(tq, tk, tv, ti, O, L, tdo, bs, scale, dq=poisoned(tq.shape, f32),
                         dk=poisoned(tk.shape, f32), dv=poisoned(tv.shape, f32))
    torch.cuda.synchronize()
    return [g.cpu().numpy().astype(np.float64) for g in grads]


U16 = 2.0 ** -11  # fp16 unit roundoff
KAPPA = 4         # units of u per element (see the module docstring)


def assert_elementwise(name, g, ex, mag, what=""):
    """|g - ex| <= KAPPA * U16 * mag at every element."""
    assert np.isfinite(g).all(), f"{what} {name}: non-finite"
    bound = KAPPA * U16 * mag
    err = np.abs(g - ex)
    bad = err > bound
    if bad.any():
        i = np.unravel_index(np.argmax(np.where(bad, err - bound, -np.inf)), err.shape)
        raise AssertionError(
            f"{what} {name}: {int(bad.sum())} of {err.size} elements out of bound; worst at "
            f"{tuple(int(x) for x in i)}: got {g[i]:.6e} exact {ex[i]:.6e} bound {bound[i]:.3e}")


def _check(got, q, k, v, idx, dO, bs, scale=None, what=""):
    exact = oracle.sel_attn_bwd(q, k, v, idx, dO, bs, scale)
    mags = oracle.sel_attn_bwd(q, k, v, idx, dO, bs, scale, magnitudes=True)
    for name, g, ex, mg in zip(("dQ", "dK", "dV"), got, exact, mags):
        assert_elementwise(name, g, ex, mg, what)


@pytest.mark.parametrize("B,M,N,D,bs,T,rule", [
    (2, 700, 700, 128, 64, 5, "first_two_local"),
    (1, 900, 900, 64, 32, 4, "local"),
    (1, 500, 500, 128, 32, 6, "first_local"),
    (1, 300, 520, 128, 64, 3, "local"),
    (1, 520, 300, 64, 64, 3, "local"),
    (1, 520, 300, 128, 64, 3, "local"),
    (1, 410, 200, 128, 32, 5, "first_two_local"),
    (1, 640, 640, 128, 64, 10, "all_causal"),
])
def test_bwd_matches_oracle(B, M, N, D, bs, T, rule):
    q, k, v, idx = small_inputs(B, M, N, 16, 2, D, bs, T, rule, seed=M + T)
    dO = np.random.default_rng(M).standard_normal(q.shape).astype(np.float32)
    got = _run(q, k, v, idx, dO, bs)
    _check(got, q, k, v, idx, dO, bs, what=f"M{M} N{N} D{D} bs{bs}")


def test_bwd_padding_out_of_range_future_and_empty_rows():
    q, k, v, idx = small_inputs(1, 400, 400, 16, 2, 128, 64, 6, "first_two_local", seed=9)
    rng = np.random.default_rng(10)
    idx = rng.permuted(idx, axis=-1).copy()
    pads = idx < 0
    idx[pads] = rng.choice(np.array([-1, -3, 7, 1 << 29], np.int32), size=int(pads.sum()))
    idx[0, 5:9] = -1  # empty rows
    dO = rng.standard_normal(q.shape).astype(np.float32)
    got = _run(q, k, v, idx, dO, 64, scale=0.1)
    _check(got, q, k, v, idx, dO, 64, scale=0.1, what="padding")
    assert np.all(got[0][0, 5:9] == 0)  # dQ of empty rows


@pytest.mark.parametrize("bs", [64, 32])
def test_bwd_local_blocks_taken_by_some_rows_only(bs):
    """The local-block kernel (D = 128) takes each row's entries of its own
    block c and of block c - 1. Here rows of one block row differ: some
    list both, some one, some neither, and one block row (queries 4 bs ..
    5 bs - 1) lists neither anywhere, so its CTA runs no step and stores
    zero dQ rows before the key-major kernel adds their other blocks."""
    M = 9 * bs + 5
    q, k, v, idx = small_inputs(1, M, M, 16, 2, 128, bs, 6, "first_two_local", seed=bs + 3)
    rng = np.random.default_rng(bs)
    c = (np.arange(M) // bs)[None, :, None, None]
    drop_c = rng.random(idx.shape[:3])[..., None] < 0.3
    drop_p = rng.random(idx.shape[:3])[..., None] < 0.3
    row4 = (c == 4)
    idx = np.where(((idx == c) & (drop_c | row4)) | ((idx == c - 1) & (drop_p | row4)), -1,
                   idx).astype(np.int32)
    dO = rng.standard_normal(q.shape).astype(np.float32)
    got = _run(q, k, v, idx, dO, bs)
    _check(got, q, k, v, idx, dO, bs, what=f"local rows bs{bs}")


@pytest.mark.parametrize("T,N", [(0, 256), (3, 0)])
def test_bwd_degenerate(T, N):
    import torch

    q, k, v, idx = small_inputs(1, 256, 256, 8, 1, 64, 32, 3, "local", seed=11)
    if T == 0:
        idx = np.zeros((1, 256, 1, 0), np.int32)
    k, v = k[:, :N].copy(), v[:, :N].copy()
    dO = np.ones(q.shape, np.float32)
    dq, dk, dv = _run(q, k, v, idx, dO, 32)
    assert np.all(dq == 0) and np.all(dk == 0) and np.all(dv == 0)


@pytest.mark.parametrize("name", ["m64k_bs64", "m32k_bs32"])
def test_bwd_full_size(name):
    """Full-size workloads: dQ on sampled rows and dK/dV of sampled blocks vs
    the oracle; dV column sums equal the summed upstream gradient of every
    non-empty row and dK column sums vanish (exact identities)."""
    import torch

    from nsa_block_selection_gb300 import inputs as gen
    from _parity import sample_rows

    w = gen.workload(name)
    q, k, v, idx = gen.make_inputs(w)
    dO = np.random.default_rng(1).standard_normal(q.shape, dtype=np.float32)
    dq, dk, dv = _run(q, k, v, idx, dO, w.block_size)
    hpg = w.H // w.G
    # dQ, sampled rows
    rows = sample_rows(w.B, w.M, w.G, w.block_size, seed=7, n_random=512)
    ex = oracle.sel_attn_bwd_dq_rows(q, k, v, idx, dO, rows, w.block_size)
    mg = oracle.sel_attn_bwd_dq_rows(q, k, v, idx, dO, rows, w.block_size, magnitudes=True)
    got = np.stack([dq[b, m, g * hpg:(g + 1) * hpg] for b, m, g in rows])
    assert_elementwise("dQ", got, ex, mg, "sampled rows")
    # dK / dV of sampled blocks (the first, a middle, the last)
    nblk = -(-w.N // w.block_size)
    for b, g, t in ((0, 0, 1), (w.B - 1, w.G - 1, nblk // 2), (0, w.G // 2, nblk - 1)):
        ek, ev = oracle.sel_attn_bwd_block(q, k, v, idx, dO, b, g, t, w.block_size)
        mk, mv = oracle.sel_attn_bwd_block(q, k, v, idx, dO, b, g, t, w.block_size,
                                           magnitudes=True)
        sl = slice(t * w.block_size, min((t + 1) * w.block_size, w.N))
        assert_elementwise("dK", dk[b, sl, g], ek, mk, f"block {t}")
        assert_elementwise("dV", dv[b, sl, g], ev, mv, f"block {t}")
    # identities over all keys
    nonempty = (idx >= 0).any(-1)  # every row lists its own block here
    assert nonempty.all()
    want = dO.astype(np.float64).reshape(w.B, w.M, w.G, hpg, w.D).sum(axis=(1, 3))
    np.testing.assert_allclose(dv.sum(axis=1), want, rtol=1e-4, atol=1e-3 * np.abs(want).max())
    assert np.abs(dk.sum(axis=1)).max() <= 1e-4 * np.abs(dk).sum(axis=1).max()


@pytest.mark.parametrize("H,G,bs", [(4, 4, 64), (6, 2, 32), (16, 4, 64), (32, 2, 32)])
def test_bwd_heads_per_group(H, G, bs):
    """1, 3, 4 and 16 query heads per KV group."""
    q, k, v, idx = small_inputs(1, 500, 500, H, G, 128, bs, 5, "first_two_local", seed=H + G)
    dO = np.random.default_rng(H).standard_normal(q.shape).astype(np.float32)
    got = _run(q, k, v, idx, dO, bs)
    _check(got, q, k, v, idx, dO, bs, what=f"H{H} G{G}")


U_BF16 = 2.0 ** -8  # bf16 unit roundoff


@pytest.mark.parametrize("B,M,N,D,bs,T,rule", [
    (2, 700, 700, 128, 64, 5, "first_two_local"),
    (1, 900, 900, 64, 32, 4, "local"),
    (1, 500, 500, 128, 32, 6, "first_local"),
    (1, 300, 520, 128, 64, 3, "local"),
])
def test_bwd_bf16_matches_oracle(B, M, N, D, bs, T, rule):
    """bf16 inputs (nsa_sel_attn_bwd_ex): the same per-element bound with the
    bf16 unit roundoff, 4 u |terms| (dO, P and dS rounded to bf16 once each;
    the forward's bf16 P enters delta through O)."""
    import torch

    from nsa_block_selection_gb300 import inputs as gen
    from nsa_block_selection_gb300 import sel_attn_fwd
    from nsa_block_selection_gb300._lib import sel_attn_bwd

    w = gen.Workload("bwd_bf16", B, M, N, 16, 2, D, bs, T, 1.0, rule)
    q, k, v = gen.make_qkv(w, M + T, "bf16")
    idx = gen.make_block_indices(w.replace(N=min(M, N)) if M <= N else w, M + T)
    dO = np.random.default_rng(M + 1).standard_normal(q.shape).astype(np.float32)
    tq, tk, tv = (torch.from_numpy(np.asarray(x)).cuda().to(torch.bfloat16) for x in (q, k, v))
    ti, tdo = to_dev(idx, dO)
    f32 = torch.float32
    O, L = sel_attn_fwd(tq, tk, tv, ti, bs, out=poisoned((B, M, 16, D), f32),
                        lse=poisoned((B, 16, M), f32))
    grads = sel_attn_bwd(tq, tk, tv, ti, O, L, tdo, bs, dq=poisoned(tq.shape, f32),
                         dk=poisoned(tk.shape, f32), dv=poisoned(tv.shape, f32))
    torch.cuda.synchronize()
    got = [g.cpu().numpy().astype(np.float64) for g in grads]
    qd, kd, vd = (np.asarray(x, dtype=np.float64) for x in (q, k, v))
    exact = oracle.sel_attn_bwd(qd, kd, vd, idx, dO, bs)
    mags = oracle.sel_attn_bwd(qd, kd, vd, idx, dO, bs, magnitudes=True)
    for name, g, ex, mg in zip(("dQ", "dK", "dV"), got, exact, mags):
        assert np.isfinite(g).all(), f"bf16 {name}: non-finite"
        err = np.abs(g - ex)
        bound = KAPPA * U_BF16 * mg
        assert np.all(err <= bound), \
            f"bf16 {name}: {int((err > bound).sum())} elements beyond 4u|terms|"


def test_bwd_bf16_full_size():
    """m64k_bs64 with bf16 inputs: dQ on sampled rows and dK/dV of sampled
    blocks against the oracle on the same bf16 values, per element under
    4 u |terms| with the bf16 unit roundoff; the dV and dK column identities."""
    import torch

    from nsa_block_selection_gb300 import inputs as gen
    from nsa_block_selection_gb300 import sel_attn_fwd
    from nsa_block_selection_gb300._lib import sel_attn_bwd
    from _parity import sample_rows

    w = gen.workload("m64k_bs64")
    seed = gen.default_seed(w.name)
    q, k, v = gen.make_qkv(w, seed, "bf16")
    idx = gen.make_block_indices(w, seed)
    dO = np.random.default_rng(2).standard_normal(q.shape, dtype=np.float32)
    tq, tk, tv = (torch.from_numpy(x).cuda().to(torch.bfloat16) for x in (q, k, v))
    ti, tdo = to_dev(idx, dO)
    f32 = torch.float32
    O, L = sel_attn_fwd(tq, tk, tv, ti, w.block_size, out=poisoned(tuple(tq.shape), f32),
                        lse=poisoned((w.B, w.H, w.M), f32))
    dq, dk, dv = sel_attn_bwd(tq, tk, tv, ti, O, L, tdo, w.block_size,
                              dq=poisoned(tuple(tq.shape), f32), dk=poisoned(tuple(tk.shape), f32),
                              dv=poisoned(tuple(tv.shape), f32))
    torch.cuda.synchronize()
    del O, L, tq, tk, tv, ti, tdo
    dq, dk, dv = (x.cpu().numpy().astype(np.float64) for x in (dq, dk, dv))
    hpg = w.H // w.G
    rows = sample_rows(w.B, w.M, w.G, w.block_size, seed=9, n_random=256)
    ex = oracle.sel_attn_bwd_dq_rows(q, k, v, idx, dO, rows, w.block_size)
    mg = oracle.sel_attn_bwd_dq_rows(q, k, v, idx, dO, rows, w.block_size, magnitudes=True)
    got = np.stack([dq[b, m, g * hpg:(g + 1) * hpg] for b, m, g in rows])

    def check(name, g, e, m):
        assert np.isfinite(g).all(), f"bf16 {name}: non-finite"
        bad = np.abs(g - e) > KAPPA * U_BF16 * m
        assert not bad.any(), f"bf16 {name}: {int(bad.sum())} elements beyond 4u|terms|"

    check("dQ", got, ex, mg)
    nblk = -(-w.N // w.block_size)
    for b, g, t in ((0, 0, 1), (0, w.G - 1, nblk // 2), (0, w.G // 2, nblk - 1)):
        ek, ev = oracle.sel_attn_bwd_block(q, k, v, idx, dO, b, g, t, w.block_size)
        mk, mv = oracle.sel_attn_bwd_block(q, k, v, idx, dO, b, g, t, w.block_size,
                                           magnitudes=True)
        sl = slice(t * w.block_size, min((t + 1) * w.block_size, w.N))
        check(f"dK block {t}", dk[b, sl, g], ek, mk)
        check(f"dV block {t}", dv[b, sl, g], ev, mv)
    # the same identities; bf16 rounds P and dS 8 times more coarsely than fp16
    want = dO.astype(np.float64).reshape(w.B, w.M, w.G, hpg, w.D).sum(axis=(1, 3))
    np.testing.assert_allclose(dv.sum(axis=1), want, rtol=8e-4, atol=8e-3 * np.abs(want).max())
    assert np.abs(dk.sum(axis=1)).max() <= 8e-4 * np.abs(dk).sum(axis=1).max()
