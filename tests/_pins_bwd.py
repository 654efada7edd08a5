"""Pins for the oracle's backward (gradients of the selection-attention
forward), against facts other than the oracle itself:

* autograd through a library routine: torch ``scaled_dot_product_attention``
  in float64 under the boolean mask the index rows describe (K/V expanded
  from groups to heads, so autograd sums the heads of a group);
* central finite differences of the (pinned) oracle forward, float64;
* closed forms: a single visible key gives dQ = dK = 0 and dV = the sum of
  the upstream gradients that reach it;
* an exact invariant: for every query row and head the dS terms sum to zero,
  so dK summed over all keys of a (b, g) vanishes and dQ does not change when
  a constant vector is added to every key;
* the per-element magnitudes that scale the GPU tolerance: above |gradient|
  everywhere, equal to dV when every term is non-negative, zero when V is,
  and a closed form for one visible key.
"""

from __future__ import annotations

import numpy as np
import torch

from nsa_block_selection_gb300 import inputs as gen


def _rand(shape, seed, dtype=np.float64):
    return np.random.default_rng(seed).standard_normal(shape).astype(dtype)


def _rows_mask(idx, M, N, H, G, bs):
    """Boolean [B, H, M, N]: key n visible to (b, m, head h) per the rows."""
    B = idx.shape[0]
    mask = np.zeros((B, H, M, N), bool)
    hpg = H // G
    nblk = -(-N // bs)
    for b in range(B):
        for m in range(M):
            for g in range(G):
                for t in idx[b, m, g]:
                    if 0 <= t < nblk:
                        lo, hi = t * bs, min(t * bs + bs, N, m + 1)
                        mask[b, g * hpg:(g + 1) * hpg, m, lo:hi] = True
    return mask


def _library_grads(Q, K, V, idx, dO, bs, scale):
    B, M, H, D = Q.shape
    N, G = K.shape[1], K.shape[2]
    hpg = H // G
    q = torch.tensor(Q, dtype=torch.float64, requires_grad=True)
    k = torch.tensor(K, dtype=torch.float64, requires_grad=True)
    v = torch.tensor(V, dtype=torch.float64, requires_grad=True)
    qh = q.permute(0, 2, 1, 3)
    kh = k.permute(0, 2, 1, 3).repeat_interleave(hpg, 1)
    vh = v.permute(0, 2, 1, 3).repeat_interleave(hpg, 1)
    mask = torch.from_numpy(_rows_mask(idx, M, N, H, G, bs))
    o = torch.nn.functional.scaled_dot_product_attention(qh, kh, vh, attn_mask=mask,
                                                         scale=scale)
    o.backward(torch.tensor(dO, dtype=torch.float64).permute(0, 2, 1, 3))
    return q.grad.numpy(), k.grad.numpy(), v.grad.numpy()


def _close(a, b, tol, what):
    err = np.abs(np.asarray(a) - np.asarray(b))
    bound = tol * (1.0 + np.abs(np.asarray(b)))
    assert np.all(err <= bound), f"{what}: max err {err.max():.3e}"


def bpin_matches_library_autograd(S):
    """Sparse rows (N not a multiple of bs, GQA 2 heads per group, B=2)."""
    w = gen.Workload("t", 2, 37, 37, 4, 2, 8, 4, 4, 1.0, "first_local")
    idx = gen.make_block_indices(w, 5)
    rng = np.random.default_rng(6)
    idx = np.ascontiguousarray(rng.permuted(idx, axis=-1))
    Q, K, V = _rand((2, 37, 4, 8), 1), _rand((2, 37, 2, 8), 2), _rand((2, 37, 2, 8), 3)
    dO = _rand((2, 37, 4, 8), 4)
    got = S.sel_attn_bwd(Q, K, V, idx, dO, 4, 0.3)
    want = _library_grads(Q, K, V, idx, dO, 4, 0.3)
    for name, a, b in zip(("dQ", "dK", "dV"), got, want):
        _close(a, b, 1e-10, name)


def bpin_finite_differences(S):
    """Central differences of sum(O * dO) in float64 on a tiny case."""
    B, M, H, G, D, bs = 1, 6, 2, 1, 3, 2
    Q, K, V = _rand((B, M, H, D), 11), _rand((B, M, G, D), 12), _rand((B, M, G, D), 13)
    dO = _rand((B, M, H, D), 14)
    idx = np.array([[0, -1], [0, -1], [1, -1], [1, 0], [2, 0], [1, 2]], np.int32)
    idx = idx.reshape(1, M, 1, 2)
    scale = 0.7
    dQ, dK, dV = S.sel_attn_bwd(Q, K, V, idx, dO, bs, scale)

    def loss(q, k, v):
        O, _ = S.sel_attn_fwd(q, k, v, idx, bs, scale)
        return float((O * dO).sum())

    eps = 1e-6
    for name, X, G_ in (("Q", Q, dQ), ("K", K, dK), ("V", V, dV)):
        num = np.zeros_like(X)
        for i in np.ndindex(X.shape):
            Xp, Xm = X.copy(), X.copy()
            Xp[i] += eps
            Xm[i] -= eps
            args_p = {"Q": (Xp, K, V), "K": (Q, Xp, V), "V": (Q, K, Xp)}[name]
            args_m = {"Q": (Xm, K, V), "K": (Q, Xm, V), "V": (Q, K, Xm)}[name]
            num[i] = (loss(*args_p) - loss(*args_m)) / (2 * eps)
        _close(G_, num, 1e-7, "d" + name + " vs finite differences")


def bpin_single_key_closed_form(S):
    """One visible key per row: p = 1, so dS = 0 (dQ = dK = 0) and dV[n] is
    the sum of dO over the heads and queries that see key n."""
    B, M, H, G, D, bs = 1, 8, 4, 2, 5, 4
    Q, K, V = _rand((B, M, H, D), 21), _rand((B, M, G, D), 22), _rand((B, M, G, D), 23)
    dO = _rand((B, M, H, D), 24)
    idx = np.full((B, M, G, 1), -1, np.int32)
    idx[0, 0] = 0  # query 0 sees key 0 only
    idx[0, 4] = 1  # query 4 sees key 4 only (block 1 = keys 4..7)
    dQ, dK, dV = S.sel_attn_bwd(Q, K, V, idx, dO, bs, 0.5)
    assert np.all(dQ == 0) and np.all(dK == 0)
    want = np.zeros_like(dV)
    for m, n in ((0, 0), (4, 4)):
        for g in range(G):
            want[0, n, g] = dO[0, m, 2 * g] + dO[0, m, 2 * g + 1]
    _close(dV, want, 1e-14, "dV single key")


def bpin_dk_sums_to_zero(S):
    """sum_n dS_n = 0 for every row and head, so sum over keys of dK is 0 and
    dQ is unchanged by a constant shift of every key."""
    w = gen.Workload("t", 1, 48, 48, 8, 2, 16, 8, 4, 1.0, "first_two_local")
    idx = gen.make_block_indices(w, 31)
    Q, K, V = _rand((1, 48, 8, 16), 32), _rand((1, 48, 2, 16), 33), _rand((1, 48, 2, 16), 34)
    dO = _rand((1, 48, 8, 16), 35)
    dQ, dK, dV = S.sel_attn_bwd(Q, K, V, idx, dO, 8, 0.25)
    assert np.abs(dK.sum(axis=1)).max() < 1e-10, np.abs(dK.sum(axis=1)).max()
    shift = _rand((1, 1, 2, 16), 36)
    # shifting keys changes the scores by q.c, a per-row constant: p unchanged
    dQ2, _, _ = S.sel_attn_bwd(Q, K + shift, V, idx, dO, 8, 0.25)
    _close(dQ2, dQ, 1e-9, "dQ under key shift")
    # and dV does not depend on dO's component along ... nothing: check
    # linearity in dO instead
    dQ3, dK3, dV3 = S.sel_attn_bwd(Q, K, V, idx, 2.5 * dO, 8, 0.25)
    for a, b in ((dQ3, dQ), (dK3, dK), (dV3, dV)):
        _close(a, 2.5 * b, 1e-12, "linearity in dO")


def bpin_magnitudes(S):
    """The per-element magnitudes (``magnitudes=True``) that scale the GPU
    tolerance: they bound the autograd-pinned gradients from above
    (triangle inequality); with dO >= 0 every dV term is >= 0, so dV's
    magnitude equals dV; with V = 0 every dS bound is 0, so dQ's and dK's
    magnitudes vanish; with one visible key per row p = 1 and dP = delta =
    dO.v, so the dS bound is 2 |dO.v| for V, dO >= 0 and dQ's magnitude is
    scale * 2 (dO.v) |k| (a value the exact dQ = 0 never shows)."""
    w = gen.Workload("t", 2, 30, 30, 4, 2, 8, 4, 4, 1.0, "first_local")
    idx = gen.make_block_indices(w, 41)
    Q, K, V = _rand((2, 30, 4, 8), 42), _rand((2, 30, 2, 8), 43), _rand((2, 30, 2, 8), 44)
    dO = _rand((2, 30, 4, 8), 45)
    exact = _library_grads(Q, K, V, idx, dO, 4, 0.4)
    mags = S.sel_attn_bwd(Q, K, V, idx, dO, 4, 0.4, magnitudes=True)
    for name, e, mg in zip(("dQ", "dK", "dV"), exact, mags):
        assert np.all(mg >= np.abs(e) - 1e-12), f"{name} magnitude below |gradient|"
        assert np.all(mg >= 0)
    dOp = np.abs(dO)
    _, _, dVp = _library_grads(Q, K, V, idx, dOp, 4, 0.4)
    _close(S.sel_attn_bwd(Q, K, V, idx, dOp, 4, 0.4, magnitudes=True)[2], dVp, 1e-12,
           "dV magnitude with dO >= 0")
    mq, mk, _ = S.sel_attn_bwd(Q, K, np.zeros_like(V), idx, dO, 4, 0.4, magnitudes=True)
    assert np.all(mq == 0) and np.all(mk == 0)
    # one visible key per row (as in the single-key pin): query 0 sees key 0
    B, M, H, G, D, bs = 1, 8, 4, 2, 5, 4
    Q1, K1 = _rand((B, M, H, D), 51), _rand((B, M, G, D), 52)
    V1, dO1 = np.abs(_rand((B, M, G, D), 53)), np.abs(_rand((B, M, H, D), 54))
    idx1 = np.full((B, M, G, 1), -1, np.int32)
    idx1[0, 0] = 0
    mq, _, _ = S.sel_attn_bwd(Q1, K1, V1, idx1, dO1, bs, 0.5, magnitudes=True)
    for h in range(H):
        g = h // 2
        want = 0.5 * 2 * float(dO1[0, 0, h] @ V1[0, 0, g]) * np.abs(K1[0, 0, g])
        _close(mq[0, 0, h], want, 1e-12, "dQ magnitude, one key")
    # the restricted helpers give the same magnitudes
    rows = [(1, 29, 0), (0, 3, 1)]
    got = S.sel_attn_bwd_dq_rows(Q, K, V, idx, dO, rows, 4, 0.4, magnitudes=True)
    for r, (b, m, g) in enumerate(rows):
        _close(got[r], mags[0][b, m, 2 * g:2 * g + 2], 1e-12, "dQ rows magnitude")
    bk, bv = S.sel_attn_bwd_block(Q, K, V, idx, dO, 1, 1, 2, 4, 0.4, magnitudes=True)
    _close(bk, mags[1][1, 8:12, 1], 1e-12, "dK block magnitude")
    _close(bv, mags[2][1, 8:12, 1], 1e-12, "dV block magnitude")


BPINS = [
    bpin_matches_library_autograd,
    bpin_finite_differences,
    bpin_single_key_closed_form,
    bpin_dk_sums_to_zero,
    bpin_magnitudes,
]
