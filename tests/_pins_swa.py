"""Pins of the sliding-window attention oracle, as functions of the module
under test (so planted mistakes can be run against them).

They check it against: torch's scaled_dot_product_attention in float64 for
the dense, causal and arbitrary-window cases (the window mask built here by
brute force over (i, j) pairs), a log-sum-exp recomputed with math.fsum, the
selection-attention oracle with one-key blocks listing exactly the window
(a second, independent implementation), closed forms and a hand-worked case.
"""

from __future__ import annotations

import math

import numpy as np


def _inputs(rng, B, M, N, H, Hkv, D):
    q = rng.standard_normal((B, M, H, D)).astype(np.float16)
    k = rng.standard_normal((B, N, Hkv, D)).astype(np.float16)
    v = rng.standard_normal((B, N, Hkv, D)).astype(np.float16)
    return q, k, v


def _sdpa(q, k, v, mask, scale):
    """torch SDPA in float64; mask [M, N] bool (True = attend); K/V expanded per group."""
    import torch

    H, Hkv = q.shape[2], k.shape[2]
    tq = torch.from_numpy(q.astype(np.float64)).permute(0, 2, 1, 3)
    tk = torch.from_numpy(k.astype(np.float64)).repeat_interleave(H // Hkv, dim=2).permute(0, 2, 1, 3)
    tv = torch.from_numpy(v.astype(np.float64)).repeat_interleave(H // Hkv, dim=2).permute(0, 2, 1, 3)
    m = torch.from_numpy(mask)
    o = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, attn_mask=m, scale=scale)
    s = (tq @ tk.transpose(-1, -2)) * scale
    lse = torch.logsumexp(s.masked_fill(~m, -math.inf), dim=-1)
    return o.permute(0, 2, 1, 3).numpy(), lse.numpy()


def _brute_mask(M, N, left, right):
    mask = np.zeros((M, N), dtype=bool)
    for i in range(M):
        for j in range(N):
            ok = True
            if left >= 0 and j < i - left:
                ok = False
            if right >= 0 and j > i + right:
                ok = False
            mask[i, j] = ok
    return mask


def pin_sdpa_windows(W):
    rng = np.random.default_rng(11)
    q, k, v = _inputs(rng, 2, 37, 37, 6, 2, 16)
    scale = 1 / 4
    for left, right in ((-1, -1), (-1, 0), (5, 0), (0, 0), (3, 4), (-1, 2), (9, -1), (40, 40)):
        mask = _brute_mask(37, 37, left, right)
        o_ref, l_ref = _sdpa(q, k, v, mask, scale)
        O, L = W.swa_fwd(q, k, v, left, right, scale)
        np.testing.assert_allclose(O, o_ref, atol=1e-12, rtol=1e-12)
        np.testing.assert_allclose(L, l_ref, atol=1e-12, rtol=1e-12)


def pin_queries_and_keys_differ(W):
    rng = np.random.default_rng(12)
    for M, N in ((20, 31), (31, 20)):
        q, k, v = _inputs(rng, 1, M, N, 4, 4, 8)
        for left, right in ((3, 2), (-1, 0)):
            mask = _brute_mask(M, N, left, right)
            O, L = W.swa_fwd(q, k, v, left, right, 0.3)
            keep = mask.any(1)
            o_ref, l_ref = _sdpa(q, k, v, mask | ~keep[:, None], 0.3)  # SDPA wants a key per row
            np.testing.assert_allclose(O[:, keep], o_ref[:, keep], atol=1e-12)
            np.testing.assert_allclose(L[:, :, keep], l_ref[:, :, keep], atol=1e-12)
            assert (O[:, ~keep] == 0).all() and np.isneginf(L[:, :, ~keep]).all()


def pin_lse_fsum(W):
    rng = np.random.default_rng(13)
    q, k, v = _inputs(rng, 1, 12, 12, 2, 1, 8)
    _, L = W.swa_fwd(q, k, v, 4, 1, 0.5)
    for i in range(12):
        for h in range(2):
            js = [j for j in range(12) if i - 4 <= j <= i + 1]
            s = [0.5 * float(np.dot(q[0, i, h].astype(np.float64), k[0, j, 0].astype(np.float64)))
                 for j in js]
            mx = max(s)
            want = mx + math.log(math.fsum(math.exp(x - mx) for x in s))
            assert abs(L[0, h, i] - want) < 1e-12


def pin_matches_selection_oracle(W):
    """(LEFT, 0) windows equal selection attention with one-key blocks
    listing exactly the window."""
    import oracle.sel_attn as S

    rng = np.random.default_rng(14)
    q, k, v = _inputs(rng, 1, 40, 40, 8, 2, 16)
    for left in (0, 3, 17):
        T = left + 1
        idx = np.full((1, 40, 2, T), -1, np.int32)
        for i in range(40):
            blocks = list(range(max(0, i - left), i + 1))
            idx[0, i, :, :len(blocks)] = blocks
        O1, L1 = S.sel_attn_fwd(q, k, v, idx, 1, 0.25)
        O2, L2 = W.swa_fwd(q, k, v, left, 0, 0.25)
        np.testing.assert_allclose(O2, O1, atol=1e-12)
        np.testing.assert_allclose(L2, L1, atol=1e-12)


def pin_closed_forms(W):
    rng = np.random.default_rng(15)
    q, k, v = _inputs(rng, 1, 30, 30, 4, 2, 8)
    # K = 0: uniform weights over the window, LSE = ln(window size)
    O, L = W.swa_fwd(q, np.zeros_like(k), v, 4, 2, 0.7)
    for i in (0, 1, 10, 28, 29):
        js = np.arange(max(0, i - 4), min(29, i + 2) + 1)
        for h in range(4):
            np.testing.assert_allclose(O[0, i, h], v[0, js, h // 2].astype(np.float64).mean(0),
                                       atol=1e-12)
            assert abs(L[0, h, i] - math.log(len(js))) < 1e-12
    # window (0, 0): each query sees only its own key
    O, L = W.swa_fwd(q, k, v, 0, 0, 0.7)
    for i in (0, 7, 29):
        for h in range(4):
            np.testing.assert_array_equal(O[0, i, h], v[0, i, h // 2].astype(np.float64))
            want = 0.7 * float(q[0, i, h].astype(np.float64) @ k[0, i, h // 2].astype(np.float64))
            assert abs(L[0, h, i] - want) < 1e-12
    # V = const: O = const wherever a key is visible
    O, _ = W.swa_fwd(q, k, np.full_like(v, 1.5), 3, 3, 0.7)
    np.testing.assert_allclose(O, 1.5, atol=1e-12)


def pin_hand_case(W):
    # D = 2, one head, N = 3, scale 1, window (1, 0):
    # q1 = (1, 0) sees k0 = (1, 0) (score 1) and k1 = (0, 2) (score 0)
    q = np.zeros((1, 3, 1, 2)); q[0, 1, 0] = (1, 0)
    k = np.zeros((1, 3, 1, 2)); k[0, 0, 0] = (1, 0); k[0, 1, 0] = (0, 2); k[0, 2, 0] = (5, 5)
    v = np.zeros((1, 3, 1, 2)); v[0, 0, 0] = (1, 0); v[0, 1, 0] = (0, 1); v[0, 2, 0] = (9, 9)
    O, L = W.swa_fwd(q, k, v, 1, 0, 1.0)
    e = math.e
    np.testing.assert_allclose(O[0, 1, 0], [e / (e + 1), 1 / (e + 1)], atol=1e-15)
    assert abs(L[0, 0, 1] - math.log(e + 1)) < 1e-15
    # query 0 sees only k0 (score 0): O = v0, LSE = 0
    np.testing.assert_allclose(O[0, 0, 0], [1, 0], atol=1e-15)
    assert abs(L[0, 0, 0]) < 1e-15


PINS = [pin_sdpa_windows, pin_queries_and_keys_differ, pin_lse_fsum,
        pin_matches_selection_oracle, pin_closed_forms, pin_hand_case]
