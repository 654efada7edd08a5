"""Pins for the CPU oracle: facts fixed by the pages or by mathematics.

Each pin takes the oracle module and raises AssertionError when the oracle
disagrees with something other than itself:

* textbook causal softmax attention through a library routine
  (torch ``scaled_dot_product_attention`` in float64 on the CPU), with the
  LSE read back through an added zero-score "sink" key;
* closed forms (first query, K = 0, one visible key, constant V, per-group
  constant V for the head -> group map, equal keys);
* hand-worked cases whose scores, weights, O and LSE are derived below;
* brute force with explicit Python loops on tiny inputs;
* invariances (order of the index row, padding position, values of rows
  that are never selected);
* agreement of the two routes (plain definition vs. online block loop).

``tests/test_oracle_pins.py`` runs them on the oracle; ``tests/
test_oracle_mutants.py`` plants one mistake at a time in the oracle and checks
that some pin fails.
"""

from __future__ import annotations

import math

import numpy as np
import torch

from nsa_block_selection_gb300 import inputs as gen


def _rand(shape, seed, sigma=1.0):
    rng = np.random.default_rng(seed)
    return (rng.standard_normal(shape) * sigma).astype(np.float16)


def _sdpa_reference(Q, K, V, scale, mask=None, causal=False):
    """Library attention in float64: O [B,M,H,D] and LSE [B,H,M].

    K and V are expanded from G groups to H heads with head h reading group
    h // (H/G). LSE comes from a prepended key with score exactly 0 (a zero
    key) and a value that is 1 in an extra column: that column of the output
    equals 1 / (1 + exp(LSE)).
    """
    B, M, H, D = Q.shape
    N, G = K.shape[1], K.shape[2]
    hpg = H // G
    q = torch.from_numpy(Q.astype(np.float64)).permute(0, 2, 1, 3)
    k = torch.from_numpy(K.astype(np.float64)).permute(0, 2, 1, 3).repeat_interleave(hpg, 1)
    v = torch.from_numpy(V.astype(np.float64)).permute(0, 2, 1, 3).repeat_interleave(hpg, 1)
    # sink key at position 0
    k = torch.cat([torch.zeros(B, H, 1, D, dtype=torch.float64), k], dim=2)
    v = torch.cat([torch.zeros(B, H, 1, D, dtype=torch.float64), v], dim=2)
    col = torch.zeros(B, H, N + 1, 1, dtype=torch.float64)
    col[:, :, 0, 0] = 1.0
    v = torch.cat([v, col], dim=3)
    if causal:
        allow = torch.ones(M, N, dtype=torch.bool).tril()
        mask = allow
    if mask is None:
        mask = torch.ones(M, N, dtype=torch.bool)
    mask = torch.as_tensor(mask)
    if mask.dim() == 2:
        mask = mask[None, None]
    full = torch.cat([torch.ones(*mask.shape[:-1], 1, dtype=torch.bool), mask], dim=-1)
    out = torch.nn.functional.scaled_dot_product_attention(q, k, v, attn_mask=full, scale=scale)
    w_sink = out[..., D]
    o = out[..., :D] / (1.0 - w_sink)[..., None]
    lse = torch.log((1.0 - w_sink) / w_sink)
    return o.permute(0, 2, 1, 3).numpy(), lse.numpy()


def _close(a, b, tol=1e-10, what=""):
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    assert a.shape == b.shape, (what, a.shape, b.shape)
    both_inf = np.isinf(a) & np.isinf(b) & (np.sign(a) == np.sign(b))
    err = np.where(both_inf, 0.0, np.abs(a - b))
    assert np.all(err <= tol * (1 + np.abs(np.where(both_inf, 0, b)))), \
        f"{what}: max err {np.nanmax(err)}"


# --------------------------------------------------------------------------
# Pins
# --------------------------------------------------------------------------

def pin_dense_matches_library_attention(S):
    """Every causal block listed -> textbook causal softmax attention."""
    B, M, H, G, D, bs = 2, 40, 4, 2, 8, 4
    Q, K, V = _rand((B, M, H, D), 1), _rand((B, M, G, D), 2), _rand((B, M, G, D), 3)
    idx = gen.dense_causal_indices(B, M, G, 12, bs)  # 10 blocks + 2 pads
    rng = np.random.default_rng(4)
    idx = np.ascontiguousarray(rng.permuted(idx, axis=-1))  # order must not matter
    scale = 0.37
    O, L = S.sel_attn_fwd(Q, K, V, idx, bs, scale)
    Oref, Lref = _sdpa_reference(Q, K, V, scale, causal=True)
    _close(O, Oref, 1e-10, "O dense")
    _close(L, Lref, 1e-10, "LSE dense")


def pin_sparse_matches_library_masked_attention(S):
    """Sparse rows == library attention under the mask the rows describe.

    The mask marks key n visible for (b, m, g) iff n <= m and block
    floor(n/bs) is listed. N is not a multiple of bs, so the last block is
    short.
    """
    B, M, H, G, D, bs, T = 1, 30, 4, 2, 16, 4, 3
    N = M
    Q, K, V = _rand((B, M, H, D), 11), _rand((B, N, G, D), 12), _rand((B, N, G, D), 13)
    rng = np.random.default_rng(14)
    nblk = -(-N // bs)
    idx = np.full((B, M, G, T), -1, np.int32)
    mask = np.zeros((B, H, M, N), bool)
    for m in range(M):
        for g in range(G):
            c = m // bs
            pick = rng.choice(c + 1, size=min(T, c + 1), replace=False)
            row = list(pick) + [-1] * (T - len(pick))
            rng.shuffle(row)
            idx[0, m, g] = row
            for t in pick:
                for n in range(t * bs, min(t * bs + bs, N)):
                    if n <= m:
                        mask[0, g * (H // G):(g + 1) * (H // G), m, n] = True
    assert nblk * bs > N
    O, L = S.sel_attn_fwd(Q, K, V, idx, bs, 0.25)
    Oref, Lref = _sdpa_reference(Q, K, V, 0.25, mask=torch.from_numpy(mask))
    _close(O, Oref, 1e-10, "O sparse")
    _close(L, Lref, 1e-10, "LSE sparse")


def pin_routes_agree(S):
    """Plain definition == online block loop, for arbitrary block order."""
    w = gen.Workload("t", 2, 70, 70, 8, 2, 16, 8, 5, 1.0, "first_two_local")
    Q, K, V = gen.make_qkv(w, 21)
    idx = gen.make_block_indices(w, 21)
    rng = np.random.default_rng(22)
    idx = np.ascontiguousarray(rng.permuted(idx, axis=-1))
    O1, L1 = S.sel_attn_fwd(Q, K, V, idx, w.block_size)
    O2, L2 = S.sel_attn_fwd(Q, K, V, idx, w.block_size, route="online")
    _close(O1, O2, 1e-12, "O routes")
    _close(L1, L2, 1e-12, "LSE routes")


def pin_order_and_padding_position_invariance(S):
    """Permuting a row (padding included) changes nothing."""
    w = gen.Workload("t", 1, 64, 64, 4, 1, 8, 4, 6, 1.0, "first_local")
    Q, K, V = gen.make_qkv(w, 31)
    idx = gen.make_block_indices(w, 31)
    rng = np.random.default_rng(32)
    for route in ("set", "online"):
        O1, L1 = S.sel_attn_fwd(Q, K, V, idx, w.block_size, route=route)
        O2, L2 = S.sel_attn_fwd(Q, K, V, np.ascontiguousarray(rng.permuted(idx, axis=-1)),
                                w.block_size, route=route)
        _close(O1, O2, 1e-12, "O order " + route)
        _close(L1, L2, 1e-12, "LSE order " + route)


def pin_first_query_closed_form(S):
    """m = 0 sees only key 0: O = V[0, g], LSE = scale * q . k_0."""
    B, M, H, G, D, bs = 2, 8, 6, 3, 4, 4
    Q, K, V = _rand((B, M, H, D), 41), _rand((B, M, G, D), 42), _rand((B, M, G, D), 43)
    idx = np.full((B, M, G, 2), -1, np.int32)
    idx[:, :, :, 1] = 0
    O, L = S.sel_attn_fwd(Q, K, V, idx, bs, 0.5)
    for b in range(B):
        for h in range(H):
            g = h // 2
            np.testing.assert_array_equal(O[b, 0, h], V[b, 0, g].astype(np.float64))
            want = 0.5 * sum(float(Q[b, 0, h, d]) * float(K[b, 0, g, d]) for d in range(D))
            assert abs(L[b, h, 0] - want) < 1e-12, (L[b, h, 0], want)


def pin_zero_keys_closed_form(S):
    """K = 0: every score is 0, so O = mean of the visible V rows, LSE = ln|S|.

    N = 10, bs = 4: blocks are {0..3}, {4..7}, {8, 9}. Row for m = 9 lists
    [2, -1, 0]: visible keys 0, 1, 2, 3, 8, 9 (6 keys). Row for m = 5 lists
    [1, 0]: keys 0..5 visible (block 1 cut at 5 by the causal mask). Row for
    m = 7 lists [2, 1]: block 2 starts at 8 > 7, so keys 4..7 (4 keys).
    """
    N, bs, D = 10, 4, 3
    Q = _rand((1, N, 1, D), 51)
    K = np.zeros((1, N, 1, D), np.float16)
    V = _rand((1, N, 1, D), 52)
    idx = np.full((1, N, 1, 3), -1, np.int32)
    idx[0, 9, 0] = [2, -1, 0]
    idx[0, 5, 0] = [1, 0, -1]
    idx[0, 7, 0] = [2, 1, -1]
    O, L = S.sel_attn_fwd(Q, K, V, idx, bs, 1.0)
    v = V[0, :, 0].astype(np.float64)
    for m, keys in ((9, [0, 1, 2, 3, 8, 9]), (5, [0, 1, 2, 3, 4, 5]), (7, [4, 5, 6, 7])):
        _close(O[0, m, 0], v[keys].mean(axis=0), 1e-14, f"O K=0 m={m}")
        assert abs(L[0, 0, m] - math.log(len(keys))) < 1e-14, (m, L[0, 0, m])


def pin_single_key_and_constant_value(S):
    """One visible key -> O is its V row; constant V -> O is that constant."""
    N, bs, D = 12, 4, 5
    Q, K = _rand((1, N, 2, D), 61), _rand((1, N, 1, D), 62)
    V = _rand((1, N, 1, D), 63)
    idx = np.full((1, N, 1, 2), -1, np.int32)
    idx[0, 8, 0] = [-1, 2]  # m = 8: block 2 = keys 8..11, only key 8 visible
    O, L = S.sel_attn_fwd(Q, K, V, idx, bs, 0.3)
    for h in range(2):
        np.testing.assert_array_equal(O[0, 8, h], V[0, 8, 0].astype(np.float64))
        want = 0.3 * sum(float(Q[0, 8, h, d]) * float(K[0, 8, 0, d]) for d in range(D))
        assert abs(L[0, h, 8] - want) < 1e-12
    Vc = np.full((1, N, 1, D), 1.75, np.float16)
    idx2 = gen.dense_causal_indices(1, N, 1, 3, bs)
    O2, _ = S.sel_attn_fwd(Q, K, Vc, idx2, bs, 0.3)
    _close(O2, np.full(O2.shape, 1.75), 1e-14, "constant V")


def pin_hand_worked_case(S):
    """D = 2, bs = 2, N = 4, one head, scale = 1.

    k_0 = (1, 0), k_1 = (0, 1), k_2 = (1, 1), k_3 = (0, 0);
    v_0 = (1, 0), v_1 = (0, 1), v_2 = (2, 0), v_3 = (0, 2); q_m = (1, 0).
    Scores q.k = 1, 0, 1, 0.

    m = 3, row [1, 0]: all four keys. LSE = ln(2e + 2); weights e/(2e+2) on
      keys 0 and 2, 1/(2e+2) on keys 1 and 3; O = (3e, 3) / (2e + 2).
    m = 1, row [1, 0]: block 1 (keys 2, 3) is in the future; keys 0, 1.
      LSE = ln(e + 1); O = (e, 1) / (e + 1).
    m = 2, row [1, -1]: block 1, key 3 masked; key 2 alone. LSE = 1, O = (2, 0).
    m = 0, row [-1, -1]: nothing visible. O = (0, 0), LSE = -inf.
    """
    e = math.e
    K = np.array([[1, 0], [0, 1], [1, 1], [0, 0]], np.float16).reshape(1, 4, 1, 2)
    V = np.array([[1, 0], [0, 1], [2, 0], [0, 2]], np.float16).reshape(1, 4, 1, 2)
    Q = np.tile(np.array([1, 0], np.float16), (1, 4, 1, 1))
    idx = np.array([[-1, -1], [1, 0], [1, -1], [1, 0]], np.int32).reshape(1, 4, 1, 2)
    O, L = S.sel_attn_fwd(Q, K, V, idx, 2, 1.0)
    _close(O[0, 3, 0], [3 * e / (2 * e + 2), 3 / (2 * e + 2)], 1e-14, "hand m=3")
    _close(L[0, 0, 3], math.log(2 * e + 2), 1e-14, "hand lse m=3")
    _close(O[0, 1, 0], [e / (e + 1), 1 / (e + 1)], 1e-14, "hand m=1")
    _close(L[0, 0, 1], math.log(e + 1), 1e-14, "hand lse m=1")
    _close(O[0, 2, 0], [2.0, 0.0], 0.0, "hand m=2")
    _close(L[0, 0, 2], 1.0, 1e-15, "hand lse m=2")
    _close(O[0, 0, 0], [0.0, 0.0], 0.0, "hand m=0")
    assert L[0, 0, 0] == -np.inf


def pin_group_map_closed_form(S):
    """K = 0 and V[:, :, g] = g + 1: head h reads group h // (H/G)."""
    B, M, H, G, D, bs = 1, 9, 8, 4, 2, 3
    Q = _rand((B, M, H, D), 71)
    K = np.zeros((B, M, G, D), np.float16)
    V = np.zeros((B, M, G, D), np.float16)
    for g in range(G):
        V[:, :, g] = g + 1
    idx = gen.dense_causal_indices(B, M, G, 3, bs)
    O, _ = S.sel_attn_fwd(Q, K, V, idx, bs)
    for h in range(H):
        _close(O[0, :, h], np.full((M, D), h // 2 + 1.0), 1e-14, f"group of head {h}")


def pin_equal_keys_closed_form(S):
    """All keys equal to k: every score is s = scale q.k, LSE = s + ln|S|."""
    N, bs, D = 16, 4, 4
    Q = _rand((1, N, 1, D), 81)
    K = np.tile(_rand((1, 1, 1, D), 82), (1, N, 1, 1))
    V = _rand((1, N, 1, D), 83)
    idx = np.full((1, N, 1, 2), -1, np.int32)
    idx[0, 13, 0] = [3, 1]  # keys 4..7 and 12, 13
    _, L = S.sel_attn_fwd(Q, K, V, idx, bs, 0.5)
    s = 0.5 * sum(float(Q[0, 13, 0, d]) * float(K[0, 0, 0, d]) for d in range(D))
    assert abs(L[0, 0, 13] - (s + math.log(6))) < 1e-12


def pin_brute_force_loops(S):
    """Tiny random case against explicit Python loops (math.exp / fsum)."""
    B, M, H, G, D, bs, T = 1, 7, 2, 1, 3, 2, 3
    Q, K, V = _rand((B, M, H, D), 91), _rand((B, M, G, D), 92), _rand((B, M, G, D), 93)
    rng = np.random.default_rng(94)
    idx = np.full((B, M, G, T), -1, np.int32)
    for m in range(M):
        c = m // bs
        pick = rng.choice(c + 1, size=min(T, c + 1), replace=False)
        idx[0, m, 0, :len(pick)] = pick
    scale = 0.8
    O, L = S.sel_attn_fwd(Q, K, V, idx, bs, scale)
    for m in range(M):
        listed = [int(t) for t in idx[0, m, 0] if t >= 0]
        for h in range(H):
            sc = {}
            for n in range(M):
                if n // bs in listed and n <= m:
                    sc[n] = scale * math.fsum(float(Q[0, m, h, d]) * float(K[0, n, 0, d])
                                              for d in range(D))
            top = max(sc.values())
            z = math.fsum(math.exp(x - top) for x in sc.values())
            lse = top + math.log(z)
            assert abs(L[0, h, m] - lse) < 1e-12
            for d in range(D):
                o = math.fsum(math.exp(sc[n] - lse) * float(V[0, n, 0, d]) for n in sc)
                assert abs(O[0, m, h, d] - o) < 1e-12


def pin_unselected_rows_never_read(S):
    """NaN/Inf in rows no index selects, and out-of-range ids, change nothing."""
    w = gen.Workload("t", 1, 48, 48, 4, 2, 8, 4, 3, 1.0, "first_local")
    Q, K, V = gen.make_qkv(w, 101)
    idx = gen.make_block_indices(w, 101)
    O1, L1 = S.sel_attn_fwd(Q, K, V, idx, w.block_size)
    # blocks 9..11 are selected by nobody for query rows below 36: poison them
    # for a truncated problem that only has those queries
    M2 = 36
    Q2, idx2 = Q[:, :M2], idx[:, :M2].copy()
    K2, V2 = K.copy(), V.copy()
    K2[:, M2:] = np.float16(np.nan)
    V2[:, M2:] = np.float16(np.inf)
    # out-of-range ids are padding: replace the pads by ids >= ceil(N/bs)
    idx2[idx2 < 0] = 12 + (np.arange((idx2 < 0).sum()) % 5)
    O2, L2 = S.sel_attn_fwd(Q2, K2, V2, idx2, w.block_size)
    assert np.isfinite(O2).all() and np.isfinite(L2).all()
    _close(O2, O1[:, :M2], 0.0, "poisoned O")
    _close(L2, L1[:, :, :M2], 0.0, "poisoned LSE")


def pin_convex_hull(S):
    """Each O[d] lies within [min, max] of the attended V rows."""
    w = gen.Workload("t", 1, 40, 40, 4, 2, 8, 4, 4, 1.0, "local")
    Q, K, V = gen.make_qkv(w, 111)
    idx = gen.make_block_indices(w, 111)
    O, _ = S.sel_attn_fwd(Q, K, V, idx, w.block_size)
    for m in range(w.M):
        for g in range(w.G):
            keys = [n for n in range(w.N) if n <= m and n // w.block_size in set(idx[0, m, g])]
            vv = V[0, keys, g].astype(np.float64)
            for h in range(g * 2, g * 2 + 2):
                assert np.all(O[0, m, h] >= vv.min(0) - 1e-15)
                assert np.all(O[0, m, h] <= vv.max(0) + 1e-15)


def pin_duplicates_rejected(S):
    """A row listing a block twice is outside the contract (top-k output)."""
    Q, K, V = _rand((1, 4, 1, 2), 121), _rand((1, 4, 1, 2), 122), _rand((1, 4, 1, 2), 123)
    idx = np.array([[-1, -1], [0, -1], [1, 1], [0, 1]], np.int32).reshape(1, 4, 1, 2)
    try:
        S.sel_attn_fwd(Q, K, V, idx, 2)
    except ValueError:
        return
    raise AssertionError("duplicate block accepted")


def pin_default_scale(S):
    """scale defaults to 1/sqrt(D): single visible key, LSE = q.k / sqrt(D)."""
    D = 16
    Q, K, V = _rand((1, 1, 1, D), 131), _rand((1, 1, 1, D), 132), _rand((1, 1, 1, D), 133)
    idx = np.zeros((1, 1, 1, 1), np.int32)
    _, L = S.sel_attn_fwd(Q, K, V, idx, 32)
    want = sum(float(Q[0, 0, 0, d]) * float(K[0, 0, 0, d]) for d in range(D)) / 4.0
    assert abs(L[0, 0, 0] - want) < 1e-12


PINS = [
    pin_dense_matches_library_attention,
    pin_sparse_matches_library_masked_attention,
    pin_routes_agree,
    pin_order_and_padding_position_invariance,
    pin_first_query_closed_form,
    pin_zero_keys_closed_form,
    pin_single_key_and_constant_value,
    pin_hand_worked_case,
    pin_group_map_closed_form,
    pin_equal_keys_closed_form,
    pin_brute_force_loops,
    pin_unselected_rows_never_read,
    pin_convex_hull,
    pin_duplicates_rejected,
    pin_default_scale,
]
