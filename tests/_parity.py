"""Shared helpers of the GPU parity tests: run the CUDA path, pick rows,
compare with the CPU oracle under the stated tolerance.

Tolerance: |O - O*| <= 2e-3 + 2e-3 |O*| elementwise and |LSE - LSE*| <= 1e-3,
with an empty row's LSE exactly -inf and its O exactly 0.
"""

from __future__ import annotations

import numpy as np

import oracle.sel_attn as oracle

O_ATOL = 2e-3
O_RTOL = 2e-3
LSE_ATOL = 1e-3


def poisoned(shape, dtype, device="cuda"):
    """An output buffer the kernel must overwrite: NaN for floating types,
    a value no index can take (2^31 - 1) for int32. A row the kernel never
    writes then fails the comparison instead of passing on whatever an
    earlier result left in recycled memory."""
    import torch

    fill = float("nan") if dtype.is_floating_point else 2 ** 31 - 1
    return torch.full(tuple(shape), fill, dtype=dtype, device=device)


def to_dev(*arrays):
    import torch

    return [torch.from_numpy(np.ascontiguousarray(a)).cuda() for a in arrays]


def run_cuda(q, k, v, idx, bs, scale=None, stream=None):
    """Inputs as numpy or CUDA tensors; returns CUDA tensors (O, LSE)."""
    import torch

    from nsa_block_selection_gb300 import sel_attn_fwd

    t = [x if isinstance(x, torch.Tensor) else to_dev(x)[0] for x in (q, k, v, idx)]
    B, M, H, D = t[0].shape
    out = sel_attn_fwd(*t, bs, scale, stream=stream,
                       out=poisoned((B, M, H, D), torch.float32, t[0].device),
                       lse=poisoned((B, H, M), torch.float32, t[0].device))
    torch.cuda.synchronize()
    return out


def gather_rows(O, L, rows, hpg):
    """O [R, hpg, D] and LSE [R, hpg] of rows (b, m, g) from device tensors."""
    import torch

    r = torch.as_tensor(np.asarray(rows, np.int64).reshape(-1, 3), device=O.device)
    b, m, g = r[:, 0:1], r[:, 1:2], r[:, 2:3]
    h = g * hpg + torch.arange(hpg, device=O.device)[None, :]
    return O[b, m, h].cpu().numpy().astype(np.float64), L[b, h, m].cpu().numpy().astype(np.float64)


def compare(o, l, o_ref, l_ref, what="", extra=0.0):
    """Assert the tolerance (plus ``extra``, elementwise, for the variants
    whose rounding adds a derived term); returns (max O error / bound, max
    LSE error)."""
    assert o.shape == o_ref.shape and l.shape == l_ref.shape
    empty = np.isneginf(l_ref)
    assert np.array_equal(np.isneginf(l), empty), f"{what}: -inf LSE mismatch"
    assert np.all(o[empty] == 0.0), f"{what}: empty rows must give O = 0"
    bound = O_ATOL + O_RTOL * np.abs(o_ref) + extra
    err = np.abs(o - o_ref)
    assert np.isfinite(o).all(), f"{what}: non-finite O"
    ratio = float((err / bound).max()) if err.size else 0.0
    lerr = float(np.abs(np.where(empty, 0.0, l - np.where(empty, 0.0, l_ref))).max()) \
        if l.size else 0.0
    assert ratio <= 1.0, f"{what}: O error {ratio:.3f} x tolerance"
    assert lerr <= LSE_ATOL, f"{what}: LSE error {lerr:.2e}"
    return ratio, lerr


def check_all_rows(q, k, v, idx, bs, O, L, scale=None, what=""):
    B, M, H, D = q.shape
    G = k.shape[2]
    rows = [(b, m, g) for b in range(B) for m in range(M) for g in range(G)]
    return check_rows(q, k, v, idx, bs, O, L, rows, scale, what)


def check_rows(q, k, v, idx, bs, O, L, rows, scale=None, what=""):
    hpg = q.shape[2] // k.shape[2]
    o, l = gather_rows(O, L, rows, hpg)
    o_ref, l_ref = oracle.sel_attn_rows(q, k, v, idx, rows, bs, scale)
    return compare(o, l, o_ref, l_ref, what)


def sample_rows(B, M, G, bs, seed, n_random=4096):
    """A fixed sample of (b, m, g) rows: random ones plus the edges -- the
    first two blocks, rows around block boundaries and the last 64 rows."""
    rng = np.random.default_rng(seed)
    rows = set()
    for _ in range(n_random):
        rows.add((int(rng.integers(B)), int(rng.integers(M)), int(rng.integers(G))))
    edge_m = set(range(min(M, 2 * bs)))
    for c in rng.integers(1, max(2, M // bs), size=16):
        edge_m.update(x for x in (c * bs - 1, c * bs, c * bs + 1) if 0 <= x < M)
    edge_m.update(range(max(0, M - 64), M))
    for m in edge_m:
        b = int(rng.integers(B))
        for g in range(G):
            rows.add((b, int(m), g))
    return sorted(rows)


def small_inputs(B, M, N, H, G, D, bs, T, rule, seed, sigma=1.0):
    """Seeded inputs for a small problem; index rows from the workload rules
    (rows for M > N may name blocks past N: they are padding)."""
    from nsa_block_selection_gb300 import inputs as gen

    w = gen.Workload("small", B, M, N, H, G, D, bs, T, sigma, rule)
    q, k, v = gen.make_qkv(w, seed)
    idx = gen.make_block_indices(w.replace(N=min(M, N)) if M <= N else w, seed)
    return q, k, v, idx
