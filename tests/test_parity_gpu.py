"""CUDA path vs the CPU oracle (GB300): edge cases on small problems compared
on every row, then the five workloads at full size on sampled rows."""

import numpy as np
import pytest

from nsa_block_selection_gb300 import inputs as gen
from _parity import (check_all_rows, check_rows, gather_rows, run_cuda, sample_rows,
                     to_dev)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _need_gpu(cuda_lib):
    import torch

    assert torch.cuda.is_available(), "GPU tests need a CUDA device"


def _small(B, M, N, H, G, D, bs, T, rule, seed, sigma=1.0):
    w = gen.Workload("small", B, M, N, H, G, D, bs, T, sigma, rule)
    q, k, v = gen.make_qkv(w, seed)
    if M <= N:
        idx = gen.make_block_indices(w.replace(N=M), seed)
    else:
        idx = gen.make_block_indices(w, seed)
    return q, k, v, idx


def test_tiny_bs32_every_row():
    w = gen.workload("tiny_bs32")
    q, k, v, idx = gen.make_inputs(w)
    O, L = run_cuda(q, k, v, idx, w.block_size)
    check_all_rows(q, k, v, idx, w.block_size, O, L, what="tiny_bs32")


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("bs", [32, 64])
@pytest.mark.parametrize("rule,T", [("first_two_local", 5), ("local", 3), ("all_causal", 40)])
def test_ragged_small(D, bs, rule, T):
    """N not a multiple of the block size (short last block), B = 2, G = 2."""
    M = N = 1000
    if rule == "all_causal":
        T = -(-M // bs)
    q, k, v, idx = _small(2, M, N, 16, 2, D, bs, T, rule, seed=D + bs + T)
    O, L = run_cuda(q, k, v, idx, bs)
    check_all_rows(q, k, v, idx, bs, O, L, what=f"ragged D{D} bs{bs} {rule}")


@pytest.mark.parametrize("M,N", [(300, 520), (520, 300)])
def test_queries_and_keys_differ(M, N):
    """M != N: key n is visible to query m iff n <= m and n < N; index ids
    >= ceil(N/bs) are padding."""
    q, k, v, _ = _small(1, M, N, 8, 1, 128, 64, 4, "local", seed=3)
    rng = np.random.default_rng(4)
    nb = -(-max(M, N) // 64)
    idx = np.stack([rng.permutation(nb)[:4] for _ in range(M)]).astype(np.int32)
    idx = idx.reshape(1, M, 1, 4)
    O, L = run_cuda(q, k, v, idx, 64, scale=0.2)
    check_all_rows(q, k, v, idx, 64, O, L, scale=0.2, what=f"M{M} N{N}")


def test_empty_rows_T0_and_N0():
    import torch

    q, k, v, idx = _small(1, 64, 64, 8, 1, 64, 32, 2, "local", seed=5)
    # all padding
    idx_pad = np.full_like(idx, -1)
    O, L = run_cuda(q, k, v, idx_pad, 32)
    assert torch.all(O == 0) and torch.all(torch.isneginf(L))
    # T = 0
    O, L = run_cuda(q, k, v, np.zeros((1, 64, 1, 0), np.int32), 32)
    assert torch.all(O == 0) and torch.all(torch.isneginf(L))
    # N = 0
    O, L = run_cuda(q, k[:, :0].copy(), v[:, :0].copy(), idx, 32)
    assert torch.all(O == 0) and torch.all(torch.isneginf(L))


def test_padding_anywhere_out_of_range_and_future_blocks():
    """-1 in any position, ids >= ceil(N/bs), ids < -1 and blocks wholly in
    the causal future all contribute nothing."""
    q, k, v, idx = _small(2, 512, 512, 16, 2, 128, 64, 6, "first_two_local", seed=6)
    rng = np.random.default_rng(7)
    idx2 = rng.permuted(idx, axis=-1).copy()
    pads = idx2 < 0
    idx2[pads] = rng.choice(np.array([-1, -7, 8, 9, 1 << 30, -(1 << 30)], np.int32),
                            size=int(pads.sum()))
    # list the next (future) block where there is room
    c = (np.arange(512) // 64)[None, :, None]
    fut = np.broadcast_to(c + 1, idx2.shape[:3])
    room = (idx2 < 0).any(-1) & (fut < 8)
    for b, m, g in zip(*np.nonzero(room)):
        j = int(np.nonzero(idx2[b, m, g] < 0)[0][0])
        idx2[b, m, g, j] = fut[b, m, g]
    O, L = run_cuda(q, k, v, idx2, 64)
    check_all_rows(q, k, v, idx2, 64, O, L, what="padding/out-of-range/future")


def test_order_invariance():
    q, k, v, idx = _small(1, 2048, 2048, 8, 1, 128, 64, 16, "first_two_local", seed=8)
    rng = np.random.default_rng(9)
    O1, L1 = run_cuda(q, k, v, idx, 64)
    idx_p = rng.permuted(idx, axis=-1).copy()
    O2, L2 = run_cuda(q, k, v, idx_p, 64)
    check_all_rows(q, k, v, idx_p, 64, O2, L2, what="permuted rows")
    assert float((O1 - O2).abs().max()) < 2e-3


def test_unselected_and_future_rows_may_hold_nan():
    """K/V rows in every query's future, and blocks no row selects, never
    reach the output: NaN/Inf there leaves it bit-identical."""
    import torch

    M, N, bs = 384, 640, 32
    q, k, v, idx = _small(1, M, N, 16, 2, 128, bs, 6, "first_local", seed=10)
    used = np.zeros(-(-N // bs), bool)
    used[idx[idx >= 0]] = True
    O1, L1 = run_cuda(q, k, v, idx, bs)
    k2, v2 = k.copy(), v.copy()
    k2[:, M:] = np.float16(np.nan)
    v2[:, M:] = np.float16(np.inf)
    for t in np.nonzero(~used)[0]:
        k2[:, t * bs:(t + 1) * bs] = np.float16(-np.inf)
        v2[:, t * bs:(t + 1) * bs] = np.float16(np.nan)
    # inside diagonal blocks, rows past the query are masked: poison V there
    # for a problem with one query per block start
    O2, L2 = run_cuda(q, k2, v2, idx, bs)
    assert torch.equal(O1, O2) and torch.equal(L1, L2)
    assert torch.isfinite(O2).all()


def test_diagonal_future_rows_never_reach_output():
    """Within the query's own tile, keys after m never reach the output even
    when K and V hold NaN there (queries 0..5, keys 6.. poisoned)."""
    import torch

    D, bs = 64, 32
    q, k, v, _ = _small(1, 32, 32, 8, 1, D, bs, 1, "local", seed=11)
    idx = np.zeros((1, 32, 1, 1), np.int32)
    O1, L1 = run_cuda(q, k, v, idx, bs)
    k2, v2 = k.copy(), v.copy()
    k2[:, 6:] = np.float16(np.nan)
    v2[:, 6:] = np.float16(np.nan)
    O2, L2 = run_cuda(q[:, :6].copy(), k2, v2, idx[:, :6].copy(), bs)
    assert torch.equal(O1[:, :6], O2) and torch.equal(L1[:, :, :6], L2)


def test_deterministic_and_streams():
    import torch

    q, k, v, idx = _small(1, 1024, 1024, 16, 2, 128, 64, 8, "first_local", seed=12)
    tq, tk, tv, ti = to_dev(q, k, v, idx)
    O1, L1 = run_cuda(tq, tk, tv, ti, 64)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        O2, L2 = run_cuda(tq, tk, tv, ti, 64, stream=s)
    assert torch.equal(O1, O2) and torch.equal(L1, L2)


def test_scale_argument():
    q, k, v, idx = _small(1, 256, 256, 8, 1, 64, 32, 4, "local", seed=13)
    O, L = run_cuda(q, k, v, idx, 32, scale=0.05)
    check_all_rows(q, k, v, idx, 32, O, L, scale=0.05, what="scale 0.05")


# --------------------------------------------------------------------------
# Full-size workloads, sampled rows
# --------------------------------------------------------------------------

@pytest.mark.parametrize("name", ["m8k_bs64", "m64k_bs64", "m32k_bs32", "dense_m16k"])
def test_full_size_sampled(name):
    import torch

    w = gen.workload(name)
    q, k, v, idx = gen.make_inputs(w)
    O, L = run_cuda(q, k, v, idx, w.block_size)
    # every row lists its own block, so every LSE is finite and O is finite
    assert bool(torch.isfinite(L).all()) and bool(torch.isfinite(O).all())
    rows = sample_rows(w.B, w.M, w.G, w.block_size, seed=gen.default_seed(name))
    ratio, lerr = check_rows(q, k, v, idx, w.block_size, O, L, rows, what=name)
    print(f"{name}: {len(rows)} rows, O err {ratio:.3f} x tol, LSE err {lerr:.2e}")


def test_bounded_wait_reports_timeout():
    """A wait nothing completes gives up after its limit and is reported by
    nsa_sync_status; the context stays usable and the status clears."""
    from nsa_block_selection_gb300 import _lib

    assert _lib.sync_status() == 0
    assert _lib.selftest_wait_timeout(2_000_000) == 0  # 2 ms
    assert _lib.sync_status() == -8
    assert _lib.sync_status() == 0
    q, k, v, idx = _small(1, 128, 128, 8, 1, 64, 32, 2, "local", seed=14)
    O, L = run_cuda(q, k, v, idx, 32)
    check_all_rows(q, k, v, idx, 32, O, L, what="after timeout")
    assert _lib.sync_status() == 0


@pytest.mark.parametrize("B,M,N,T,bs,chunk", [
    (1, 1000, 1000, 5, 64, 0), (2, 777, 777, 4, 32, 100), (2, 600, 450, 6, 64, 64),
    (1, 300, 520, 3, 32, 1000), (1, 256, 256, 0, 32, 64)])
def test_host_entry_matches_device_entry(B, M, N, T, bs, chunk):
    """Host buffers through the chunked pipeline == device entry, bit for bit."""
    import torch

    from nsa_block_selection_gb300 import _lib

    rule = "first_two_local" if T >= 3 else "local"
    q, k, v, idx = _small(B, M, N, 16, 2, 128, bs, max(T, 1), rule, seed=M + T)
    if T == 0:
        idx = np.zeros((B, M, 2, 0), np.int32)
    else:
        nb = -(-N // bs)
        idx = np.where(idx < nb, idx, -1).astype(np.int32)  # M > N: ids past N are padding
    O_d, L_d = run_cuda(q, k, v, idx, bs)
    pin = [torch.from_numpy(x).pin_memory() for x in (q, k, v, idx)]
    O_h, L_h = _lib.sel_attn_fwd_host(*pin, bs, chunk_m=chunk,
                                      out=_nan_pinned(O_d.shape), lse=_nan_pinned(L_d.shape))
    assert torch.equal(O_h, O_d.cpu()) and torch.equal(L_h, L_d.cpu())
    # pageable host memory is also accepted
    O_p, L_p = _lib.sel_attn_fwd_host(*[torch.from_numpy(x) for x in (q, k, v, idx)], bs,
                                      out=torch.full_like(O_h, float("nan")),
                                      lse=torch.full_like(L_h, float("nan")),
                                      chunk_m=chunk)
    assert torch.equal(O_p, O_d.cpu()) and torch.equal(L_p, L_d.cpu())
    if T:
        check_all_rows(q, k, v, idx, bs, O_d, L_d, what="host entry")


def _nan_pinned(shape):
    """Pinned host output the host entry point must overwrite (NaN-filled)."""
    import torch

    return torch.full(tuple(shape), float("nan"), dtype=torch.float32).pin_memory()


@pytest.mark.parametrize("M,bs,T,perm", [(2047, 32, 64, False), (1531, 64, 24, True),
                                          (13, 32, 1, False)])
def test_cta_shared_blocks(M, bs, T, perm):
    """Consecutive queries list many common blocks (every causal block), more
    than one CTA shares, in rows longer than 32 entries, with a partial last
    CTA; optionally each row permuted."""
    q, k, v, _ = _small(1, M, M, 8, 1, 128, bs, 1, "local", seed=M + bs)
    idx = gen.dense_causal_indices(1, M, 1, -(-M // bs), bs)
    idx = np.ascontiguousarray(idx[..., :T])  # the first T causal blocks
    if perm:
        idx = np.random.default_rng(1).permuted(idx, axis=-1).copy()
    O, L = run_cuda(q, k, v, idx, bs)
    check_all_rows(q, k, v, idx, bs, O, L, what=f"shared M{M} bs{bs} T{T}")


@pytest.mark.parametrize("H,G", [(4, 4), (8, 4), (6, 2), (16, 4), (32, 2)])
def test_heads_per_group(H, G):
    """1, 2, 3, 4 and 16 query heads per KV group (padded or split into
    sub-groups of 8), forward through the device and host entry points."""
    import torch

    from nsa_block_selection_gb300 import _lib

    q, k, v, idx = _small(2, 600, 600, H, G, 128, 64, 5, "first_two_local", seed=H * 10 + G)
    O, L = run_cuda(q, k, v, idx, 64)
    check_all_rows(q, k, v, idx, 64, O, L, what=f"H{H} G{G}")
    pin = [torch.from_numpy(x).pin_memory() for x in (q, k, v, idx)]
    O_h, L_h = _lib.sel_attn_fwd_host(*pin, 64, chunk_m=128, out=_nan_pinned(O.shape),
                                      lse=_nan_pinned(L.shape))
    assert torch.equal(O_h, O.cpu()) and torch.equal(L_h, L.cpu())
