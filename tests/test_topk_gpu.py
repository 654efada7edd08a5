"""nsa_topk_blocks against the top-k oracle: bit for bit (integer output).

Covers every register layout of the kernel (up to 256, 1024, 2048 and 4096
blocks per row), rows whose length is and is not a multiple of 4 (16-byte
and scalar loads), both selection paths (few survivors; many ties or more
than 32 free picks), rows with at most T candidates, queries past the last
key, no keys, ties, NaN, infinities, signed zeros and subnormal scores,
forced block counts from 0 to T, and the 64k-query workload on sampled rows with
the structure of every row checked on the device. Its output then drives
the selection-attention forward.
"""

import numpy as np
import pytest

import oracle.topk as K
from _parity import poisoned

pytestmark = pytest.mark.gpu


def _scores(rng, shape, kind):
    if kind == "uniform":
        return rng.random(shape, dtype=np.float32)
    if kind == "ties":
        return rng.integers(0, 3, shape).astype(np.float32)
    if kind == "quantized":
        # a few equal scores at the threshold: ties decided by block among
        # the fast path's survivors
        return np.floor(rng.random(shape, dtype=np.float32) * 256) / np.float32(256)
    if kind == "zeros_on_top":
        # negative scores with a few +0.0 and -0.0 on top (equal scores)
        x = -rng.random(shape, dtype=np.float32) - np.float32(0.5)
        pick = rng.random(shape) < 0.01
        x[pick] = np.where(rng.random(int(pick.sum())) < 0.5, np.float32(0.0), np.float32(-0.0))
        return x
    if kind == "special":
        pool = np.float32([0.0, -0.0, 0.5, -0.5, np.inf, -np.inf, np.nan, 1e-45, -1e-45,
                           3e-39, -3e-39, 1.0])
        return pool[rng.integers(0, pool.size, shape)]
    raise ValueError(kind)


def _run(sc, N, bs, T, n_init, n_local):
    import torch

    from nsa_block_selection_gb300 import topk_blocks

    B, M, G = sc.shape[:3]
    out = topk_blocks(torch.from_numpy(sc).cuda(), N, bs, T, n_init, n_local,
                      out=poisoned((B, M, G, T), torch.int32))
    torch.cuda.synchronize()
    return out.cpu().numpy()


@pytest.mark.parametrize("kind", ["uniform", "ties", "quantized", "zeros_on_top", "special"])
@pytest.mark.parametrize("B,M,N,G,bs,T,n_init,n_local", [
    (2, 700, 700, 3, 32, 6, 1, 2),       # <= 256 blocks
    (1, 1000, 1000, 2, 4, 16, 0, 0),     # <= 256 blocks, no forced
    (1, 1024, 1024, 2, 4, 12, 1, 2),     # 256 blocks: a multiple of 4 (bulk copies)
    (1, 2000, 2000, 2, 2, 9, 4, 5),      # <= 1024 blocks, all forced
    (1, 1200, 900, 1, 1, 33, 3, 1),      # <= 1024, queries past the keys, T > 32
    (1, 1800, 1800, 1, 1, 20, 1, 2),     # <= 2048 blocks
    (1, 4000, 4000, 1, 1, 40, 2, 2),     # <= 4096 blocks
])
def test_topk_matches_oracle(kind, B, M, N, G, bs, T, n_init, n_local):
    rng = np.random.default_rng(B * M + N + T)
    nblk = -(-N // bs)
    sc = _scores(rng, (B, M, G, nblk), kind)
    got = _run(sc, N, bs, T, n_init, n_local)
    want = K.topk_blocks(sc, N, bs, T, n_init, n_local)
    bad = np.argwhere((got != want).any(-1))
    assert bad.size == 0, (bad[:3].tolist(), got[tuple(bad[0])], want[tuple(bad[0])])


def test_topk_no_keys_and_all_forced():
    sc = np.zeros((1, 50, 2, 0), np.float32)
    assert (_run(sc, 0, 64, 5, 1, 2) == -1).all()
    rng = np.random.default_rng(9)
    sc = rng.random((1, 300, 1, 300), dtype=np.float32)
    got = _run(sc, 300, 1, 7, 3, 4)
    np.testing.assert_array_equal(got, K.topk_blocks(sc, 300, 1, 7, 3, 4))


def test_topk_full_size_sampled_and_structure():
    """m64k_bs64 shape: scores [1, 65536, 8, 1024] drawn on the device;
    sampled rows bit for bit against the oracle, every row's structure on
    the device (ascending, causal, block 0 and the two most recent present,
    count min(T, c+1))."""
    import torch

    from nsa_block_selection_gb300 import inputs as gen
    from nsa_block_selection_gb300 import topk_blocks

    B, M, G, bs, T = 1, 65536, 8, 64, 16
    sc = gen.make_block_scores_torch(B, M, G, M // bs, 17, "cuda")
    idx = topk_blocks(sc, M, bs, T, 1, 2, out=poisoned((B, M, G, T), torch.int32))
    torch.cuda.synchronize()
    m = torch.arange(M, device="cuda").view(1, M, 1, 1)
    c = m // bs
    valid = idx >= 0
    assert not (valid[..., 1:] & ~valid[..., :-1]).any()
    assert ((idx[..., 1:] > idx[..., :-1]) | ~valid[..., 1:]).all()
    assert (idx <= c).all()
    assert (valid.sum(-1) == torch.clamp(c[..., 0] + 1, max=T)).all()
    for blk in (torch.zeros_like(c), c, torch.clamp(c - 1, min=0)):
        assert (idx == blk).any(-1).all()
    rng = np.random.default_rng(3)
    ms = np.concatenate([rng.integers(0, M, 300), [0, 1, 63, 64, 1023, 1024, M - 1]])
    gs = rng.integers(0, G, ms.size)
    rows_sc = sc[0, ms, gs].cpu().numpy()
    got = idx[0, ms, gs].cpu().numpy()
    for r in range(ms.size):
        want = K.topk_row(rows_sc[r], int(ms[r]), M, bs, T, 1, 2)
        np.testing.assert_array_equal(got[r], want)


def test_topk_drives_the_forward():
    """scores -> nsa_topk_blocks -> nsa_sel_attn_fwd, against both oracles."""
    import torch

    from _parity import check_rows, sample_rows
    from nsa_block_selection_gb300 import inputs as gen
    from nsa_block_selection_gb300 import sel_attn_fwd, topk_blocks

    w = gen.Workload("topk", 1, 3000, 3000, 16, 2, 128, 64, 8, 1.0, "first_two_local")
    q, k, v = gen.make_qkv(w, 5)
    sc = gen.make_block_scores(1, w.M, w.G, -(-w.N // w.block_size), 5)
    idx = topk_blocks(torch.from_numpy(sc).cuda(), w.N, w.block_size, w.T, 1, 2,
                      out=poisoned((w.B, w.M, w.G, w.T), torch.int32))
    idx_np = idx.cpu().numpy()
    np.testing.assert_array_equal(idx_np, K.topk_blocks(sc, w.N, w.block_size, w.T, 1, 2))
    tq, tk, tv = (torch.from_numpy(x).cuda() for x in (q, k, v))
    O, L = sel_attn_fwd(tq, tk, tv, idx, w.block_size,
                        out=poisoned((w.B, w.M, w.H, w.D), torch.float32),
                        lse=poisoned((w.B, w.H, w.M), torch.float32))
    torch.cuda.synchronize()
    rows = sample_rows(w.B, w.M, w.G, w.block_size, 1, n_random=512)
    check_rows(q, k, v, idx_np, w.block_size, O, L, rows, what="topk->fwd")
