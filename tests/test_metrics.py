"""Work counting used by the benchmark, checked against brute force."""

import numpy as np
import pytest
import torch

import oracle.sel_attn as oracle
from nsa_block_selection_gb300 import inputs as gen
from nsa_block_selection_gb300.metrics import count_rows, count_work


@pytest.mark.parametrize("M,N,bs", [(300, 300, 32), (200, 330, 64), (330, 200, 64)])
def test_counts_match_brute_force(M, N, bs):
    rng = np.random.default_rng(M + N)
    G, T, hpg, D = 2, 5, 8, 128
    nb = -(-max(M, N) // bs)
    idx = np.stack([rng.permutation(nb + 3)[:T] - 1 for _ in range(M * G)]).astype(np.int32)
    idx = idx.reshape(1, M, G, T)
    keys = blocks = block_keys = 0
    nblk = -(-N // bs)
    for m in range(M):
        for g in range(G):
            keys += len(oracle.visible_keys(idx[0, m, g], m, N, bs))
            for t in idx[0, m, g]:
                if 0 <= t < nblk and t * bs <= min(m, N - 1):
                    blocks += 1
                    block_keys += min(bs, N - t * bs)
    w = count_work(torch.from_numpy(idx), N, bs, hpg, D, chunk_rows=97)
    assert w["visible_keys"] == keys
    assert w["flops"] == 4 * D * hpg * keys
    assert w["blocks"] == blocks
    assert w["gathered_bytes"] == 4 * D * block_keys
    ms = np.repeat(np.arange(M), G)
    assert count_rows(idx.reshape(-1, T), ms, N, bs, hpg, D) == w["flops"]


def test_target_workload_totals_scale():
    """m64k_bs64 totals land where the row rules put them (~16 blocks/row)."""
    w = gen.workload("m8k_bs64")
    idx = gen.make_block_indices(w, 1)
    r = count_work(torch.from_numpy(idx), w.N, w.block_size, 8, w.D)
    assert r["rows"] == w.M * w.G
    assert 15.0 < r["blocks"] / r["rows"] <= 16.0
    assert r["gathered_bytes"] == r["blocks"] * 64 * 128 * 4
