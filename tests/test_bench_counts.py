"""bench.py's count of the backward's local entries (the entries of a
query's own block c and of block c - 1, which the local-block kernel sums
in place instead of reducing into dQ), against a loop over every entry."""

import numpy as np
import torch

import bench
from nsa_block_selection_gb300 import inputs as gen


def _by_loop(idx, w):
    nblk = (w.N + w.block_size - 1) // w.block_size
    vis = loc = 0
    B, M, G, T = idx.shape
    for b in range(B):
        for m in range(M):
            c = m // w.block_size
            last = min(m, w.N - 1)
            for g in range(G):
                for t in idx[b, m, g]:
                    t = int(t)
                    if t < 0 or t >= nblk or t * w.block_size > last:
                        continue
                    vis += 1
                    loc += t in (c, c - 1)
    return vis, loc


def test_local_entries_match_a_loop():
    w = gen.Workload("small", 1, 300, 200, 4, 2, 64, 32, 5, 1.0, "first_two_local")
    idx = gen.make_block_indices(w.replace(N=w.M), 5)  # rows may name blocks past N
    rng = np.random.default_rng(6)
    idx = rng.permuted(idx, axis=-1).copy()
    pads = idx < 0
    idx[pads] = rng.choice(np.array([-1, 9, 1 << 20], np.int32), size=int(pads.sum()))
    got = bench.local_entries(torch.from_numpy(idx), w)
    assert got == _by_loop(idx, w)
    assert 0 < got[1] < got[0]
