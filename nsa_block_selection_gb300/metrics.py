"""Algorithmic work of one selection-attention forward, counted exactly from
the index tensor (host-side bookkeeping for the benchmark; no attention
arithmetic).

* FLOPs: 4*D per (query, head, visible gathered key) -- 2*D for QK^T and
  2*D for PV.
* gathered bytes: every whole selected block that holds at least one
  visible key, K and V, fp16: 2 tensors * keys_in_block * D * 2 bytes. A
  block is [t*bs, (t+1)*bs) clipped to N; padding (< 0 or >= ceil(N/bs)) and
  blocks wholly after the query are not gathered.
"""

from __future__ import annotations


def count_work(idx, N: int, block_size: int, heads_per_group: int, D: int,
               chunk_rows: int = 1 << 22) -> dict:
    """idx: int32 torch tensor [B, M, G, T] (any device). Returns exact integer
    totals: flops, gathered_bytes, visible_keys (per (b,m,g) row, summed),
    blocks (gathered), rows."""
    import torch

    B, M, G, T = idx.shape
    dev = idx.device
    bs = int(block_size)
    nblk = -(-int(N) // bs)
    tot_keys = 0
    tot_blocks = 0
    tot_block_keys = 0
    flat = idx.reshape(B * M * G, T)
    m_of_row = torch.arange(M, device=dev, dtype=torch.int64).repeat_interleave(G).repeat(B)
    for lo in range(0, flat.shape[0], max(1, chunk_rows // max(T, 1))):
        hi = min(flat.shape[0], lo + max(1, chunk_rows // max(T, 1)))
        t = flat[lo:hi].to(torch.int64)
        m = m_of_row[lo:hi, None]
        last = torch.clamp(m, max=int(N) - 1)  # last visible key
        start = t * bs
        valid = (t >= 0) & (t < nblk) & (start <= last)
        end_block = torch.clamp(start + bs, max=int(N))
        end_vis = torch.minimum(end_block, last + 1)
        keys = torch.where(valid, end_vis - start, torch.zeros_like(t))
        bkeys = torch.where(valid, end_block - start, torch.zeros_like(t))
        tot_keys += int(keys.sum().item())
        tot_blocks += int(valid.sum().item())
        tot_block_keys += int(bkeys.sum().item())
    return {
        "flops": 4 * D * heads_per_group * tot_keys,
        "gathered_bytes": 2 * 2 * D * tot_block_keys,
        "visible_keys": tot_keys,
        "blocks": tot_blocks,
        "rows": B * M * G,
    }


def count_rows(idx_rows, m_rows, N: int, block_size: int, heads_per_group: int, D: int) -> int:
    """FLOPs of a list of rows: idx_rows int [R, T] (numpy), m_rows [R]."""
    import numpy as np

    t = np.asarray(idx_rows, np.int64)
    m = np.asarray(m_rows, np.int64)[:, None]
    bs = int(block_size)
    nblk = -(-int(N) // bs)
    last = np.minimum(m, int(N) - 1)
    start = t * bs
    valid = (t >= 0) & (t < nblk) & (start <= last)
    end_vis = np.minimum(np.minimum(start + bs, int(N)), last + 1)
    keys = np.where(valid, end_vis - start, 0).sum()
    return int(4 * D * heads_per_group * keys)
