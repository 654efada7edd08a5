"""CPU oracle for top-k block selection -- TEST INFRASTRUCTURE ONLY.

Only the tests, the smoke check and the benchmark's CPU-baseline leg may use
this module. The product path never imports or calls it, and shares no code
with it.

The selection-attention pages take ``block_indices [B,M,G,T]`` as given and
name the kernel that supplies them: "[wave] NSA: selection attention forward
kernel", section "Depends on" (a top-k selection kernel, for block_indices);
section "Operation" fixes the output (T = number of selected blocks per
query) and section "Requirements" that the heads of a GQA group share one
index row, so a row is chosen per (b, m, g). The pages do not say how the
blocks are scored, so the operation takes one score per candidate block as
its input: ``scores [B, M, G, ceil(N/block_size)]``, float32.

Readings taken where the pages are silent:

* candidates of query m: the key blocks holding at least one key visible to
  m (causal, n <= m and n < N), i.e. t = 0 .. c with
  c = floor(min(m, N-1) / block_size); none when N = 0;
* forced blocks: the first ``n_init`` and the last ``n_local`` candidates are
  always selected (the workloads' "block 0 and the most recent blocks" rule;
  n_init + n_local <= T);
* the other T - (forced) slots go to the remaining candidates with the
  highest scores; equal scores rank the lower block index first (-0.0 equals
  +0.0); NaN ranks below every number, NaNs by block index;
* a row with at most T candidates selects all of them;
* the row is written in ascending block order, padded with -1 at the end.

Plain, unblocked code: one row at a time, ranking by a library sort.
"""

from __future__ import annotations

from typing import Sequence

import numpy as np

__all__ = ["last_candidate", "forced_blocks", "rank_order", "topk_row", "topk_blocks"]


def last_candidate(m: int, N: int, block_size: int) -> int:
    """Last block with a key visible to query m (-1: no candidate)."""
    if N <= 0:
        return -1
    return min(m, N - 1) // block_size


def forced_blocks(c: int, n_init: int, n_local: int) -> set:
    """The first n_init and the last n_local of the candidates 0..c."""
    cand = range(c + 1)
    return {t for t in cand if t < n_init or t > c - n_local}


def rank_order(scores: np.ndarray, blocks: Sequence[int]) -> list:
    """``blocks`` from most to least preferred: score descending, NaN last,
    ties to the lower block index."""
    blocks = np.asarray(list(blocks), dtype=np.int64)
    if blocks.size == 0:
        return []
    s = np.asarray(scores, dtype=np.float64)[blocks]
    nan = np.isnan(s)
    neg = np.where(nan, 0.0, -s) + 0.0  # + 0.0 turns -0.0 into +0.0
    # lexsort: last key is the primary one
    order = np.lexsort((blocks, neg, nan))
    return [int(t) for t in blocks[order]]


def topk_row(scores_row: np.ndarray, m: int, N: int, block_size: int, T: int,
             n_init: int, n_local: int) -> np.ndarray:
    """The T block indices of one (b, m, g) row."""
    if n_init < 0 or n_local < 0 or n_init + n_local > T:
        raise ValueError("need 0 <= n_init, n_local and n_init + n_local <= T")
    c = last_candidate(m, N, block_size)
    if c + 1 <= T:
        chosen = list(range(c + 1))
    else:
        forced = forced_blocks(c, n_init, n_local)
        rest = [t for t in range(c + 1) if t not in forced]
        chosen = sorted(forced) + rank_order(scores_row, rest)[:T - len(forced)]
    out = np.full(T, -1, dtype=np.int32)
    chosen = sorted(chosen)
    out[:len(chosen)] = chosen
    return out


def topk_blocks(scores: np.ndarray, N: int, block_size: int, T: int, n_init: int,
                n_local: int) -> np.ndarray:
    """block_indices [B, M, G, T] from scores [B, M, G, ceil(N/block_size)]."""
    B, M, G, S = scores.shape
    if S != -(-N // block_size):
        raise ValueError("scores must have ceil(N/block_size) entries per row")
    out = np.empty((B, M, G, T), dtype=np.int32)
    for b in range(B):
        for m in range(M):
            for g in range(G):
                out[b, m, g] = topk_row(scores[b, m, g], m, N, block_size, T, n_init, n_local)
    return out
