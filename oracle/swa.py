"""CPU oracle for GQA sliding-window attention forward -- TEST INFRASTRUCTURE ONLY.

Only the tests, the smoke check and the benchmark's CPU-baseline leg may use
this module. The product path never imports or calls it, and shares no code
with it.

What it computes (float64 from the 16-bit inputs), following "[Kernel][MI350]
Add 8 wave GQA sliding-window attention kernel", sections "Summary" and "What
it does":

* grouped-query attention: H query heads share H_kv key/value heads,
  H / H_kv consecutive query heads per KV head (the page's head remap sends
  query head h to KV head h // (H / H_kv));
* dense attention, or sliding-window attention with (LEFT, RIGHT) window
  semantics: query i attends to the keys in [i - LEFT, i + RIGHT];
* O [B, M, H, D] (the inputs' 16-bit type on the GPU; float64 here).

Readings taken where the page is silent (parameters of the definition):

* layouts Q [B, M, H, D], K and V [B, N, H_kv, D] (the page passes one row
  stride per tensor);
* query i is aligned with key i; keys outside [0, N) do not exist;
* a negative LEFT (RIGHT) leaves that side unbounded: (-1, -1) is dense,
  (-1, 0) causal;
* scores are multiplied by ``scale`` (1/sqrt(D) unless given);
* LSE [B, H, M] is the natural log of the sum of exp of the scaled scores
  over the window (returned for use by a backward pass or a branch merge);
  a row with no key gives O = 0 and LSE = -inf.

Plain definition, one (b, i, kv-group) row at a time, no blocking.
"""

from __future__ import annotations

import math
from typing import Iterable, Optional, Tuple

import numpy as np

__all__ = ["window_keys", "swa_row", "swa_rows", "swa_fwd"]


def window_keys(i: int, N: int, left: int, right: int) -> np.ndarray:
    """Keys visible to query i: [i - left, i + right] clipped to [0, N)."""
    lo = 0 if left < 0 else max(0, i - left)
    hi = N - 1 if right < 0 else min(N - 1, i + right)
    return np.arange(lo, hi + 1, dtype=np.int64) if hi >= lo else np.zeros(0, np.int64)


def swa_row(Q, K, V, b: int, i: int, g: int, left: int, right: int,
            scale: Optional[float] = None) -> Tuple[np.ndarray, np.ndarray]:
    """O [H/H_kv, D] and LSE [H/H_kv] for the query heads of KV head g."""
    H, D = Q.shape[2], Q.shape[3]
    N, Hkv = K.shape[1], K.shape[2]
    hpg = H // Hkv
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    q = np.asarray(Q[b, i, g * hpg:(g + 1) * hpg], dtype=np.float64)
    n = window_keys(i, N, left, right)
    if n.size == 0:
        return np.zeros((hpg, D)), np.full(hpg, -np.inf)
    k = np.asarray(K[b, n, g], dtype=np.float64)
    v = np.asarray(V[b, n, g], dtype=np.float64)
    s = scale * (q @ k.T)
    mx = s.max(axis=1, keepdims=True)
    e = np.exp(s - mx)
    tot = e.sum(axis=1)
    lse = mx[:, 0] + np.log(tot)
    return (e / tot[:, None]) @ v, lse


def swa_rows(Q, K, V, rows: Iterable[Tuple[int, int, int]], left: int, right: int,
             scale: Optional[float] = None):
    """O [R, H/H_kv, D] and LSE [R, H/H_kv] for rows (b, i, g)."""
    rows = list(rows)
    H, D = Q.shape[2], Q.shape[3]
    hpg = H // K.shape[2]
    O = np.empty((len(rows), hpg, D))
    L = np.empty((len(rows), hpg))
    for r, (b, i, g) in enumerate(rows):
        O[r], L[r] = swa_row(Q, K, V, b, i, g, left, right, scale)
    return O, L


def swa_fwd(Q, K, V, left: int, right: int, scale: Optional[float] = None):
    """Full oracle: O [B, M, H, D] and LSE [B, H, M], float64."""
    B, M, H, D = Q.shape
    Hkv = K.shape[2]
    if H % Hkv:
        raise ValueError("H must be a multiple of H_kv")
    hpg = H // Hkv
    O = np.zeros((B, M, H, D))
    L = np.zeros((B, H, M))
    for b in range(B):
        for i in range(M):
            for g in range(Hkv):
                o, lse = swa_row(Q, K, V, b, i, g, left, right, scale)
                O[b, i, g * hpg:(g + 1) * hpg] = o
                L[b, g * hpg:(g + 1) * hpg, i] = lse
    return O, L
