"""CPU oracle for NSA selection-attention forward -- TEST INFRASTRUCTURE ONLY.

Only the tests, the smoke check and the benchmark's CPU-baseline leg may use
this module. The product path (the CUDA library and its Python binding) never
imports or calls it, and shares no code with it.

What it computes (all in float64 from the fp16 inputs), following
"[wave] NSA: selection attention forward kernel":

* section "Operation": Q [B,M,H,D], K and V [B,N,G,D],
  block_indices [B,M,G,T] in; O_slc [B,M,H,D] and LSE_slc [B,H,M] out,
  T being the number of selected blocks per query;
* section "Algorithm": for query m, each selected block t contributes the
  keys [t*block_size, (t+1)*block_size); scores are Q K^T, causally masked,
  softmaxed; the softmax is taken over all selected blocks together;
* section "Requirements": the heads of a GQA group share one index row;
  the softmax is the online (running max + log-sum-exp) one across all T
  blocks; the causal mask applies inside the gathered blocks; LSE is returned.

Readings taken where the pages are silent (each is a parameter of the
definition below, stated once here):

* scale: scores are multiplied by ``scale`` (1/sqrt(D) unless given);
* causal alignment: key n is visible to query m iff n <= m;
* head -> group: head h belongs to group h // (H/G) (contiguous heads);
* padding: any index < 0 is padding, wherever it sits in the row;
* an index >= ceil(N/block_size) is padding too (it names no keys);
* duplicates: a row must not list a block twice (ValueError here);
* a row with no visible key gives O = 0 and LSE = -inf;
* LSE is the natural log of the sum of exp of the scaled, masked scores.

Two routes compute the same numbers:

* ``route="set"``: the plain definition. The visible key set is
  S = {n : n < N, n <= m, floor(n/bs) listed}; LSE = log sum_{n in S} exp(s_n)
  and O = sum_{n in S} exp(s_n - LSE) V[n]. This is exact up to rounding.
* ``route="online"``: the block loop in the order the row lists the blocks,
  carrying a running max, a running sum and a running weighted V sum (the
  online softmax named in the Algorithm and Requirements sections).
  ``emulate_kernel_rounding=True`` (or ``"f16"``) carries the running sums in
  float32 and rounds the probabilities to fp16 for the V product only (the
  "FP16 matmuls, FP32 accumulation" requirement), to measure how much of the
  parity tolerance that rounding uses; ``"bf16"`` rounds them to bfloat16
  instead (the same requirement read for bf16 operands).

Every step is pinned by tests (textbook attention through a library routine,
closed forms, hand-worked cases, order invariance, planted mistakes); no
function here is parity-unpinned.
"""

from __future__ import annotations

import math
from typing import Iterable, Optional, Sequence, Tuple

import numpy as np

__all__ = [
    "head_group",
    "num_blocks",
    "selected_blocks",
    "block_keys",
    "causal_visible",
    "visible_keys",
    "scores",
    "logsumexp_rows",
    "attend",
    "round_bf16",
    "sel_attn_row",
    "sel_attn_rows",
    "sel_attn_fwd",
    "softmax_grad_terms",
    "softmax_grad_magnitudes",
    "sel_attn_bwd",
    "sel_attn_bwd_dq_rows",
    "sel_attn_bwd_block",
]


# --------------------------------------------------------------------------
# Index-side steps (section "Operation" and "Algorithm", step 2)
# --------------------------------------------------------------------------

def head_group(h: int, H: int, G: int) -> int:
    """KV group of query head h: heads of one group share an index row
    (section "Requirements", GQA support); contiguous-heads reading."""
    return h // (H // G)


def num_blocks(N: int, block_size: int) -> int:
    """Number of blocks the N keys form: ceil(N / block_size)."""
    return -(-N // block_size)


def selected_blocks(idx_row: Sequence[int], N: int, block_size: int) -> list:
    """Block ids a row selects, in the row's order, padding dropped.

    Entries < 0 and entries >= ceil(N/bs) name no keys and are skipped. A
    block listed twice is rejected: the rows come from a top-k selection.
    """
    nblk = num_blocks(N, block_size)
    out = [int(t) for t in idx_row if 0 <= int(t) < nblk]
    if len(set(out)) != len(out):
        raise ValueError(f"index row lists a block twice: {list(idx_row)}")
    return out


def block_keys(t: int, block_size: int, N: int) -> np.ndarray:
    """Keys gathered for block t: [t*bs, (t+1)*bs), clipped to [0, N)
    (section "Algorithm", step 2, the gather)."""
    return np.arange(t * block_size, min((t + 1) * block_size, N), dtype=np.int64)


def causal_visible(n: np.ndarray, m: int) -> np.ndarray:
    """Causal mask inside a gathered block: key n is seen by query m iff n <= m."""
    return n <= m


def visible_keys(idx_row: Sequence[int], m: int, N: int, block_size: int) -> np.ndarray:
    """The visible key set S of one (b, m, g) row, sorted ascending."""
    parts = [block_keys(t, block_size, N) for t in selected_blocks(idx_row, N, block_size)]
    if not parts:
        return np.zeros(0, dtype=np.int64)
    n = np.sort(np.concatenate(parts))
    return n[causal_visible(n, m)]


# --------------------------------------------------------------------------
# Arithmetic steps (section "Algorithm", step 2: QK^T, softmax, weighted V)
# --------------------------------------------------------------------------

def scores(q: np.ndarray, k: np.ndarray, scale: float) -> np.ndarray:
    """s[h, j] = scale * sum_d q[h, d] * k[j, d], float64."""
    return scale * (q @ k.T)


def logsumexp_rows(s: np.ndarray) -> np.ndarray:
    """log sum_j exp(s[h, j]) per row, stabilised by the row max; -inf if empty."""
    if s.shape[1] == 0:
        return np.full(s.shape[0], -np.inf)
    mu = s.max(axis=1)
    return mu + np.log(np.exp(s - mu[:, None]).sum(axis=1))


def attend(s: np.ndarray, lse: np.ndarray, v: np.ndarray) -> np.ndarray:
    """O[h, :] = sum_j exp(s[h, j] - lse[h]) * v[j, :]; zero rows if empty."""
    if s.shape[1] == 0:
        return np.zeros((s.shape[0], v.shape[1]))
    return np.exp(s - lse[:, None]) @ v


# --------------------------------------------------------------------------
# One (b, m, g) row: both routes
# --------------------------------------------------------------------------

def _row_operands(Q, K, V, b, m, g, H, G):
    hpg = H // G
    heads = [h for h in range(H) if head_group(h, H, G) == g]
    if len(heads) != hpg:
        raise ValueError("heads do not split evenly into groups")
    q = np.asarray(Q[b, m, heads], dtype=np.float64)
    return heads, q, K[b, :, g], V[b, :, g]


def _route_set(q, Kg, Vg, idx_row, m, N, bs, scale):
    n = visible_keys(idx_row, m, N, bs)
    k = np.asarray(Kg[n], dtype=np.float64)
    v = np.asarray(Vg[n], dtype=np.float64)
    s = scores(q, k, scale)
    lse = logsumexp_rows(s)
    return attend(s, lse, v), lse


def round_bf16(x: np.ndarray) -> np.ndarray:
    """Nearest bfloat16 of float32 values (ties to even), as float32.

    bfloat16 is the upper half of an IEEE binary32: rounding adds half a unit
    of the dropped 16 bits (minus one when the kept part is even, so that
    exact ties go to the even neighbour) and clears them. Finite inputs only.
    """
    u = np.asarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    u = (u + 0x7FFF + ((u >> 16) & 1)) >> 16 << 16
    return u.astype(np.uint32).view(np.float32)


def _round_p(p: np.ndarray, how) -> np.ndarray:
    if how == "bf16":
        return round_bf16(p)
    if how is True or how == "f16":
        return p.astype(np.float16).astype(np.float32)
    raise ValueError(f"unknown rounding {how!r}")


def _route_online(q, Kg, Vg, idx_row, m, N, bs, scale, emulate_kernel_rounding):
    hpg, D = q.shape
    acc_t = np.float32 if emulate_kernel_rounding else np.float64
    run_max = np.full(hpg, -np.inf)
    run_sum = np.zeros(hpg, dtype=acc_t)
    acc = np.zeros((hpg, D), dtype=acc_t)
    for t in selected_blocks(idx_row, N, bs):
        n = block_keys(t, bs, N)
        n = n[causal_visible(n, m)]
        if n.size == 0:
            continue  # a block wholly in the future contributes nothing
        k = np.asarray(Kg[n], dtype=np.float64)
        v = np.asarray(Vg[n], dtype=np.float64)
        s = scores(q, k, scale)
        new_max = np.maximum(run_max, s.max(axis=1))
        alpha = np.exp(run_max - new_max)  # exp(-inf) = 0 on the first block
        p = np.exp(s - new_max[:, None])
        if emulate_kernel_rounding:
            p = p.astype(np.float32)
            alpha = alpha.astype(np.float32)
            run_sum = run_sum * alpha + p.sum(axis=1, dtype=np.float32)
            p16 = _round_p(p, emulate_kernel_rounding)
            acc = acc * alpha[:, None] + (p16 @ v.astype(np.float32)).astype(np.float32)
        else:
            run_sum = run_sum * alpha + p.sum(axis=1)
            acc = acc * alpha[:, None] + p @ v
        run_max = new_max
    run_sum = run_sum.astype(np.float64)
    acc = acc.astype(np.float64)
    empty = run_sum == 0
    with np.errstate(divide="ignore", invalid="ignore"):
        o = np.where(empty[:, None], 0.0, acc / np.where(empty, 1.0, run_sum)[:, None])
        lse = np.where(empty, -np.inf, run_max + np.log(np.where(empty, 1.0, run_sum)))
    return o, lse


def sel_attn_row(Q, K, V, idx, b: int, m: int, g: int, block_size: int,
                 scale: Optional[float] = None, route: str = "set",
                 emulate_kernel_rounding: bool = False) -> Tuple[np.ndarray, np.ndarray, list]:
    """O [H/G, D] and LSE [H/G] for the heads of group g at query (b, m).

    Returns (O_rows, LSE_rows, heads) where ``heads`` lists the head ids.
    """
    B, M, H, D = Q.shape
    N, G = K.shape[1], K.shape[2]
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    heads, q, Kg, Vg = _row_operands(Q, K, V, b, m, g, H, G)
    row = np.asarray(idx[b, m, g])
    if route == "set":
        o, lse = _route_set(q, Kg, Vg, row, m, N, block_size, scale)
    elif route == "online":
        o, lse = _route_online(q, Kg, Vg, row, m, N, block_size, scale,
                               emulate_kernel_rounding)
    else:
        raise ValueError(route)
    return o, lse, heads


def sel_attn_rows(Q, K, V, idx, rows: Iterable[Tuple[int, int, int]], block_size: int,
                  scale: Optional[float] = None, route: str = "set",
                  emulate_kernel_rounding: bool = False):
    """Oracle on a list of (b, m, g) rows.

    Returns O [R, H/G, D] and LSE [R, H/G] (float64), row r matching rows[r];
    the heads of row r are g*(H/G) .. g*(H/G)+H/G-1.
    """
    rows = list(rows)
    H, D = Q.shape[2], Q.shape[3]
    hpg = H // K.shape[2]
    O = np.empty((len(rows), hpg, D))
    L = np.empty((len(rows), hpg))
    for r, (b, m, g) in enumerate(rows):
        O[r], L[r], _ = sel_attn_row(Q, K, V, idx, b, m, g, block_size, scale, route,
                                     emulate_kernel_rounding)
    return O, L


def sel_attn_fwd(Q, K, V, idx, block_size: int, scale: Optional[float] = None,
                 route: str = "set", emulate_kernel_rounding: bool = False):
    """Full oracle: O_slc [B,M,H,D] and LSE_slc [B,H,M], float64."""
    B, M, H, D = Q.shape
    G = K.shape[2]
    O = np.zeros((B, M, H, D))
    L = np.zeros((B, H, M))
    for b in range(B):
        for m in range(M):
            for g in range(G):
                o, lse, heads = sel_attn_row(Q, K, V, idx, b, m, g, block_size, scale,
                                             route, emulate_kernel_rounding)
                O[b, m, heads] = o
                L[b, heads, m] = lse
    return O, L


# --------------------------------------------------------------------------
# Backward (gradients of the forward above)
# --------------------------------------------------------------------------
#
# The issue's "Requirements" section returns LSE because the backward pass
# needs it. The gradient of the definition above, per (b, m, g) row and head
# h, with p_n = exp(s_n - LSE), dP_n = dO . v_n and
# delta = sum_n p_n dP_n (= dO . O):
#
#   dV[n] += p_n dO                  dS_n = p_n (dP_n - delta)
#   dQ    += scale sum_n dS_n k_n    dK[n] += scale dS_n q
#
# summed over every (m, h) whose visible set contains key n.

def softmax_grad_terms(s: np.ndarray, lse: np.ndarray, v: np.ndarray, do: np.ndarray):
    """p, dS for one row: s [H', n], lse [H'], v [n, D], do [H', D]."""
    p = np.exp(s - lse[:, None])
    dp = do @ v.T
    delta = (p * dp).sum(axis=1)
    return p, p * (dp - delta[:, None])


def softmax_grad_magnitudes(s: np.ndarray, lse: np.ndarray, v: np.ndarray, do: np.ndarray):
    """p and an upper bound of |dS| for one row, built from absolute values
    only: |dP_n| <= sum_d |dO_d| |v_nd| and |delta| <= sum_d |dO_d|
    sum_n p_n |v_nd| (since O = sum_n p_n v_n), so |dS_n| <= p_n (those two
    sums added). Each term is the magnitude an operand's relative error is
    taken of, so a rounding error of relative size r in dO, V, O or dS moves
    dS_n by at most r times this bound."""
    p = np.exp(s - lse[:, None])
    av, ado = np.abs(v), np.abs(do)
    dp_mag = ado @ av.T
    delta_mag = (ado * (p @ av)).sum(axis=1)
    return p, p * (dp_mag + delta_mag[:, None])


def _fp16(x: np.ndarray) -> np.ndarray:
    return x.astype(np.float16).astype(np.float64)


def sel_attn_bwd(Q, K, V, idx, dO, block_size: int, scale: Optional[float] = None,
                 emulate_kernel_rounding: bool = False, magnitudes: bool = False):
    """Gradients dQ [B,M,H,D], dK [B,N,G,D], dV [B,N,G,D] (float64) of the
    forward for the upstream gradient dO [B,M,H,D] (LSE is recomputed).

    ``emulate_kernel_rounding=True`` rounds to fp16 the operands that enter
    fp16 matrix products on the GPU (dO, P for dV, dS for dQ and dK), all
    else in float64: it measures what fp16 operands alone cost.

    ``magnitudes=True`` returns instead, per element, the sum of the absolute
    values of the terms that make it up (dS replaced by the bound of
    :func:`softmax_grad_magnitudes`, q, k, dO by their absolute values): the
    scale against which the rounding of those terms is measured, per
    element, in the GPU parity tolerance."""
    B, M, H, D = Q.shape
    N, G = K.shape[1], K.shape[2]
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    dQ = np.zeros((B, M, H, D))
    dK = np.zeros((B, N, G, D))
    dV = np.zeros((B, N, G, D))
    for b in range(B):
        for m in range(M):
            for g in range(G):
                heads, q, Kg, Vg = _row_operands(Q, K, V, b, m, g, H, G)
                n = visible_keys(idx[b, m, g], m, N, block_size)
                if n.size == 0:
                    continue
                k = np.asarray(Kg[n], dtype=np.float64)
                v = np.asarray(Vg[n], dtype=np.float64)
                do = np.asarray(dO[b, m, heads], dtype=np.float64)
                s = scores(q, k, scale)
                if magnitudes:
                    p, ds = softmax_grad_magnitudes(s, logsumexp_rows(s), v, do)
                    q, k, do = np.abs(q), np.abs(k), np.abs(do)
                elif emulate_kernel_rounding:
                    lse = logsumexp_rows(s)
                    p = np.exp(s - lse[:, None])
                    dp = _fp16(do) @ v.T
                    delta = (do * attend(s, lse, v)).sum(axis=1)
                    ds = _fp16(p * (dp - delta[:, None]))
                    p, do = _fp16(p), _fp16(do)
                else:
                    p, ds = softmax_grad_terms(s, logsumexp_rows(s), v, do)
                dQ[b, m, heads] = scale * (ds @ k)
                dK[b, n, g] += scale * (ds.T @ q)
                dV[b, n, g] += p.T @ do
    return dQ, dK, dV


def sel_attn_bwd_dq_rows(Q, K, V, idx, dO, rows, block_size: int,
                         scale: Optional[float] = None, magnitudes: bool = False) -> np.ndarray:
    """dQ [R, H/G, D] of the listed (b, m, g) rows (each row's dQ depends on
    that row only); with ``magnitudes=True`` the per-element magnitudes of
    :func:`sel_attn_bwd` instead."""
    B, M, H, D = Q.shape
    N, G = K.shape[1], K.shape[2]
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    out = np.zeros((len(rows), H // G, D))
    for r, (b, m, g) in enumerate(rows):
        heads, q, Kg, Vg = _row_operands(Q, K, V, b, m, g, H, G)
        n = visible_keys(idx[b, m, g], m, N, block_size)
        if n.size == 0:
            continue
        k = np.asarray(Kg[n], dtype=np.float64)
        v = np.asarray(Vg[n], dtype=np.float64)
        s = scores(q, k, scale)
        do = np.asarray(dO[b, m, heads], dtype=np.float64)
        if magnitudes:
            _, ds = softmax_grad_magnitudes(s, logsumexp_rows(s), v, do)
            k = np.abs(k)
        else:
            _, ds = softmax_grad_terms(s, logsumexp_rows(s), v, do)
        out[r] = scale * (ds @ k)
    return out


def sel_attn_bwd_block(Q, K, V, idx, dO, b: int, g: int, t: int, block_size: int,
                       scale: Optional[float] = None, magnitudes: bool = False):
    """dK, dV rows [keys of block t, D] of (b, g): contributions of every row
    of group g that selects block t; with ``magnitudes=True`` the
    per-element magnitudes of :func:`sel_attn_bwd` instead."""
    B, M, H, D = Q.shape
    N, G = K.shape[1], K.shape[2]
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    keys = block_keys(t, block_size, N)
    dK = np.zeros((keys.size, D))
    dV = np.zeros((keys.size, D))
    for m in np.nonzero((np.asarray(idx[b, :, g]) == t).any(axis=-1))[0]:
        m = int(m)
        heads, q, Kg, Vg = _row_operands(Q, K, V, b, m, g, H, G)
        n = visible_keys(idx[b, m, g], m, N, block_size)
        k = np.asarray(Kg[n], dtype=np.float64)
        v = np.asarray(Vg[n], dtype=np.float64)
        s = scores(q, k, scale)
        do = np.asarray(dO[b, m, heads], dtype=np.float64)
        if magnitudes:
            p, ds = softmax_grad_magnitudes(s, logsumexp_rows(s), v, do)
            q, do = np.abs(q), np.abs(do)
        else:
            p, ds = softmax_grad_terms(s, logsumexp_rows(s), v, do)
        sel = (n >= keys[0]) & (n <= keys[-1])
        dK[n[sel] - keys[0]] += scale * (ds[:, sel].T @ q)
        dV[n[sel] - keys[0]] += p[:, sel].T @ do
    return dK, dV
