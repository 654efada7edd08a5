"""Host-side checks of the two-pass forward (no GPU).

* The records: their definition, restated in ``_records.py`` and compared
  exactly with the list pass on the GPU, checked here on rows worked out by
  hand.
* The decomposition the two passes rely on: the softmax over a row's keys
  splits over the recorded blocks and the rest. The state the first pass
  leaves, (O_A, row sum 1, reference LSE_A), continued over the remaining
  keys gives the oracle's O and LSE. It is checked in fp64 on the oracle's
  own partial results ("[wave] NSA: selection attention forward kernel",
  section "Algorithm": one online softmax across the selected blocks; the
  online softmax is an order of the same sums).
"""

import numpy as np
import pytest

import oracle.sel_attn as oracle
from _records import MAXREC, records_ref
from nsa_block_selection_gb300 import inputs as gen


def _rows(M, T, fill):
    idx = np.full((1, M, 1, T), -1, np.int32)
    for m in range(M):
        r = fill(m)
        idx[0, m, 0, :len(r)] = r
    return idx


def test_records_by_hand():
    bs, N, M = 32, 160, 80
    # every query lists blocks 1, 0, 2 in that order (plus padding)
    idx = _rows(M, 4, lambda m: [1, 0, 2])
    rec = records_ref(idx, N, bs)[0, 0]
    # tiles of 16 queries: m0 = 0, 16, 32, 48, 64; a block qualifies when its
    # first key e * 32 is <= m0 and its keys end by min(M, N) = 80
    assert rec[0].tolist() == [1, 0] + [-1] * 6            # m0 = 0: block 0 (the tile's own)
    assert rec[1].tolist() == [1, 0] + [-1] * 6            # m0 = 16: block 0 still
    assert rec[2].tolist() == [2, 1, 0] + [-1] * 5         # m0 = 32: blocks 1, 0 (first row's order)
    assert rec[3].tolist() == [2, 1, 0] + [-1] * 5         # m0 = 48
    assert rec[4].tolist() == [2, 1, 0] + [-1] * 5         # m0 = 64: block 2 runs to key 95 >= M


def test_records_need_every_query_and_skip_padding_and_repeats():
    bs, N, M = 32, 160, 48
    # m0 = 32 tile: query 40 does not list block 0 -> nothing recorded
    idx = _rows(M, 4, lambda m: [1] if m == 40 else [0, 1])
    assert records_ref(idx, N, bs)[0, 0, 2, 0] == 0
    # padding, out-of-range ids and a repeat in the first row
    idx = _rows(M, 6, lambda m: [-1, 99, 0, 0, -5, 1])
    assert records_ref(idx, N, bs)[0, 0, 2].tolist() == [1, 0] + [-1] * 6
    # ids past N: nblk = ceil(N / bs) bounds them
    assert records_ref(idx, 40, bs)[0, 0, 2].tolist() == [1, 0] + [-1] * 6
    # a block whose keys run past N is not recorded (queries past N, M > N)
    idx = _rows(80, 2, lambda m: [0, 1])
    assert records_ref(idx, 160, bs)[0, 0, 4].tolist() == [2, 0, 1] + [-1] * 5
    assert records_ref(idx, 40, bs)[0, 0, 4].tolist() == [1, 0] + [-1] * 6


def test_records_cap():
    bs, M = 32, 512
    idx = gen.dense_causal_indices(1, M, 1, M // bs, bs)
    rec = records_ref(idx, M, bs)[0, 0]
    assert rec[:, 0].max() == MAXREC
    last = rec[-1]  # m0 = 496: blocks 0..15 qualify; the first 7 in row order
    assert last.tolist() == [MAXREC] + list(range(MAXREC))


def _restrict(idx, keep):
    """idx with every entry outside ``keep`` (a per-row boolean) made padding."""
    return np.where(keep, idx, -1).astype(np.int32)


@pytest.mark.parametrize("bs,rule,T", [(64, "first_two_local", 6), (32, "first_two_local", 5),
                                       (32, "all_causal", 0)])
def test_partial_state_continued_equals_the_oracle(bs, rule, T):
    M = N = 300
    if rule == "all_causal":
        T = -(-M // bs)
    w = gen.Workload("two_pass_host", 1, M, N, 16, 2, 128, bs, T, 1.0, rule)
    q, k, v = gen.make_qkv(w, 7 + bs)
    idx = gen.make_block_indices(w, 7 + bs)
    rec = records_ref(idx, N, bs)  # [B, G, tiles, 8]
    # per row: is the entry one of its tile's recorded blocks?
    tiles = np.arange(M) // 16
    shared = np.zeros(idx.shape, bool)
    for g in range(w.G):
        r = rec[0, g, tiles]  # [M, 8]
        ids = np.where(np.arange(7)[None, :] < r[:, :1], r[:, 1:], -2)  # -2 matches nothing
        shared[0, :, g] = (idx[0, :, g, :, None] == ids[:, None, :]).any(-1) & (idx[0, :, g] >= 0)
    assert shared.any()
    O, L = oracle.sel_attn_fwd(q, k, v, idx, bs)
    OA, LA = oracle.sel_attn_fwd(q, k, v, _restrict(idx, shared), bs)
    OB, LB = oracle.sel_attn_fwd(q, k, v, _restrict(idx, ~shared), bs)
    # continue from (OA, 1, LA) over the remaining keys: with weights relative
    # to LA, the rest adds exp(LB - LA) of row sum and exp(LB - LA) * OB of O
    with np.errstate(invalid="ignore", over="ignore"):
        wB = np.where(np.isneginf(LA), 1.0, np.exp(LB - np.where(np.isneginf(LA), 0.0, LA)))
        wA = np.where(np.isneginf(LA), 0.0, 1.0)
    wB = np.where(np.isneginf(LB), 0.0, wB)
    den = wA + wB  # [B, H, M]
    Om = (wA[..., None] * OA.transpose(0, 2, 1, 3) + wB[..., None] * OB.transpose(0, 2, 1, 3))
    Om = (Om / den[..., None]).transpose(0, 2, 1, 3)
    Lm = np.where(np.isneginf(LA), LB, LA + np.log(den))
    assert np.abs(Om - O).max() < 1e-12
    assert np.abs(Lm - L).max() < 1e-12
