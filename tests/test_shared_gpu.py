"""The two-pass forward (nsa_sel_attn_fwd_shared) against the CPU oracle.

Per tile of 16 queries the list pass records the blocks every query of the
tile lists whose first key the tile's first query sees and whose keys all
lie below M and N; the tile-shared pass attends to them on the tcgen05
tensor cores (masking the keys after each row's query in the block the
tile sits in), and the gather kernel continues from that state. The
records are integer work and are compared exactly with a restatement of
their definition here; O and LSE are compared with the oracle under the
forward's tolerance (bf16 inputs add the bf16 rounding term of P, as in the
dtype tests).
"""

import numpy as np
import pytest

import oracle.sel_attn as oracle
from _parity import (check_all_rows, check_rows, compare, gather_rows, poisoned, run_cuda,
                     sample_rows, to_dev)
from _records import MAXREC, TILE, records_ref

pytestmark = pytest.mark.gpu

@pytest.fixture(scope="module", autouse=True)
def _need_gpu(cuda_lib):
    import torch

    assert torch.cuda.is_available(), "GPU tests need a CUDA device"


def run_shared(q, k, v, idx, bs, dtype=None, scale=None):
    import torch

    from nsa_block_selection_gb300 import _lib

    tq, tk, tv, ti = to_dev(q, k, v, idx)
    if dtype is not None:
        tq, tk, tv = tq.to(dtype), tk.to(dtype), tv.to(dtype)
    B, M, H, D = q.shape
    G = k.shape[2]
    ws = torch.zeros(_lib.shared_workspace_bytes(B, M, G) + 256, dtype=torch.uint8,
                     device="cuda")
    O, L = _lib.sel_attn_fwd_shared(tq, tk, tv, ti, bs, scale, workspace=ws,
                                    out=poisoned((B, M, H, D), torch.float32),
                                    lse=poisoned((B, H, M), torch.float32))
    torch.cuda.synchronize()
    assert _lib.sync_status() == 0
    ntiles = -(-M // TILE)
    rec = ws[:B * G * ntiles * 32].view(torch.int32).reshape(B, G, ntiles, 8).cpu().numpy()
    return O, L, rec, ws


def _inputs(B, M, N, H, G, D, bs, T, rule, seed):
    from nsa_block_selection_gb300 import inputs as gen

    w = gen.Workload("two_pass", B, M, N, H, G, D, bs, T, 1.0, rule)
    q, k, v = gen.make_qkv(w, seed)
    idx = gen.make_block_indices(w, seed)
    return q, k, v, idx


@pytest.mark.parametrize("rule,T", [("first_two_local", 6), ("first_local", 4),
                                    ("all_causal", 0)])
def test_records_and_every_row(rule, T):
    """Ragged M (a partial last tile), B = 2, G = 2; the records are exact."""
    bs = 64
    M = N = 1000
    if rule == "all_causal":
        T = -(-M // bs)
    q, k, v, idx = _inputs(2, M, N, 16, 2, 128, bs, T, rule, seed=bs + T)
    O, L, rec, _ = run_shared(q, k, v, idx, bs)
    ref = records_ref(idx, N, bs)
    assert np.array_equal(rec, ref)
    assert (ref[..., 0] > 0).mean() > 0.8  # the path is exercised
    check_all_rows(q, k, v, idx, bs, O, L, what=f"two-pass bs{bs} {rule}")


def test_bf16_every_row():
    import torch

    bs = 64
    q, k, v, idx = _inputs(1, 700, 700, 16, 2, 128, bs, 6, "first_two_local", seed=5)
    O, L, rec, _ = run_shared(q, k, v, idx, bs, dtype=torch.bfloat16)
    qb, kb, vb = (torch.from_numpy(x).to(torch.bfloat16).float().numpy().astype(np.float64)
                  for x in (q, k, v))
    rows = [(0, m, g) for m in range(700) for g in range(2)]
    o, l = gather_rows(O, L, rows, 8)
    o_ref, l_ref = oracle.sel_attn_rows(qb, kb, vb, idx, rows, bs)
    a_ref, _ = oracle.sel_attn_rows(qb, kb, np.abs(vb), idx, rows, bs)
    compare(o, l, o_ref, l_ref, "two-pass bf16", extra=2.0 ** -8 * a_ref)
    assert np.array_equal(rec, records_ref(idx, 700, bs))


def test_permuted_rows_and_padding_anywhere():
    """Rows in any order with -1 and out-of-range ids mixed in: the records
    follow the first query's order and skip padding."""
    bs = 64
    M = N = 777
    q, k, v, idx = _inputs(1, M, N, 16, 2, 128, bs, 8, "first_two_local", seed=9)
    rng = np.random.default_rng(3)
    idx = rng.permuted(idx, axis=-1).copy()
    pad = rng.random(idx.shape) < 0.15
    idx[pad] = -1
    idx[rng.random(idx.shape) < 0.05] = 10 ** 6
    idx = idx.astype(np.int32)
    O, L, rec, _ = run_shared(q, k, v, idx, bs)
    assert np.array_equal(rec, records_ref(idx, N, bs))
    check_all_rows(q, k, v, idx, bs, O, L, what="two-pass permuted")


def test_more_common_blocks_than_a_record_holds():
    """Every causal block listed (dense rows, T up to 64): only the first 7
    common blocks are recorded; the gather kernel takes the rest."""
    from nsa_block_selection_gb300 import inputs as gen

    bs, M = 64, 2047
    q, k, v, _ = _inputs(1, M, M, 8, 1, 128, bs, 1, "local", seed=M)
    idx = gen.dense_causal_indices(1, M, 1, -(-M // bs), bs)  # 32 blocks per row
    O, L, rec, _ = run_shared(q, k, v, idx, bs)
    ref = records_ref(idx, M, bs)
    assert np.array_equal(rec, ref) and ref[..., 0].max() == MAXREC
    check_all_rows(q, k, v, idx, bs, O, L, what="two-pass dense")


def test_no_common_block():
    """Random rows without forced blocks: most tiles record nothing and the
    gather kernel does all the work, from the empty state."""
    bs, M = 64, 512
    q, k, v, _ = _inputs(1, M, M, 8, 1, 128, bs, 1, "local", seed=21)
    rng = np.random.default_rng(21)
    nb = M // bs
    idx = np.stack([rng.permutation(nb)[:3] for _ in range(M)]).astype(np.int32)
    idx = idx.reshape(1, M, 1, 3)
    O, L, rec, _ = run_shared(q, k, v, idx, bs)
    ref = records_ref(idx, M, bs)
    assert np.array_equal(rec, ref)
    check_all_rows(q, k, v, idx, bs, O, L, what="two-pass no common block")


@pytest.mark.parametrize("M", [384, 376])
def test_unselected_and_future_rows_may_hold_nan(M):
    """As for the one-pass call: rows past every query and blocks no row
    lists never reach the output (M = 376: poisoned rows inside the last
    tile's own block, past its last query)."""
    import torch

    bs = 64
    N = 640
    q, k, v, idx = _inputs(1, M, N, 16, 2, 128, bs, 6, "first_two_local", seed=10)
    used = np.zeros(-(-N // bs), bool)
    used[idx[idx >= 0]] = True
    O1, L1, _, _ = run_shared(q, k, v, idx, bs)
    k2, v2 = k.copy(), v.copy()
    k2[:, M:] = np.float16(np.nan)
    v2[:, M:] = np.float16(np.inf)
    for t in np.nonzero(~used)[0]:
        k2[:, t * bs:(t + 1) * bs] = np.float16(-np.inf)
        v2[:, t * bs:(t + 1) * bs] = np.float16(np.nan)
    O2, L2, _, _ = run_shared(q, k2, v2, idx, bs)
    assert torch.equal(O1, O2) and torch.equal(L1, L2)
    assert torch.isfinite(O2).all()


def test_keys_past_a_tiles_last_query_never_reach_it():
    """The tile-shared pass takes the block its queries sit in, masked per
    row; the keys of that block past the tile's last query enter no product
    of the tile. K/V rows 80..127 poisoned: the rows of queries 0..79 are
    bit-identical to the clean run (queries 80.. see those keys and are not
    compared)."""
    import torch

    bs, M = 64, 512
    q, k, v, idx = _inputs(1, M, M, 16, 2, 128, bs, 6, "first_two_local", seed=12)
    O1, L1, rec, _ = run_shared(q, k, v, idx, bs)
    assert (rec[0, :, 64 // TILE, 1:4] == 1).any(-1).all()  # tile of queries 64..79 shares block 1
    k2, v2 = k.copy(), v.copy()
    k2[:, 80:128] = np.float16(np.nan)
    v2[:, 80:128] = np.float16(np.nan)
    O2, L2, _, _ = run_shared(q, k2, v2, idx, bs)
    assert torch.equal(O1[:, :80], O2[:, :80]) and torch.equal(L1[:, :, :80], L2[:, :, :80])


@pytest.mark.parametrize("H,G,D,M,bs", [(8, 2, 128, 300, 64), (16, 2, 64, 300, 64),
                                        (16, 2, 128, 13, 64), (16, 2, 128, 700, 32)])
def test_other_shapes_take_the_one_pass_kernel(H, G, D, M, bs):
    """4 heads per group, D = 64, fewer than 16 queries, or 32-key blocks:
    the one-pass kernel runs (bit-identical to nsa_sel_attn_fwd) and the
    records stay untouched."""
    import torch

    q, k, v, idx = _inputs(1, M, M, H, G, D, bs, 4, "first_two_local", seed=H + D + M)
    O, L, _, ws = run_shared(q, k, v, idx, bs)
    assert int(ws.count_nonzero()) == 0
    O1, L1 = run_cuda(q, k, v, idx, bs)
    assert torch.equal(O, O1) and torch.equal(L, L1)


def test_close_to_one_pass():

    bs = 64
    q, k, v, idx = _inputs(1, 2048, 2048, 16, 2, 128, bs, 16, "first_two_local", seed=2)
    O, L, _, _ = run_shared(q, k, v, idx, bs)
    O1, L1 = run_cuda(q, k, v, idx, bs)
    assert float((O - O1).abs().max()) < 1e-3
    assert float((L - L1).abs().max()) < 1e-4


@pytest.mark.parametrize("name", ["m64k_bs64", "m32k_bs32"])
def test_full_size_sampled(name):
    import torch

    from nsa_block_selection_gb300 import _lib
    from nsa_block_selection_gb300 import inputs as gen

    w = gen.workload(name)
    q, k, v, idx = gen.make_inputs(w)
    tq, tk, tv, ti = to_dev(q, k, v, idx)
    O, L = _lib.sel_attn_fwd_shared(tq, tk, tv, ti, w.block_size,
                                    out=poisoned((w.B, w.M, w.H, w.D), torch.float32),
                                    lse=poisoned((w.B, w.H, w.M), torch.float32))
    torch.cuda.synchronize()
    assert _lib.sync_status() == 0
    assert bool(torch.isfinite(L).all()) and bool(torch.isfinite(O).all())
    rows = sample_rows(w.B, w.M, w.G, w.block_size, seed=gen.default_seed(name))
    ratio, lerr = check_rows(q, k, v, idx, w.block_size, O, L, rows, what=name)
    print(f"two-pass {name}: {len(rows)} rows, O err {ratio:.3f} x tol, LSE err {lerr:.2e}")
