"""nsa_swa_fwd (tcgen05 sliding-window / dense GQA attention) against the
CPU oracle.

The oracle computes in float64 from the same 16-bit inputs. Tolerance: the
forward's 2e-3 + 2e-3 |O*| plus the two roundings the kernel adds, each
bounded through the unit roundoff u of the input type (fp16 2^-11, bf16
2^-8): P rounded before the PV product moves O by at most u * sum_n p_n |V[n]|
(the oracle's O for |V|), and the 16-bit O by at most u |O*|. LSE within
1e-3; a row without keys gives O = 0 and LSE = -inf exactly.
"""

import numpy as np
import pytest

import oracle.swa as W
from _parity import compare, poisoned

pytestmark = pytest.mark.gpu

U = {"f16": 2.0 ** -11, "bf16": 2.0 ** -8}


def _inputs(B, M, N, H, Hkv, D, dtype, seed, sigma=1.0):
    from nsa_block_selection_gb300 import inputs as gen

    w = gen.Workload("swa", B, M, N, H, Hkv, D, 64, 1, sigma, "local")
    return gen.make_qkv(w, seed, dtype)


def _run(q, k, v, window, dtype, scale=None, lse=True):
    import torch

    from nsa_block_selection_gb300 import swa_fwd

    dt = torch.bfloat16 if dtype == "bf16" else torch.float16
    t = [torch.from_numpy(x).cuda().to(dt) for x in (q, k, v)]
    B, M, H, D = t[0].shape
    O, L = swa_fwd(*t, window=window, scale=scale, return_lse=lse, out=poisoned((B, M, H, D), dt),
                   lse=poisoned((B, H, M), torch.float32) if lse else None)
    torch.cuda.synchronize()
    assert O.dtype == dt
    return O, L


def _check(q, k, v, window, dtype, O, L, rows, scale=None, what=""):
    import torch

    H, Hkv = q.shape[2], k.shape[2]
    hpg = H // Hkv
    r = torch.as_tensor(np.asarray(rows, np.int64).reshape(-1, 3), device=O.device)
    b, i, g = r[:, 0:1], r[:, 1:2], r[:, 2:3]
    hs = g * hpg + torch.arange(hpg, device=O.device)[None, :]
    o = O[b, i, hs].float().cpu().numpy().astype(np.float64)
    l = L[b, hs, i].cpu().numpy().astype(np.float64)
    o_ref, l_ref = W.swa_rows(q, k, v, rows, window[0], window[1], scale)
    a_ref, _ = W.swa_rows(q, k, np.abs(v), rows, window[0], window[1], scale)
    u = U[dtype]
    return compare(o, l, o_ref, l_ref, what, extra=u * a_ref + u * np.abs(o_ref))


def _all_rows(B, M, Hkv):
    return [(b, i, g) for b in range(B) for i in range(M) for g in range(Hkv)]


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("dtype", ["bf16", "f16"])
@pytest.mark.parametrize("window", [(-1, -1), (-1, 0), (100, 0), (0, 0), (37, 53), (300, -1)])
def test_swa_every_row(D, dtype, window):
    B, M, N, H, Hkv = 2, 700, 700, 8, 2
    q, k, v = _inputs(B, M, N, H, Hkv, D, dtype, 40 + D)
    O, L = _run(q, k, v, window, dtype)
    _check(q, k, v, window, dtype, O, L, _all_rows(B, M, Hkv), what=f"{window}")


@pytest.mark.parametrize("M,N", [(300, 520), (520, 300), (130, 1000)])
@pytest.mark.parametrize("window", [(64, 0), (-1, 0), (10, 200)])
def test_swa_queries_and_keys_differ(M, N, window):
    q, k, v = _inputs(1, M, N, 4, 1, 128, "bf16", 7)
    O, L = _run(q, k, v, window, "bf16")
    _check(q, k, v, window, "bf16", O, L, _all_rows(1, M, 1), what=f"{M}x{N} {window}")


@pytest.mark.parametrize("H,Hkv", [(4, 4), (6, 2), (16, 1)])
def test_swa_head_groups_and_scale(H, Hkv):
    q, k, v = _inputs(1, 260, 260, H, Hkv, 64, "bf16", 8, sigma=1.5)
    O, L = _run(q, k, v, (90, 10), "bf16", scale=0.2)
    _check(q, k, v, (90, 10), "bf16", O, L, _all_rows(1, 260, Hkv), scale=0.2)


def test_swa_no_keys_and_no_lse():
    import torch

    from nsa_block_selection_gb300 import swa_fwd

    q = torch.randn(1, 200, 4, 64, device="cuda").bfloat16()
    k = torch.zeros(1, 0, 2, 64, device="cuda").bfloat16()
    O, L = swa_fwd(q, k, k, window=(-1, 0), out=poisoned(q.shape, q.dtype),
                   lse=poisoned((1, 4, 200), torch.float32))
    torch.cuda.synchronize()
    assert (O == 0).all() and torch.isneginf(L).all()
    # queries past the last key, window (5, 5): rows 306.. see nothing
    qq, kk, vv = _inputs(1, 400, 300, 4, 2, 64, "bf16", 9)
    O, L = _run(qq, kk, vv, (5, 5), "bf16")
    _check(qq, kk, vv, (5, 5), "bf16", O, L, _all_rows(1, 400, 2))
    O2, L2 = _run(qq, kk, vv, (5, 5), "bf16", lse=False)
    assert L2 is None and torch.equal(O, O2)


def test_swa_deterministic():
    import torch

    q, k, v = _inputs(1, 1000, 1000, 8, 2, 128, "bf16", 10)
    a = _run(q, k, v, (256, 0), "bf16")
    b = _run(q, k, v, (256, 0), "bf16")
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])


@pytest.mark.parametrize("window", [(1024, 0), (-1, 0)])
def test_swa_large_sampled(window):
    """M = N = 8192, H = 64, H_kv = 8, D = 128: sampled rows, plus the sync
    status (no timed-out wait)."""
    from nsa_block_selection_gb300 import _lib

    M = 8192
    q, k, v = _inputs(1, M, M, 64, 8, 128, "bf16", 11)
    O, L = _run(q, k, v, window, "bf16")
    import torch

    assert _lib.sync_status(torch.cuda.current_stream()) == 0
    rng = np.random.default_rng(1)
    ms = np.concatenate([rng.integers(0, M, 200), [0, 1, 127, 128, 1023, 1024, M - 1]])
    rows = sorted({(0, int(m), int(rng.integers(8))) for m in ms})
    _check(q, k, v, window, "bf16", O, L, rows, what=f"8k {window}")


@pytest.mark.parametrize("D", [64, 128])
def test_swa_output_alignment(D):
    """The head-pair kernel stores O rows with 32-byte stores when O is
    32-byte aligned and 16-byte stores otherwise: an O that starts 16 bytes
    into an allocation gives the same bits."""
    import torch

    from nsa_block_selection_gb300 import swa_fwd

    q, k, v = _inputs(1, 700, 700, 8, 2, D, "bf16", 12)
    t = [torch.from_numpy(x).cuda().to(torch.bfloat16) for x in (q, k, v)]
    shape = tuple(t[0].shape)
    n = t[0].numel()
    flat = torch.full((n + 8,), float("nan"), dtype=torch.bfloat16, device="cuda")
    o16 = flat[8:].view(shape)  # 16-byte aligned, not 32
    assert o16.data_ptr() % 32 == 16
    O16, L16 = swa_fwd(*t, window=(600, 0), out=o16)
    O32, L32 = swa_fwd(*t, window=(600, 0), out=poisoned(shape, torch.bfloat16))
    torch.cuda.synchronize()
    assert torch.equal(O16, O32) and torch.equal(L16, L32)
    _check(q, k, v, (600, 0), "bf16", O32, L32, _all_rows(1, 700, 2))
