"""The backward's no-allocation entry point (scratch in a fixed device array
inside the library), against the workspace entry point and the oracle.

Callers that may not allocate device memory (a plugin given no allocator by
its host application, a service that reserves all memory at start-up) use
nsa_sel_attn_bwd_noalloc. This file is collected last so that a run that
stops at its first failure has run every other test already; it also passes
alone in a fresh process.

Tolerance: the per-element bound of the backward parity tests, |GPU - exact|
<= 4 u |terms| (u = 2^-11, |terms| the oracle's per-element magnitude).
"""

import ctypes

import numpy as np
import pytest

import oracle.sel_attn as oracle
from _parity import small_inputs, to_dev

pytestmark = pytest.mark.gpu

U16 = 2.0 ** -11
KAPPA = 4


def _noalloc(lib, tq, tk, tv, ti, O, L, tdo, dq, dk, dv, bs, stream):
    B, M, H, D = tq.shape
    N, G = tk.shape[1], tk.shape[2]
    T = ti.shape[-1]
    vp = ctypes.c_void_p
    return lib.nsa_sel_attn_bwd_noalloc(
        vp(tq.data_ptr()), vp(tk.data_ptr()), vp(tv.data_ptr()), vp(ti.data_ptr()),
        vp(O.data_ptr()), vp(L.data_ptr()), vp(tdo.data_ptr()), vp(dq.data_ptr()),
        vp(dk.data_ptr()), vp(dv.data_ptr()), B, M, N, H, G, D, T, bs, ctypes.c_float(0.0),
        vp(stream.cuda_stream))


def _nan_outputs(O, tk):
    import torch

    dq = torch.full_like(O, float("nan"))
    dk = torch.full(tk.shape, float("nan"), dtype=torch.float32, device=tk.device)
    return dq, dk, torch.full_like(dk, float("nan"))


def _within(name, g, ex, mag, what):
    assert np.isfinite(g).all(), f"{what} {name}: non-finite"
    err = np.abs(g - ex)
    bound = KAPPA * U16 * mag
    assert np.all(err <= bound), \
        f"{what} {name}: {int((err > bound).sum())} elements beyond 4u|terms|"


def _problem(B, M, H, G, D, bs, T, rule, seed):
    q, k, v, idx = small_inputs(B, M, M, H, G, D, bs, T, rule, seed=seed)
    dO = np.random.default_rng(seed + 1).standard_normal(q.shape).astype(np.float32)
    exact = oracle.sel_attn_bwd(q, k, v, idx, dO, bs)
    mags = oracle.sel_attn_bwd(q, k, v, idx, dO, bs, magnitudes=True)
    return (q, k, v, idx, dO), exact, mags


def test_noalloc_backward_matches_workspace_entry():
    """Two shapes in a row through the one shared array: first D = 64,
    bs = 32 with more rows and a longer index row (the query-major dQ kernel
    writes the records there), then D = 128, bs = 64 twice. Each call must
    rebuild every part of the scratch it uses; outputs start as NaN."""
    import torch

    from nsa_block_selection_gb300 import _lib, sel_attn_fwd

    lib = _lib.load()
    stream = torch.cuda.current_stream()
    cases = [
        (dict(B=2, M=900, H=16, G=2, D=64, bs=32, T=8, rule="first_two_local", seed=61), 1),
        (dict(B=2, M=700, H=16, G=2, D=128, bs=64, T=5, rule="first_two_local", seed=77), 2),
    ]
    for spec, calls in cases:
        bs = spec["bs"]
        (q, k, v, idx, dO), exact, mags = _problem(**spec)
        tq, tk, tv, ti, tdo = to_dev(q, k, v, idx, dO)
        O, L = sel_attn_fwd(tq, tk, tv, ti, bs)
        ref = [g.cpu().numpy().astype(np.float64)
               for g in _lib.sel_attn_bwd(tq, tk, tv, ti, O, L, tdo, bs)]
        what = f"D{spec['D']} bs{bs}"
        for name, r, ex, mg in zip(("dQ", "dK", "dV"), ref, exact, mags):
            _within(name, r, ex, mg, what + " workspace entry")
        for call in range(calls):
            dq, dk, dv = _nan_outputs(O, tk)
            assert _noalloc(lib, tq, tk, tv, ti, O, L, tdo, dq, dk, dv, bs, stream) == 0
            torch.cuda.synchronize()
            got = [g.cpu().numpy().astype(np.float64) for g in (dq, dk, dv)]
            for name, g, r, ex, mg in zip(("dQ", "dK", "dV"), got, ref, exact, mags):
                _within(name, g, ex, mg, f"{what} no-alloc call {call}")
                # both entries run the same kernels; only the order of fp32
                # atomics differs between runs
                assert np.all(np.abs(g - r) <= 2 * KAPPA * U16 * mg), \
                    f"{what} {name}: no-alloc vs workspace entry"
    assert _lib.sync_status() == 0


def test_noalloc_rejects_problems_beyond_its_scratch():
    from nsa_block_selection_gb300 import _lib

    lib = _lib.load()
    fake = ctypes.c_void_p(4096)
    # m64k_bs64 with 2 batches: its fp16 dO copy alone is 2 GiB, far beyond
    # the fixed 64 MiB; rejected before anything is launched
    st = lib.nsa_sel_attn_bwd_noalloc(fake, fake, fake, fake, fake, fake, fake, fake, fake, fake,
                                      2, 65536, 65536, 64, 8, 128, 16, 64, ctypes.c_float(0.0),
                                      None)
    assert st == -10
    assert "scratch" in _lib.status_string(st)
    need = _lib.bwd_workspace_bytes(2, 65536, 65536, 64, 8, 128, 16, 64)
    assert need > 64 << 20


def test_noalloc_without_queries_needs_no_scratch():
    """M == 0: the call needs no scratch (the size limit is not applied);
    dK and dV are zeroed."""
    import torch

    from nsa_block_selection_gb300 import _lib

    lib = _lib.load()
    N = 4096
    dk = torch.full((1, N, 8, 64), float("nan"), device="cuda")
    dv = torch.full_like(dk, float("nan"))
    vp = ctypes.c_void_p
    st = lib.nsa_sel_attn_bwd_noalloc(None, vp(4096), vp(4096), None, None, None, None, None,
                                      vp(dk.data_ptr()), vp(dv.data_ptr()), 1, 0, N, 64, 8, 64,
                                      16, 64, ctypes.c_float(0.0),
                                      vp(torch.cuda.current_stream().cuda_stream))
    assert st == 0
    torch.cuda.synchronize()
    assert bool((dk == 0).all()) and bool((dv == 0).all())
