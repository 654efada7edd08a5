"""The backward's no-allocation entry point (scratch in a fixed device array
inside the library), against the workspace entry point.

Callers that may not allocate device memory (a plugin given no allocator by
its host application, a service that reserves all memory at start-up) use
nsa_sel_attn_bwd_noalloc. This file is collected last so that a run that
stops at its first failure has run every other test already; it also passes
alone in a fresh process.
"""

import ctypes

import numpy as np
import pytest

import oracle.sel_attn as oracle
from _parity import small_inputs, to_dev

pytestmark = pytest.mark.gpu


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


def test_noalloc_backward_matches_workspace_entry():
    import torch

    from nsa_block_selection_gb300 import _lib, sel_attn_fwd

    lib = _lib.load()
    bs = 64
    q, k, v, idx = small_inputs(2, 700, 700, 16, 2, 128, bs, 5, "first_two_local", seed=77)
    dO = np.random.default_rng(78).standard_normal(q.shape).astype(np.float32)
    tq, tk, tv, ti, tdo = to_dev(q, k, v, idx, dO)
    O, L = sel_attn_fwd(tq, tk, tv, ti, bs)
    ref = [g.cpu().numpy().astype(np.float64)
           for g in _lib.sel_attn_bwd(tq, tk, tv, ti, O, L, tdo, bs)]
    # tolerance of the backward parity tests: 4x the fp16-operand error + 1e-5 max
    exact = oracle.sel_attn_bwd(q, k, v, idx, dO, bs)
    emul = oracle.sel_attn_bwd(q, k, v, idx, dO, bs, emulate_kernel_rounding=True)
    tol = [4 * np.abs(em - ex).max() + 1e-5 * np.abs(ex).max() for em, ex in zip(emul, exact)]
    stream = torch.cuda.current_stream()
    for call in range(2):  # the second call finds the first call's scratch
        dq = torch.full_like(O, float("nan"))
        dk = torch.full(tk.shape, float("nan"), dtype=torch.float32, device=tk.device)
        dv = torch.full_like(dk, float("nan"))
        assert _noalloc(lib, tq, tk, tv, ti, O, L, tdo, dq, dk, dv, bs, stream) == 0
        torch.cuda.synchronize()
        got = [g.cpu().numpy().astype(np.float64) for g in (dq, dk, dv)]
        for name, g, r, ex, t in zip(("dQ", "dK", "dV"), got, ref, exact, tol):
            assert np.isfinite(g).all(), f"call {call} {name}: non-finite"
            assert np.abs(g - r).max() <= t, f"call {call} {name} vs workspace entry"
            assert np.abs(g - ex).max() <= t, f"call {call} {name} vs oracle"
    assert _lib.sync_status() == 0


def test_noalloc_rejects_problems_beyond_its_scratch():
    from nsa_block_selection_gb300 import _lib

    lib = _lib.load()
    fake = ctypes.c_void_p(4096)
    # m64k_bs64 x 2 batches: ~100 MB of scratch > 64 MiB; nothing is launched
    st = lib.nsa_sel_attn_bwd_noalloc(fake, fake, fake, fake, fake, fake, fake, fake, fake, fake,
                                      2, 65536, 65536, 64, 8, 128, 16, 64, ctypes.c_float(0.0),
                                      None)
    assert st == -10
    assert "scratch" in _lib.status_string(st)
