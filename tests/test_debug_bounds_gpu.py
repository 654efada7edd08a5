"""The NSA_DEBUG_BOUNDS build: the selection forward's kernels check every
K/V tile they copy (16-key boundary, at or before the query's last visible
key, inside a block of the index range) and report a failed check through
nsa_sync_status as NSA_ERR_BOUNDS. A stand-in for a memory checker on a pool
where none runs: the library is built a second time with the checks, the
problems below (padding anywhere, ids out of range, blocks wholly after the
query, ragged sizes, both entry points) must pass every check, and the
outputs must equal the normal build's bit for bit (the checks change no
arithmetic).
"""

import ctypes
import os

import numpy as np
import pytest

from _parity import poisoned, small_inputs, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def debug_lib():
    from nsa_block_selection_gb300 import _lib
    from nsa_block_selection_gb300.build import LIB_DIR, build

    path = build(out=os.path.join(LIB_DIR, "libnsa_sel_attn_debug.so"),
                 defines=["NSA_DEBUG_BOUNDS"])
    return _lib.load(path)


def _fwd(lib, tq, tk, tv, ti, bs, shared_ws=None):
    import torch

    B, M, H, D = tq.shape
    N, G = tk.shape[1], tk.shape[2]
    T = ti.shape[-1]
    O = poisoned((B, M, H, D), torch.float32)
    L = poisoned((B, H, M), torch.float32)
    vp = ctypes.c_void_p
    st = vp(torch.cuda.current_stream().cuda_stream)
    ptrs = [vp(t.data_ptr() if t.numel() else 0) for t in (tq, tk, tv, ti, O, L)]
    if shared_ws is None:
        rc = lib.nsa_sel_attn_fwd(*ptrs, B, M, N, H, G, D, T, bs, ctypes.c_float(0.0), st)
    else:
        rc = lib.nsa_sel_attn_fwd_shared(*ptrs, B, M, N, H, G, D, T, bs, ctypes.c_float(0.0), 0,
                                         vp(shared_ws.data_ptr()), shared_ws.numel(), st)
    assert rc == 0
    return O, L, lib.nsa_sync_status(st)


@pytest.mark.parametrize("case", ["padding", "ragged_bs32_d64", "two_pass", "no_keys"])
def test_debug_build_passes_every_check_and_matches(debug_lib, case):
    import torch

    from nsa_block_selection_gb300 import _lib

    lib = _lib.load()
    ws = None
    if case == "padding":
        q, k, v, idx = small_inputs(2, 400, 400, 16, 2, 128, 64, 6, "first_two_local", seed=5)
        rng = np.random.default_rng(6)
        idx = rng.permuted(idx, axis=-1).copy()
        pads = idx < 0
        idx[pads] = rng.choice(np.array([-1, -7, 7, 1 << 30], np.int32), size=int(pads.sum()))
        idx[0, 10, 0, :] = -1
        idx[0, 10, 0, 3] = 6  # a block wholly after query 10: never copied
        bs = 64
    elif case == "ragged_bs32_d64":
        q, k, v, idx = small_inputs(1, 777, 700, 8, 1, 64, 32, 9, "first_local", seed=7)
        bs = 32
    elif case == "two_pass":
        q, k, v, idx = small_inputs(1, 1000, 1000, 16, 2, 128, 64, 6, "first_two_local", seed=8)
        bs = 64
        B, M, G = 1, 1000, 2
        ws = torch.zeros(_lib.shared_workspace_bytes(B, M, G) + 256, dtype=torch.uint8,
                         device="cuda")
    else:  # every row empty: T = 0
        q, k, v, _ = small_inputs(1, 128, 128, 8, 1, 128, 64, 2, "local", seed=9)
        idx = np.zeros((1, 128, 1, 0), np.int32)
        bs = 64
    tq, tk, tv, ti = to_dev(q, k, v, idx)
    O_d, L_d, st_d = _fwd(debug_lib, tq, tk, tv, ti, bs, ws)
    O_n, L_n, st_n = _fwd(lib, tq, tk, tv, ti, bs, None if ws is None else ws.clone())
    assert st_d == 0, f"debug build: {_lib.status_string(st_d)}"
    assert st_n == 0
    assert torch.equal(O_d, O_n) and torch.equal(L_d, L_n)
