"""nsa_sel_attn_fwd_strided: Q, K, V as views into one fused projection and
O as a slice of a larger buffer give the contiguous call's results bit for
bit (same kernel arithmetic, other addresses), and the oracle's."""

import numpy as np
import pytest

from _parity import check_rows, poisoned, sample_rows

pytestmark = pytest.mark.gpu


def _fused(B, M, H, G, D, bs, T, seed, dtype):
    import torch

    from nsa_block_selection_gb300 import inputs as gen

    w = gen.Workload("fused", B, M, M, H, G, D, bs, T, 1.0, "first_two_local")
    q, k, v = gen.make_qkv(w, seed, "bf16" if dtype == torch.bfloat16 else "f16")
    idx = gen.make_block_indices(w, seed)
    qkv = torch.empty((B, M, H + 2 * G, D), dtype=dtype, device="cuda")
    qkv[:, :, :H] = torch.from_numpy(np.asarray(q)).cuda().to(dtype)
    qkv[:, :, H:H + G] = torch.from_numpy(np.asarray(k)).cuda().to(dtype)
    qkv[:, :, H + G:] = torch.from_numpy(np.asarray(v)).cuda().to(dtype)
    return w, q, k, v, idx, qkv


@pytest.mark.parametrize("dtype_name,out_name", [("f16", "f32"), ("bf16", "f32"),
                                                 ("bf16", "bf16"), ("f16", "f16")])
@pytest.mark.parametrize("D", [64, 128])
def test_fused_qkv_views_and_sliced_out(dtype_name, out_name, D):
    import torch

    from nsa_block_selection_gb300 import sel_attn_fwd

    dt = {"f16": torch.float16, "bf16": torch.bfloat16}[dtype_name]
    ot = torch.float32 if out_name == "f32" else dt
    B, M, H, G = 2, 900, 16, 2
    w, q, k, v, idx, qkv = _fused(B, M, H, G, D, 64, 6, 3 + D, dt)
    tq, tk, tv = qkv[:, :, :H], qkv[:, :, H:H + G], qkv[:, :, H + G:]
    assert not tq.is_contiguous() and not tk.is_contiguous()
    ti = torch.from_numpy(idx).cuda()
    big = torch.full((B, M, H + 8, D), 7.0, dtype=ot, device="cuda")
    out = big[:, :, 3:3 + H]
    out.fill_(float("nan"))  # the kernel must overwrite every element of the slice
    O, L = sel_attn_fwd(tq, tk, tv, ti, 64, out=out, lse=poisoned((B, H, M), torch.float32))
    Oc, Lc = sel_attn_fwd(tq.contiguous(), tk.contiguous(), tv.contiguous(), ti, 64,
                          out=poisoned((B, M, H, D), ot), lse=poisoned((B, H, M), torch.float32))
    torch.cuda.synchronize()
    assert O.data_ptr() == out.data_ptr()
    assert torch.equal(O, Oc) and torch.equal(L, Lc)
    # the rest of the buffer is untouched
    assert (big[:, :, :3] == 7.0).all() and (big[:, :, 3 + H:] == 7.0).all()
    if dtype_name == "f16" and out_name == "f32":
        rows = sample_rows(B, M, G, 64, 2, n_random=256)
        check_rows(q, k, v, idx, 64, O, L, rows, what="fused views")


def test_strided_misaligned_view_is_rejected():
    import torch

    from nsa_block_selection_gb300 import NsaError, sel_attn_fwd

    qkv = torch.zeros((1, 64, 20, 132), dtype=torch.float16, device="cuda")
    q = qkv[:, :, :16, :128]  # strides (20*132, 132, 1): 132 is not a multiple of 8
    k = qkv[:, :, 16:18, :128]
    v = qkv[:, :, 18:20, :128]
    idx = torch.zeros((1, 64, 2, 1), dtype=torch.int32, device="cuda")
    with pytest.raises(NsaError):
        sel_attn_fwd(q, k, v, idx, 64)
