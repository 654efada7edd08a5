"""bf16 inputs and 16-bit O (nsa_sel_attn_fwd_ex) against the CPU oracle.

The oracle computes in float64 from the same (bf16- or fp16-valued) inputs.
Tolerance: the forward's 2e-3 + 2e-3 |O*|, plus the terms the variant's
rounding adds, each derived from the unit roundoff u of the type:
  * bf16 operands: P is rounded to bf16 (u = 2^-8) before PV while the row
    sums use the unrounded P, so O moves by at most u * sum_n p_n |V[n]| --
    exactly the oracle's O for |V| (pinned on the CPU by the bf16 emulation);
  * 16-bit O: the fp32 result rounded once, at most u |O| (fp16 2^-11,
    bf16 2^-8).
A 16-bit O must also equal the fp32 O of the same call rounded to nearest
even, bit for bit, and LSE must not depend on the O type.
"""

import numpy as np
import pytest

import oracle.sel_attn as oracle
from _parity import compare, gather_rows, poisoned, sample_rows

pytestmark = pytest.mark.gpu

U = {"f16": 2.0 ** -11, "bf16": 2.0 ** -8, "f32": 0.0}


def _torch_dtype(name):
    import torch

    return {"f16": torch.float16, "bf16": torch.bfloat16, "f32": torch.float32}[name]


def _run(w, seed, qkv, out, rows=None):
    import torch

    from nsa_block_selection_gb300 import inputs as gen
    from nsa_block_selection_gb300 import sel_attn_fwd

    q, k, v = gen.make_qkv(w, seed, qkv)
    idx = gen.make_block_indices(w, seed)
    dt = _torch_dtype(qkv)
    tq, tk, tv = (torch.from_numpy(x).cuda().to(dt) for x in (q, k, v))
    ti = torch.from_numpy(idx).cuda()
    shp, lshp = (w.B, w.M, w.H, w.D), (w.B, w.H, w.M)
    O, L = sel_attn_fwd(tq, tk, tv, ti, w.block_size, out=poisoned(shp, _torch_dtype(out)),
                        lse=poisoned(lshp, torch.float32))
    O32, L32 = sel_attn_fwd(tq, tk, tv, ti, w.block_size, out=poisoned(shp, torch.float32),
                            lse=poisoned(lshp, torch.float32))
    torch.cuda.synchronize()
    assert O.dtype == _torch_dtype(out) and O32.dtype == torch.float32
    assert torch.equal(L, L32), "LSE depends on the O type"
    if out != "f32":
        assert torch.equal(O, O32.to(O.dtype)), "16-bit O is not the rounded fp32 O"
    if rows is None:
        rows = [(b, m, g) for b in range(w.B) for m in range(w.M) for g in range(w.G)]
    o, l = gather_rows(O.float(), L, rows, w.heads_per_group)
    o_ref, l_ref = oracle.sel_attn_rows(q, k, v, idx, rows, w.block_size)
    extra = U[out] * np.abs(o_ref)
    if qkv == "bf16":
        a_ref, _ = oracle.sel_attn_rows(q, k, np.abs(v), idx, rows, w.block_size)
        extra = extra + U["bf16"] * a_ref
    return compare(o, l, o_ref, l_ref, f"{w.name} {qkv}->{out}", extra=extra)


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("bs", [32, 64])
@pytest.mark.parametrize("qkv,out", [("f16", "f16"), ("bf16", "f32"), ("bf16", "bf16")])
def test_dtype_variants_every_row(D, bs, qkv, out):
    from nsa_block_selection_gb300 import inputs as gen

    w = gen.Workload("ragged", 2, 700, 700, 16, 2, D, bs, 6, 1.0, "first_two_local")
    _run(w, 31 + D + bs, qkv, out)


@pytest.mark.parametrize("H,G", [(6, 2), (32, 2)])
def test_dtype_variants_head_layouts(H, G):
    from nsa_block_selection_gb300 import inputs as gen

    w = gen.Workload("heads", 1, 400, 400, H, G, 128, 64, 4, 1.5, "first_local")
    _run(w, 77, "bf16", "bf16")


@pytest.mark.parametrize("qkv,out", [("bf16", "f32"), ("f16", "f16")])
def test_dtype_variants_full_size_sampled(qkv, out):
    from nsa_block_selection_gb300 import inputs as gen

    w = gen.workload("m8k_bs64")
    rows = sample_rows(w.B, w.M, w.G, w.block_size, 5, n_random=1024)
    _run(w, gen.default_seed(w.name), qkv, out, rows)


@pytest.mark.parametrize("qkv,out", [("bf16", "f32"), ("bf16", "bf16"), ("f16", "f16")])
def test_host_entry_dtypes_match_device_entry(qkv, out):
    """The host-buffer entry point with bf16 inputs and / or a 16-bit O:
    bit-identical to the device entry point on the same inputs."""
    import torch

    from nsa_block_selection_gb300 import _lib
    from nsa_block_selection_gb300 import inputs as gen
    from nsa_block_selection_gb300 import sel_attn_fwd

    w = gen.Workload("host_dt", 2, 700, 700, 16, 2, 128, 64, 6, 1.0, "first_two_local")
    q, k, v = gen.make_qkv(w, 21, qkv)
    idx = gen.make_block_indices(w, 21)
    dt, ot = _torch_dtype(qkv), _torch_dtype(out)
    hq, hk, hv = (torch.from_numpy(x).to(dt).pin_memory() for x in (q, k, v))
    hi = torch.from_numpy(idx).pin_memory()
    ho = torch.full((w.B, w.M, w.H, w.D), float("nan"), dtype=ot).pin_memory()
    hl = torch.full((w.B, w.H, w.M), float("nan"), dtype=torch.float32).pin_memory()
    O_h, L_h = _lib.sel_attn_fwd_host(hq, hk, hv, hi, w.block_size, out=ho, lse=hl, chunk_m=128)
    O_d, L_d = sel_attn_fwd(*(t.cuda() for t in (hq, hk, hv, hi)), w.block_size,
                            out=poisoned((w.B, w.M, w.H, w.D), ot),
                            lse=poisoned((w.B, w.H, w.M), torch.float32))
    torch.cuda.synchronize()
    assert O_h.dtype == ot
    assert torch.equal(O_h, O_d.cpu()) and torch.equal(L_h, L_d.cpu())
