"""Host-side checks of the C ABI (no GPU): the library loads, exports every
function the headers declare, and rejects bad arguments before touching
CUDA."""

import ctypes
import glob
import os
import re

import pytest

from nsa_block_selection_gb300 import _lib
from nsa_block_selection_gb300.build import INCLUDE

# Sizes of a valid call: B, M, N, H, G, D, T, block_size
GOOD = dict(B=1, M=128, N=128, H=16, G=2, D=128, T=4, bs=64)
FAKE = 4096  # a 16-byte aligned non-null address that is never dereferenced


def declared_functions():
    names = set()
    for h in glob.glob(os.path.join(INCLUDE, "*.h")):
        text = open(h).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        for m in re.finditer(r"^[A-Za-z_][\w \*]*?\b(nsa_\w+)\s*\(", text, flags=re.M):
            names.add(m.group(1))
    return sorted(names)


@pytest.fixture(scope="module")
def lib():
    path = _lib.LIB_PATH
    if not os.path.exists(path):
        from nsa_block_selection_gb300.build import build

        build()
    return _lib.load()


def call(lib, q=FAKE, k=FAKE, v=FAKE, idx=FAKE, o=FAKE, lse=FAKE, scale=0.0, **over):
    a = dict(GOOD)
    a.update(over)
    vp = ctypes.c_void_p
    return lib.nsa_sel_attn_fwd(vp(q), vp(k), vp(v), vp(idx), vp(o), vp(lse), a["B"], a["M"],
                                a["N"], a["H"], a["G"], a["D"], a["T"], a["bs"], scale, None)


def test_exports_match_header(lib):
    names = declared_functions()
    assert set(names) >= {"nsa_sel_attn_fwd", "nsa_status_string", "nsa_version"}
    for n in names:
        assert hasattr(lib, n), f"{n} declared in include/ but not exported"
    assert set(_lib.EXPORTS) <= set(names)


def test_status_strings(lib):
    for code in range(0, -13, -1):
        s = lib.nsa_status_string(code).decode()
        assert s and s != "unknown status"
    assert lib.nsa_status_string(-99).decode() == "unknown status"
    assert lib.nsa_version() >= 100


@pytest.mark.parametrize("over,status", [
    (dict(B=-1), -2), (dict(M=-3), -2), (dict(N=-1), -2), (dict(T=-1), -2),
    (dict(H=0), -2), (dict(G=0), -2), (dict(D=0), -2),
    (dict(H=24, G=2), -5), (dict(H=20, G=2), -5), (dict(H=15, G=2), -5),
    (dict(D=96), -4), (dict(D=256), -4),
    (dict(bs=16), -3), (dict(bs=128), -3), (dict(bs=0), -3),
    (dict(M=1 << 31), -2), (dict(N=1 << 40), -2),
])
def test_bad_sizes(lib, over, status):
    assert call(lib, **over) == status


@pytest.mark.parametrize("which", ["q", "k", "v", "idx", "o", "lse"])
def test_null_pointers(lib, which):
    assert call(lib, **{which: None}) == -1


@pytest.mark.parametrize("which,addr", [("q", FAKE + 8), ("k", FAKE + 2), ("v", FAKE + 4),
                                        ("o", FAKE + 4), ("lse", FAKE + 2), ("idx", FAKE + 1)])
def test_misaligned(lib, which, addr):
    assert call(lib, **{which: addr}) == -6


@pytest.mark.parametrize("over", [dict(B=0), dict(M=0), dict(B=0, M=0)])
def test_empty_problem_is_a_no_op(lib, over):
    # returns before any CUDA call, so it runs without a GPU; pointers unused
    assert call(lib, q=None, k=None, v=None, idx=None, o=None, lse=None, **over) == 0


def test_host_workspace_bytes(lib):
    f = lib.nsa_sel_attn_fwd_host_workspace_bytes
    n = f(1, 65536, 65536, 64, 8, 128, 16, 64, 8192)
    kv = 2 * 65536 * 8 * 128 * 2
    per_slot = 8192 * 64 * 128 * 2 + 8192 * 8 * 16 * 4 + 8192 * 64 * 128 * 4 + 64 * 8192 * 4
    assert n == kv + 2 * per_slot
    per_slot2 = 2048 * 64 * 128 * 2 + 2048 * 8 * 16 * 4 + 2048 * 64 * 128 * 4 + 64 * 2048 * 4
    assert f(1, 65536, 65536, 64, 8, 128, 16, 64, 0) == kv + 2 * per_slot2  # default: M/32
    assert f(1, 100, 100, 16, 2, 64, 4, 32, 1000) > 0       # chunk clipped to M
    assert f(1, 100, 100, 16, 2, 64, 4, 48, 0) == -3
    assert f(1, 100, 100, 24, 2, 64, 4, 32, 0) == -5  # 12 heads per group


def call_host(lib, q=FAKE, k=FAKE, v=FAKE, idx=FAKE, o=FAKE, lse=FAKE, ws=FAKE, ws_bytes=1 << 40,
              chunk=0, **over):
    a = dict(GOOD)
    a.update(over)
    vp = ctypes.c_void_p
    return lib.nsa_sel_attn_fwd_host(vp(q), vp(k), vp(v), vp(idx), vp(o), vp(lse), a["B"], a["M"],
                                     a["N"], a["H"], a["G"], a["D"], a["T"], a["bs"], 0.0, vp(ws),
                                     ws_bytes, chunk, None)


@pytest.mark.parametrize("which", ["q", "k", "v", "idx", "o", "lse"])
def test_host_null_pointers(lib, which):
    assert call_host(lib, **{which: None}) == -1


def test_host_workspace_checks(lib):
    need = lib.nsa_sel_attn_fwd_host_workspace_bytes(1, 128, 128, 16, 2, 128, 4, 64, 0)
    assert call_host(lib, ws=None) == -9
    assert call_host(lib, ws_bytes=need - 1) == -9
    assert call_host(lib, ws=FAKE + 16, ws_bytes=need) == -6
    assert call_host(lib, bs=16) == -3
    assert call_host(lib, B=0, q=None, k=None, v=None, idx=None, o=None, lse=None, ws=None) == 0


def call_shared(lib, q=FAKE, k=FAKE, v=FAKE, idx=FAKE, o=FAKE, lse=FAKE, ws=FAKE,
                ws_bytes=1 << 40, dtype=0, **over):
    a = dict(GOOD)
    a.update(over)
    vp = ctypes.c_void_p
    return lib.nsa_sel_attn_fwd_shared(vp(q), vp(k), vp(v), vp(idx), vp(o), vp(lse), a["B"],
                                       a["M"], a["N"], a["H"], a["G"], a["D"], a["T"], a["bs"],
                                       0.0, dtype, vp(ws), ws_bytes, None)


def test_shared_workspace_bytes(lib):
    f = lib.nsa_sel_attn_fwd_shared_workspace_bytes
    assert f(1, 65536, 8) == 8 * 4096 * 32  # one 32-byte record per (b, g, 16 queries)
    assert f(2, 1000, 2) == -(-(2 * 2 * 63 * 32) // 256) * 256
    assert f(1, 0, 8) == 0
    assert f(1, 16, 0) == -2 and f(-1, 16, 8) == -2
    assert f(1 << 20, 1 << 30, 64) == -2  # records past 2^31


def test_shared_argument_checks(lib):
    need = lib.nsa_sel_attn_fwd_shared_workspace_bytes(1, 128, 2)
    assert call_shared(lib, ws=None) == -9
    assert call_shared(lib, ws_bytes=need - 1) == -9
    assert call_shared(lib, ws=FAKE + 8, ws_bytes=need) == -6
    assert call_shared(lib, o=None) == -1
    assert call_shared(lib, bs=16) == -3
    assert call_shared(lib, dtype=2) == -11
    assert call_shared(lib, H=24) == -5
    assert call_shared(lib, B=0, q=None, k=None, v=None, idx=None, o=None, lse=None, ws=None) == 0


@pytest.mark.parametrize("H,G", [(16, 16), (16, 8), (12, 4), (16, 2), (64, 4), (96, 3)])
def test_heads_per_group_accepted(lib, H, G):
    # 1..8 heads per group, or a multiple of 8: the size checks pass (the
    # empty problem then returns before any CUDA call)
    assert call(lib, q=None, k=None, v=None, idx=None, o=None, lse=None, B=0, H=H, G=G) == 0


def call_ex(lib, qkv_dtype, o_dtype, q=FAKE, k=FAKE, v=FAKE, idx=FAKE, o=FAKE, lse=FAKE, **over):
    a = dict(GOOD)
    a.update(over)
    vp = ctypes.c_void_p
    return lib.nsa_sel_attn_fwd_ex(vp(q), vp(k), vp(v), vp(idx), vp(o), vp(lse), a["B"], a["M"],
                                   a["N"], a["H"], a["G"], a["D"], a["T"], a["bs"], 0.0,
                                   qkv_dtype, o_dtype, None)


@pytest.mark.parametrize("qkv,o,status", [
    (_lib.NSA_F16, _lib.NSA_F32, 0), (_lib.NSA_BF16, _lib.NSA_F32, 0),
    (_lib.NSA_F16, _lib.NSA_F16, 0), (_lib.NSA_BF16, _lib.NSA_BF16, 0),
    (_lib.NSA_F16, _lib.NSA_BF16, -11), (_lib.NSA_BF16, _lib.NSA_F16, -11),
    (_lib.NSA_F32, _lib.NSA_F32, -11), (3, _lib.NSA_F32, -11), (_lib.NSA_F16, -1, -11),
])
def test_ex_dtype_combinations(lib, qkv, o, status):
    # the dtype check runs after the size checks and before the empty-problem
    # return, so an empty problem shows it without any CUDA call
    assert call_ex(lib, qkv, o, q=None, k=None, v=None, idx=None, o=None, lse=None, B=0) == status


def test_ex_shares_the_size_checks(lib):
    assert call_ex(lib, _lib.NSA_BF16, _lib.NSA_BF16, bs=16) == -3
    assert call_ex(lib, _lib.NSA_BF16, _lib.NSA_F32, D=96) == -4
    assert call_ex(lib, _lib.NSA_F16, _lib.NSA_F16, o=None) == -1
    assert call_ex(lib, _lib.NSA_BF16, _lib.NSA_BF16, k=FAKE + 2) == -6


def test_binding_rejects_mixed_dtypes():
    torch = pytest.importorskip("torch")
    q = torch.zeros(1, 4, 8, 64, dtype=torch.bfloat16)
    k = torch.zeros(1, 4, 1, 64, dtype=torch.float16)
    idx = torch.zeros(1, 4, 1, 1, dtype=torch.int32)
    with pytest.raises(TypeError):
        _lib.sel_attn_fwd(q, k, k, idx, 32)
    with pytest.raises(TypeError):
        _lib.sel_attn_fwd(q.float(), k.float(), k.float(), idx, 32)


def call_topk(lib, scores=FAKE, idx=FAKE, B=1, M=128, N=128, G=2, T=4, bs=64, n_init=1,
              n_local=1):
    vp = ctypes.c_void_p
    return lib.nsa_topk_blocks(vp(scores), vp(idx), B, M, N, G, T, bs, n_init, n_local, None)


@pytest.mark.parametrize("over,status", [
    (dict(B=-1), -2), (dict(M=-1), -2), (dict(N=-1), -2), (dict(T=-1), -2), (dict(G=0), -2),
    (dict(bs=0), -3), (dict(n_init=-1), -2), (dict(n_local=-1), -2),
    (dict(n_init=3, n_local=2), -2), (dict(N=4097 * 64), -2), (dict(N=4097, bs=1), -2),
    (dict(idx=None), -1), (dict(scores=None), -1), (dict(idx=FAKE + 2), -6),
    (dict(scores=FAKE + 1), -6),
])
def test_topk_bad_arguments(lib, over, status):
    assert call_topk(lib, **over) == status


@pytest.mark.parametrize("over", [dict(B=0), dict(M=0), dict(T=0, n_init=0, n_local=0)])
def test_topk_empty_output_is_a_no_op(lib, over):
    assert call_topk(lib, scores=None, idx=None, **over) == 0


def call_swa(lib, q=FAKE, k=FAKE, v=FAKE, o=FAKE, lse=FAKE, B=1, M=128, N=128, H=8, Hkv=2, D=128,
             left=-1, right=0, dtype=1):
    vp = ctypes.c_void_p
    return lib.nsa_swa_fwd(vp(q), vp(k), vp(v), vp(o), vp(lse), B, M, N, H, Hkv, D, left, right,
                           0.0, dtype, None)


@pytest.mark.parametrize("over,status", [
    (dict(B=-1), -2), (dict(M=-1), -2), (dict(N=-1), -2), (dict(H=0), -2), (dict(Hkv=0), -2),
    (dict(H=8, Hkv=3), -5), (dict(D=96), -4), (dict(dtype=2), -11), (dict(dtype=7), -11),
    (dict(M=(1 << 30) + 1), -2), (dict(q=None), -1), (dict(o=None), -1), (dict(k=None), -1),
    (dict(v=FAKE + 8), -6), (dict(o=FAKE + 2), -6), (dict(lse=FAKE + 1), -6),
])
def test_swa_bad_arguments(lib, over, status):
    assert call_swa(lib, **over) == status


@pytest.mark.parametrize("over", [dict(B=0), dict(M=0)])
def test_swa_empty_is_a_no_op(lib, over):
    assert call_swa(lib, q=None, k=None, v=None, o=None, lse=None, **over) == 0


def call_strided(lib, strides, q=FAKE, k=FAKE, v=FAKE, idx=FAKE, o=FAKE, lse=FAKE, **over):
    a = dict(GOOD)
    a.update(over)
    vp = ctypes.c_void_p
    arr = (ctypes.c_int64 * 12)(*strides) if strides is not None else None
    return lib.nsa_sel_attn_fwd_strided(vp(q), vp(k), vp(v), vp(idx), vp(o), vp(lse), a["B"],
                                        a["M"], a["N"], a["H"], a["G"], a["D"], a["T"], a["bs"],
                                        0.0, 0, 2, arr, None)


def _contig_strides(B=1, M=128, N=128, H=16, G=2, D=128):
    return [M * H * D, H * D, D, N * G * D, G * D, D, N * G * D, G * D, D, M * H * D, H * D, D]


@pytest.mark.parametrize("i,value,status", [
    (0, 4, -6), (1, 12, -6), (2, 1, -6), (4, 100, -6), (8, 3, -6), (11, 6, -6),
    (3, -8, -2), (9, (1 << 41), -2),
])
def test_strided_checks(lib, i, value, status):
    st = _contig_strides()
    st[i] = value
    assert call_strided(lib, st) == status


def test_strided_empty_and_null_strides(lib):
    assert call_strided(lib, None, q=None, k=None, v=None, idx=None, o=None, lse=None, B=0) == 0
    assert call_strided(lib, _contig_strides(), q=None, k=None, v=None, idx=None, o=None,
                        lse=None, M=0) == 0


def call_probe(lib, k=FAKE, v=FAKE, N=4096, G=8, D=128, g=0, bs=64, ctas=152, warps=4, slots=2,
               loads=16, rows=16, rec=None):
    vp = ctypes.c_void_p
    return lib.nsa_probe_l2_gather(vp(k), vp(v), N, G, D, g, bs, ctas, warps, slots, loads, rows,
                                   1, vp(rec), None)


@pytest.mark.parametrize("over,status", [
    (dict(k=None), -1), (dict(v=None), -1), (dict(k=FAKE + 8), -6), (dict(rec=FAKE + 4), -6),
    (dict(D=96), -4), (dict(bs=16), -3), (dict(N=63), -2), (dict(G=0), -2), (dict(g=8), -2),
    (dict(g=-2), -2), (dict(ctas=0), -2), (dict(warps=0), -2), (dict(warps=33), -2),
    (dict(slots=0), -2), (dict(slots=17), -2), (dict(loads=-1), -2),
    (dict(warps=32, slots=2), -2),  # 256 KB of shared memory per CTA
    (dict(rows=8), -2), (dict(rows=64, bs=32), -2), (dict(rows=64, warps=8, slots=4), -2),
])
def test_probe_rejects_bad_arguments(lib, over, status):
    assert call_probe(lib, **over) == status


def test_probe_bytes(lib):
    f = lib.nsa_probe_l2_gather_bytes
    assert f(128, 152, 4, 1000, 16) == 152 * 4 * 1000 * 4096
    assert f(64, 10, 2, 3, 16) == 10 * 2 * 3 * 2048
    assert f(128, 1, 1, 1, 64) == 16384
    assert f(96, 1, 1, 1, 16) == -2
    assert f(128, 1, 1, 1, 48) == -2


def call_rows_probe(lib, k=FAKE, v=FAKE, idx=FAKE, B=1, M=256, N=256, G=8, D=128, T=4, bs=64,
                    ctas=152, warps=4, slots=2, pad=0):
    vp = ctypes.c_void_p
    return lib.nsa_probe_gather_rows(vp(k), vp(v), vp(idx), B, M, N, G, D, T, bs, ctas, warps,
                                     slots, pad, None)


@pytest.mark.parametrize("over,status", [
    (dict(k=None), -1), (dict(idx=None), -1), (dict(v=FAKE + 4), -6), (dict(idx=FAKE + 2), -6),
    (dict(D=96), -4), (dict(bs=16), -3), (dict(M=-1), -2), (dict(ctas=0), -2),
    (dict(warps=33), -2), (dict(slots=0), -2), (dict(warps=32, slots=2), -2),
    (dict(pad=-1), -2), (dict(pad=200 * 1024), -2),
])
def test_rows_probe_rejects_bad_arguments(lib, over, status):
    assert call_rows_probe(lib, **over) == status


def test_rows_probe_empty_is_a_no_op(lib):
    assert call_rows_probe(lib, k=None, v=None, idx=None, M=0) == 0


@pytest.mark.parametrize("over,status", [
    (dict(buf=None), -1), (dict(buf=FAKE + 4), -6), (dict(rows=0), -2), (dict(stride=512), -2),
    (dict(stride=1026), -2), (dict(ctas=0), -2), (dict(warps=33), -2), (dict(iters=-1), -2),
])
def test_reduce_probe_rejects_bad_arguments(lib, over, status):
    a = dict(buf=FAKE, rows=1024, stride=8192, ctas=152, warps=4, iters=16)
    a.update(over)
    vp = ctypes.c_void_p
    assert lib.nsa_probe_reduce_rows(vp(a["buf"]), a["rows"], a["stride"], a["ctas"], a["warps"],
                                     a["iters"], 1, None) == status


def test_host_ex_rejects_bad_dtypes(lib):
    a = dict(GOOD)
    vp = ctypes.c_void_p
    for qkv, o in ((2, 2), (0, 1), (1, 0), (3, 2)):
        st = lib.nsa_sel_attn_fwd_host_ex(vp(FAKE), vp(FAKE), vp(FAKE), vp(FAKE), vp(FAKE),
                                          vp(FAKE), a["B"], a["M"], a["N"], a["H"], a["G"], a["D"],
                                          a["T"], a["bs"], 0.0, qkv, o, vp(FAKE), 1 << 40, 0, None)
        assert st == -11, (qkv, o)


def test_bwd_ex_rejects_bad_dtypes(lib):
    vp = ctypes.c_void_p
    for dt in (2, 3, -1):
        st = lib.nsa_sel_attn_bwd_ex(*([vp(FAKE)] * 10), 1, 128, 128, 16, 2, 128, 4, 64, 0.0, dt,
                                     vp(FAKE), 1 << 40, None)
        assert st == -11, dt
