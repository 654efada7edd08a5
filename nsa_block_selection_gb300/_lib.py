"""ctypes binding of ``libnsa_sel_attn.so`` (argument marshalling only).

Every step of the selection-attention forward runs in the library's CUDA
kernels; this module only checks tensor dtypes/devices, allocates outputs
with torch and passes raw pointers, sizes and the current CUDA stream. There
is no fallback: if the library is missing, calls raise.
"""

from __future__ import annotations

import ctypes
import os
from typing import Optional

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "lib", "libnsa_sel_attn.so")

NSA_OK = 0
NSA_F16, NSA_BF16, NSA_F32 = 0, 1, 2

EXPORTS = ("nsa_status_string", "nsa_version", "nsa_sel_attn_fwd", "nsa_sel_attn_fwd_ex",
           "nsa_sel_attn_fwd_strided", "nsa_sync_status",
           "nsa_selftest_wait_timeout", "nsa_sel_attn_fwd_host_workspace_bytes",
           "nsa_sel_attn_fwd_host", "nsa_sel_attn_bwd_workspace_bytes", "nsa_sel_attn_bwd",
           "nsa_sel_attn_bwd_noalloc", "nsa_topk_blocks", "nsa_swa_fwd",
           "nsa_sel_attn_fwd_shared_workspace_bytes", "nsa_sel_attn_fwd_shared",
           "nsa_probe_l2_gather", "nsa_probe_l2_gather_bytes", "nsa_probe_gather_rows",
           "nsa_probe_reduce_rows", "nsa_sel_attn_fwd_host_ex", "nsa_sel_attn_bwd_ex")

_lib = None


class NsaError(RuntimeError):
    def __init__(self, status: int, what: str):
        super().__init__(f"{what} failed: {status_string(status)} ({status})")
        self.status = status


def load(path: Optional[str] = None) -> ctypes.CDLL:
    """Load the library (once) and declare the C signatures."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    p = path or LIB_PATH
    if not os.path.exists(p):
        raise RuntimeError(
            f"{p} is missing: build it with `python -m nsa_block_selection_gb300.build` "
            "(the CUDA library is the only implementation)")
    lib = ctypes.CDLL(p)
    i64, c_int, vp = ctypes.c_int64, ctypes.c_int, ctypes.c_void_p
    lib.nsa_status_string.restype = ctypes.c_char_p
    lib.nsa_status_string.argtypes = [c_int]
    lib.nsa_version.restype = c_int
    lib.nsa_version.argtypes = []
    lib.nsa_sel_attn_fwd.restype = c_int
    lib.nsa_sel_attn_fwd.argtypes = [vp, vp, vp, vp, vp, vp, i64, i64, i64, i64, i64, i64, i64,
                                     c_int, ctypes.c_float, vp]
    lib.nsa_sel_attn_fwd_ex.restype = c_int
    lib.nsa_sel_attn_fwd_ex.argtypes = [vp, vp, vp, vp, vp, vp, i64, i64, i64, i64, i64, i64,
                                        i64, c_int, ctypes.c_float, c_int, c_int, vp]
    lib.nsa_sel_attn_fwd_strided.restype = c_int
    lib.nsa_sel_attn_fwd_strided.argtypes = [vp, vp, vp, vp, vp, vp, i64, i64, i64, i64, i64,
                                             i64, i64, c_int, ctypes.c_float, c_int, c_int, vp,
                                             vp]
    lib.nsa_sel_attn_fwd_shared_workspace_bytes.restype = i64
    lib.nsa_sel_attn_fwd_shared_workspace_bytes.argtypes = [i64, i64, i64]
    lib.nsa_sel_attn_fwd_shared.restype = c_int
    lib.nsa_sel_attn_fwd_shared.argtypes = [vp, vp, vp, vp, vp, vp, i64, i64, i64, i64, i64, i64,
                                            i64, c_int, ctypes.c_float, c_int, vp, i64, vp]
    lib.nsa_sync_status.restype = c_int
    lib.nsa_sync_status.argtypes = [vp]
    lib.nsa_selftest_wait_timeout.restype = c_int
    lib.nsa_selftest_wait_timeout.argtypes = [i64, vp]
    lib.nsa_sel_attn_fwd_host_workspace_bytes.restype = i64
    lib.nsa_sel_attn_fwd_host_workspace_bytes.argtypes = [i64, i64, i64, i64, i64, i64, i64,
                                                          c_int, i64]
    lib.nsa_sel_attn_bwd_workspace_bytes.restype = i64
    lib.nsa_sel_attn_bwd_workspace_bytes.argtypes = [i64, i64, i64, i64, i64, i64, i64, c_int]
    lib.nsa_sel_attn_bwd.restype = c_int
    lib.nsa_sel_attn_bwd.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, i64, i64, i64, i64,
                                     i64, i64, i64, c_int, ctypes.c_float, vp, i64, vp]
    lib.nsa_sel_attn_bwd_ex.restype = c_int
    lib.nsa_sel_attn_bwd_ex.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, i64, i64, i64,
                                        i64, i64, i64, i64, c_int, ctypes.c_float, c_int, vp, i64,
                                        vp]
    lib.nsa_sel_attn_bwd_noalloc.restype = c_int
    lib.nsa_sel_attn_bwd_noalloc.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, i64, i64,
                                             i64, i64, i64, i64, i64, c_int, ctypes.c_float, vp]
    lib.nsa_swa_fwd.restype = c_int
    lib.nsa_swa_fwd.argtypes = [vp, vp, vp, vp, vp, i64, i64, i64, i64, i64, i64, i64, i64,
                                ctypes.c_float, c_int, vp]
    lib.nsa_topk_blocks.restype = c_int
    lib.nsa_topk_blocks.argtypes = [vp, vp, i64, i64, i64, i64, i64, c_int, c_int, c_int, vp]
    lib.nsa_sel_attn_fwd_host_ex.restype = c_int
    lib.nsa_sel_attn_fwd_host_ex.argtypes = [vp, vp, vp, vp, vp, vp, i64, i64, i64, i64, i64,
                                             i64, i64, c_int, ctypes.c_float, c_int, c_int, vp,
                                             i64, i64, vp]
    lib.nsa_sel_attn_fwd_host.restype = c_int
    lib.nsa_sel_attn_fwd_host.argtypes = [vp, vp, vp, vp, vp, vp, i64, i64, i64, i64, i64, i64,
                                          i64, c_int, ctypes.c_float, vp, i64, i64, vp]
    lib.nsa_probe_l2_gather.restype = c_int
    lib.nsa_probe_l2_gather.argtypes = [vp, vp, i64, i64, i64, i64, c_int, i64, c_int, c_int,
                                        i64, c_int, ctypes.c_uint32, vp, vp]
    lib.nsa_probe_l2_gather_bytes.restype = i64
    lib.nsa_probe_l2_gather_bytes.argtypes = [i64, i64, c_int, i64, c_int]
    lib.nsa_probe_reduce_rows.restype = c_int
    lib.nsa_probe_reduce_rows.argtypes = [vp, i64, i64, i64, c_int, i64, ctypes.c_uint32, vp]
    lib.nsa_probe_gather_rows.restype = c_int
    lib.nsa_probe_gather_rows.argtypes = [vp, vp, vp, i64, i64, i64, i64, i64, i64, c_int, i64,
                                          c_int, c_int, i64, vp]
    if path is None:
        _lib = lib
    return lib


def status_string(status: int) -> str:
    return load().nsa_status_string(int(status)).decode()


def _ptr(t) -> Optional[int]:
    return t.data_ptr() if t is not None and t.numel() > 0 else None


def _dtype_code(dt) -> int:
    import torch

    return {torch.float16: NSA_F16, torch.bfloat16: NSA_BF16, torch.float32: NSA_F32}[dt]


def sel_attn_fwd(q, k, v, block_indices, block_size: int, scale: Optional[float] = None,
                 out=None, lse=None, stream=None, out_dtype=None):
    """NSA selection-attention forward on the GPU.

    q: fp16 or bf16 [B, M, H, D]; k, v: [B, N, G, D] of q's dtype;
    block_indices: int32 [B, M, G, T] (-1 = padding), contiguous; all on one
    CUDA device. q, k, v (and a preallocated ``out``) may be strided views
    (for example slices of one fused projection) whose last dimension is
    contiguous and whose strides are multiples of 8 elements. Returns
    (O [B, M, H, D], LSE fp32 [B, H, M]). O is fp32 unless ``out_dtype`` (or
    a preallocated ``out``) is q's dtype. ``stream`` defaults to torch's
    current stream.
    """
    import torch

    lib = load()
    B, M, N, H, G, D, T = _check_common(q, k, v, block_indices, device_expected=True,
                                        qkv_dtypes=(torch.float16, torch.bfloat16),
                                        strided=True)
    if out_dtype is None:
        out_dtype = out.dtype if out is not None else torch.float32
    if out_dtype not in (torch.float32, q.dtype):
        raise TypeError(f"O must be fp32 or {q.dtype}, got {out_dtype}")
    if out is None:
        out = torch.empty((B, M, H, D), dtype=out_dtype, device=q.device)
    if lse is None:
        lse = torch.empty((B, H, M), dtype=torch.float32, device=q.device)
    if out.dtype != out_dtype or tuple(out.shape) != (B, M, H, D) or out.stride(-1) != 1:
        raise ValueError(f"out must be {out_dtype} [B, M, H, D] with a contiguous last dim")
    if lse.dtype != torch.float32 or tuple(lse.shape) != (B, H, M) or not lse.is_contiguous():
        raise ValueError("lse must be contiguous fp32 [B, H, M]")
    if stream is None:
        stream = torch.cuda.current_stream(q.device)
    sc = float(scale) if scale is not None else 0.0  # the ABI: <= 0 selects 1/sqrt(D)
    args = (_ptr(q), _ptr(k), _ptr(v), _ptr(block_indices), _ptr(out), _ptr(lse), B, M, N, H,
            G, D, T, int(block_size), sc)
    if not all(t.is_contiguous() or t.numel() == 0 for t in (q, k, v, out)):
        strides = (ctypes.c_int64 * 12)(*(list(q.stride()[:3]) + list(k.stride()[:3]) +
                                          list(v.stride()[:3]) + list(out.stride()[:3])))
        st = lib.nsa_sel_attn_fwd_strided(*args, _dtype_code(q.dtype), _dtype_code(out.dtype),
                                          strides, ctypes.c_void_p(stream.cuda_stream))
        what = "nsa_sel_attn_fwd_strided"
    elif q.dtype == torch.float16 and out.dtype == torch.float32:
        st = lib.nsa_sel_attn_fwd(*args, ctypes.c_void_p(stream.cuda_stream))
        what = "nsa_sel_attn_fwd"
    else:
        st = lib.nsa_sel_attn_fwd_ex(*args, _dtype_code(q.dtype), _dtype_code(out.dtype),
                                     ctypes.c_void_p(stream.cuda_stream))
        what = "nsa_sel_attn_fwd_ex"
    if st != NSA_OK:
        raise NsaError(st, what)
    return out, lse


def shared_workspace_bytes(B, M, G) -> int:
    n = load().nsa_sel_attn_fwd_shared_workspace_bytes(B, M, G)
    if n < 0:
        raise NsaError(int(n), "nsa_sel_attn_fwd_shared_workspace_bytes")
    return int(n)


def sel_attn_fwd_shared(q, k, v, block_indices, block_size: int, scale: Optional[float] = None,
                        out=None, lse=None, workspace=None, stream=None):
    """The two-pass forward (nsa_sel_attn_fwd_shared): blocks common to a tile
    of 16 consecutive queries are gathered once per tile. Contiguous fp16 or
    bf16 q, k, v; O fp32. ``workspace``: a CUDA uint8 tensor of at least
    shared_workspace_bytes(B, M, G) bytes (allocated when None). Returns
    (O, LSE); the per-tile records stay in ``workspace``.
    """
    import torch

    lib = load()
    B, M, N, H, G, D, T = _check_common(q, k, v, block_indices, device_expected=True,
                                        qkv_dtypes=(torch.float16, torch.bfloat16))
    if out is None:
        out = torch.empty((B, M, H, D), dtype=torch.float32, device=q.device)
    if lse is None:
        lse = torch.empty((B, H, M), dtype=torch.float32, device=q.device)
    if out.dtype != torch.float32 or tuple(out.shape) != (B, M, H, D) or not out.is_contiguous():
        raise ValueError("out must be contiguous fp32 [B, M, H, D]")
    if lse.dtype != torch.float32 or tuple(lse.shape) != (B, H, M) or not lse.is_contiguous():
        raise ValueError("lse must be contiguous fp32 [B, H, M]")
    if workspace is None:
        workspace = torch.empty(max(shared_workspace_bytes(B, M, G), 1), dtype=torch.uint8,
                                device=q.device)
    if stream is None:
        stream = torch.cuda.current_stream(q.device)
    sc = float(scale) if scale is not None else 0.0  # the ABI: <= 0 selects 1/sqrt(D)
    st = lib.nsa_sel_attn_fwd_shared(_ptr(q), _ptr(k), _ptr(v), _ptr(block_indices), _ptr(out),
                                     _ptr(lse), B, M, N, H, G, D, T, int(block_size), sc,
                                     _dtype_code(q.dtype), _ptr(workspace), workspace.numel(),
                                     ctypes.c_void_p(stream.cuda_stream))
    if st != NSA_OK:
        raise NsaError(st, "nsa_sel_attn_fwd_shared")
    return out, lse


def _check_common(q, k, v, block_indices, device_expected: bool, qkv_dtypes=None,
                  strided: bool = False):
    import torch

    qkv_dtypes = qkv_dtypes or (torch.float16,)
    if q.dtype not in qkv_dtypes:
        raise TypeError(f"q must be one of {qkv_dtypes}, got {q.dtype}")

    B, M, H, D = q.shape
    Bk, N, G, Dk = k.shape
    T = block_indices.shape[-1]
    if (Bk, Dk) != (B, D) or tuple(v.shape) != tuple(k.shape) or \
            tuple(block_indices.shape) != (B, M, G, T):
        raise ValueError("shape mismatch: q [B,M,H,D], k/v [B,N,G,D], "
                         "block_indices [B,M,G,T]")
    named = (("q", q, q.dtype), ("k", k, q.dtype), ("v", v, q.dtype),
             ("block_indices", block_indices, torch.int32))
    for name, t, dt in named:
        if t.dtype != dt:
            raise TypeError(f"{name} must be {dt}, got {t.dtype}")
    for name, t, _ in named:
        if t.is_cuda != device_expected:
            raise ValueError(f"{name} must be a {'CUDA' if device_expected else 'CPU'} tensor")
        if strided and name != "block_indices":
            if t.numel() > 0 and t.stride(-1) != 1:
                raise ValueError(f"{name} must have a contiguous last dimension")
        elif not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous")
    return B, M, N, H, G, D, T


def host_workspace_bytes(B, M, N, H, G, D, T, block_size, chunk_m=0) -> int:
    n = load().nsa_sel_attn_fwd_host_workspace_bytes(B, M, N, H, G, D, T, int(block_size),
                                                     int(chunk_m))
    if n < 0:
        raise NsaError(int(n), "nsa_sel_attn_fwd_host_workspace_bytes")
    return int(n)


def sel_attn_fwd_host(q, k, v, block_indices, block_size: int, scale: Optional[float] = None,
                      out=None, lse=None, chunk_m: int = 0, workspace=None, device=None,
                      stream=None, sync: bool = True, out_dtype=None):
    """Forward with host (CPU) tensors in and out, through the library's
    pipelined host entry point (pin the tensors for overlapped copies).

    q, k, v fp16 or bf16. Returns (O, LSE) as CPU tensors: O fp32 unless
    ``out_dtype`` (or a preallocated ``out``) is q's dtype, LSE fp32.
    ``workspace`` is a CUDA uint8 tensor of at least
    :func:`host_workspace_bytes`; one is allocated when omitted. With
    ``sync=False`` the call returns once everything is enqueued on ``stream``.
    """
    import torch

    lib = load()
    B, M, N, H, G, D, T = _check_common(q, k, v, block_indices, device_expected=False,
                                        qkv_dtypes=(torch.float16, torch.bfloat16))
    if out_dtype is None:
        out_dtype = out.dtype if out is not None else torch.float32
    if out_dtype not in (torch.float32, q.dtype):
        raise TypeError(f"O must be fp32 or {q.dtype}, got {out_dtype}")
    device = torch.device(device) if device is not None else torch.device("cuda",
                                                                        torch.cuda.current_device())
    need = host_workspace_bytes(B, M, N, H, G, D, T, block_size, chunk_m)
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=device)
    if out is None:
        out = torch.empty((B, M, H, D), dtype=out_dtype, pin_memory=True)
    if lse is None:
        lse = torch.empty((B, H, M), dtype=torch.float32, pin_memory=True)
    if out.is_cuda or lse.is_cuda or out.dtype != out_dtype or lse.dtype != torch.float32:
        raise ValueError(f"out must be a {out_dtype} CPU tensor and lse an fp32 one")
    if tuple(out.shape) != (B, M, H, D) or tuple(lse.shape) != (B, H, M):
        raise ValueError("out must be [B, M, H, D] and lse [B, H, M]")
    if stream is None:
        stream = torch.cuda.current_stream(device)
    sc = float(scale) if scale is not None else 0.0  # the ABI: <= 0 selects 1/sqrt(D)
    args = (_ptr(q), _ptr(k), _ptr(v), _ptr(block_indices), _ptr(out), _ptr(lse), B, M, N, H,
            G, D, T, int(block_size), sc)
    tail = (workspace.data_ptr(), workspace.numel(), int(chunk_m),
            ctypes.c_void_p(stream.cuda_stream))
    if q.dtype == torch.float16 and out.dtype == torch.float32:
        st = lib.nsa_sel_attn_fwd_host(*args, *tail)
        what = "nsa_sel_attn_fwd_host"
    else:
        st = lib.nsa_sel_attn_fwd_host_ex(*args, _dtype_code(q.dtype), _dtype_code(out.dtype),
                                          *tail)
        what = "nsa_sel_attn_fwd_host_ex"
    if st != NSA_OK:
        raise NsaError(st, what)
    if sync:
        stream.synchronize()
    return out, lse


def bwd_workspace_bytes(B, M, N, H, G, D, T, block_size) -> int:
    n = load().nsa_sel_attn_bwd_workspace_bytes(B, M, N, H, G, D, T, int(block_size))
    if n < 0:
        raise NsaError(int(n), "nsa_sel_attn_bwd_workspace_bytes")
    return int(n)


def sel_attn_bwd(q, k, v, block_indices, o, lse, do, block_size: int,
                 scale: Optional[float] = None, dq=None, dk=None, dv=None, workspace=None,
                 stream=None):
    """Gradients of :func:`sel_attn_fwd`: returns (dQ, dK, dV) fp32 CUDA tensors.

    q, k, v fp16 or bf16 (as passed to the forward). ``o`` and ``lse`` are
    the forward's fp32 outputs, ``do`` the fp32 upstream gradient
    [B, M, H, D]. ``workspace`` (CUDA uint8) is allocated when omitted.
    """
    import torch

    lib = load()
    B, M, N, H, G, D, T = _check_common(q, k, v, block_indices, device_expected=True,
                                        qkv_dtypes=(torch.float16, torch.bfloat16))
    for name, t, shape in (("o", o, (B, M, H, D)), ("lse", lse, (B, H, M)),
                           ("do", do, (B, M, H, D))):
        if t.dtype != torch.float32 or tuple(t.shape) != shape or not t.is_contiguous() \
                or not t.is_cuda:
            raise ValueError(f"{name} must be a contiguous fp32 CUDA tensor of shape {shape}")
    dev = q.device
    dq = torch.empty((B, M, H, D), dtype=torch.float32, device=dev) if dq is None else dq
    dk = torch.empty((B, N, G, D), dtype=torch.float32, device=dev) if dk is None else dk
    dv = torch.empty((B, N, G, D), dtype=torch.float32, device=dev) if dv is None else dv
    need = bwd_workspace_bytes(B, M, N, H, G, D, T, block_size)
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=dev)
    if stream is None:
        stream = torch.cuda.current_stream(dev)
    sc = float(scale) if scale is not None else 0.0  # the ABI: <= 0 selects 1/sqrt(D)
    args = (_ptr(q), _ptr(k), _ptr(v), _ptr(block_indices), _ptr(o), _ptr(lse), _ptr(do),
            _ptr(dq), _ptr(dk), _ptr(dv), B, M, N, H, G, D, T, int(block_size), sc)
    tail = (workspace.data_ptr(), workspace.numel(), ctypes.c_void_p(stream.cuda_stream))
    if q.dtype == torch.float16:
        st = lib.nsa_sel_attn_bwd(*args, *tail)
        what = "nsa_sel_attn_bwd"
    else:
        st = lib.nsa_sel_attn_bwd_ex(*args, _dtype_code(q.dtype), *tail)
        what = "nsa_sel_attn_bwd_ex"
    if st != NSA_OK:
        raise NsaError(st, what)
    return dq, dk, dv


def sync_status(stream=None) -> int:
    """Wait for ``stream`` (default: torch's current stream) and return the
    library's device status (NSA_OK, or -8 after a timed-out device wait)."""
    import torch

    if stream is None:
        stream = torch.cuda.current_stream()
    return load().nsa_sync_status(ctypes.c_void_p(stream.cuda_stream))


def selftest_wait_timeout(limit_ns: int, stream=None) -> int:
    """Launch the self-test kernel whose wait can only time out."""
    import torch

    if stream is None:
        stream = torch.cuda.current_stream()
    return load().nsa_selftest_wait_timeout(int(limit_ns), ctypes.c_void_p(stream.cuda_stream))


def topk_blocks(scores, N: int, block_size: int, T: int, n_init: int = 0, n_local: int = 0,
                out=None, stream=None):
    """Top-k block selection on the GPU (nsa_topk_blocks).

    scores: fp32 [B, M, G, ceil(N/block_size)], contiguous on a CUDA device.
    Returns block_indices int32 [B, M, G, T] (ascending, -1 padded): per
    (b, m, g) the first n_init and last n_local causal blocks and the
    highest-scoring others.
    """
    import torch

    lib = load()
    if scores.dtype != torch.float32 or not scores.is_cuda or not scores.is_contiguous():
        raise TypeError("scores must be a contiguous fp32 CUDA tensor")
    B, M, G, S = scores.shape
    if S != -(-int(N) // int(block_size)):
        raise ValueError("scores must have ceil(N/block_size) entries per row")
    if out is None:
        out = torch.empty((B, M, G, T), dtype=torch.int32, device=scores.device)
    if out.dtype != torch.int32 or tuple(out.shape) != (B, M, G, T) or not out.is_contiguous():
        raise ValueError("out must be contiguous int32 [B, M, G, T]")
    if stream is None:
        stream = torch.cuda.current_stream(scores.device)
    st = lib.nsa_topk_blocks(_ptr(scores), _ptr(out), B, M, int(N), G, int(T), int(block_size),
                             int(n_init), int(n_local), ctypes.c_void_p(stream.cuda_stream))
    if st != NSA_OK:
        raise NsaError(st, "nsa_topk_blocks")
    return out


def swa_fwd(q, k, v, window=(-1, -1), scale: Optional[float] = None, out=None, lse=None,
            return_lse: bool = True, stream=None):
    """GQA sliding-window attention forward on the GPU (nsa_swa_fwd).

    q: bf16 or fp16 [B, M, H, D]; k, v: [B, N, H_kv, D] of q's dtype, all
    contiguous on one CUDA device. ``window`` = (left, right): query i sees
    keys [i - left, i + right]; a negative side is unbounded. Returns
    (O [B, M, H, D] in q's dtype, LSE fp32 [B, H, M] or None).
    """
    import torch

    lib = load()
    if q.dtype not in (torch.float16, torch.bfloat16):
        raise TypeError(f"q must be fp16 or bf16, got {q.dtype}")
    for name, t in (("k", k), ("v", v)):
        if t.dtype != q.dtype:
            raise TypeError(f"{name} must be {q.dtype}, got {t.dtype}")
    for name, t in (("q", q), ("k", k), ("v", v)):
        if not t.is_cuda or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous CUDA tensor")
    B, M, H, D = q.shape
    Bk, N, Hkv, Dk = k.shape
    if (Bk, Dk) != (B, D) or tuple(v.shape) != tuple(k.shape):
        raise ValueError("shape mismatch: q [B,M,H,D], k/v [B,N,H_kv,D]")
    if out is None:
        out = torch.empty((B, M, H, D), dtype=q.dtype, device=q.device)
    if out.dtype != q.dtype or tuple(out.shape) != (B, M, H, D) or not out.is_contiguous():
        raise ValueError(f"out must be contiguous {q.dtype} [B, M, H, D]")
    if lse is None and return_lse:
        lse = torch.empty((B, H, M), dtype=torch.float32, device=q.device)
    if lse is not None and (lse.dtype != torch.float32 or tuple(lse.shape) != (B, H, M)
                            or not lse.is_contiguous()):
        raise ValueError("lse must be contiguous fp32 [B, H, M]")
    if stream is None:
        stream = torch.cuda.current_stream(q.device)
    left, right = (int(window[0]), int(window[1])) if window is not None else (-1, -1)
    sc = float(scale) if scale is not None else 0.0  # the ABI: <= 0 selects 1/sqrt(D)
    st = lib.nsa_swa_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), B, M, N, H, Hkv, D,
                         left, right, sc, _dtype_code(q.dtype),
                         ctypes.c_void_p(stream.cuda_stream))
    if st != NSA_OK:
        raise NsaError(st, "nsa_swa_fwd")
    return out, lse


def probe_l2_gather(k, v, g: int, block_size: int, ctas: int, warps_per_cta: int,
                    slots_per_warp: int, loads_per_warp: int, seed: int = 1, record=None,
                    stream=None, rows_per_box: int = 16) -> int:
    """Launch the gather-bandwidth probe (nsa_probe_l2_gather) on K, V
    [N, G, D] fp16 (one batch) and return the bytes it moves. ``record``: an
    int64 CUDA tensor [ctas, 3] for per-CTA (SM id, start ns, end ns), or
    None."""
    import torch

    lib = load()
    for name, t in (("k", k), ("v", v)):
        if t.dtype != torch.float16 or not t.is_cuda or not t.is_contiguous() or t.dim() != 3:
            raise ValueError(f"{name} must be a contiguous fp16 CUDA tensor [N, G, D]")
    if tuple(v.shape) != tuple(k.shape):
        raise ValueError("k and v must have the same shape")
    N, G, D = k.shape
    if record is not None and (record.dtype != torch.int64 or not record.is_cuda
                               or tuple(record.shape) != (ctas, 3)
                               or not record.is_contiguous()):
        raise ValueError("record must be a contiguous int64 CUDA tensor [ctas, 3]")
    if stream is None:
        stream = torch.cuda.current_stream(k.device)
    st = lib.nsa_probe_l2_gather(_ptr(k), _ptr(v), N, G, D, int(g), int(block_size), int(ctas),
                                 int(warps_per_cta), int(slots_per_warp), int(loads_per_warp),
                                 int(rows_per_box), int(seed) & 0xFFFFFFFF, _ptr(record),
                                 ctypes.c_void_p(stream.cuda_stream))
    if st != NSA_OK:
        raise NsaError(st, "nsa_probe_l2_gather")
    n = lib.nsa_probe_l2_gather_bytes(D, int(ctas), int(warps_per_cta), int(loads_per_warp),
                                      int(rows_per_box))
    if n < 0:
        raise NsaError(int(n), "nsa_probe_l2_gather_bytes")
    return int(n)


def probe_gather_rows(k, v, block_indices, block_size: int, ctas: int, warps_per_cta: int,
                      slots_per_warp: int, stream=None, extra_smem_bytes: int = 0) -> None:
    """Launch the index-driven gather probe (nsa_probe_gather_rows): the
    forward's copies for these rows alone. k, v: fp16 [B, N, G, D];
    block_indices: int32 [B, M, G, T], all contiguous on one CUDA device."""
    import torch

    lib = load()
    for name, t in (("k", k), ("v", v)):
        if t.dtype != torch.float16 or not t.is_cuda or not t.is_contiguous() or t.dim() != 4:
            raise ValueError(f"{name} must be a contiguous fp16 CUDA tensor [B, N, G, D]")
    if block_indices.dtype != torch.int32 or not block_indices.is_contiguous():
        raise ValueError("block_indices must be contiguous int32 [B, M, G, T]")
    B, N, G, D = k.shape
    Bi, M, Gi, T = block_indices.shape
    if (Bi, Gi) != (B, G) or tuple(v.shape) != tuple(k.shape):
        raise ValueError("shape mismatch: k/v [B, N, G, D], block_indices [B, M, G, T]")
    if stream is None:
        stream = torch.cuda.current_stream(k.device)
    st = lib.nsa_probe_gather_rows(_ptr(k), _ptr(v), _ptr(block_indices), B, M, N, G, D, T,
                                   int(block_size), int(ctas), int(warps_per_cta),
                                   int(slots_per_warp), int(extra_smem_bytes),
                                   ctypes.c_void_p(stream.cuda_stream))
    if st != NSA_OK:
        raise NsaError(st, "nsa_probe_gather_rows")


def probe_reduce_rows(buf, rows: int, stride: int, ctas: int, warps_per_cta: int,
                      iters_per_warp: int, seed: int = 1, stream=None) -> int:
    """Launch the reduction-rate probe (nsa_probe_reduce_rows) on an fp32
    CUDA tensor of at least rows * stride elements; returns the bytes it
    reduces. Adds zeros: the tensor's values are unchanged."""
    import torch

    lib = load()
    if buf.dtype != torch.float32 or not buf.is_cuda or buf.numel() < rows * stride:
        raise ValueError("buf must be an fp32 CUDA tensor of at least rows * stride elements")
    if stream is None:
        stream = torch.cuda.current_stream(buf.device)
    st = lib.nsa_probe_reduce_rows(_ptr(buf), int(rows), int(stride), int(ctas),
                                   int(warps_per_cta), int(iters_per_warp), int(seed) & 0xFFFFFFFF,
                                   ctypes.c_void_p(stream.cuda_stream))
    if st != NSA_OK:
        raise NsaError(st, "nsa_probe_reduce_rows")
    return int(ctas) * int(warps_per_cta) * int(iters_per_warp) * 4096
