"""Seeded synthetic inputs for NSA selection attention.

This module is shared by the CPU oracle's tests and by the CUDA path's tests
and benchmark. It draws numbers and lays out index rows; it holds none of the
attention arithmetic (no scores, no softmax, no masking of scores).

Shapes follow the operation statement of "[wave] NSA: selection attention
forward kernel" (section "Operation"): Q [B, M, H, D], K and V [B, N, G, D],
block_indices [B, M, G, T]. Index rows are what an upstream top-k selection
would hand over: distinct block ids, sorted ascending, padded with -1 at the
end, always causal (block id <= floor(m / block_size)).

Workloads (sizes and index rules):

=========== = ===== ===== == = === == ==== ===== ==================================
name        B M=N   H     G  D bs  T  sigma rule
=========== = ===== ===== == = === == ==== ===== ==================================
tiny_bs32   1  1024 16    2  64 32  4  1.0 {c} + 3 random from [0, c)
m8k_bs64    1  8192 64    8 128 64  16 1.0 {0, c} + 14 random from [1, c)
m64k_bs64   1 65536 64    8 128 64  16 1.0 {0, c-1, c} + 13 random from [1, c-1)
m32k_bs32   2 32768 32    4 128 32  32 1.5 {0, c-1, c} + 29 random from [1, c-1)
dense_m16k  1 16384 64    8 128 64 256 1.0 every block of [0, c]
dense_m64k  1 65536 64    8 128 64 1024 1.0 every block of [0, c]
m16k_bs64   1 16384 64    8 128 64  16 1.0 as m64k_bs64 (profiling size)
=========== = ===== ===== == = === == ==== ===== ==================================

Here c = floor(m / bs) is the query's own (diagonal) block. A row whose
causal prefix holds no more than T blocks lists all of them. Random picks are
uniform without replacement (Floyd's subset sampling). "sigma" is the standard
deviation of the normal draws for Q, K and V, which are then rounded to fp16
(round to nearest even).

Seeds: Q, K and V are tensors 0, 1, 2 of ``SeedSequence([seed, tensor])``
(numpy PCG64, filled in 4 Mi-element chunks with one spawned stream each);
the index picks come from ``Generator(PCG64(seed + 1000))``.
"""

from __future__ import annotations

import dataclasses
from typing import Optional

import numpy as np

__all__ = [
    "Workload",
    "WORKLOADS",
    "workload",
    "default_seed",
    "make_qkv",
    "make_block_indices",
    "make_inputs",
    "dense_causal_indices",
    "dense_causal_indices_torch",
]


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    B: int
    M: int
    N: int
    H: int
    G: int
    D: int
    block_size: int
    T: int
    sigma: float
    rule: str  # "local" | "first_local" | "first_two_local" | "all_causal"

    @property
    def heads_per_group(self) -> int:
        return self.H // self.G

    @property
    def scale(self) -> float:
        return 1.0 / float(np.sqrt(self.D))

    def replace(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


WORKLOADS = {
    "tiny_bs32": Workload("tiny_bs32", 1, 1024, 1024, 16, 2, 64, 32, 4, 1.0, "local"),
    "m8k_bs64": Workload("m8k_bs64", 1, 8192, 8192, 64, 8, 128, 64, 16, 1.0, "first_local"),
    "m64k_bs64": Workload("m64k_bs64", 1, 65536, 65536, 64, 8, 128, 64, 16, 1.0,
                          "first_two_local"),
    "m32k_bs32": Workload("m32k_bs32", 2, 32768, 32768, 32, 4, 128, 32, 32, 1.5,
                          "first_two_local"),
    "dense_m16k": Workload("dense_m16k", 1, 16384, 16384, 64, 8, 128, 64, 256, 1.0,
                           "all_causal"),
    "dense_m64k": Workload("dense_m64k", 1, 65536, 65536, 64, 8, 128, 64, 1024, 1.0,
                           "all_causal"),
    # m64k_bs64 cut to 16k queries: same row rule, ~0.9 GB on the device
    "m16k_bs64": Workload("m16k_bs64", 1, 16384, 16384, 64, 8, 128, 64, 16, 1.0,
                          "first_two_local"),
}

# Order of the parity workloads; position i seeds with 20260000 + i.
_SEED_ORDER = ["tiny_bs32", "m8k_bs64", "m64k_bs64", "m32k_bs32", "dense_m16k"]


def workload(name: str) -> Workload:
    return WORKLOADS[name]


def default_seed(name: str) -> int:
    if name in _SEED_ORDER:
        return 20260000 + _SEED_ORDER.index(name)
    return 20260000 + 100 + sorted(WORKLOADS).index(name)


_CHUNK = 1 << 22  # elements per independently seeded stream


def _normal_fp16(seed: int, tensor_id: int, shape, sigma: float) -> np.ndarray:
    return _normal(seed, tensor_id, shape, sigma, np.float16)


def _normal_f32(seed: int, tensor_id: int, shape, sigma: float) -> np.ndarray:
    return _normal(seed, tensor_id, shape, sigma, np.float32)


def _normal(seed: int, tensor_id: int, shape, sigma: float, dtype) -> np.ndarray:
    """normal(0, sigma) float32 draws stored as ``dtype`` (float16: rounded to
    nearest even), filled in fixed-size chunks.

    Chunk i uses ``PCG64(SeedSequence([seed, tensor_id]).spawn(...)[i])``, so
    the values depend only on (seed, tensor_id, shape), never on how many
    threads fill them.
    """
    n = int(np.prod(shape))
    out = np.empty(n, dtype=dtype)
    nchunks = (n + _CHUNK - 1) // _CHUNK
    children = np.random.SeedSequence([seed, tensor_id]).spawn(nchunks)

    def fill(i: int) -> None:
        lo, hi = i * _CHUNK, min(n, (i + 1) * _CHUNK)
        x = np.random.Generator(np.random.PCG64(children[i])).standard_normal(
            hi - lo, dtype=np.float32)
        if sigma != 1.0:
            x *= np.float32(sigma)
        out[lo:hi] = x  # float32 -> float16 rounds to nearest even

    if nchunks <= 1:
        for i in range(nchunks):
            fill(i)
    else:
        import concurrent.futures as cf
        import os

        with cf.ThreadPoolExecutor(max_workers=min(nchunks, os.cpu_count() or 1)) as ex:
            list(ex.map(fill, range(nchunks)))
    return out.reshape(shape)


def make_qkv(w: Workload, seed: int, dtype: str = "f16"):
    """Q [B,M,H,D], K and V [B,N,G,D], normal(0, sigma) then RNE.

    dtype "f16": float16 arrays. dtype "bf16": float32 arrays whose values
    are bfloat16 numbers (the same float32 draws rounded to nearest-even
    bfloat16 by torch), ready for ``torch.from_numpy(a).bfloat16()``.
    """
    if dtype == "f16":
        return (
            _normal_fp16(seed, 0, (w.B, w.M, w.H, w.D), w.sigma),
            _normal_fp16(seed, 1, (w.B, w.N, w.G, w.D), w.sigma),
            _normal_fp16(seed, 2, (w.B, w.N, w.G, w.D), w.sigma),
        )
    if dtype != "bf16":
        raise ValueError(dtype)
    import torch

    return tuple(
        torch.from_numpy(_normal_f32(seed, i, shape, w.sigma)).bfloat16().float().numpy()
        for i, shape in enumerate([(w.B, w.M, w.H, w.D), (w.B, w.N, w.G, w.D),
                                   (w.B, w.N, w.G, w.D)]))


def _floyd_subsets(rng: np.random.Generator, pool: np.ndarray, k: int) -> np.ndarray:
    """k distinct uniform picks from [0, pool[r]) for every row r (pool >= k).

    Floyd's algorithm: for i = n-k .. n-1 draw t uniform in [0, i]; keep t
    unless already taken, in which case keep i. Vectorised over rows.
    """
    rows = pool.shape[0]
    out = np.empty((rows, k), dtype=np.int64)
    for j in range(k):
        i = pool - k + j
        t = rng.integers(0, i + 1)
        if j:
            taken = (out[:, :j] == t[:, None]).any(axis=1)
            t = np.where(taken, i, t)
        out[:, j] = t
    return out


def make_block_indices(w: Workload, seed: int) -> np.ndarray:
    """block_indices int32 [B, M, G, T].

    Each (b, m, g) row holds distinct causal block ids sorted ascending and
    padded with -1 at the end; see the module docstring for the rules.
    """
    bs, T = w.block_size, w.T
    ms = np.arange(w.M, dtype=np.int64)
    nrows = w.B * ms.shape[0] * w.G
    # row order: b, m, g
    c = np.broadcast_to(ms[None, :, None] // bs, (w.B, ms.shape[0], w.G)).reshape(-1)
    out = np.full((nrows, T), -1, dtype=np.int32)

    full = (c + 1) <= T
    if full.any():
        tt = np.arange(T, dtype=np.int64)[None, :]
        cf = c[full][:, None]
        out[full] = np.where(tt <= cf, tt, -1).astype(np.int32)
    if w.rule == "all_causal":
        if not full.all():
            raise ValueError(f"{w.name}: T={T} cannot list every causal block")
        return out.reshape(w.B, ms.shape[0], w.G, T)

    rng = np.random.Generator(np.random.PCG64(seed + 1000))
    sel = ~full
    cs = c[sel]
    if w.rule == "local":
        fixed = [cs]
        lo, hi = np.zeros_like(cs), cs
    elif w.rule == "first_local":
        fixed = [np.zeros_like(cs), cs]
        lo, hi = np.ones_like(cs), cs
    elif w.rule == "first_two_local":
        fixed = [np.zeros_like(cs), cs - 1, cs]
        lo, hi = np.ones_like(cs), cs - 1
    else:
        raise ValueError(f"unknown index rule {w.rule!r}")
    k = T - len(fixed)
    picks = _floyd_subsets(rng, hi - lo, k) + lo[:, None]
    rows = np.concatenate([np.stack(fixed, axis=1), picks], axis=1)
    rows.sort(axis=1)
    out[sel] = rows.astype(np.int32)
    return out.reshape(w.B, ms.shape[0], w.G, T)


def make_inputs(w: Workload, seed: Optional[int] = None):
    """(Q, K, V, block_indices) as numpy arrays for workload ``w``."""
    if seed is None:
        seed = default_seed(w.name)
    q, k, v = make_qkv(w, seed)
    idx = make_block_indices(w, seed)
    return q, k, v, idx


def dense_causal_indices(B: int, M: int, G: int, T: int, block_size: int) -> np.ndarray:
    """Index rows listing every causal block 0..floor(m/bs), -1 padded."""
    c = np.arange(M, dtype=np.int64) // block_size
    if (c[-1] + 1 if M else 0) > T:
        raise ValueError("T too small to list every causal block")
    tt = np.arange(T, dtype=np.int64)
    rows = np.where(tt[None, :] <= c[:, None], tt[None, :], -1).astype(np.int32)
    return np.ascontiguousarray(np.broadcast_to(rows[None, :, None, :], (B, M, G, T)))


def dense_causal_indices_torch(B: int, M: int, G: int, T: int, block_size: int, device):
    """Same rows as :func:`dense_causal_indices`, built directly on ``device``."""
    import torch

    c = torch.arange(M, device=device, dtype=torch.int64) // block_size
    if M and int(c[-1].item()) + 1 > T:
        raise ValueError("T too small to list every causal block")
    tt = torch.arange(T, device=device, dtype=torch.int64)
    rows = torch.where(tt[None, :] <= c[:, None], tt[None, :], torch.full_like(tt[None, :], -1))
    return rows.to(torch.int32)[None, :, None, :].expand(B, M, G, T).contiguous()


def make_block_scores(B: int, M: int, G: int, nblk: int, seed: int) -> np.ndarray:
    """Block scores [B, M, G, nblk] for top-k selection: i.i.d. uniform [0, 1)
    float32 (with the initial and local blocks forced, a top-k over them
    picks the other blocks of a row uniformly, as the index rules do)."""
    n = B * M * G * nblk
    out = np.empty(n, dtype=np.float32)
    nchunks = (n + _CHUNK - 1) // _CHUNK
    children = np.random.SeedSequence([seed, 7]).spawn(max(nchunks, 1))
    for i in range(nchunks):
        lo, hi = i * _CHUNK, min(n, (i + 1) * _CHUNK)
        out[lo:hi] = np.random.Generator(np.random.PCG64(children[i])).random(
            hi - lo, dtype=np.float32)
    return out.reshape(B, M, G, nblk)


def make_block_scores_torch(B: int, M: int, G: int, nblk: int, seed: int, device):
    """The same kind of scores drawn on the device by torch (for sizes too
    large to draw on the host quickly); seeded, not equal to the host draw."""
    import torch

    g = torch.Generator(device=device).manual_seed(seed)
    return torch.rand((B, M, G, nblk), generator=g, device=device, dtype=torch.float32)
