"""NSA selection-attention forward for GB300 (sm_103a).

Public API (GPU only; the CUDA library must be built):

* :func:`sel_attn_fwd` -- O [B,M,H,D] and LSE [B,H,M] fp32 from fp16 or
  bf16 Q [B,M,H,D], K/V [B,N,G,D] and int32 block_indices [B,M,G,T];
* :func:`sel_attn_bwd` -- dQ, dK, dV from dO and the forward's O and LSE;
* :func:`topk_blocks` -- block_indices from per-block scores (top-k with
  forced initial and local blocks);
* :func:`sel_attn_fwd_shared` -- the same forward in two passes: the blocks
  common to a tile of 16 consecutive queries are gathered once per tile;
* :func:`sel_attn_fwd_host` -- the forward with host buffers in and out;
* :func:`swa_fwd` -- GQA sliding-window (or dense) attention forward on the
  tcgen05 tensor cores.

The C ABI is declared in ``include/nsa_sel_attn.h``; ``inputs`` draws the
seeded synthetic workloads.
"""

from ._lib import (NsaError, load, sel_attn_bwd, sel_attn_fwd, sel_attn_fwd_host,  # noqa: F401
                   sel_attn_fwd_shared, status_string, swa_fwd, topk_blocks)

__all__ = ["sel_attn_fwd", "sel_attn_fwd_shared", "sel_attn_bwd", "sel_attn_fwd_host",
           "topk_blocks", "swa_fwd", "load", "status_string", "NsaError"]
