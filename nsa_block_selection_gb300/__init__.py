"""NSA selection-attention forward for GB300 (sm_103a).

Public API (GPU only; the CUDA library must be built):

* :func:`sel_attn_fwd` -- O [B,M,H,D] fp32 and LSE [B,H,M] fp32 from fp16
  Q [B,M,H,D], K/V [B,N,G,D] and int32 block_indices [B,M,G,T].

The C ABI is declared in ``include/nsa_sel_attn.h``; ``inputs`` draws the
seeded synthetic workloads.
"""

from ._lib import NsaError, load, sel_attn_fwd, status_string  # noqa: F401

__all__ = ["sel_attn_fwd", "load", "status_string", "NsaError"]
