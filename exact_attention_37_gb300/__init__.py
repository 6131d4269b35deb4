"""Exact scaled-dot-product attention for GB300 (sm_103a): fused forward with online
softmax and a key-block-parallel backward, behind a small C ABI.

    import exact_attention_37_gb300 as fa
    o, lse = fa.forward(q, k, v, causal=True)          # q: [B, H, N_q, d], k, v: [B, H_kv, N_k, d]
    dq, dk, dv = fa.backward(q, k, v, o, lse, dout, causal=True)

H_kv may be smaller than H (grouped-query / multi-query attention) and N_k may
differ from N_q (the causal mask is then aligned at the bottom right).

``forward``/``backward`` allocate their outputs with torch and call the C ABI;
``fa_fwd``/``fa_bwd`` take caller-owned outputs.  All compute runs in the
library's CUDA kernels; there is no CPU fallback.
"""
from __future__ import annotations

import math

from ._lib import (  # noqa: F401
    FA_BF16,
    FA_FP16,
    FaError,
    fa_bwd,
    fa_profile_begin,
    fa_profile_end,
    fa_bwd_workspace_size,
    fa_check_device_status,
    fa_fwd,
    fa_fwd_bwd_host,
    fa_fwd_host,
    fa_cta_head_group,
    fa_host_chunk_plan,
    fa_host_scratch_size,
    fa_status_string,
    fa_version,
    load,
)

__all__ = ["forward", "backward", "fa_fwd", "fa_bwd", "fa_bwd_workspace_size", "fa_check_device_status",
           "fa_fwd_host", "fa_fwd_bwd_host", "fa_host_scratch_size", "fa_host_chunk_plan", "fa_cta_head_group",
           "FaError", "load"]


def _default_scale(d: int) -> float:
    return 1.0 / math.sqrt(d)


def forward(q, k, v, scale: float | None = None, causal: bool = False, stream=None):
    """Returns (O, L): O like q, L fp32 [B, H, N]."""
    import torch

    B, H, N, d = q.shape
    o = torch.empty_like(q)
    lse = torch.empty((B, H, N), dtype=torch.float32, device=q.device)
    fa_fwd(q, k, v, o, lse, _default_scale(d) if scale is None else scale, causal, stream)
    return o, lse


def backward(q, k, v, o, lse, dout, scale: float | None = None, causal: bool = False, stream=None, workspace=None):
    """Returns (dQ, dK, dV) like q, k, v.  ``workspace`` (uint8 CUDA tensor) is allocated if not given."""
    import torch

    B, H, N, d = q.shape
    dq = torch.empty_like(q)
    dk = torch.empty_like(k)
    dv = torch.empty_like(v)
    if workspace is None:
        workspace = torch.empty(max(1, fa_bwd_workspace_size(B, H, N, d)), dtype=torch.uint8, device=q.device)
    fa_bwd(q, k, v, o, dout, lse, dq, dk, dv, workspace, _default_scale(d) if scale is None else scale, causal,
           stream)
    return dq, dk, dv
