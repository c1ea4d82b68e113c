"""A torch.library operator over the C ABI: ``torch.ops.bos.attention_fwd``.

Importing this module registers the operator, so the kernel can sit inside
torch programs (fake-tensor shape propagation, graph capture) with no compute
on the torch side: the operator's CUDA implementation only allocates O and LSE
and marshals the arguments into ``attn_fwd`` on torch's current stream; its
fake implementation only states the output shapes. There is no CPU
implementation (the library has no CPU path), and no autograd formula is
registered: this is the forward pass only, so differentiating through it
raises.

    import blocked_online_softmax_gb300.torch_op
    o, lse = torch.ops.bos.attention_fwd(q, k, v, scale, causal)
"""
from __future__ import annotations

import torch

from . import attention as _attention


@torch.library.custom_op("bos::attention_fwd", mutates_args=(), device_types="cuda")
def attention_fwd(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, scale: float,
                  causal: bool) -> tuple[torch.Tensor, torch.Tensor]:
    """O (bf16 [B,H,N,d]) and LSE (fp32 [B,H,N], natural log) of softmax(scale q k^T [causal]) v."""
    return _attention(q, k, v, scale=scale, causal=causal)


@attention_fwd.register_fake
def _attention_fwd_fake(q, k, v, scale, causal):
    if q.dim() != 4 or q.shape != k.shape or q.shape != v.shape:
        raise ValueError("q, k, v must be [B,H,N,d] with one shape")
    B, H, N, _ = q.shape
    return torch.empty_like(q), q.new_empty((B, H, N), dtype=torch.float32)
