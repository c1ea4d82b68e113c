"""torch.library operators over the C ABI: ``torch.ops.bos.attention_fwd`` and
``torch.ops.bos.attention_bwd``, with an autograd formula joining them.

Importing this module registers the operators, so the kernels can sit inside
torch programs (fake-tensor shape propagation, graph capture, autograd) with
no compute on the torch side: each CUDA implementation only allocates its
outputs (and the backward's workspace) and marshals the arguments into
``attn_fwd`` / ``attn_bwd`` on torch's current stream; the fake
implementations only state the output shapes. There is no CPU implementation
(the library has no CPU path).

The forward accepts strided q, k, v (head dim contiguous); O comes back
contiguous. Autograd: the forward saves q, k, v and its outputs O and LSE;
the backward passes dL/dO and, when the loss also uses LSE, dL/dLSE to
``attn_bwd`` (the derivative of LSE_i in the score S_ij is P_ij, which the
kernel folds into its row term D). ``scale`` and ``causal`` get no gradient.

    import blocked_online_softmax_gb300.torch_op
    o, lse = torch.ops.bos.attention_fwd(q, k, v, scale, causal)
"""
from __future__ import annotations

from typing import Optional

import torch

from . import attention as _attention
from . import attention_backward as _attention_backward


@torch.library.custom_op("bos::attention_fwd", mutates_args=(), device_types="cuda")
def attention_fwd(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, scale: float,
                  causal: bool) -> tuple[torch.Tensor, torch.Tensor]:
    """O ([B,H,N,d], q's dtype: bf16 or fp16) and LSE (fp32 [B,H,N], natural log) of softmax(scale q k^T [causal]) v."""
    return _attention(q, k, v, scale=scale, causal=causal)


@attention_fwd.register_fake
def _attention_fwd_fake(q, k, v, scale, causal):
    if q.dim() != 4 or q.shape != k.shape or q.shape != v.shape:
        raise ValueError("q, k, v must be [B,H,N,d] with one shape")
    B, H, N, _ = q.shape
    return torch.empty(q.shape, dtype=q.dtype, device=q.device), q.new_empty((B, H, N), dtype=torch.float32)


@torch.library.custom_op("bos::attention_bwd", mutates_args=(), device_types="cuda")
def attention_bwd(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, o: torch.Tensor, lse: torch.Tensor,
                  dout: torch.Tensor, dlse: Optional[torch.Tensor], scale: float,
                  causal: bool) -> tuple[torch.Tensor, torch.Tensor, torch.Tensor]:
    """dq, dk, dv ([B,H,N,d], q's dtype) for the forward's o, lse and the gradients dout (and dlse, optional)."""
    return _attention_backward(q, k, v, o, lse, dout, scale=scale, causal=causal, dlse=dlse)


@attention_bwd.register_fake
def _attention_bwd_fake(q, k, v, o, lse, dout, dlse, scale, causal):
    return torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)


def _setup_context(ctx, inputs, output):
    q, k, v, scale, causal = inputs
    o, lse = output
    ctx.save_for_backward(q, k, v, o, lse)
    ctx.scale = scale
    ctx.causal = causal


def _backward(ctx, grad_o, grad_lse):
    q, k, v, o, lse = ctx.saved_tensors
    q, k, v = q.contiguous(), k.contiguous(), v.contiguous()   # the backward takes dense [B,H,N,d]
    if grad_o is None:
        grad_o = torch.zeros_like(o)
    grad_o = grad_o.to(q.dtype).contiguous()
    if grad_lse is not None:
        grad_lse = grad_lse.to(torch.float32).contiguous()
    dq, dk, dv = torch.ops.bos.attention_bwd(q, k, v, o, lse, grad_o, grad_lse, ctx.scale, ctx.causal)
    return dq, dk, dv, None, None


attention_fwd.register_autograd(_backward, setup_context=_setup_context)
