"""The torch.library operators over the C ABI, and their autograd formula."""
import numpy as np
import pytest
import torch

import blocked_online_softmax_gb300.torch_op  # noqa: F401  (registers torch.ops.bos.attention_fwd)


def test_operator_registered():
    assert hasattr(torch.ops.bos, "attention_fwd")
    assert hasattr(torch.ops.bos, "attention_bwd")


def test_fake_tensor_shapes():
    """Shape propagation needs no GPU and runs no kernel."""
    from torch._subclasses.fake_tensor import FakeTensorMode
    with FakeTensorMode():
        q = torch.empty(2, 3, 100, 64, dtype=torch.bfloat16, device="cuda")
        o, lse = torch.ops.bos.attention_fwd(q, q, q, 0.125, True)
        assert o.shape == q.shape and o.dtype == torch.bfloat16
        assert lse.shape == (2, 3, 100) and lse.dtype == torch.float32


def test_meta_backward_shapes():
    """Autograd through the operator on meta tensors: the fake implementations give
    the shapes of both passes, and no kernel runs (the autograd engine needs a
    real CUDA device for fake CUDA tensors, so meta stands in for them here)."""
    q, k, v = (torch.empty(2, 3, 100, 64, dtype=torch.bfloat16, device="meta", requires_grad=True)
               for _ in range(3))
    o, lse = torch.ops.bos.attention_fwd(q, k, v, 0.125, False)
    assert o.shape == q.shape and lse.shape == (2, 3, 100)
    (o.float().sum() + lse.sum()).backward()
    for t in (q, k, v):
        assert t.grad is not None and t.grad.shape == t.shape and t.grad.dtype == torch.bfloat16


def test_no_cpu_implementation():
    x = torch.zeros(1, 1, 4, 8, dtype=torch.bfloat16)
    with pytest.raises(NotImplementedError):
        torch.ops.bos.attention_fwd(x, x, x, 0.1, False)


@pytest.mark.gpu
def test_operator_matches_oracle():
    import __graft_entry__
    import oracle
    from blocked_online_softmax_gb300.workloads import make_qkv
    from parity_util import assert_parity
    __graft_entry__.build()
    q, k, v = make_qkv(2, 3, 333, 128, seed=41)
    scale = float(np.float32(128 ** -0.5))
    o, lse = torch.ops.bos.attention_fwd(q.cuda(), k.cuda(), v.cuda(), scale, True)
    torch.cuda.synchronize()
    o_ref, lse_ref = oracle.attention(q, k, v, scale, True)
    assert_parity(o.float().cpu().numpy(), lse.cpu().numpy(), o_ref, lse_ref, "torch op")


@pytest.mark.gpu
@pytest.mark.parametrize("use_lse", [False, True])
def test_autograd_matches_oracle(use_lse):
    """loss = sum(O * g) [+ sum(LSE * gl)] through torch autograd, against the fp64 oracle's gradients."""
    import __graft_entry__
    import oracle
    from blocked_online_softmax_gb300.workloads import make_qkv
    __graft_entry__.build()
    B, H, N, d = 1, 2, 300, 64
    q, k, v = make_qkv(B, H, N, d, seed=43)
    gen = torch.Generator().manual_seed(44)
    g = torch.randn(q.shape, generator=gen).to(torch.bfloat16)
    gl = torch.randn(B, H, N, generator=gen)
    qd, kd, vd = (t.cuda().requires_grad_(True) for t in (q, k, v))
    o, lse = torch.ops.bos.attention_fwd(qd, kd, vd, 0.125, True)
    loss = (o.float() * g.cuda().float()).sum()
    if use_lse:
        loss = loss + (lse * gl.cuda()).sum()
    loss.backward()
    torch.cuda.synchronize()
    ref = oracle.attention_bwd(q, k, v, g, 0.125, True, dlse=gl.numpy() if use_lse else None)
    for name, t, r in zip(("dq", "dk", "dv"), (qd, kd, vd), ref):
        err = np.abs(t.grad.float().cpu().numpy() - r).max()
        assert err <= 2e-2 * np.abs(r).max() + 1e-3, f"{name}: {err}"


@pytest.mark.gpu
def test_operator_on_transposed_inputs():
    """[B,N,H,d] tensors transposed to [B,H,N,d] go through attn_fwd_strided;
    the gradients (dense, from attn_bwd) match the oracle's."""
    import __graft_entry__
    import oracle
    from blocked_online_softmax_gb300.workloads import make_qkv
    __graft_entry__.build()
    B, H, N, d = 2, 3, 200, 128
    q, k, v = make_qkv(B, H, N, d, seed=45)
    g = torch.randn(q.shape, generator=torch.Generator().manual_seed(46)).to(torch.bfloat16)
    views = [t.permute(0, 2, 1, 3).contiguous().cuda().requires_grad_(True) for t in (q, k, v)]
    qd, kd, vd = (x.permute(0, 2, 1, 3) for x in views)
    o, lse = torch.ops.bos.attention_fwd(qd, kd, vd, float(np.float32(d ** -0.5)), False)
    (o.float() * g.cuda().float()).sum().backward()
    torch.cuda.synchronize()
    o_ref, _ = oracle.attention(q, k, v, float(np.float32(d ** -0.5)), False)
    assert np.abs(o.detach().float().cpu().numpy() - o_ref).max() <= 2e-2
    ref = oracle.attention_bwd(q, k, v, g, float(np.float32(d ** -0.5)), False)
    for name, x, r in zip(("dq", "dk", "dv"), views, ref):
        grad = x.grad.permute(0, 2, 1, 3).float().cpu().numpy()
        err = np.abs(grad - r).max()
        assert err <= 2e-2 * np.abs(r).max() + 1e-3, f"{name}: {err}"


@pytest.mark.gpu
def test_wide_head_dim_forward_and_backward_limit():
    """d = 256 runs forward through the operator; its backward reports the
    backward's head-dim limit (128) instead of computing anything."""
    import oracle
    import blocked_online_softmax_gb300 as bos
    from blocked_online_softmax_gb300.workloads import make_qkv
    from parity_util import assert_parity
    qh, kh, vh = make_qkv(1, 2, 200, 256, seed=88)
    q, k, v = (t.cuda().requires_grad_(True) for t in (qh, kh, vh))
    o, lse = torch.ops.bos.attention_fwd(q, k, v, 0.0625, True)
    o_ref, lse_ref = oracle.attention(qh, kh, vh, 0.0625, True)
    assert_parity(o.detach().float().cpu().numpy(), lse.detach().cpu().numpy(), o_ref, lse_ref, "op d=256")
    with pytest.raises(bos.AttnError) as ei:
        o.float().sum().backward()
    assert ei.value.status == bos.ATTN_ERR_UNSUPPORTED_D
