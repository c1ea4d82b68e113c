"""The torch.library operator over the C ABI (forward only)."""
import numpy as np
import pytest
import torch

import blocked_online_softmax_gb300.torch_op  # noqa: F401  (registers torch.ops.bos.attention_fwd)


def test_operator_registered():
    assert hasattr(torch.ops.bos, "attention_fwd")


def test_fake_tensor_shapes():
    """Shape propagation needs no GPU and runs no kernel."""
    from torch._subclasses.fake_tensor import FakeTensorMode
    with FakeTensorMode():
        q = torch.empty(2, 3, 100, 64, dtype=torch.bfloat16, device="cuda")
        o, lse = torch.ops.bos.attention_fwd(q, q, q, 0.125, True)
        assert o.shape == q.shape and o.dtype == torch.bfloat16
        assert lse.shape == (2, 3, 100) and lse.dtype == torch.float32


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
