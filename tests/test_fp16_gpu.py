"""fp16 inputs (the pages' examples call their kernels on fp16 tensors): the
same kernels with fp16 operands on the tensor cores, against the fp64 oracle
on the same fp16 values (widened exactly). O is fp16, LSE fp32; the
tolerances are those of the bf16 path (fp16 rounds O more finely)."""
import numpy as np
import pytest
import torch

import blocked_online_softmax_gb300 as bos
import oracle
from blocked_online_softmax_gb300.workloads import make_qkv
from parity_util import assert_parity

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()
    torch.cuda.set_device(0)


def _check(q, k, v, scale, causal, what, layout=None):
    qd, kd, vd = (t.cuda() for t in (q, k, v))
    if layout == "bnhd":
        qd, kd, vd = (t.permute(0, 2, 1, 3).contiguous().permute(0, 2, 1, 3) for t in (qd, kd, vd))
    o, lse = bos.attention(qd, kd, vd, scale=scale, causal=causal)
    torch.cuda.synchronize()
    assert o.dtype == torch.float16
    o_ref, lse_ref = oracle.attention(q.double(), k.double(), v.double(), scale, causal)
    assert_parity(o.float().cpu().numpy(), lse.cpu().numpy(), o_ref, lse_ref, what)


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("d", [40, 64, 128, 200, 256])
@pytest.mark.parametrize("N", [1, 300, 1000])
def test_fp16_against_oracle(N, d, causal):
    q, k, v = make_qkv(2, 2, N, d, seed=600 + N + d, dtype=torch.float16)
    _check(q, k, v, float(np.float32(d ** -0.5)), causal, f"fp16 N={N} d={d} causal={causal}")


@pytest.mark.parametrize("d", [64, 128, 256])
def test_fp16_large_logits_and_strided(d):
    q, k, v = make_qkv(1, 3, 700, d, seed=650 + d, logit_mult=4.0, dtype=torch.float16)
    _check(q, k, v, 0.125, True, f"fp16 x4 d={d}", layout="bnhd")


def test_fp16_many_units_full_compare():
    q, k, v = make_qkv(2, 40, 900, 128, seed=660, dtype=torch.float16)
    _check(q, k, v, float(np.float32(128 ** -0.5)), True, "fp16 80 heads N=900")


def test_fp16_operator_forward():
    import blocked_online_softmax_gb300.torch_op  # noqa: F401
    q, k, v = make_qkv(1, 2, 333, 128, seed=670, dtype=torch.float16)
    o, lse = torch.ops.bos.attention_fwd(q.cuda(), k.cuda(), v.cuda(), 0.0884, False)
    torch.cuda.synchronize()
    o_ref, lse_ref = oracle.attention(q.double(), k.double(), v.double(), 0.0884, False)
    assert_parity(o.float().cpu().numpy(), lse.cpu().numpy(), o_ref, lse_ref, "fp16 operator")


@pytest.mark.parametrize("d,causal,N", [(64, False, 300), (128, True, 700), (40, True, 129), (128, False, 1000)])
def test_fp16_backward_against_oracle(d, causal, N):
    q, k, v = make_qkv(1, 2, N, d, seed=690 + d + N, dtype=torch.float16)
    g = torch.randn(q.shape, generator=torch.Generator().manual_seed(691)).to(torch.float16)
    scale = float(np.float32(d ** -0.5))
    qd, kd, vd, gd = (t.cuda() for t in (q, k, v, g))
    o, lse = bos.attention(qd, kd, vd, scale=scale, causal=causal)
    grads = bos.attention_backward(qd, kd, vd, o, lse, gd, scale=scale, causal=causal)
    torch.cuda.synchronize()
    refs = oracle.attention_bwd(q, k, v, g, scale, causal)
    for name, gpu, ref in zip(("dq", "dk", "dv"), grads, refs):
        assert gpu.dtype == torch.float16
        err = float(np.max(np.abs(gpu.float().cpu().numpy() - ref)))
        bound = 2e-2 * float(np.max(np.abs(ref))) + 1e-3
        assert err <= bound, f"fp16 {name} d={d} causal={causal} N={N}: {err:.3g} > {bound:.3g}"


def test_fp16_autograd_through_operator():
    import blocked_online_softmax_gb300.torch_op  # noqa: F401
    q, k, v = make_qkv(1, 2, 300, 64, seed=695, dtype=torch.float16)
    qd, kd, vd = (t.cuda().requires_grad_(True) for t in (q, k, v))
    o, lse = torch.ops.bos.attention_fwd(qd, kd, vd, 0.125, True)
    o.float().sum().backward()
    g = torch.ones(q.shape, dtype=torch.float16)
    refs = oracle.attention_bwd(q, k, v, g, 0.125, True)
    for name, gpu, ref in zip(("dq", "dk", "dv"), (qd.grad, kd.grad, vd.grad), refs):
        err = float(np.max(np.abs(gpu.float().cpu().numpy() - ref)))
        assert err <= 2e-2 * float(np.max(np.abs(ref))) + 1e-3, name
