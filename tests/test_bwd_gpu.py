"""GPU parity of the backward pass (attn_bwd) against the fp64 oracle.

The GPU backward takes its own forward's O (bf16) and LSE, as a training step
would; the oracle recomputes everything in fp64 from q, k, v and dO.
Tolerance, per gradient tensor: max |g - g_ref| <= 2e-2 * max |g_ref| + 1e-3.
The outputs are bf16 (a rounding of 2^-9 relative), P and dS enter the tensor
cores as bf16 (2^-9 relative per term), and D comes from the bf16 O; with
accumulation in fp32 the expected error is a few parts in 10^3 of the
largest gradient, and the bound leaves a margin of several times that.
"""
import numpy as np
import pytest
import torch

import blocked_online_softmax_gb300 as bos
import oracle
from blocked_online_softmax_gb300.workloads import make_qkv

pytestmark = pytest.mark.gpu

SENT = -12288.0


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()
    oracle.build()
    torch.cuda.set_device(0)


def grads_gpu(q, k, v, g, scale, causal, dlse=None):
    B, H, N, d = q.shape
    dev = torch.device("cuda")
    qd, kd, vd, gd = (t.to(dev) for t in (q, k, v, g))
    dl = None if dlse is None else dlse.to(dev).contiguous()
    o = torch.empty_like(qd)
    lse = torch.empty(B, H, N, dtype=torch.float32, device=dev)
    bos.attn_fwd(qd, kd, vd, o, lse, B, H, N, d, scale, causal, None)
    n = B * H * N * d
    outs = []
    for _ in range(3):   # dq, dk, dv with sentinels after the last element
        buf = torch.full((n + 64,), SENT, dtype=torch.bfloat16, device=dev)
        outs.append(buf)
    nbytes = bos.attn_bwd_workspace_bytes(B, H, N, d)
    ws = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    bos.attn_bwd(qd, kd, vd, o, gd, lse, dl, outs[0], outs[1], outs[2], ws, nbytes, B, H, N, d, scale, causal, None)
    torch.cuda.synchronize()
    res = []
    for buf in outs:
        h = buf.float().cpu()
        assert torch.all(h[n:] == SENT), "wrote past the gradient tensor"
        res.append(h[:n].view(B, H, N, d).numpy().astype(np.float64))
    return res


def check(gpu, ref, what):
    for name, a, b in zip(("dq", "dk", "dv"), gpu, ref):
        bound = 2e-2 * np.abs(b).max() + 1e-3
        err = np.abs(a - b).max()
        assert err <= bound, f"{what} {name}: max err {err:.3e} > {bound:.3e} (max |ref| {np.abs(b).max():.3e})"


def dout_like(q, seed):
    g = torch.Generator().manual_seed(seed)
    return torch.randn(q.shape, generator=g).to(torch.bfloat16)


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("d", [64, 128, 80])
@pytest.mark.parametrize("N", [1, 64, 128, 129, 300])
def test_backward_small(N, d, causal):
    q, k, v = make_qkv(1, 2, N, d, seed=500 + N + d)
    g = dout_like(q, 600 + N + d)
    scale = float(np.float32(d ** -0.5))
    gpu = grads_gpu(q, k, v, g, scale, causal)
    ref = oracle.attention_bwd(q, k, v, g, scale, causal)
    check(gpu, ref, f"N={N} d={d} causal={causal}")


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("d", [8, 40, 104])
def test_backward_other_head_dims(d, causal):
    """Head dims below each kernel width: partial dQ boxes and zero-filled columns."""
    q, k, v = make_qkv(1, 2, 300, d, seed=700 + d)
    g = dout_like(q, 800 + d)
    scale = float(np.float32(d ** -0.5))
    gpu = grads_gpu(q, k, v, g, scale, causal)
    ref = oracle.attention_bwd(q, k, v, g, scale, causal)
    check(gpu, ref, f"d={d} causal={causal}")


@pytest.mark.parametrize("causal", [False, True])
def test_backward_several_blocks(causal):
    q, k, v = make_qkv(2, 3, 700, 128, seed=71)
    g = dout_like(q, 72)
    gpu = grads_gpu(q, k, v, g, 0.0883883, causal)
    ref = oracle.attention_bwd(q, k, v, g, float(np.float32(0.0883883)), causal)
    check(gpu, ref, f"B2H3N700 causal={causal}")


def test_backward_large_logits():
    q, k, v = make_qkv(1, 2, 400, 64, seed=73, logit_mult=4.0)
    g = dout_like(q, 74)
    gpu = grads_gpu(q, k, v, g, 0.125, True)
    ref = oracle.attention_bwd(q, k, v, g, 0.125, True)
    check(gpu, ref, "x4 logits")


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("d", [64, 128])
def test_backward_lse_gradient(d, causal):
    """A gradient on the LSE output as well: the kernel takes D - dLSE."""
    q, k, v = make_qkv(1, 2, 333, d, seed=80 + d)
    g = dout_like(q, 81)
    gl = torch.randn(1, 2, 333, generator=torch.Generator().manual_seed(82), dtype=torch.float32)
    scale = float(np.float32(d ** -0.5))
    gpu = grads_gpu(q, k, v, g, scale, causal, dlse=gl)
    ref = oracle.attention_bwd(q, k, v, g, scale, causal, dlse=gl.numpy())
    check(gpu, ref, f"dlse d={d} causal={causal}")


@pytest.mark.parametrize("d,causal", [(64, False), (128, True), (32, True), (120, False)])
def test_backward_long(d, causal):
    """Many query blocks per key block: both Q/dO stages and LSE buffers are reused many times."""
    q, k, v = make_qkv(1, 1, 2000, d, seed=90 + d)
    g = dout_like(q, 91)
    scale = float(np.float32(d ** -0.5))
    gpu = grads_gpu(q, k, v, g, scale, causal)
    ref = oracle.attention_bwd(q, k, v, g, scale, causal)
    check(gpu, ref, f"N=2000 d={d} causal={causal}")


def test_backward_full_size_sampled_head():
    """The 8K causal workload (B=2, H=16, N=8192, d=128) in one call; one head
    (b=1, h=9) checked in full against the oracle, every other gradient finite."""
    from blocked_online_softmax_gb300.workloads import CAUSAL_8K as w
    B, H, N, d = w.B, w.H, w.N, w.d
    q, k, v = make_qkv(B, H, N, d, w.seed)
    g = dout_like(q, 97)
    dq, dk, dv = grads_gpu(q, k, v, g, w.scale, True)
    for t in (dq, dk, dv):
        assert np.isfinite(t).all()
    b, h = 1, 9
    sl = (slice(b, b + 1), slice(h, h + 1))
    ref = oracle.attention_bwd(q[sl], k[sl], v[sl], g[sl], w.scale, True)
    check([t[sl] for t in (dq, dk, dv)], ref, "B2H16N8192 head (1, 9)")


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("scale", [0.0, -0.2])
def test_backward_zero_and_negative_scale(scale, causal):
    """Scale 0 (uniform attention over the valid keys) and a negative scale,
    with a ragged tail: the masked blocks must still drop the invalid keys."""
    q, k, v = make_qkv(1, 2, 300, 128, seed=85)
    g = dout_like(q, 86)
    gpu = grads_gpu(q, k, v, g, scale, causal)
    ref = oracle.attention_bwd(q, k, v, g, scale, causal)
    check(gpu, ref, f"scale={scale} causal={causal}")
