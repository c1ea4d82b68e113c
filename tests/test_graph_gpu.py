"""The forward and backward inside CUDA graphs: both entry points allocate
nothing and only enqueue kernels on the caller's stream, so a captured call
replays with new inputs copied into the captured buffers and gives, bit for
bit, what an eager call on those inputs gives."""
import numpy as np
import pytest
import torch

import blocked_online_softmax_gb300 as bos
from blocked_online_softmax_gb300.workloads import make_qkv

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()
    torch.cuda.set_device(0)


@pytest.mark.parametrize("d,causal", [(128, True), (64, False), (256, True)])
def test_forward_graph_replays_match_eager(d, causal):
    B, H, N = 2, 3, 700
    scale = float(np.float32(d ** -0.5))
    sq, sk, sv = (t.cuda() for t in make_qkv(B, H, N, d, seed=500))
    so = torch.empty_like(sq)
    sl = torch.empty((B, H, N), dtype=torch.float32, device="cuda")
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):   # first call outside the capture: one-time set-up
        bos.attn_fwd(sq, sk, sv, so, sl, B, H, N, d, scale, causal, s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        bos.attn_fwd(sq, sk, sv, so, sl, B, H, N, d, scale, causal, s)
    for seed in (501, 502, 503):
        q, k, v = (t.cuda() for t in make_qkv(B, H, N, d, seed=seed))
        sq.copy_(q), sk.copy_(k), sv.copy_(v)
        g.replay()
        torch.cuda.synchronize()
        o, lse = bos.attention(q, k, v, scale=scale, causal=causal)
        torch.cuda.synchronize()
        assert torch.equal(so, o) and torch.equal(sl, lse), f"replay with seed {seed} differs from eager"


def test_backward_graph_replay_matches_eager():
    B, H, N, d = 1, 2, 500, 128
    scale = float(np.float32(d ** -0.5))
    q, k, v = (t.cuda() for t in make_qkv(B, H, N, d, seed=510))
    dout = torch.randn(q.shape, generator=torch.Generator().manual_seed(511)).to(torch.bfloat16).cuda()
    o, lse = bos.attention(q, k, v, scale=scale, causal=True)
    grads_eager = bos.attention_backward(q, k, v, o, lse, dout, scale=scale, causal=True)
    torch.cuda.synchronize()
    nbytes = bos.attn_bwd_workspace_bytes(B, H, N, d)
    ws = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        bos.attn_bwd(q, k, v, o, dout, lse, None, dq, dk, dv, ws, nbytes, B, H, N, d, scale, True, s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        bos.attn_bwd(q, k, v, o, dout, lse, None, dq, dk, dv, ws, nbytes, B, H, N, d, scale, True, s)
    g.replay()
    torch.cuda.synchronize()
    # dK and dV are deterministic; dQ is summed by reductions in no fixed order
    assert torch.equal(dk, grads_eager[1]) and torch.equal(dv, grads_eager[2])
    err = (dq.float() - grads_eager[0].float()).abs().max().item()
    assert err <= 1e-2 * grads_eager[0].float().abs().max().item()
