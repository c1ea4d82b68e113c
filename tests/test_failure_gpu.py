"""Failure detection without a GPU fault: every wait inside the kernel is bounded.

The test hook makes the MMA thread wait on a barrier that nothing signals (a
flag nothing sets). With a 20 ms wait limit the wait runs out; the kernel must
record ATTN_ERR_TIMEOUT, drain its own copies and MMAs, free tensor memory and
return. The host reads the status and the context stays usable.
"""
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


def _run(q, k, v, scale, causal):
    B, H, N, d = q.shape
    o = torch.empty_like(q)
    lse = torch.empty((B, H, N), dtype=torch.float32, device=q.device)
    bos.attn_fwd(q, k, v, o, lse, B, H, N, d, scale, causal)
    return o, lse


def test_status_ok_after_normal_runs():
    q, k, v = (t.cuda() for t in make_qkv(1, 2, 300, 128, seed=21))
    assert bos.attn_device_status() == bos.ATTN_OK
    _run(q, k, v, 0.088, True)
    assert bos.attn_device_status() == bos.ATTN_OK


@pytest.mark.parametrize("d,causal", [(64, False), (128, True), (256, True), (192, False)])
def test_wait_timeout_is_reported_and_context_survives(d, causal):
    qh, kh, vh = make_qkv(2, 8, 1024, d, seed=22)
    q, k, v = (t.cuda() for t in (qh, kh, vh))
    assert bos.attn_device_status() == bos.ATTN_OK
    bos.attn_set_wait_limit_ns(20_000_000)          # 20 ms
    bos.attn_set_test_stall(True)
    try:
        _run(q, k, v, 0.1, causal)
        status = bos.attn_device_status()
    finally:
        bos.attn_set_test_stall(False)
        bos.attn_set_wait_limit_ns(0)
    assert status == bos.ATTN_ERR_TIMEOUT
    assert bos.attn_device_status() == bos.ATTN_OK  # read clears it
    # the context is still usable and the next launch is correct
    o, lse = _run(q, k, v, 0.1, causal)
    assert bos.attn_device_status() == bos.ATTN_OK
    o_ref, lse_ref = oracle.attention(qh, kh, vh, float(np.float32(0.1)), causal)
    assert_parity(o.float().cpu().numpy(), lse.cpu().numpy(), o_ref, lse_ref, "after timeout")


@pytest.mark.parametrize("d,causal", [(64, False), (128, True)])
def test_backward_wait_timeout_is_reported_and_context_survives(d, causal):
    """The same hook on attn_bwd: its S/dV issuer waits on a barrier nothing
    signals, every role gives up after the limit (the other MMA thread, the
    producer and the dQ warps with work in flight drain it first), the status
    reads ATTN_ERR_TIMEOUT, and the next backward is correct."""
    qh, kh, vh = make_qkv(1, 4, 700, d, seed=23)
    gh = torch.randn(qh.shape, generator=torch.Generator().manual_seed(24)).to(torch.bfloat16)
    q, k, v, g = (t.cuda() for t in (qh, kh, vh, gh))
    scale = float(np.float32(d ** -0.5))
    o, lse = bos.attention(q, k, v, scale=scale, causal=causal)
    torch.cuda.synchronize()
    assert bos.attn_device_status() == bos.ATTN_OK
    bos.attn_set_wait_limit_ns(20_000_000)          # 20 ms
    bos.attn_set_test_stall(True)
    try:
        bos.attention_backward(q, k, v, o, lse, g, scale=scale, causal=causal)
        status = bos.attn_device_status()
    finally:
        bos.attn_set_test_stall(False)
        bos.attn_set_wait_limit_ns(0)
    assert status == bos.ATTN_ERR_TIMEOUT
    assert bos.attn_device_status() == bos.ATTN_OK
    grads = bos.attention_backward(q, k, v, o, lse, g, scale=scale, causal=causal)
    torch.cuda.synchronize()
    assert bos.attn_device_status() == bos.ATTN_OK
    for name, gpu, ref in zip(("dq", "dk", "dv"), grads, oracle.attention_bwd(qh, kh, vh, gh, scale, causal)):
        err = np.abs(gpu.float().cpu().numpy() - ref).max()
        assert err <= 2e-2 * np.abs(ref).max() + 1e-3, f"{name}: {err}"


@pytest.mark.parametrize("d,causal", [(64, False), (128, True), (256, False)])
def test_busy_counter_slot_is_reported_not_shared(d, causal):
    """A launch whose work-counter slot is still held by another launch takes no
    work units and records ATTN_ERR_SCHED_BUSY (it never shares the other
    launch's counter). The hook marks the slot as held; no wait is involved.
    The outputs stay untouched, and the next launch on a free slot is correct."""
    qh, kh, vh = make_qkv(2, 8, 1024, d, seed=25)
    q, k, v = (t.cuda() for t in (qh, kh, vh))
    assert bos.attn_device_status() == bos.ATTN_OK
    o = torch.full_like(q, -12288.0)
    lse = torch.full((2, 8, 1024), -7.0e30, dtype=torch.float32, device=q.device)
    bos.attn_set_test_sched_busy(True)
    try:
        bos.attn_fwd(q, k, v, o, lse, 2, 8, 1024, d, 0.1, causal)
        status = bos.attn_device_status()
    finally:
        bos.attn_set_test_sched_busy(False)
    assert status == bos.ATTN_ERR_SCHED_BUSY
    assert torch.all(o == -12288.0) and torch.all(lse == -7.0e30), "a launch without its slot wrote output"
    o, lse = _run(q, k, v, 0.1, causal)
    assert bos.attn_device_status() == bos.ATTN_OK
    o_ref, lse_ref = oracle.attention(qh, kh, vh, float(np.float32(0.1)), causal)
    assert_parity(o.float().cpu().numpy(), lse.cpu().numpy(), o_ref, lse_ref, "after a busy slot")
