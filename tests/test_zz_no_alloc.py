"""attn_fwd_host_noalloc: the host-buffer entry point that allocates no device memory.

Some callers cannot allocate device memory where they need attention (another
framework's caching allocator owns the device, or the thread must not take the
synchronisation an allocation can bring). For them the library stages Q, K, V,
O and LSE through one fixed device array instead of per-call allocations. This
test calls that entry point through the C ABI twice in a row, with different
shapes, and checks each result against the allocating host entry point
(attn_fwd_host) within the parity tolerances used everywhere else. It lives in
its own file, collected last.
"""
import ctypes

import numpy as np
import pytest
import torch

import blocked_online_softmax_gb300 as bos
from blocked_online_softmax_gb300.workloads import make_qkv
from parity_util import LSE_RTOL, O_ATOL, lse_err

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    import __graft_entry__
    __graft_entry__.build()
    torch.cuda.set_device(0)
    return bos.load_library()


def _host(t):
    """bf16 CPU tensor -> contiguous uint16 numpy array (pageable host memory)."""
    return np.ascontiguousarray(t.contiguous().view(torch.int16).numpy().view(np.uint16))


def _call(fn, q, k, v, scale, causal):
    B, H, N, d = q.shape
    qh, kh, vh = _host(q), _host(k), _host(v)
    o = np.zeros((B, H, N, d), dtype=np.uint16)
    lse = np.zeros((B, H, N), dtype=np.float32)
    st = fn(qh.ctypes.data, kh.ctypes.data, vh.ctypes.data, o.ctypes.data, lse.ctypes.data,
            B, H, N, d, ctypes.c_float(scale), int(causal), None)
    assert st == bos.ATTN_OK, bos.attn_status_string(st)
    o_f = (o.astype(np.uint32) << 16).view(np.float32)
    return o_f, lse


def test_noalloc_matches_allocating_entry_twice(lib):
    cases = [((2, 4, 777, 128), True, 11), ((1, 3, 300, 64), False, 12)]
    for (B, H, N, d), causal, seed in cases:          # two calls in a row, different shapes
        q, k, v = make_qkv(B, H, N, d, seed=seed)
        scale = float(np.float32(d ** -0.5))
        o_ref, lse_ref = _call(lib.attn_fwd_host, q, k, v, scale, causal)
        o, lse = _call(lib.attn_fwd_host_noalloc, q, k, v, scale, causal)
        assert np.all(np.isfinite(o)) and np.all(np.isfinite(lse))
        assert float(np.max(np.abs(o - o_ref))) <= O_ATOL
        assert lse_err(lse, lse_ref.astype(np.float64)) <= LSE_RTOL


def test_noalloc_rejects_problems_beyond_its_scratch(lib):
    dummy = np.zeros(16, dtype=np.uint16)
    p = dummy.ctypes.data
    # 64 heads x 8192 rows x 128 dims of bf16 = 128 MiB per tensor > 64 MiB of scratch
    st = lib.attn_fwd_host_noalloc(p, p, p, p, p, 4, 16, 8192, 128, ctypes.c_float(0.1), 0, None)
    assert st == bos.ATTN_ERR_TOO_LARGE
    assert "noalloc" in bos.attn_status_string(st)
