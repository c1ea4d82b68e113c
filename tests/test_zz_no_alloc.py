"""attn_fwd_host_noalloc: the host-buffer entry point that allocates no device memory.

Some callers cannot allocate device memory where they need attention (another
framework's caching allocator owns the device, or the thread must not take the
synchronisation an allocation can bring). For them the library stages Q, K, V,
O and LSE through one fixed device array instead of per-call allocations.

This test calls that entry point through the C ABI, twice in a row for each of
several shapes (head dims 64, 96, 128 and 256, causal and not), and checks

* each result against the fp64 oracle, within the parity tolerances used
  everywhere else;
* each result byte for byte against the allocating host entry point
  (attn_fwd_host): the same kernel on the same inputs gives the same bits;
* that the second round of calls changes neither the device's free memory
  (cudaMemGetInfo) nor torch's allocated bytes, i.e. the call allocates
  nothing. The first round loads the library's modules and kernels, which
  takes device memory once.

It lives in its own file, collected last, and passes alone in a fresh process
as well as after the other tests.
"""
import ctypes
import gc

import numpy as np
import pytest
import torch

import blocked_online_softmax_gb300 as bos
import oracle
from blocked_online_softmax_gb300.workloads import make_qkv
from parity_util import assert_parity

pytestmark = pytest.mark.gpu

CASES = [((2, 4, 777, 128), True, 11), ((1, 3, 300, 64), False, 12), ((1, 2, 333, 256), True, 13),
         ((2, 1, 200, 96), False, 14)]


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
    """One call of a host-buffer entry point; returns O's raw bf16 bits and LSE."""
    B, H, N, d = q.shape
    qh, kh, vh = _host(q), _host(k), _host(v)
    o = np.zeros((B, H, N, d), dtype=np.uint16)
    lse = np.zeros((B, H, N), dtype=np.float32)
    st = fn(qh.ctypes.data, kh.ctypes.data, vh.ctypes.data, o.ctypes.data, lse.ctypes.data,
            B, H, N, d, ctypes.c_float(scale), int(causal), None)
    assert st == bos.ATTN_OK, bos.attn_status_string(st)
    return o, lse


def _widen(o_bits):
    return (o_bits.astype(np.uint32) << 16).view(np.float32)


def test_noalloc_matches_oracle_and_allocating_entry_twice(lib):
    inputs, refs = [], []
    for (B, H, N, d), causal, seed in CASES:
        q, k, v = make_qkv(B, H, N, d, seed=seed)
        scale = float(np.float32(d ** -0.5))
        inputs.append((q, k, v, scale, causal))
        refs.append((_call(lib.attn_fwd_host, q, k, v, scale, causal), oracle.attention(q, k, v, scale, causal)))
    torch.cuda.synchronize()

    def one_round():
        for (q, k, v, scale, causal), ((o_host, lse_host), (o_ref, lse_ref)) in zip(inputs, refs):
            o, lse = _call(lib.attn_fwd_host_noalloc, q, k, v, scale, causal)
            what = f"noalloc {tuple(q.shape)} causal={causal}"
            assert_parity(_widen(o), lse, o_ref, lse_ref, what)
            assert np.array_equal(o, o_host), f"{what}: O differs from attn_fwd_host"
            assert np.array_equal(lse.view(np.uint32), lse_host.view(np.uint32)), \
                f"{what}: LSE differs from attn_fwd_host"

    one_round()                       # loads the modules and kernels it needs (once per process)
    # Python's collector could free tensors of earlier tests in the middle of the
    # measurement; keep it out of the measured calls
    gc.collect()
    gc.disable()
    try:
        torch.cuda.synchronize()
        free0, _ = torch.cuda.mem_get_info()
        alloc0 = torch.cuda.memory_allocated()
        one_round()                   # the same calls again: nothing may be allocated now
        torch.cuda.synchronize()
        free1, _ = torch.cuda.mem_get_info()
        alloc1 = torch.cuda.memory_allocated()
    finally:
        gc.enable()
    assert free1 == free0, f"free device memory moved by {free0 - free1} bytes across no-alloc calls"
    assert alloc1 == alloc0, f"torch's allocated bytes moved by {alloc1 - alloc0} across no-alloc calls"


def test_noalloc_rejects_problems_beyond_its_scratch(lib):
    dummy = np.zeros(16, dtype=np.uint16)
    p = dummy.ctypes.data
    # 64 heads x 8192 rows x 128 dims of bf16 = 128 MiB per tensor > 64 MiB of scratch
    st = lib.attn_fwd_host_noalloc(p, p, p, p, p, 4, 16, 8192, 128, ctypes.c_float(0.1), 0, None)
    assert st == bos.ATTN_ERR_TOO_LARGE
    assert "noalloc" in bos.attn_status_string(st)
    # the argument checks of attn_fwd_host come first, in its order
    assert lib.attn_fwd_host_noalloc(p, p, p, p, p, 1, 1, 16, 100, ctypes.c_float(0.1), 0, None) == \
        bos.ATTN_ERR_UNSUPPORTED_D
    assert lib.attn_fwd_host_noalloc(p, p, p, p, p, 1 << 22, 1 << 22, 1 << 20, 128, ctypes.c_float(0.1), 0,
                                     None) == bos.ATTN_ERR_BAD_SHAPE
