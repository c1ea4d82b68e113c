"""The C-ABI library: it loads, exports every declared symbol, and rejects bad
arguments on the host before touching the GPU (no compute call here)."""
import ctypes
import os
import re

import pytest

import blocked_online_softmax_gb300 as bos
from blocked_online_softmax_gb300 import _build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    _build.build()
    return bos.load_library()


def _declared_functions():
    names = []
    for path in sorted(os.listdir(os.path.join(ROOT, "include"))):
        if not path.endswith(".h"):
            continue
        text = open(os.path.join(ROOT, "include", path)).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        names += re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*((?:attn|softmax)_\w+)\s*\(", text, flags=re.M)
    return names


def test_exports_every_declared_symbol(lib):
    declared = _declared_functions()
    assert set(declared) >= {"attn_fwd", "attn_fwd_host", "attn_fwd_host_noalloc", "attn_device_status",
                             "attn_set_wait_limit_ns", "attn_set_test_stall", "attn_status_string",
                             "attn_abi_version"}
    for name in declared:
        assert hasattr(lib, name), f"{name} declared in include/ but not exported"
    assert set(declared) == set(bos.EXPORTED_SYMBOLS)


def test_status_strings(lib):
    for code in range(0, 13):
        s = bos.attn_status_string(code)
        assert s and s != "unknown status"
    assert bos.attn_status_string(12345) == "unknown status"
    assert bos.attn_abi_version() >= 1


def _call(lib, q=16, k=32, v=48, o=64, lse=80, B=1, H=1, N=8, d=64, scale=0.125, causal=0):
    return lib.attn_fwd(q, k, v, o, lse, B, H, N, d, ctypes.c_float(scale), causal, None)


@pytest.mark.parametrize("kw,code", [
    (dict(q=0), bos.ATTN_ERR_NULLPTR), (dict(lse=0), bos.ATTN_ERR_NULLPTR),
    (dict(B=0), bos.ATTN_ERR_BAD_SHAPE), (dict(H=-1), bos.ATTN_ERR_BAD_SHAPE),
    (dict(N=0), bos.ATTN_ERR_BAD_SHAPE), (dict(B=1 << 20, H=1 << 20), bos.ATTN_ERR_BAD_SHAPE),
    (dict(d=60), bos.ATTN_ERR_UNSUPPORTED_D), (dict(d=0), bos.ATTN_ERR_UNSUPPORTED_D),
    (dict(d=264), bos.ATTN_ERR_UNSUPPORTED_D), (dict(d=4), bos.ATTN_ERR_UNSUPPORTED_D),
    (dict(d=260), bos.ATTN_ERR_UNSUPPORTED_D),
    (dict(scale=float("nan")), bos.ATTN_ERR_BAD_SCALE), (dict(scale=float("inf")), bos.ATTN_ERR_BAD_SCALE),
    (dict(causal=2), bos.ATTN_ERR_BAD_ARG),
    (dict(q=17), bos.ATTN_ERR_MISALIGNED), (dict(o=72), bos.ATTN_ERR_MISALIGNED),
    (dict(lse=82), bos.ATTN_ERR_MISALIGNED),
])
def test_host_validation_before_any_launch(lib, kw, code):
    assert _call(lib, **kw) == code


@pytest.mark.parametrize("d", [8, 64, 72, 128, 136, 200, 256])
def test_head_dims_pass_validation(lib, d):
    """Every multiple of 8 up to 256 gets past the host checks (here the call
    then fails only for want of a GPU)."""
    st = _call(lib, d=d)
    assert st not in (bos.ATTN_ERR_UNSUPPORTED_D, bos.ATTN_ERR_BAD_ARG, bos.ATTN_ERR_BAD_SHAPE)


def test_backward_head_dims_stop_at_128(lib):
    lib.attn_bwd_workspace_bytes.restype = ctypes.c_size_t
    assert lib.attn_bwd_workspace_bytes(1, 2, 300, 128) > 0
    assert lib.attn_bwd_workspace_bytes(1, 2, 300, 136) == 0
    assert lib.attn_bwd_workspace_bytes(1, 2, 300, 256) == 0


def _call_strided(lib, qs=(8 * 64, 8 * 64, 64), os_=(8 * 64, 8 * 64, 64), B=1, H=1, N=8, d=64, null=None):
    arrs = [(ctypes.c_longlong * 3)(*st) for st in (qs, qs, qs, os_)]
    ptrs = [ctypes.addressof(a) for a in arrs]
    if null is not None:
        ptrs[null] = None
    return lib.attn_fwd_strided(16, 32, 48, 64, 80, B, H, N, d, *ptrs, ctypes.c_float(0.125), 0, None)


@pytest.mark.parametrize("kw,code", [
    (dict(null=0), bos.ATTN_ERR_NULLPTR), (dict(null=3), bos.ATTN_ERR_NULLPTR),
    (dict(qs=(512, 512, 60)), bos.ATTN_ERR_BAD_ARG),          # row stride not a multiple of 8
    (dict(qs=(512, 0, 64)), bos.ATTN_ERR_BAD_ARG),            # zero stride
    (dict(qs=(512, 512, 56)), bos.ATTN_ERR_BAD_ARG),          # rows overlap in the head dim
    (dict(os_=(512, 512, 56)), bos.ATTN_ERR_BAD_ARG),         # output rows overlap
    (dict(os_=(64, 64, 8), B=2, H=2, N=8, d=8), bos.ATTN_ERR_BAD_ARG),   # output (b, h) planes overlap
    (dict(qs=(1 << 40, 512, 64)), bos.ATTN_ERR_BAD_ARG),      # past the TMA stride range
])
def test_strided_validation(lib, kw, code):
    assert _call_strided(lib, **kw) == code


def test_strided_accepts_transposed_layouts(lib):
    """[B, N, H, d] viewed as [B, H, N, d]: rows H*d apart, heads d apart. With
    valid strides the call only fails for want of a GPU, after validation."""
    B, H, N, d = 2, 4, 8, 64
    bnhd = (N * H * d, d, H * d)
    st = _call_strided(lib, qs=bnhd, os_=bnhd, B=B, H=H, N=N, d=d)
    assert st not in (bos.ATTN_ERR_BAD_ARG, bos.ATTN_ERR_NULLPTR, bos.ATTN_ERR_MISALIGNED)


def test_host_entry_validation(lib):
    st = lib.attn_fwd_host(None, 8, 8, 8, 8, 1, 1, 4, 64, ctypes.c_float(1.0), 0, None)
    assert st == bos.ATTN_ERR_NULLPTR
    st = lib.attn_fwd_host(8, 8, 8, 8, 8, 1, 1, 4, 81, ctypes.c_float(1.0), 0, None)
    assert st == bos.ATTN_ERR_UNSUPPORTED_D


def test_binding_raises_on_error(lib):
    with pytest.raises(bos.AttnError) as ei:
        bos.attn_fwd(0, 16, 16, 16, 16, 1, 1, 8, 64, 0.1, 0, stream=0)
    assert ei.value.status == bos.ATTN_ERR_NULLPTR


def test_fwd_ex_validation(lib):
    """attn_fwd_ex: unknown dtype and bad strides are refused on the host; NULL
    strides mean dense tensors, so a valid call fails only for want of a GPU."""
    def call(dtype=0, qs=None):
        arr = None if qs is None else (ctypes.c_longlong * 3)(*qs)
        ptr = None if arr is None else ctypes.addressof(arr)
        return lib.attn_fwd_ex(16, 32, 48, 64, 80, 1, 1, 8, 64, ptr, None, None, None, ctypes.c_float(0.125), 0,
                               dtype, None)
    assert call(dtype=2) == bos.ATTN_ERR_BAD_ARG
    assert call(dtype=-1) == bos.ATTN_ERR_BAD_ARG
    assert call(qs=(512, 512, 60)) == bos.ATTN_ERR_BAD_ARG
    for dt in (bos.ATTN_DTYPE_BF16, bos.ATTN_DTYPE_F16):
        assert call(dtype=dt) not in (bos.ATTN_ERR_BAD_ARG, bos.ATTN_ERR_NULLPTR, bos.ATTN_ERR_MISALIGNED)
