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
    for code in range(0, 12):
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
    (dict(d=136), bos.ATTN_ERR_UNSUPPORTED_D), (dict(d=4), bos.ATTN_ERR_UNSUPPORTED_D),
    (dict(scale=float("nan")), bos.ATTN_ERR_BAD_SCALE), (dict(scale=float("inf")), bos.ATTN_ERR_BAD_SCALE),
    (dict(causal=2), bos.ATTN_ERR_BAD_ARG),
    (dict(q=17), bos.ATTN_ERR_MISALIGNED), (dict(o=72), bos.ATTN_ERR_MISALIGNED),
    (dict(lse=82), bos.ATTN_ERR_MISALIGNED),
])
def test_host_validation_before_any_launch(lib, kw, code):
    assert _call(lib, **kw) == code


def test_host_entry_validation(lib):
    st = lib.attn_fwd_host(None, 8, 8, 8, 8, 1, 1, 4, 64, ctypes.c_float(1.0), 0, None)
    assert st == bos.ATTN_ERR_NULLPTR
    st = lib.attn_fwd_host(8, 8, 8, 8, 8, 1, 1, 4, 81, ctypes.c_float(1.0), 0, None)
    assert st == bos.ATTN_ERR_UNSUPPORTED_D


def test_binding_raises_on_error(lib):
    with pytest.raises(bos.AttnError) as ei:
        bos.attn_fwd(0, 16, 16, 16, 16, 1, 1, 8, 64, 0.1, 0, stream=0)
    assert ei.value.status == bos.ATTN_ERR_NULLPTR
