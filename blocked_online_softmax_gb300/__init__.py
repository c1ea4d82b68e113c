"""Python binding of the GB300 attention-forward library (ctypes over the C ABI).

Argument marshalling only: every step of the computation runs in the CUDA
library ``libbos_attn.so`` built from ``csrc/`` (see ``include/attn.h`` for the
contract). There is no CPU or PyTorch fallback: if the library is missing or
the GPU is not sm_103a, the calls raise.

Names follow the C ABI: ``attn_fwd``, ``attn_fwd_host``, ``attn_status_string``,
``softmax_rows_fwd``. ``attention`` and ``softmax`` are conveniences that
allocate their outputs with torch (device memory only) and call the C entry.
"""
from __future__ import annotations

import ctypes
import math
import os

from . import workloads  # noqa: F401  (seeded inputs; no attention arithmetic)

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libbos_attn.so")

# status codes, mirrored from include/attn.h
ATTN_OK = 0
ATTN_ERR_NULLPTR = 1
ATTN_ERR_BAD_SHAPE = 2
ATTN_ERR_UNSUPPORTED_D = 3
ATTN_ERR_BAD_SCALE = 4
ATTN_ERR_MISALIGNED = 5
ATTN_ERR_UNSUPPORTED_DEVICE = 6
ATTN_ERR_LAUNCH = 7
ATTN_ERR_TIMEOUT = 8
ATTN_ERR_CUDA = 9
ATTN_ERR_BAD_ARG = 10
ATTN_ERR_TOO_LARGE = 11
ATTN_ERR_SCHED_BUSY = 12

# every symbol include/attn.h declares
EXPORTED_SYMBOLS = ("attn_fwd", "attn_fwd_host", "attn_fwd_host_noalloc", "attn_device_status",
                    "attn_set_wait_limit_ns", "attn_set_test_stall", "attn_status_string", "attn_abi_version",
                    "softmax_rows_fwd", "attn_bwd", "attn_bwd_workspace_bytes", "attn_fwd_strided", "attn_fwd_ex", "attn_bwd_ex",
                    "attn_set_test_sched_busy")

_lib = None


class AttnError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = int(status)
        super().__init__(f"{where}: status {status}: {attn_status_string(status)}")


def load_library(path: str = LIB_PATH):
    """Load the CUDA library; raises if it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(f"CUDA library not built ({path} missing): run "
                           "`python -c 'import __graft_entry__ as g; g.build()'` first")
    lib = ctypes.CDLL(path)
    vp, i, f = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
    for name in ("attn_fwd", "attn_fwd_host", "attn_fwd_host_noalloc"):
        fn = getattr(lib, name)
        fn.restype = i
        fn.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, f, i, vp]
    lib.attn_device_status.restype = i
    lib.attn_device_status.argtypes = [vp]
    lib.attn_set_wait_limit_ns.restype = i
    lib.attn_set_wait_limit_ns.argtypes = [ctypes.c_ulonglong]
    lib.attn_set_test_stall.restype = i
    lib.attn_set_test_stall.argtypes = [i]
    lib.attn_set_test_sched_busy.restype = i
    lib.attn_set_test_sched_busy.argtypes = [i]
    lib.attn_status_string.restype = ctypes.c_char_p
    lib.attn_status_string.argtypes = [i]
    lib.attn_abi_version.restype = i
    lib.attn_abi_version.argtypes = []
    lib.softmax_rows_fwd.restype = i
    lib.softmax_rows_fwd.argtypes = [vp, vp, i, i, ctypes.c_longlong, ctypes.c_longlong, vp]
    lib.attn_bwd.restype = i
    lib.attn_bwd.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, ctypes.c_size_t, i, i, i, i, f, i, vp]
    lib.attn_fwd_strided.restype = i
    lib.attn_fwd_strided.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, vp, vp, vp, vp, f, i, vp]
    lib.attn_fwd_ex.restype = i
    lib.attn_fwd_ex.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, vp, vp, vp, vp, f, i, i, vp]
    lib.attn_bwd_ex.restype = i
    lib.attn_bwd_ex.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, ctypes.c_size_t, i, i, i, i, f, i, i, vp]
    lib.attn_bwd_workspace_bytes.restype = ctypes.c_size_t
    lib.attn_bwd_workspace_bytes.argtypes = [i, i, i, i]
    _lib = lib
    return lib


def attn_status_string(status: int) -> str:
    return load_library().attn_status_string(int(status)).decode()


def attn_abi_version() -> int:
    return int(load_library().attn_abi_version())


def _ptr(x) -> int:
    if x is None:
        return 0
    if isinstance(x, int):
        return x
    if hasattr(x, "data_ptr"):
        return int(x.data_ptr())
    if hasattr(x, "ctypes"):           # numpy array
        return int(x.ctypes.data)
    raise TypeError(f"cannot take a pointer from {type(x)!r}")


def _stream_handle(stream) -> int:
    if stream is None:
        import torch
        return int(torch.cuda.current_stream().cuda_stream)
    if isinstance(stream, int):
        return stream
    return int(stream.cuda_stream)


def attn_fwd(q, k, v, o, lse, B: int, H: int, N: int, d: int, scale: float, causal,
             stream=None) -> None:
    """Enqueue the forward kernel (C ``attn_fwd``); raises AttnError on a nonzero status.

    q, k, v, o: bf16 device tensors (or raw device pointers), contiguous [B,H,N,d];
    lse: fp32 device tensor [B,H,N]; stream: torch stream, raw handle, or None
    for torch's current stream.
    """
    st = load_library().attn_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), int(B), int(H),
                                 int(N), int(d), float(scale), int(causal), _stream_handle(stream))
    if st != ATTN_OK:
        raise AttnError(st, "attn_fwd")


def attn_fwd_strided(q, k, v, o, lse, B: int, H: int, N: int, d: int, q_strides, k_strides, v_strides,
                     o_strides, scale: float, causal, stream=None) -> None:
    """Enqueue the forward kernel on strided q, k, v, o (C ``attn_fwd_strided``).

    Each ``*_strides`` is three element strides (batch, head, row); the head dim
    is contiguous. Raises AttnError on a nonzero status.
    """
    arrs = [(ctypes.c_longlong * 3)(*[int(x) for x in st]) for st in (q_strides, k_strides, v_strides, o_strides)]
    st = load_library().attn_fwd_strided(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), int(B), int(H), int(N),
                                         int(d), *[ctypes.addressof(a) for a in arrs], float(scale), int(causal),
                                         _stream_handle(stream))
    if st != ATTN_OK:
        raise AttnError(st, "attn_fwd_strided")


ATTN_DTYPE_BF16 = 0
ATTN_DTYPE_F16 = 1


def attn_fwd_ex(q, k, v, o, lse, B: int, H: int, N: int, d: int, q_strides, k_strides, v_strides, o_strides,
                scale: float, causal, dtype: int, stream=None) -> None:
    """Enqueue the forward kernel for bf16 or fp16 tensors (C ``attn_fwd_ex``).

    ``dtype`` is ATTN_DTYPE_BF16 or ATTN_DTYPE_F16; each ``*_strides`` is three
    element strides (batch, head, row) or None for a dense tensor. Raises
    AttnError on a nonzero status.
    """
    arrs = [None if st is None else (ctypes.c_longlong * 3)(*[int(x) for x in st])
            for st in (q_strides, k_strides, v_strides, o_strides)]
    ptrs = [None if a is None else ctypes.addressof(a) for a in arrs]
    st = load_library().attn_fwd_ex(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), int(B), int(H), int(N), int(d),
                                    *ptrs, float(scale), int(causal), int(dtype), _stream_handle(stream))
    if st != ATTN_OK:
        raise AttnError(st, "attn_fwd_ex")


def attn_fwd_host(q_h, k_h, v_h, o_h, lse_h, B: int, H: int, N: int, d: int, scale: float,
                  causal, stream=None) -> None:
    """Host-buffer entry (C ``attn_fwd_host``): copies in, runs, copies out, synchronises."""
    st = load_library().attn_fwd_host(_ptr(q_h), _ptr(k_h), _ptr(v_h), _ptr(o_h), _ptr(lse_h),
                                      int(B), int(H), int(N), int(d), float(scale), int(causal),
                                      _stream_handle(stream))
    if st != ATTN_OK:
        raise AttnError(st, "attn_fwd_host")


def attn_fwd_host_noalloc(q_h, k_h, v_h, o_h, lse_h, B: int, H: int, N: int, d: int, scale: float,
                          causal, stream=None) -> None:
    """Host-buffer entry that allocates no device memory (C ``attn_fwd_host_noalloc``).

    For callers that cannot allocate device memory at the call site: staging goes
    through one fixed device array shared by all calls, so calls must not overlap
    on the GPU. Raises AttnError (ATTN_ERR_TOO_LARGE past the array's size).
    """
    st = load_library().attn_fwd_host_noalloc(_ptr(q_h), _ptr(k_h), _ptr(v_h), _ptr(o_h), _ptr(lse_h),
                                              int(B), int(H), int(N), int(d), float(scale), int(causal),
                                              _stream_handle(stream))
    if st != ATTN_OK:
        raise AttnError(st, "attn_fwd_host_noalloc")


def attn_device_status(stream=None) -> int:
    """Synchronise the stream, return and clear the kernel's sticky status word (C ``attn_device_status``)."""
    return int(load_library().attn_device_status(_stream_handle(stream)))


def attn_set_wait_limit_ns(ns: int) -> None:
    """Wall-time limit of each wait inside the kernel (0 = default 2 s)."""
    load_library().attn_set_wait_limit_ns(int(ns))


def attn_set_test_stall(on: bool) -> None:
    """Test hook: make every launch's MMA thread wait on a barrier nothing signals."""
    load_library().attn_set_test_stall(int(bool(on)))


def attn_set_test_sched_busy(on: bool) -> None:
    """Test hook: mark each forward launch's work-counter slot as held by another launch."""
    load_library().attn_set_test_sched_busy(int(bool(on)))


def attn_bwd_workspace_bytes(B: int, H: int, N: int, d: int) -> int:
    """Device workspace bytes ``attn_bwd`` needs (C ``attn_bwd_workspace_bytes``)."""
    return int(load_library().attn_bwd_workspace_bytes(int(B), int(H), int(N), int(d)))


def attn_bwd(q, k, v, o, dout, lse, dlse, dq, dk, dv, workspace, workspace_bytes: int, B: int, H: int, N: int,
             d: int, scale: float, causal, stream=None) -> None:
    """Enqueue the backward pass (C ``attn_bwd``; dlse may be None); raises AttnError on a nonzero status."""
    st = load_library().attn_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(dout), _ptr(lse), _ptr(dlse), _ptr(dq),
                                 _ptr(dk),
                                 _ptr(dv), _ptr(workspace), int(workspace_bytes), int(B), int(H), int(N), int(d),
                                 float(scale), int(causal), _stream_handle(stream))
    if st != ATTN_OK:
        raise AttnError(st, "attn_bwd")


def attention_backward(q, k, v, o, lse, dout, scale: float | None = None, causal: bool = False, stream=None,
                       dlse=None):
    """dq, dk, dv (q's dtype: bf16 or fp16) for the attention() forward outputs o, lse and the gradients
    dout (and dlse, optional)."""
    import torch
    B, H, N, d = q.shape
    if q.dtype not in (torch.bfloat16, torch.float16):
        raise ValueError("q, k, v, o, dout must be bf16 or fp16")
    for t in (q, k, v, o, dout):
        if t.shape != q.shape or t.dtype != q.dtype or not t.is_contiguous():
            raise ValueError("q, k, v, o, dout must be contiguous tensors of one dtype and one [B,H,N,d] shape")
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    nbytes = attn_bwd_workspace_bytes(B, H, N, d)
    ws = torch.empty(nbytes, dtype=torch.uint8, device=q.device)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    if dlse is not None:
        if dlse.dtype != torch.float32 or not dlse.is_contiguous() or tuple(dlse.shape) != (B, H, N):
            raise ValueError("dlse must be a contiguous fp32 [B,H,N] tensor")
    if q.dtype == torch.float16:
        st = load_library().attn_bwd_ex(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(dout), _ptr(lse), _ptr(dlse),
                                        _ptr(dq), _ptr(dk), _ptr(dv), _ptr(ws), int(nbytes), int(B), int(H), int(N),
                                        int(d), float(scale), int(causal), ATTN_DTYPE_F16, _stream_handle(stream))
        if st != ATTN_OK:
            raise AttnError(st, "attn_bwd_ex")
    else:
        attn_bwd(q, k, v, o, dout, lse, dlse, dq, dk, dv, ws, nbytes, B, H, N, d, scale, causal, stream)
    return dq, dk, dv


def softmax_rows_fwd(x, y, rows: int, cols: int, x_row_stride: int, y_row_stride: int, stream=None) -> None:
    """Row softmax of an fp32 device matrix (C ``softmax_rows_fwd``); strides in elements."""
    lib = load_library()
    st = lib.softmax_rows_fwd(_ptr(x), _ptr(y), int(rows), int(cols), int(x_row_stride), int(y_row_stride),
                              _stream_handle(stream))
    if st != ATTN_OK:
        raise AttnError(st, "softmax_rows_fwd")


def softmax(x, out=None, stream=None):
    """Softmax over the last dimension of a 2-D fp32 CUDA tensor (rows may be strided)."""
    import torch
    if x.dim() != 2 or x.dtype != torch.float32 or not x.is_cuda or x.stride(1) != 1:
        raise ValueError("x must be a 2-D fp32 CUDA tensor with unit column stride")
    if out is None:
        out = torch.empty_like(x, memory_format=torch.contiguous_format)
    softmax_rows_fwd(x, out, x.shape[0], x.shape[1], x.stride(0), out.stride(0), stream)
    return out


def attention(q, k, v, scale: float | None = None, causal: bool = False, stream=None, out=None):
    """O, LSE for bf16 or fp16 CUDA tensors [B,H,N,d]; scale defaults to 1/sqrt(d) rounded to fp32.

    q, k, v (and ``out``, an optional preallocated O) may be strided views, e.g.
    [B,N,H,d] tensors transposed to [B,H,N,d], as long as the head dim is
    contiguous and the other strides are multiples of 8 elements; O is
    allocated contiguous unless ``out`` is given.
    """
    import torch
    if q.dim() != 4 or q.shape != k.shape or q.shape != v.shape:
        raise ValueError("q, k, v must be [B,H,N,d] with one shape")
    if q.dtype not in (torch.bfloat16, torch.float16):
        raise ValueError("q, k, v must be bf16 or fp16 CUDA tensors")
    for t in (q, k, v):
        if t.dtype != q.dtype or not t.is_cuda:
            raise ValueError("q, k, v must be CUDA tensors of one dtype (bf16 or fp16)")
    B, H, N, d = q.shape
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    o = torch.empty_like(q, memory_format=torch.contiguous_format) if out is None else out
    if o.shape != q.shape or o.dtype != q.dtype:
        raise ValueError("out must be a tensor shaped like q, of q's dtype")
    lse = torch.empty((B, H, N), dtype=torch.float32, device=q.device)
    if q.dtype == torch.float16:
        for t in (q, k, v, o):
            if t.stride(3) != 1:
                raise ValueError("the head dim (last) of q, k, v and out must be contiguous")
        attn_fwd_ex(q, k, v, o, lse, B, H, N, d, *[t.stride()[:3] for t in (q, k, v, o)], scale, causal,
                    ATTN_DTYPE_F16, stream)
    elif all(t.is_contiguous() for t in (q, k, v, o)):
        attn_fwd(q, k, v, o, lse, B, H, N, d, scale, causal, stream)
    else:
        for t in (q, k, v, o):
            if t.stride(3) != 1:
                raise ValueError("the head dim (last) of q, k, v and out must be contiguous")
        attn_fwd_strided(q, k, v, o, lse, B, H, N, d, *[t.stride()[:3] for t in (q, k, v, o)], scale, causal,
                         stream)
    return o, lse
