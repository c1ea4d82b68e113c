"""fp64 CPU oracle for the attention forward pass (test infrastructure).

Only the test suite, ``__graft_entry__.smoke()`` and the bench's CPU-baseline
leg may import this package. The product path is the CUDA library in
``blocked_online_softmax_gb300``; it shares no code with this oracle and never
calls it.

The arithmetic lives in ``attn_oracle.c`` (plain C, fp64, OpenMP over rows).
It follows the plain definition that the blocked online softmax reaches exactly
("4.4 Writing GPU Kernels with Triton", Kernel 4 "A Simplified FlashAttention":
the streamed output equals a full softmax-then-matmul), with the three-pass
stable softmax of Kernel 2 "Fused Softmax" on the same page.

Every function here is pinned by the CPU tests (closed forms, invariants, the
page's worked exercise, brute force in extended precision); none is "parity
unpinned".
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "attn_oracle.c")
_LIB = os.path.join(_HERE, "liboracle_attn.so")
_lib = None


def build(force: bool = False) -> str:
    """Compile attn_oracle.c with gcc (-O2, OpenMP, no fast-math) in place."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c11",
               "-o", tmp, _SRC, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        i64p = ctypes.POINTER(ctypes.c_int64)
        dp = ctypes.POINTER(ctypes.c_double)
        for name in ("oracle_attn_fwd_bf16", "oracle_attn_fwd_f64"):
            fn = getattr(lib, name)
            fn.restype = ctypes.c_int
            fn.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                           ctypes.c_int, ctypes.c_int, ctypes.c_int64, ctypes.c_int,
                           ctypes.c_double, ctypes.c_int, i64p, ctypes.c_int64,
                           dp, dp, ctypes.c_int]
        lib.oracle_softmax_row_f64.restype = ctypes.c_double
        lib.oracle_softmax_row_f64.argtypes = [dp, ctypes.c_int64, dp]
        lib.oracle_max_threads.restype = ctypes.c_int
        lib.oracle_max_threads.argtypes = []
        _lib = lib
    return _lib


def _as_host_array(x):
    """bf16 torch tensor -> uint16 bit array; numpy uint16 / float64 pass through."""
    if isinstance(x, np.ndarray):
        if x.dtype not in (np.uint16, np.float64):
            raise TypeError("oracle inputs are bf16 bit patterns (uint16) or float64")
        return np.ascontiguousarray(x)
    import torch
    if x.dtype == torch.bfloat16:
        return np.ascontiguousarray(x.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16))
    if x.dtype == torch.float64:
        return np.ascontiguousarray(x.detach().cpu().numpy())
    raise TypeError(f"unsupported oracle input dtype {x.dtype}")


def max_threads() -> int:
    return int(_load().oracle_max_threads())


def attention(q, k, v, scale: float, causal: bool, rows=None, nthreads: int = 0):
    """O and LSE in fp64 for inputs shaped [B,H,N,d].

    ``q``, ``k``, ``v``: bf16 torch tensors, uint16 bf16 bit arrays, or float64
    arrays (all three the same kind). ``scale`` is used as given (pass the fp32
    value the CUDA library receives). ``rows`` (optional) is a sequence of
    flattened row ids ``(b*H + h)*N + i``; then O is [len(rows), d] and LSE is
    [len(rows)], else O is [B,H,N,d] and LSE [B,H,N].
    """
    qa, ka, va = (_as_host_array(t) for t in (q, k, v))
    if not (qa.dtype == ka.dtype == va.dtype):
        raise TypeError("q, k, v must share one input kind")
    if qa.ndim != 4 or qa.shape != ka.shape or qa.shape != va.shape:
        raise ValueError("q, k, v must all be [B,H,N,d] with one shape")
    B, H, N, d = qa.shape
    lib = _load()
    if rows is None:
        nrows = B * H * N
        rows_ptr = None
        o = np.empty((B, H, N, d), dtype=np.float64)
        lse = np.empty((B, H, N), dtype=np.float64)
    else:
        rows_arr = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
        nrows = rows_arr.size
        rows_ptr = rows_arr.ctypes.data_as(ctypes.POINTER(ctypes.c_int64))
        o = np.empty((nrows, d), dtype=np.float64)
        lse = np.empty((nrows,), dtype=np.float64)
    fn = lib.oracle_attn_fwd_bf16 if qa.dtype == np.uint16 else lib.oracle_attn_fwd_f64
    rc = fn(qa.ctypes.data, ka.ctypes.data, va.ctypes.data, B, H, N, d,
            float(scale), int(bool(causal)), rows_ptr, nrows,
            o.ctypes.data_as(ctypes.POINTER(ctypes.c_double)),
            lse.ctypes.data_as(ctypes.POINTER(ctypes.c_double)), int(nthreads))
    if rc != 0:
        raise RuntimeError(f"oracle failed with code {rc}")
    return o, lse


def softmax_row(x):
    """Three-pass stable softmax of a 1-D float64 row; returns (p, lse)."""
    xa = np.ascontiguousarray(np.asarray(x, dtype=np.float64))
    p = np.empty_like(xa)
    dp = ctypes.POINTER(ctypes.c_double)
    lse = _load().oracle_softmax_row_f64(xa.ctypes.data_as(dp), xa.size, p.ctypes.data_as(dp))
    return p, float(lse)


def attention_bwd(q, k, v, do, scale: float, causal: bool, dlse=None):
    """dq, dk, dv in fp64 for inputs shaped [B,H,N,d] (bf16 tensors or float arrays) and dO.

    The definition the backward pass computes ("4.4 Writing GPU Kernels with
    Triton", Kernel 5 "FlashAttention Backward"), per (batch, head), with the
    score matrix materialised: S = scale q k^T (causal: -inf above the
    diagonal), P = softmax(S) by rows, O = P v, dv = P^T dO, dP = dO v^T,
    D = rowsum(dO * O), dS = P * (dP - D), dq = scale dS k, dk = scale dS^T q.

    ``dlse`` ([B,H,N], optional) is a gradient on the forward's second output,
    LSE_i = log sum_j exp(S_ij). Its derivative in S_ij is P_ij, so it enters
    as dS = P * (dP - D + dlse), i.e. D is replaced by D - dlse.
    """
    qa, ka, va, ga = (_to_f64(t) for t in (q, k, v, do))
    B, H, N, d = qa.shape
    gl = None if dlse is None else _to_f64(dlse).reshape(B, H, N)
    dq = np.zeros_like(qa)
    dk = np.zeros_like(ka)
    dv = np.zeros_like(va)
    mask = np.tril(np.ones((N, N), dtype=bool)) if causal else None
    for b in range(B):
        for h in range(H):
            Q, K, V, G = qa[b, h], ka[b, h], va[b, h], ga[b, h]
            S = scale * (Q @ K.T)
            if mask is not None:
                S = np.where(mask, S, -np.inf)
            P = np.exp(S - S.max(axis=1, keepdims=True))
            P /= P.sum(axis=1, keepdims=True)
            O = P @ V
            dv[b, h] = P.T @ G
            dP = G @ V.T
            Dr = (G * O).sum(axis=1, keepdims=True)
            if gl is not None:
                Dr = Dr - gl[b, h][:, None]
            dS = P * (dP - Dr)
            dq[b, h] = scale * (dS @ K)
            dk[b, h] = scale * (dS.T @ Q)
    return dq, dk, dv


def _to_f64(t):
    """bf16 / fp16 torch tensor or array -> float64 numpy array (widened exactly)."""
    if hasattr(t, "dtype") and str(getattr(t, "dtype", "")).endswith("bfloat16"):
        return t.detach().to("cpu").float().numpy().astype(np.float64)
    if hasattr(t, "detach"):
        return t.detach().to("cpu").numpy().astype(np.float64)
    return np.asarray(t, dtype=np.float64)


def softmax_rows(x):
    """Row softmax of a 2-D array, in fp64: every row through softmax_row.

    This is the definition the fused-softmax kernel computes ("4.4 Writing GPU
    Kernels with Triton", Kernel 2 "Fused Softmax"; "Triton", fused softmax):
    y[i, j] = exp(x[i, j] - max_k x[i, k]) / sum_k exp(x[i, k] - max_k x[i, k]).
    """
    xa = np.asarray(x, dtype=np.float64)
    if xa.ndim != 2:
        raise ValueError("softmax_rows takes a 2-D array")
    out = np.empty_like(xa)
    for i in range(xa.shape[0]):
        out[i], _ = softmax_row(xa[i])
    return out
