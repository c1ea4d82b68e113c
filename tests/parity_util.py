"""Shared helpers for the GPU parity tests: tolerances, sampled rows, canaries."""
from __future__ import annotations

import numpy as np

# Tolerances for the bf16 path against the fp64 oracle:
#   O   : max |O_gpu - O_ref| <= 2e-2 (O_gpu widened from bf16)
#   LSE : |LSE_gpu - LSE_ref| <= 1e-3 * max(|LSE_ref|, 1)
# The floor of 1 keeps the relative test well posed where LSE is near 0
# (a causal row 0 has LSE = s_00, which can be ~0).
O_ATOL = 2e-2
LSE_RTOL = 1e-3


def lse_err(lse_gpu, lse_ref) -> float:
    lse_gpu = np.asarray(lse_gpu, dtype=np.float64)
    return float(np.max(np.abs(lse_gpu - lse_ref) / np.maximum(np.abs(lse_ref), 1.0)))


def o_err(o_gpu, o_ref) -> float:
    return float(np.max(np.abs(np.asarray(o_gpu, dtype=np.float64) - o_ref)))


def assert_parity(o_gpu, lse_gpu, o_ref, lse_ref, what=""):
    eo, el = o_err(o_gpu, o_ref), lse_err(lse_gpu, lse_ref)
    assert np.all(np.isfinite(np.asarray(o_gpu, dtype=np.float64))), f"{what}: non-finite O"
    assert np.all(np.isfinite(np.asarray(lse_gpu, dtype=np.float64))), f"{what}: non-finite LSE"
    assert eo <= O_ATOL, f"{what}: max|dO| = {eo:.4g} > {O_ATOL}"
    assert el <= LSE_RTOL, f"{what}: max rel dLSE = {el:.4g} > {LSE_RTOL}"
    return eo, el


def sample_rows(B, H, N, n_random=64, seed=0, heads=None):
    """Flattened row ids (grouped by head): tile edges, tails, and random rows."""
    rng = np.random.default_rng(seed)
    BH = B * H
    if heads is None:
        heads = sorted({0, BH - 1, *rng.integers(0, BH, size=4).tolist()})
    fixed = [0, 1, 2, 63, 64, 127, 128, 129, 255, 256, 257, N // 2, N - 129, N - 128,
             N - 127, N - 33, N - 32, N - 2, N - 1]
    rows = []
    for bh in heads:
        loc = sorted({i for i in fixed if 0 <= i < N} | set(rng.integers(0, N, size=n_random).tolist()))
        rows += [bh * N + i for i in loc]
    return np.array(rows, dtype=np.int64)
