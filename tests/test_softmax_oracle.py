"""Pins of the row-softmax oracle, and host-side checks of softmax_rows_fwd (no GPU).

The oracle is the definition the fused-softmax kernel computes ("4.4 Writing
GPU Kernels with Triton", Kernel 2 "Fused Softmax"): each row through the
three-pass max / exp-sum / divide. These checks tie it to values fixed by the
mathematics, not to itself.
"""
import ctypes
import math
from fractions import Fraction

import numpy as np
import pytest

import oracle


@pytest.fixture(scope="module", autouse=True)
def _built():
    oracle.build()


def test_closed_forms():
    np.testing.assert_allclose(oracle.softmax_rows([[0.0, math.log(2.0)]])[0], [1 / 3, 2 / 3], rtol=1e-15)
    np.testing.assert_allclose(oracle.softmax_rows([[0.0, math.log(3.0), math.log(6.0)]])[0], [0.1, 0.3, 0.6],
                               rtol=1e-14)
    # uniform row: 1/N everywhere
    np.testing.assert_allclose(oracle.softmax_rows(np.full((1, 7), 2.5))[0], np.full(7, 1 / 7), rtol=1e-15)


def test_rows_sum_to_one_and_shift_invariance():
    rng = np.random.default_rng(3)
    x = rng.standard_normal((20, 333)) * 10
    y = oracle.softmax_rows(x)
    np.testing.assert_allclose(y.sum(axis=1), 1.0, rtol=0, atol=1e-13)
    np.testing.assert_allclose(oracle.softmax_rows(x + 1234.5), y, rtol=1e-12, atol=1e-300)


def test_large_logits_and_masked_columns():
    y = oracle.softmax_rows([[1000.0, 0.0, -1000.0]])[0]
    assert y[0] == 1.0 and 0.0 <= y[1] < 1e-300 and y[2] == 0.0
    y = oracle.softmax_rows([[0.0, -math.inf, 0.0]])[0]
    np.testing.assert_array_equal(y, [0.5, 0.0, 0.5])


def test_brute_force_exact():
    """Tiny rows against exact rational arithmetic of exp(x_j) / sum exp(x_k) with x_j = ln(a_j)."""
    for a in ([1, 2, 3, 4], [5, 5, 1], [7], [1, 1000]):
        x = np.log(np.asarray(a, dtype=np.float64))[None, :]
        tot = sum(Fraction(v) for v in a)
        exact = [float(Fraction(v) / tot) for v in a]
        np.testing.assert_allclose(oracle.softmax_rows(x)[0], exact, rtol=1e-14)


def test_matches_an_independent_library():
    scipy_special = pytest.importorskip("scipy.special")
    rng = np.random.default_rng(4)
    x = rng.standard_normal((17, 1000)) * 30
    np.testing.assert_allclose(oracle.softmax_rows(x), scipy_special.softmax(x, axis=1), rtol=1e-12, atol=1e-300)


# ------------------------------------------------------------------ ABI, no GPU needed

@pytest.fixture(scope="module")
def lib():
    import blocked_online_softmax_gb300 as bos
    import __graft_entry__
    __graft_entry__.build()
    return bos.load_library()


@pytest.mark.parametrize("args, code", [
    ((0, 16, 4, 4, 4, 4), 1),          # NULL x
    ((16, 0, 4, 4, 4, 4), 1),          # NULL y
    ((16, 16, 0, 4, 4, 4), 2),         # no rows
    ((16, 16, 4, 0, 4, 4), 2),         # no columns
    ((16, 16, 4, 8, 7, 8), 2),         # x stride < cols
    ((16, 16, 4, 8, 8, 3), 2),         # y stride < cols
    ((18, 16, 4, 4, 4, 4), 5),         # x not 4-byte aligned
])
def test_softmax_rows_validation(lib, args, code):
    x, y, r, c, xs, ys = args
    st = lib.softmax_rows_fwd(ctypes.c_void_p(x), ctypes.c_void_p(y), r, c, xs, ys, None)
    assert st == code
