"""Pins of the backward oracle (no GPU): it is the derivative of the forward oracle.

The forward oracle is pinned separately (test_oracle_pins.py); here central
finite differences of L = sum(O * dO) through that forward, in fp64, must match
the closed-form gradients, and special cases with known answers hold.
"""
import numpy as np
import pytest

import oracle


@pytest.fixture(scope="module", autouse=True)
def _built():
    oracle.build()


def _loss(q, k, v, g, scale, causal):
    o, _ = oracle.attention(q, k, v, scale, causal)
    return float((o * g).sum())


@pytest.mark.parametrize("causal", [False, True])
def test_matches_finite_differences(causal):
    rng = np.random.default_rng(5 + causal)
    B, H, N, d = 1, 2, 5, 3
    q, k, v, g = (rng.standard_normal((B, H, N, d)) for _ in range(4))
    scale = 0.7
    dq, dk, dv = oracle.attention_bwd(q, k, v, g, scale, causal)
    eps = 1e-6
    for name, x, grad in (("q", q, dq), ("k", k, dk), ("v", v, dv)):
        num = np.zeros_like(x)
        for idx in np.ndindex(x.shape):
            xp, xm = x.copy(), x.copy()
            xp[idx] += eps
            xm[idx] -= eps
            args_p = dict(q=q, k=k, v=v)
            args_m = dict(q=q, k=k, v=v)
            args_p[name], args_m[name] = xp, xm
            num[idx] = (_loss(args_p["q"], args_p["k"], args_p["v"], g, scale, causal)
                        - _loss(args_m["q"], args_m["k"], args_m["v"], g, scale, causal)) / (2 * eps)
        np.testing.assert_allclose(grad, num, rtol=1e-6, atol=1e-8, err_msg=f"d{name}")


@pytest.mark.parametrize("causal", [False, True])
def test_lse_gradient_matches_finite_differences(causal):
    """With a gradient gl on the LSE output too, L = sum(O * dO) + sum(LSE * gl)."""
    rng = np.random.default_rng(15 + causal)
    B, H, N, d = 1, 1, 4, 3
    q, k, v, g = (rng.standard_normal((B, H, N, d)) for _ in range(4))
    gl = rng.standard_normal((B, H, N))
    scale = 0.9

    def loss(q_, k_, v_):
        o, lse = oracle.attention(q_, k_, v_, scale, causal)
        return float((o * g).sum() + (lse * gl).sum())

    dq, dk, dv = oracle.attention_bwd(q, k, v, g, scale, causal, dlse=gl)
    eps = 1e-6
    for name, grad in (("q", dq), ("k", dk), ("v", dv)):
        num = np.zeros_like(grad)
        for idx in np.ndindex(grad.shape):
            args_p, args_m = dict(q_=q.copy(), k_=k.copy(), v_=v.copy()), dict(q_=q.copy(), k_=k.copy(), v_=v.copy())
            args_p[name + "_"][idx] += eps
            args_m[name + "_"][idx] -= eps
            num[idx] = (loss(**args_p) - loss(**args_m)) / (2 * eps)
        np.testing.assert_allclose(grad, num, rtol=1e-6, atol=1e-8, err_msg=f"d{name}")
    # the LSE term changes dq and dk but never dv
    _, _, dv0 = oracle.attention_bwd(q, k, v, g, scale, causal)
    np.testing.assert_allclose(dv, dv0, rtol=0, atol=0)


def test_identical_keys_give_zero_dq():
    """Equal keys make every score row constant in q: dq = 0 (and dS sums to 0 per row)."""
    rng = np.random.default_rng(6)
    q = rng.standard_normal((1, 1, 6, 4))
    k = np.broadcast_to(rng.standard_normal((1, 1, 1, 4)), (1, 1, 6, 4)).copy()
    v, g = rng.standard_normal((2, 1, 1, 6, 4))
    dq, _, _ = oracle.attention_bwd(q, k, v, g, 0.5, False)
    np.testing.assert_allclose(dq, 0.0, atol=1e-13)


def test_constant_values_give_zero_dq_dk():
    """Equal value rows make O independent of the scores: dq = dk = 0, dv = P^T dO."""
    rng = np.random.default_rng(7)
    q, k, g = rng.standard_normal((3, 1, 2, 7, 4))
    v = np.broadcast_to(rng.standard_normal((1, 1, 1, 4)), (1, 2, 7, 4)).copy()
    dq, dk, dv = oracle.attention_bwd(q, k, v, g, 0.3, True)
    np.testing.assert_allclose(dq, 0.0, atol=1e-13)
    np.testing.assert_allclose(dk, 0.0, atol=1e-13)


def test_uniform_attention_dv_is_mean_of_do():
    """q = 0: every row attends uniformly, so dv_j = sum_i dO_i / N (non-causal)."""
    rng = np.random.default_rng(8)
    N = 9
    q = np.zeros((1, 1, N, 4))
    k, v, g = rng.standard_normal((3, 1, 1, N, 4))
    _, _, dv = oracle.attention_bwd(q, k, v, g, 1.0, False)
    np.testing.assert_allclose(dv[0, 0], np.broadcast_to(g[0, 0].sum(axis=0) / N, (N, 4)), rtol=1e-13)


def _fd_grad_q(q, k, v, g, scale, causal, eps=1e-6):
    num = np.zeros_like(q)
    for idx in np.ndindex(q.shape):
        qp, qm = q.copy(), q.copy()
        qp[idx] += eps
        qm[idx] -= eps
        num[idx] = (_loss(qp, k, v, g, scale, causal) - _loss(qm, k, v, g, scale, causal)) / (2 * eps)
    return num


def _dq_planted(q, k, v, g, scale, mistake):
    """dq of one non-causal head with one of the page's named backward mistakes
    planted (the page's failure signatures, "FlashAttention Backward" of "4.4
    Writing GPU Kernels with Triton"): the D_i term dropped, or the softmax
    scale folded in wrong (missing from dS)."""
    s = scale * q @ k.T
    p = np.exp(s - s.max(axis=1, keepdims=True))
    p /= p.sum(axis=1, keepdims=True)
    o = p @ v
    dp = g @ v.T
    dsum = (g * o).sum(axis=1, keepdims=True)
    if mistake == "no_D":
        ds = p * dp * scale
    elif mistake == "no_scale":
        ds = p * (dp - dsum)
    else:
        ds = p * (dp - dsum) * scale
    return ds @ k


@pytest.mark.parametrize("mistake", ["no_D", "no_scale"])
def test_finite_differences_catch_the_pages_backward_mistakes(mistake):
    """The finite-difference pin is sharp enough to reject each mistake the page
    names, and accepts the unmutated formula: dropping D adds scale * D_i times
    row i of P K to dq, and a missing scale multiplies dq by 1/scale."""
    rng = np.random.default_rng(41)
    q, k, v, g = (rng.standard_normal((1, 1, 5, 3)) for _ in range(4))
    scale = 0.6
    num = _fd_grad_q(q, k, v, g, scale, False)[0, 0]
    good = _dq_planted(q[0, 0], k[0, 0], v[0, 0], g[0, 0], scale, None)
    np.testing.assert_allclose(good, num, rtol=1e-6, atol=1e-8)
    bad = _dq_planted(q[0, 0], k[0, 0], v[0, 0], g[0, 0], scale, mistake)
    assert np.max(np.abs(bad - num)) > 1e-2 * np.max(np.abs(num)), f"the pin misses the planted {mistake}"
    if mistake == "no_scale":
        np.testing.assert_allclose(bad, num / scale, rtol=1e-6, atol=1e-8)
