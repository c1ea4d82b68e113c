"""Pins for the fp64 oracle: what the pages and the mathematics fix, independent of it.

Each check is chosen so that a plausible slip in the oracle (a dropped scale, a
wrong causal bound, a transposed operand, a mixed log base, a missing max
subtraction) fails at least one of them. None of them retypes the oracle's own
formula.
"""
import json
import math
import os

import numpy as np
import pytest

import oracle
from online_softmax_ref import blocked_online_attention, blocked_online_row, stale_max_row

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rand(shape, seed, scale=1.0):
    return np.random.default_rng(seed).standard_normal(shape) * scale


# ---------------------------------------------------------------- the page's worked exercise

def test_exercise5_two_key_blocks():
    """'4.4 Writing GPU Kernels with Triton', Exercises item 5 (closed forms; the page prints none)."""
    with open(os.path.join(GOLDEN, "exercise5_two_key_blocks.json")) as f:
        ex = json.load(f)
    s = np.array(ex["scores"], dtype=np.float64)
    vals = np.array(ex["values"], dtype=np.float64)
    e = math.exp
    alpha_ref = e(s[0] - s[1])                                   # e^-2
    l_ref = 1.0 + e(s[0] - s[1])                                  # 1 + e^-2
    ounorm_ref = vals[0] * e(s[0] - s[1]) + vals[1]               # e^-2 + 3
    o_ref = (vals[0] * e(s[0]) + vals[1] * e(s[1])) / (e(s[0]) + e(s[1]))
    lse_ref = s[1] + math.log1p(e(s[0] - s[1]))                   # 4 + ln(1 + e^-2)
    assert abs(o_ref - 2.761594155955765) < 1e-15
    assert abs(lse_ref - 4.126928011042972) < 1e-15

    # the streamed recurrence, one key per block
    o, lse, trace = blocked_online_row(s, vals.reshape(2, 1), block=ex["block_size"])
    assert trace[0][0] == 0.0 or trace[0][1] == 1.0  # first block starts from m = -inf
    alpha2, l2, acc2 = trace[1]
    assert alpha2 == pytest.approx(alpha_ref, rel=1e-15)
    assert l2 == pytest.approx(l_ref, rel=1e-15)
    assert acc2[0] == pytest.approx(ounorm_ref, rel=1e-15)
    assert o[0] == pytest.approx(o_ref, rel=1e-15)
    assert lse == pytest.approx(lse_ref, rel=1e-15)

    # the oracle: q = [1], k = [[2], [4]], v = [[1], [3]], scale 1
    q = np.ones((1, 1, 1, 1))
    k = s.reshape(1, 1, 2, 1).copy()
    v = vals.reshape(1, 1, 2, 1).copy()
    # the oracle needs N query rows; row 0 is the exercise's row (non-causal)
    q2 = np.concatenate([q, q], axis=2)
    oo, ll = oracle.attention(q2, k, v, scale=1.0, causal=False)
    assert oo[0, 0, 0, 0] == pytest.approx(o_ref, rel=1e-15)
    assert ll[0, 0, 0] == pytest.approx(lse_ref, rel=1e-15)


# ---------------------------------------------------------------- brute force in extended precision

def _mp_attention(q, k, v, scale, causal):
    mpmath = pytest.importorskip("mpmath")
    mpmath.mp.dps = 50
    N, d = q.shape
    o = np.zeros((N, d))
    lse = np.zeros(N)
    for i in range(N):
        keys = range(i + 1) if causal else range(N)
        s = {j: mpmath.mpf(scale) * mpmath.fsum(mpmath.mpf(q[i, t]) * mpmath.mpf(k[j, t]) for t in range(d))
             for j in keys}
        # no max subtraction here: extended precision makes the direct form safe
        w = {j: mpmath.exp(s[j]) for j in keys}
        z = mpmath.fsum(w.values())
        for t in range(d):
            o[i, t] = float(mpmath.fsum(w[j] * mpmath.mpf(v[j, t]) for j in keys) / z)
        lse[i] = float(mpmath.log(z))
    return o, lse


@pytest.mark.parametrize("N,d,causal,seed", [(1, 1, False, 0), (2, 3, False, 1), (3, 2, True, 2),
                                             (4, 3, False, 3), (4, 3, True, 4), (3, 5, False, 5)])
def test_brute_force_tiny(N, d, causal, seed):
    q = _rand((1, 1, N, d), seed)
    k = _rand((1, 1, N, d), seed + 100)          # different from q: a q/k swap shows up
    v = _rand((1, 1, N, d), seed + 200)
    scale = 0.7
    o, lse = oracle.attention(q, k, v, scale, causal)
    o_ref, lse_ref = _mp_attention(q[0, 0], k[0, 0], v[0, 0], scale, causal)
    np.testing.assert_allclose(o[0, 0], o_ref, rtol=0, atol=1e-13)
    np.testing.assert_allclose(lse[0, 0], lse_ref, rtol=0, atol=1e-13)


def test_brute_force_large_logits():
    """Logits near 700-900 overflow exp() without the max subtraction; the oracle must not."""
    N, d = 4, 2
    q = np.array([[[[30.0, 0.0], [0.0, 30.0], [20.0, 20.0], [-30.0, 1.0]]]])
    k = np.array([[[[30.0, 1.0], [29.0, 0.5], [1.0, 30.0], [-29.0, 2.0]]]])
    v = _rand((1, 1, N, d), 7)
    o, lse = oracle.attention(q, k, v, 1.0, False)
    o_ref, lse_ref = _mp_attention(q[0, 0], k[0, 0], v[0, 0], 1.0, False)
    assert np.all(np.isfinite(o)) and np.all(np.isfinite(lse))
    np.testing.assert_allclose(o[0, 0], o_ref, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse[0, 0], lse_ref, rtol=1e-15, atol=0)


# ---------------------------------------------------------------- the method equals its definition

@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("block", [1, 7, 64, 97])
def test_blocked_online_equals_three_pass(causal, block):
    B, H, N, d = 1, 2, 97, 16
    q, k, v = (_rand((B, H, N, d), s) for s in (11, 12, 13))
    o_ref, lse_ref = oracle.attention(q, k, v, 0.25, causal)
    o, lse = blocked_online_attention(q, k, v, 0.25, causal, block)
    np.testing.assert_allclose(o, o_ref, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(lse, lse_ref, rtol=1e-12, atol=1e-13)


@pytest.mark.parametrize("threshold", [0.0, 8.0, 32.0])
@pytest.mark.parametrize("reverse", [False, True])
@pytest.mark.parametrize("causal", [False, True])
def test_stale_max_recurrence_equals_three_pass(threshold, reverse, causal):
    """The kernels' stale-max rescaling (the reference max moves only when a
    block's max exceeds it by more than a threshold, 32 or 8 log2 units in the
    kernels) computes the same O and LSE as the three-pass definition, and no
    probability it forms exceeds 2^threshold. Scores rise along the keys by
    more than 32 log2 units per block, on top of logits of tens of units, so
    the reference both stays stale and moves."""
    B, H, N, d, block = 1, 2, 300, 16, 64
    rng = np.random.default_rng(41)
    q = rng.standard_normal((B, H, N, d)) * 4.0
    k = rng.standard_normal((B, H, N, d)) * 4.0
    k[..., 0] += 0.9 * np.arange(N)      # q_0 k_0 grows along the keys for rows with q_0 > 0
    v = rng.standard_normal((B, H, N, d))
    scale = 0.25
    o_ref, lse_ref = oracle.attention(q, k, v, scale, causal)
    for h in range(H):
        s_all = scale * (q[0, h] @ k[0, h].T)
        for i in range(N):
            s = s_all[i].copy()
            if causal:
                s[i + 1:] = -np.inf
            o, lse, p_max = stale_max_row(s, v[0, h], block, threshold, reverse)
            np.testing.assert_allclose(o, o_ref[0, h, i], rtol=1e-11, atol=1e-12)
            assert lse == pytest.approx(lse_ref[0, h, i], rel=1e-12, abs=1e-12)
            assert p_max <= 2.0 ** threshold * (1 + 1e-12)


def test_matches_library_sdpa_fp64():
    """torch's own fp64 scaled-dot-product attention is an independent implementation."""
    torch = pytest.importorskip("torch")
    B, H, N, d = 2, 3, 70, 24
    q, k, v = (_rand((B, H, N, d), s) for s in (21, 22, 23))
    for causal in (False, True):
        o, lse = oracle.attention(q, k, v, 0.3, causal)
        tq, tk, tv = (torch.from_numpy(x) for x in (q, k, v))
        ref = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, is_causal=causal, scale=0.3)
        s = 0.3 * tq @ tk.transpose(-1, -2)
        if causal:
            s = s.masked_fill(~torch.ones(N, N, dtype=torch.bool).tril(), float("-inf"))
        np.testing.assert_allclose(o, ref.numpy(), rtol=0, atol=1e-12)
        np.testing.assert_allclose(lse, torch.logsumexp(s, dim=-1).numpy(), rtol=1e-13, atol=1e-13)


# ---------------------------------------------------------------- invariants and closed forms

def test_softmax_rows_sum_to_one():
    for seed, n in [(0, 1), (1, 5), (2, 257), (3, 4000)]:
        x = _rand(n, seed, scale=20.0)
        p, lse = oracle.softmax_row(x)
        assert abs(p.sum() - 1.0) < 1e-12
        assert np.all(p >= 0)
        assert lse == pytest.approx(np.log(np.sum(np.exp(x - x.max()))) + x.max(), rel=1e-14)
    p, lse = oracle.softmax_row(np.array([-np.inf, 0.0, -np.inf]))
    assert list(p) == [0.0, 1.0, 0.0] and lse == 0.0


@pytest.mark.parametrize("causal", [False, True])
def test_all_ones_v_gives_ones(causal):
    B, H, N, d = 1, 2, 33, 8
    q, k = _rand((B, H, N, d), 31, 3.0), _rand((B, H, N, d), 32, 3.0)
    v = np.ones((B, H, N, d))
    o, _ = oracle.attention(q, k, v, 0.5, causal)
    np.testing.assert_allclose(o, 1.0, rtol=0, atol=1e-14)


def test_single_key_gives_v():
    B, H, N, d = 2, 3, 1, 5
    q, k, v = (_rand((B, H, N, d), s) for s in (41, 42, 43))
    for causal in (False, True):
        o, lse = oracle.attention(q, k, v, 0.8, causal)
        np.testing.assert_array_equal(o, v)
        np.testing.assert_allclose(lse[..., 0], 0.8 * np.sum(q[..., 0, :] * k[..., 0, :], axis=-1), rtol=1e-14)


def test_causal_row0_is_v0():
    B, H, N, d = 1, 2, 19, 6
    q, k, v = (_rand((B, H, N, d), s) for s in (51, 52, 53))
    o, lse = oracle.attention(q, k, v, 0.6, True)
    np.testing.assert_array_equal(o[:, :, 0], v[:, :, 0])
    np.testing.assert_allclose(lse[:, :, 0], 0.6 * np.sum(q[:, :, 0] * k[:, :, 0], axis=-1), rtol=1e-14)


def test_uniform_logits_give_mean_and_log_n():
    B, H, N, d = 1, 2, 29, 7
    q = np.zeros((B, H, N, d))
    k, v = _rand((B, H, N, d), 61), _rand((B, H, N, d), 62)
    o, lse = oracle.attention(q, k, v, 0.5, False)
    np.testing.assert_allclose(o, np.broadcast_to(v.mean(axis=2, keepdims=True), o.shape), atol=1e-14)
    np.testing.assert_allclose(lse, math.log(N), rtol=1e-15)
    o, lse = oracle.attention(q, k, v, 0.5, True)
    prefix_mean = np.cumsum(v, axis=2) / np.arange(1, N + 1).reshape(1, 1, N, 1)
    np.testing.assert_allclose(o, prefix_mean, atol=1e-14)
    np.testing.assert_allclose(lse, np.log(np.arange(1, N + 1)).reshape(1, 1, N).repeat(H, 1), rtol=1e-15)
    # scale = 0 makes any logits uniform too
    q2 = _rand((B, H, N, d), 63)
    o, lse = oracle.attention(q2, k, v, 0.0, False)
    np.testing.assert_allclose(o, np.broadcast_to(v.mean(axis=2, keepdims=True), o.shape), atol=1e-14)


def test_joint_key_value_permutation_invariance():
    B, H, N, d = 2, 2, 41, 9
    q, k, v = (_rand((B, H, N, d), s) for s in (71, 72, 73))
    perm = np.random.default_rng(74).permutation(N)
    o1, l1 = oracle.attention(q, k, v, 0.4, False)
    o2, l2 = oracle.attention(q, k[:, :, perm], v[:, :, perm], 0.4, False)
    np.testing.assert_allclose(o1, o2, rtol=0, atol=1e-13)
    np.testing.assert_allclose(l1, l2, rtol=1e-14)
    # permuting V alone must change the result (guards against V indexed by query)
    o3, _ = oracle.attention(q, k, v[:, :, perm], 0.4, False)
    assert np.max(np.abs(o3 - o1)) > 1e-3


def test_causal_row_is_prefix_attention():
    B, H, N, d = 1, 1, 23, 4
    q, k, v = (_rand((B, H, N, d), s) for s in (81, 82, 83))
    o, lse = oracle.attention(q, k, v, 0.9, True)
    for i in (0, 1, 7, 22):
        qi = np.repeat(q[:, :, i:i + 1], i + 1, axis=2)   # i+1 copies of query i
        oi, li = oracle.attention(qi, k[:, :, :i + 1], v[:, :, :i + 1], 0.9, False)
        np.testing.assert_allclose(o[0, 0, i], oi[0, 0, 0], rtol=0, atol=1e-14)
        assert lse[0, 0, i] == pytest.approx(li[0, 0, 0], rel=1e-14)


def test_shift_invariance():
    """Adding c to every logit of a row leaves O unchanged and shifts LSE by c."""
    B, H, N, d = 1, 2, 31, 5
    q, k, v = (_rand((B, H, N, d), s) for s in (91, 92, 93))
    c = 37.0
    scale = 0.5
    q_ext = np.concatenate([q, np.full((B, H, N, 1), c / scale)], axis=-1)
    k_ext = np.concatenate([k, np.ones((B, H, N, 1))], axis=-1)
    v_ext = np.concatenate([v, np.zeros((B, H, N, 1))], axis=-1)
    o1, l1 = oracle.attention(q, k, v, scale, False)
    o2, l2 = oracle.attention(q_ext, k_ext, v_ext, scale, False)
    np.testing.assert_allclose(o2[..., :d], o1, rtol=0, atol=1e-13)
    np.testing.assert_allclose(l2, l1 + c, rtol=1e-14)


def test_bf16_entry_widens_exactly():
    """The bf16 front end must widen bit patterns exactly (bf16 = top half of fp32)."""
    torch = pytest.importorskip("torch")
    B, H, N, d = 1, 2, 17, 8
    g = torch.Generator().manual_seed(5)
    q, k, v = (torch.randn(B, H, N, d, generator=g).to(torch.bfloat16) for _ in range(3))
    o1, l1 = oracle.attention(q, k, v, 0.125, True)
    o2, l2 = oracle.attention(*(t.double().numpy() for t in (q, k, v)), 0.125, True)
    np.testing.assert_array_equal(o1, o2)
    np.testing.assert_array_equal(l1, l2)


def test_row_subset_matches_full():
    B, H, N, d = 2, 2, 50, 8
    q, k, v = (_rand((B, H, N, d), s) for s in (101, 102, 103))
    o, lse = oracle.attention(q, k, v, 0.3, True)
    rows = [0, 49, 50, 77, 150, 199, 3]
    os_, ls = oracle.attention(q, k, v, 0.3, True, rows=rows)
    flat_o = o.reshape(-1, d)
    np.testing.assert_array_equal(os_, flat_o[rows])
    np.testing.assert_array_equal(ls, lse.reshape(-1)[rows])
