"""Test-only fp64 blocked online softmax attention (numpy).

Written from the recurrence of "4.4 Writing GPU Kernels with Triton"
(llm-stack-book), "The Online Softmax Recurrence" and Kernel 4: keys and values
are streamed in blocks; each query row keeps a running max m, a running sum l
and an unnormalised accumulator acc. On a block with scores s:

    m_new = max(m, max_j s_j)
    alpha = exp(m - m_new)          (the correction factor for the old state)
    p_j   = exp(s_j - m_new)
    l     = alpha * l + sum_j p_j
    acc   = alpha * acc + sum_j p_j v_j
    m     = m_new

then O = acc / l and LSE = m + ln l (natural log). Natural exp is used here:
the exp2 form with log2(e) folded into the scale is the same function.

It exists only to pin the oracle's three-pass definition to the streamed
method the pages describe (they say the two agree), and to work the page's
exercise. It shares nothing with the oracle or with the CUDA library.
"""
from __future__ import annotations

import numpy as np


def blocked_online_row(s: np.ndarray, v: np.ndarray, block: int):
    """Stream one row of (already scaled, already masked) scores s[N] against v[N, d].

    Returns (o, lse, trace) where trace lists, per block, (alpha, l, acc) after
    that block's update.
    """
    n = s.shape[0]
    m = -np.inf
    l = 0.0
    acc = np.zeros(v.shape[1], dtype=np.float64)
    trace = []
    for j0 in range(0, n, block):
        sb = s[j0:j0 + block]
        vb = v[j0:j0 + block]
        m_new = max(m, float(np.max(sb)))
        if m_new == -np.inf:            # every score so far masked: nothing to add
            trace.append((1.0, l, acc.copy()))
            continue
        alpha = 0.0 if m == -np.inf else float(np.exp(m - m_new))
        p = np.exp(sb - m_new)           # exp(-inf) = 0 for masked keys
        l = alpha * l + float(np.sum(p))
        acc = alpha * acc + p @ vb
        m = m_new
        trace.append((alpha, l, acc.copy()))
    o = acc / l
    lse = m + np.log(l)
    return o, lse, trace


def blocked_online_attention(q, k, v, scale: float, causal: bool, block: int):
    """[B,H,N,d] float64 arrays -> (O [B,H,N,d], LSE [B,H,N]) by streaming key blocks."""
    B, H, N, d = q.shape
    o = np.empty_like(q)
    lse = np.empty((B, H, N))
    for b in range(B):
        for h in range(H):
            s_all = scale * (q[b, h] @ k[b, h].T)
            for i in range(N):
                s = s_all[i].copy()
                if causal:
                    s[i + 1:] = -np.inf
                o[b, h, i], lse[b, h, i], _ = blocked_online_row(s, v[b, h], block)
    return o, lse


def stale_max_row(s: np.ndarray, v: np.ndarray, block: int, threshold_log2: float, reverse: bool):
    """The same recurrence with a stale reference max: the reference m moves
    only when a block's max exceeds it by more than `threshold_log2` (in log2
    units, as the kernels count it), so each probability is at most
    2^threshold; O and the LSE are the same quantities in exact arithmetic.
    Blocks are visited last to first when `reverse` (the kernels' order).

    Returns (o, lse, largest probability taken).
    """
    n = s.shape[0]
    t = threshold_log2 * np.log(2.0)     # natural-log units
    m = -np.inf
    l = 0.0
    acc = np.zeros(v.shape[1], dtype=np.float64)
    p_max = 0.0
    starts = list(range(0, n, block))
    for j0 in (reversed(starts) if reverse else starts):
        sb = s[j0:j0 + block]
        vb = v[j0:j0 + block]
        m_blk = float(np.max(sb))
        if m == -np.inf:
            if m_blk == -np.inf:        # every score so far masked
                continue
            m = m_blk
        elif m_blk > m + t:             # move the reference: rescale the state
            alpha = float(np.exp(m - m_blk))
            l *= alpha
            acc *= alpha
            m = m_blk
        p = np.exp(sb - m)
        p_max = max(p_max, float(np.max(p)))
        l += float(np.sum(p))
        acc += p @ vb
    return acc / l, m + np.log(l), p_max
