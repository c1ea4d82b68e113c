"""The seeded input generator: deterministic, the stated shapes, exact x4 scaling."""
import math

import torch

from blocked_online_softmax_gb300.workloads import WORKLOADS, TAIL_4000, make_qkv


def test_deterministic_and_shaped():
    a = make_qkv(1, 2, 33, 64, seed=7)
    b = make_qkv(1, 2, 33, 64, seed=7)
    c = make_qkv(1, 2, 33, 64, seed=8)
    for x, y in zip(a, b):
        assert x.dtype == torch.bfloat16 and x.shape == (1, 2, 33, 64) and x.is_contiguous()
        assert torch.equal(x, y)
    assert not torch.equal(a[0], c[0])
    assert not torch.equal(a[0], a[1])          # Q, K, V are distinct draws


def test_logit_multiplier_is_exact():
    q1, k1, v1 = make_qkv(1, 1, 40, 64, seed=3)
    q4, k4, v4 = make_qkv(1, 1, 40, 64, seed=3, logit_mult=4.0)
    assert torch.equal(q4.float(), q1.float() * 4) and torch.equal(k4.float(), k1.float() * 4)
    assert torch.equal(v4, v1)


def test_workload_table():
    assert [w.seed for w in WORKLOADS] == [1, 2, 3, 4, 5]
    assert TAIL_4000.N % 128 == 32 and TAIL_4000.logit_mult == 4.0
    for w in WORKLOADS:
        assert w.scale == float(torch.tensor(1 / math.sqrt(w.d), dtype=torch.float32))
        f = 4.0 * w.B * w.H * w.N ** 2 * w.d
        assert w.flops == (f / 2 if w.causal else f)
