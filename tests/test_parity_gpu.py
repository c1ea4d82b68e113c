"""GPU parity: the CUDA path through the C ABI against the fp64 oracle.

Every measured workload is compared element by element over every output, at
full size; only the very long single-head sequences (up to 65536 rows) are
compared on sampled rows (tile edges, the ragged tail, random rows) plus
properties that hold at any size.
"""
import numpy as np
import pytest
import torch

import blocked_online_softmax_gb300 as bos
import oracle
from blocked_online_softmax_gb300.workloads import (CAUSAL_2K, CAUSAL_4K_D256, CAUSAL_8K, MEDIUM, SMALL,
                                                    TAIL_4000, WIDE_2K_D256, make_qkv, workload_qkv)
from parity_util import assert_parity, sample_rows

pytestmark = pytest.mark.gpu

SENT_BF16 = -12288.0      # exactly representable in bf16 (-3 * 2^12)
SENT_F32 = -7.0e30


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()
    torch.cuda.set_device(0)


def run_guarded(q, k, v, scale, causal, stream=None):
    """attn_fwd into canary-guarded O / LSE; checks the guards; returns host O (float) and LSE."""
    B, H, N, d = q.shape
    pad_o, pad_l = 64, 16                       # keep 16-byte alignment of the views
    n_o, n_l = B * H * N * d, B * H * N
    dev = torch.device("cuda")
    o_buf = torch.full((pad_o + n_o + pad_o,), SENT_BF16, dtype=torch.bfloat16, device=dev)
    l_buf = torch.full((pad_l + n_l + pad_l,), SENT_F32, dtype=torch.float32, device=dev)
    o = o_buf[pad_o:pad_o + n_o].view(B, H, N, d)
    lse = l_buf[pad_l:pad_l + n_l].view(B, H, N)
    qd, kd, vd = (t.to(dev) for t in (q, k, v))
    bos.attn_fwd(qd, kd, vd, o, lse, B, H, N, d, scale, causal, stream)
    torch.cuda.synchronize()
    ob, lb = o_buf.float().cpu(), l_buf.cpu()
    assert torch.all(ob[:pad_o] == SENT_BF16) and torch.all(ob[pad_o + n_o:] == SENT_BF16), "O guard overwritten"
    assert torch.all(lb[:pad_l] == SENT_F32) and torch.all(lb[pad_l + n_l:] == SENT_F32), "LSE guard overwritten"
    return ob[pad_o:pad_o + n_o].view(B, H, N, d).numpy(), lb[pad_l:pad_l + n_l].view(B, H, N).numpy()


# ------------------------------------------------------------------ full comparison

@pytest.mark.parametrize("w", [SMALL, MEDIUM], ids=lambda w: w.name)
def test_workload_full(w):
    q, k, v = workload_qkv(w)
    o, lse = run_guarded(q, k, v, w.scale, w.causal)
    o_ref, lse_ref = oracle.attention(q, k, v, w.scale, w.causal)
    assert_parity(o, lse, o_ref, lse_ref, w.name)


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("N", [1, 2, 31, 127, 128, 129, 255, 256, 257, 383, 600])
def test_edge_lengths(N, d, causal):
    q, k, v = make_qkv(1, 2, N, d, seed=1000 + N + d)
    scale = float(np.float32(d ** -0.5))
    o, lse = run_guarded(q, k, v, scale, causal)
    o_ref, lse_ref = oracle.attention(q, k, v, scale, causal)
    assert_parity(o, lse, o_ref, lse_ref, f"N={N} d={d} causal={causal}")


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("d", [64, 128, 256])
def test_several_tiles_ragged_tail(d, causal):
    """Several query/key tiles, odd batch and head counts, a ragged tail."""
    B, H, N = 2, 3, 1000
    q, k, v = make_qkv(B, H, N, d, seed=77 + d)
    scale = float(np.float32(d ** -0.5))
    o, lse = run_guarded(q, k, v, scale, causal)
    o_ref, lse_ref = oracle.attention(q, k, v, scale, causal)
    assert_parity(o, lse, o_ref, lse_ref, f"B2H3N1000 d={d} causal={causal}")


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("d", [8, 16, 32, 48, 72, 80, 96, 112, 120])
def test_other_head_dims(d, causal):
    """Head dims below a kernel's width: the missing columns load as zero and are never stored."""
    q, k, v = make_qkv(1, 2, 300, d, seed=300 + d)
    scale = float(np.float32(d ** -0.5))
    o, lse = run_guarded(q, k, v, scale, causal)
    o_ref, lse_ref = oracle.attention(q, k, v, scale, causal)
    assert_parity(o, lse, o_ref, lse_ref, f"N=300 d={d} causal={causal}")


@pytest.mark.parametrize("d", [64, 128, 256])
@pytest.mark.parametrize("mult", [4.0, 8.0])
@pytest.mark.parametrize("causal", [False, True])
def test_large_logits_stability(mult, causal, d):
    """Logits of tens of log2 units: the running max moves often and O is rescaled in tensor memory."""
    q, k, v = make_qkv(1, 2, 700, d, seed=5 + d, logit_mult=mult)
    o, lse = run_guarded(q, k, v, 0.125, causal)
    o_ref, lse_ref = oracle.attention(q, k, v, 0.125, causal)
    assert_parity(o, lse, o_ref, lse_ref, f"x{mult} d={d} causal={causal}")


@pytest.mark.parametrize("d", [64, 128, 256])
@pytest.mark.parametrize("causal", [False, True])
def test_rescale_every_block(causal, d):
    """Scores fall by more than 50 log2 units per 128 keys, and the kernels visit
    key blocks from the last to the first, so every block's max exceeds the
    reference max by more than any stale-max threshold: O is rescaled in tensor
    memory at every block, and the result is dominated by the first keys."""
    B, H, N = 1, 2, 700
    g = torch.Generator().manual_seed(31)
    q = torch.zeros(B, H, N, d)
    q[..., 0] = 3.0 + 2.0 * torch.rand(B, H, N, generator=g)
    q[..., 1:] = 0.1 * torch.randn(B, H, N, d - 1, generator=g)
    k = torch.randn(B, H, N, d, generator=g)
    k[..., 0] = -0.75 * torch.arange(N, dtype=torch.float32)
    v = torch.randn(B, H, N, d, generator=g)
    q, k, v = (t.to(torch.bfloat16) for t in (q, k, v))
    o, lse = run_guarded(q, k, v, 0.125, causal)
    o_ref, lse_ref = oracle.attention(q, k, v, 0.125, causal)
    assert_parity(o, lse, o_ref, lse_ref, f"rescale every block d={d} causal={causal}")


def test_back_to_back_dependency():
    """A launch that reads the previous launch's output on the same stream sees all of it.

    Call A has V = 1, so its O is 1: O = P V / l with l the sum of the probabilities,
    off only by the bf16 rounding of P (relative 2^-9), so within one bf16 step of 1.
    Call B uses that O as its V, so its O is within a step of 1 as well; A's and B's
    O buffers start out as sentinels (-12288), so reading A's output early would show.
    """
    dev = torch.device("cuda")
    B, H, N, d = 2, 16, 4096, 128
    qa, ka, _ = make_qkv(B, H, N, d, seed=21)
    qa, ka = qa.to(dev), ka.to(dev)
    va = torch.ones(B, H, N, d, dtype=torch.bfloat16, device=dev)
    oa = torch.full((B, H, N, d), SENT_BF16, dtype=torch.bfloat16, device=dev)
    la = torch.empty(B, H, N, dtype=torch.float32, device=dev)
    qb, kb, _ = make_qkv(1, 4, N, d, seed=22)
    qb, kb = qb.to(dev), kb.to(dev)
    ob = torch.full((1, 4, N, d), SENT_BF16, dtype=torch.bfloat16, device=dev)
    lb = torch.empty(1, 4, N, dtype=torch.float32, device=dev)
    scale = float(np.float32(d ** -0.5))
    for _ in range(3):
        oa.fill_(SENT_BF16)
        ob.fill_(SENT_BF16)
        bos.attn_fwd(qa, ka, va, oa, la, B, H, N, d, scale, 1, None)
        vb = oa[0, :4]                            # A's first 4 heads, written by A
        bos.attn_fwd(qb, kb, vb, ob, lb, 1, 4, N, d, scale, 1, None)
        torch.cuda.synchronize()
        assert torch.all((oa.float() - 1.0).abs() <= 2.0 ** -8), "O of V = 1 must be 1"
        assert torch.all((ob.float() - 1.0).abs() <= 2.0 ** -8), \
            "the second launch read its V before the first launch wrote it"


def test_scale_zero_and_negative():
    q, k, v = make_qkv(1, 1, 300, 128, seed=9)
    for scale in (0.0, -0.2):
        o, lse = run_guarded(q, k, v, scale, False)
        o_ref, lse_ref = oracle.attention(q, k, v, scale, False)
        assert_parity(o, lse, o_ref, lse_ref, f"scale={scale}")


def test_side_stream_and_determinism():
    q, k, v = make_qkv(2, 2, 513, 128, seed=11)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        o1, l1 = run_guarded(q, k, v, 0.0883883, True, stream=s)
    o2, l2 = run_guarded(q, k, v, 0.0883883, True)
    np.testing.assert_array_equal(o1, o2)
    np.testing.assert_array_equal(l1, l2)
    o_ref, lse_ref = oracle.attention(q, k, v, float(np.float32(0.0883883)), True)
    assert_parity(o1, l1, o_ref, lse_ref, "side stream")


def test_host_buffer_entry():
    B, H, N, d = 1, 3, 333, 64
    q, k, v = make_qkv(B, H, N, d, seed=12)
    o = torch.empty_like(q).pin_memory()
    lse = torch.empty((B, H, N), dtype=torch.float32).pin_memory()
    bos.attn_fwd_host(q.pin_memory(), k.pin_memory(), v.pin_memory(), o, lse, B, H, N, d, 0.125, 1)
    o_ref, lse_ref = oracle.attention(q, k, v, 0.125, True)
    assert_parity(o.float().numpy(), lse.numpy(), o_ref, lse_ref, "host entry")


def test_host_buffer_entry_wide_head_dim():
    B, H, N, d = 1, 3, 333, 256
    q, k, v = make_qkv(B, H, N, d, seed=14)
    o = torch.empty_like(q).pin_memory()
    lse = torch.empty((B, H, N), dtype=torch.float32).pin_memory()
    bos.attn_fwd_host(q.pin_memory(), k.pin_memory(), v.pin_memory(), o, lse, B, H, N, d, 0.0625, 1)
    o_ref, lse_ref = oracle.attention(q, k, v, 0.0625, True)
    assert_parity(o.float().numpy(), lse.numpy(), o_ref, lse_ref, "host entry d=256")


def test_host_buffer_entry_chunked_matches_device_entry():
    """Large enough that attn_fwd_host pipelines several chunks of heads over its streams."""
    B, H, N, d = 2, 16, 2048, 128           # 50 MB of inputs -> 3 chunks
    q, k, v = make_qkv(B, H, N, d, seed=13)
    scale = float(np.float32(d ** -0.5))
    o_h = torch.empty_like(q).pin_memory()
    l_h = torch.empty((B, H, N), dtype=torch.float32).pin_memory()
    bos.attn_fwd_host(q.pin_memory(), k.pin_memory(), v.pin_memory(), o_h, l_h, B, H, N, d, scale, 1)
    o_d, l_d = run_guarded(q, k, v, scale, True)
    np.testing.assert_array_equal(o_h.float().numpy(), o_d)
    np.testing.assert_array_equal(l_h.numpy(), l_d)
    rows = sample_rows(B, H, N, n_random=16, seed=13)
    o_ref, lse_ref = oracle.attention(q, k, v, scale, True, rows=rows)
    assert_parity(o_h.float().numpy().reshape(-1, d)[rows], l_h.numpy().reshape(-1)[rows], o_ref, lse_ref,
                  "host entry, chunked")


# ------------------------------------------------------------------ full-size workloads, every row

@pytest.mark.parametrize("w", [CAUSAL_2K, CAUSAL_8K, TAIL_4000, CAUSAL_4K_D256, WIDE_2K_D256],
                         ids=lambda w: w.name)
def test_workload_full_size_every_row(w):
    """The measured workloads at full size, in the bench's launch configuration,
    compared with the oracle at every (batch, head, row) (the two smaller ones
    are in test_workload_full). The oracle needs about 1 s (2K causal) to 15 s
    (the 4000-row tail workload) on 16 host cores."""
    q, k, v = workload_qkv(w)
    o, lse = run_guarded(q, k, v, w.scale, w.causal)
    # a property at every row as well: O is a convex combination of the V rows it sees
    vf = v.float()
    if not w.causal:
        vmax = vf.amax(dim=2, keepdim=True).numpy()
        vmin = vf.amin(dim=2, keepdim=True).numpy()
    else:
        vmax = torch.cummax(vf, dim=2).values.numpy()
        vmin = torch.cummin(vf, dim=2).values.numpy()
    slack = 1e-2 + 2 ** -7 * np.maximum(np.abs(vmax), np.abs(vmin))
    assert np.all(o <= vmax + slack) and np.all(o >= vmin - slack), "O outside the hull of V"
    o_ref, lse_ref = oracle.attention(q, k, v, w.scale, w.causal)
    assert_parity(o, lse, o_ref, lse_ref, w.name)


# ------------------------------------------------------------------ strided layouts

def _layout(x, kind, pad=16):
    """x: host [B,H,N,d]. Returns a device view of the same values in the layout
    `kind` ("bnhd": a [B,N,H,d] tensor transposed; "padded": rows padded past d)
    and the backing tensor."""
    B, H, N, d = x.shape
    if kind == "bnhd":
        base = x.permute(0, 2, 1, 3).contiguous().cuda()
        return base.permute(0, 2, 1, 3), base
    base = torch.zeros(B, H, N, d + pad, dtype=x.dtype).cuda()
    base[..., :d] = x.cuda()
    return base[..., :d], base


@pytest.mark.parametrize("d,causal,N", [(128, True, 333), (128, False, 300), (64, True, 257), (40, False, 200),
                                         (256, True, 333), (176, False, 300)])
@pytest.mark.parametrize("kind", ["bnhd", "padded"])
def test_strided_layouts(kind, d, causal, N):
    """attn_fwd_strided on [B,N,H,d] views and on rows padded past d, inputs and
    output: equal to the oracle, and the output's padding is never written."""
    B, H = 2, 3
    q, k, v = make_qkv(B, H, N, d, seed=60 + d + N)
    scale = float(np.float32(d ** -0.5))
    (qd, _), (kd, _), (vd, _) = (_layout(t, kind) for t in (q, k, v))
    sentinel = torch.full((B, H, N, d), SENT_BF16, dtype=torch.bfloat16)
    od, obase = _layout(sentinel, kind)
    if kind == "padded":
        obase[..., d:] = SENT_BF16
    assert not qd.is_contiguous() and not od.is_contiguous()
    o, lse = bos.attention(qd, kd, vd, scale=scale, causal=causal, out=od)
    torch.cuda.synchronize()
    assert o.data_ptr() == od.data_ptr()
    o_ref, lse_ref = oracle.attention(q, k, v, scale, causal)
    assert_parity(o.float().cpu().numpy(), lse.cpu().numpy(), o_ref, lse_ref, f"{kind} d={d} causal={causal}")
    if kind == "padded":
        assert torch.all(obase[..., d:].float().cpu() == SENT_BF16), "wrote into the row padding of O"


def test_strided_matches_contiguous_bitwise():
    """The strided entry on a transposed copy gives the contiguous call's bytes."""
    q, k, v = make_qkv(1, 4, 700, 128, seed=66)
    o1, l1 = bos.attention(q.cuda(), k.cuda(), v.cuda(), causal=True)
    (qd, _), (kd, _), (vd, _) = (_layout(t, "bnhd") for t in (q, k, v))
    o2, l2 = bos.attention(qd, kd, vd, causal=True)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


# ------------------------------------------------------------------ scale and concurrency

@pytest.mark.parametrize("d,causal,N", [(128, True, 65536), (64, False, 40000), (256, True, 32768), (192, False, 20000)])
def test_long_sequence_sampled(d, causal, N):
    """One long sequence (index arithmetic at scale, 256-512 work units in one
    head): sampled rows against the oracle, every row finite."""
    q, k, v = make_qkv(1, 2, N, d, seed=77 + d)
    scale = float(np.float32(d ** -0.5))
    o, lse = run_guarded(q, k, v, scale, causal)
    assert np.all(np.isfinite(o)) and np.all(np.isfinite(lse))
    rows = sample_rows(1, 2, N, n_random=48, seed=78)
    o_ref, lse_ref = oracle.attention(q, k, v, scale, causal, rows=rows)
    assert_parity(o.reshape(-1, d)[rows], lse.reshape(-1)[rows], o_ref, lse_ref, f"N={N} d={d}")


@pytest.mark.parametrize("d", [64, 128, 256])
def test_many_short_heads(d):
    """4096 heads of 130 rows: thousands of one- and two-block units through
    the scheduler, each with a ragged tail; compared in full."""
    q, k, v = make_qkv(64, 64, 130, d, seed=79 + d)
    scale = float(np.float32(d ** -0.5))
    o, lse = run_guarded(q, k, v, scale, True)
    o_ref, lse_ref = oracle.attention(q, k, v, scale, True)
    assert_parity(o, lse, o_ref, lse_ref, f"4096 heads d={d}")


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("d", [136, 192, 200, 256])
@pytest.mark.parametrize("N", [1, 127, 129, 300, 600])
def test_wide_head_dims(N, d, causal):
    """Head dims past 128 run on the 256-wide kernel: 64-column boxes past d are
    skipped and the rest of the last box reads as zero."""
    q, k, v = make_qkv(1, 2, N, d, seed=N + d)
    scale = float(np.float32(d ** -0.5))
    o, lse = run_guarded(q, k, v, scale, causal)
    o_ref, lse_ref = oracle.attention(q, k, v, scale, causal)
    assert_parity(o, lse, o_ref, lse_ref, f"N={N} d={d} causal={causal}")


@pytest.mark.parametrize("d", [64, 128, 256])
def test_causal_mixed_units(d):
    """Causal, 80 heads of 1900 rows (15 key blocks): about four units per CTA.
    In every unit but a head's last, the upper 128 query rows see one key block
    more than the lower 128; the last unit's two tiles see the same blocks. So
    the tile that takes the upper rows changes from unit to unit in a way that
    depends on each CTA's sequence of units; every row is compared."""
    q, k, v = make_qkv(2, 40, 1900, d, seed=97 + d)
    scale = float(np.float32(d ** -0.5))
    o, lse = run_guarded(q, k, v, scale, True)
    o_ref, lse_ref = oracle.attention(q, k, v, scale, True)
    assert_parity(o, lse, o_ref, lse_ref, f"80 heads N=1900 d={d}")


def test_concurrent_host_threads():
    """Four host threads, each with its own stream and buffers, call attn_fwd
    concurrently; every result equals the single-threaded one bit for bit."""
    import threading
    shapes = [(1, 4, 700, 128, True), (2, 2, 513, 64, False), (1, 3, 1000, 96, True), (2, 1, 300, 128, False)]
    inputs, expected = [], []
    for i, (B, H, N, d, causal) in enumerate(shapes):
        q, k, v = (t.cuda() for t in make_qkv(B, H, N, d, seed=90 + i))
        inputs.append((q, k, v, causal))
        expected.append(bos.attention(q, k, v, causal=causal))
    torch.cuda.synchronize()
    errors = []

    def worker(i):
        try:
            q, k, v, causal = inputs[i]
            s = torch.cuda.Stream()
            with torch.cuda.stream(s):
                for _ in range(20):
                    o, lse = bos.attention(q, k, v, causal=causal, stream=s)
            s.synchronize()
            if not (torch.equal(o, expected[i][0]) and torch.equal(lse, expected[i][1])):
                errors.append(f"thread {i}: result differs")
        except Exception as e:  # reported below, on the main thread
            errors.append(f"thread {i}: {e!r}")

    threads = [threading.Thread(target=worker, args=(i,)) for i in range(len(shapes))]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    assert not errors, errors
    assert bos.attn_device_status() == bos.ATTN_OK
