"""GPU parity of the fused row softmax (softmax_rows_fwd) against the fp64 oracle.

Tolerance: |y - y_ref| <= 1e-6 + 1e-5 |y_ref| element by element, the check the
"Triton" page applies to its fused softmax (assert_close against the library
softmax with rtol 1e-5, atol 1e-6); fp32 output of a ~1e-7-accurate exp2.
"""
import numpy as np
import pytest
import torch

import blocked_online_softmax_gb300 as bos
import oracle

pytestmark = pytest.mark.gpu

RTOL, ATOL = 1e-5, 1e-6
SENT = -7.0e30


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()
    oracle.build()
    torch.cuda.set_device(0)


def check(y, y_ref, what):
    y = np.asarray(y, dtype=np.float64)
    err = np.abs(y - y_ref) - (ATOL + RTOL * np.abs(y_ref))
    worst = np.unravel_index(np.argmax(err), err.shape)
    assert err.max() <= 0, f"{what}: |y - y_ref| = {abs(y[worst] - y_ref[worst]):.3e} at {worst} (ref {y_ref[worst]:.3e})"


def run_strided(x_host, pad_cols=0, in_place=False):
    """x_host [rows, cols] fp32 numpy; rows may be strided (pad_cols extra columns per row).

    The output buffer is strided the same way and pre-filled with a sentinel: the
    padding columns and a guard row after the last must keep it."""
    rows, cols = x_host.shape
    ld = cols + pad_cols
    xb = torch.full((rows + 1, ld), SENT, dtype=torch.float32)
    xb[:rows, :cols] = torch.from_numpy(x_host)
    xd = xb.cuda()
    yd = xd if in_place else torch.full((rows + 1, ld), SENT, dtype=torch.float32, device="cuda")
    bos.softmax_rows_fwd(xd, yd, rows, cols, ld, ld, None)
    torch.cuda.synchronize()
    yh = yd.cpu().numpy()
    if not in_place:
        assert np.all(yh[:rows, cols:] == SENT) and np.all(yh[rows] == SENT), "wrote outside the rows"
    return yh[:rows, :cols]


@pytest.mark.parametrize("shape, mult", [((1823, 781), 1.0), ((123, 781), 10.0), ((4096, 4096), 1.0)])
def test_pages_shapes(shape, mult):
    """The pages' own examples: 1823 x 781, 123 x 781 scaled by 10, and 4096 x 4096."""
    g = torch.Generator().manual_seed(sum(shape))
    x = (torch.randn(shape, generator=g) * mult).numpy()
    xd = torch.from_numpy(x).cuda()
    y = bos.softmax(xd)
    torch.cuda.synchronize()
    check(y.cpu().numpy(), oracle.softmax_rows(x), f"{shape} x{mult}")


@pytest.mark.parametrize("cols", [1, 3, 4, 31, 128, 129, 1000, 1024, 1025, 4096, 5000, 16384, 16385, 70000])
@pytest.mark.parametrize("rows", [1, 7, 300])
def test_widths_and_paths(rows, cols):
    """One-warp rows, block rows, the widest on-chip rows and the online two-pass path."""
    if rows * cols > 6_000_000:
        pytest.skip("kept small")
    rng = np.random.default_rng(rows * 100003 + cols)
    x = (rng.standard_normal((rows, cols)) * 5).astype(np.float32)
    check(run_strided(x), oracle.softmax_rows(x), f"{rows}x{cols}")


@pytest.mark.parametrize("cols, pad", [(781, 219), (512, 512), (20000, 3)])
def test_strided_rows(cols, pad):
    rng = np.random.default_rng(cols + pad)
    x = (rng.standard_normal((37, cols)) * 3).astype(np.float32)
    check(run_strided(x, pad_cols=pad), oracle.softmax_rows(x), f"37x{cols} stride {cols + pad}")


@pytest.mark.parametrize("cols", [781, 4096, 20000])
def test_in_place(cols):
    rng = np.random.default_rng(cols)
    x = (rng.standard_normal((9, cols)) * 4).astype(np.float32)
    check(run_strided(x, in_place=True), oracle.softmax_rows(x), f"in place 9x{cols}")


@pytest.mark.parametrize("cols", [100, 3000, 30000])
def test_masked_and_large_logits(cols):
    """-inf entries contribute nothing; logits in the hundreds do not overflow."""
    rng = np.random.default_rng(7 + cols)
    x = (rng.standard_normal((5, cols)) * 200).astype(np.float32)
    x[:, ::3] = -np.inf
    x[0, :] = -np.inf
    x[0, cols // 2] = 0.0                      # a row with one finite entry -> one-hot
    check(run_strided(x), oracle.softmax_rows(x), f"masked 5x{cols}")
