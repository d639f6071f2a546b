"""GPU parity of the standalone row softmax (fa_softmax_rows) against the fp64
CPU oracle ("5.2 CUDA Online Softmax": three-pass definition and the online
(m, d) normaliser), element by element.

Tolerances (fp32 in and out, ex2 of (x - m) log2 e per element, fp32 sums merged as
a tree): |y - y_ref| <= 2e-5 |y_ref| + 1e-37 per element (the absolute term
covers results below the fp32 normal range, which the kernel flushes to zero),
and |lse - lse_ref| <= 1e-5 max(1, |lse_ref|) per row.
"""
import math

import numpy as np
import pytest
import torch

import oracle

pytestmark = pytest.mark.gpu

Y_REL = 2e-5
Y_ABS = 1e-37
LSE_TOL = 1e-5


@pytest.fixture(scope="module")
def fa():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__

    __graft_entry__.build()
    import online_softmax_04_gb300 as m

    m.fa_clear_device_status()
    yield m
    assert m.fa_get_device_status() == 0, "a kernel gave up on a barrier"


def make_rows(M, N, seed, spread=1.0, masked=0.0):
    rng = np.random.default_rng(seed)
    x = (rng.standard_normal((M, N), dtype=np.float32) * np.float32(spread)).astype(np.float32)
    if masked > 0:
        x[rng.random((M, N)) < masked] = -np.inf
        x[np.arange(M), rng.integers(0, N, M)] = rng.standard_normal(M).astype(np.float32)  # keep one finite per row
    return x


def reference(x):
    y = np.empty(x.shape, dtype=np.float64)
    lse = np.empty(x.shape[0], dtype=np.float64)
    for i in range(x.shape[0]):
        row = x[i].astype(np.float64)
        y[i] = oracle.softmax_three_pass(row)
        _, m, d = oracle.softmax_online(row)
        lse[i] = m + math.log(d)
    return y, lse


def check(y_gpu, lse_gpu, x, label):
    ref_y, ref_lse = reference(x)
    y = y_gpu.astype(np.float64)
    err = np.abs(y - ref_y) - (Y_REL * np.abs(ref_y) + Y_ABS)
    worst = np.unravel_index(np.argmax(err), err.shape)
    rel = np.abs(y - ref_y) / np.maximum(np.abs(ref_y), 1e-30)
    msg = f"{label}: max rel dy={rel.max():.2e} at {tuple(int(i) for i in worst)}"
    assert np.all(np.isfinite(y)), label
    assert err.max() <= 0, msg
    if lse_gpu is not None:
        el = np.abs(lse_gpu.astype(np.float64) - ref_lse) / np.maximum(1.0, np.abs(ref_lse))
        msg += f" max rel dlse={el.max():.2e}"
        assert el.max() <= LSE_TOL, msg
    print(msg)


SHAPES = [  # (M, N) with N % 4 == 0: one warp per chunk of rows up to N = 2048 (chunks of 8 KB, the
    # last one partial), one CTA per row up to 4N = 100 KiB; other shapes: two sweeps of HBM
    (1, 1), (1, 4), (3, 5), (2, 7), (5, 1000), (37, 128), (1000, 64), (300, 1024), (9, 2048), (16, 4096),
    (3, 25600), (2, 25604), (2, 100003), (1000, 257),
]


@pytest.mark.parametrize("M,N", SHAPES)
@pytest.mark.parametrize("spread,masked", [(1.0, 0.0), (30.0, 0.1)])
def test_rows_against_oracle(fa, M, N, spread, masked):
    x = make_rows(M, N, seed=M * 7919 + N, spread=spread, masked=masked)
    xd = torch.from_numpy(x).cuda()
    y, lse = fa.softmax(xd)
    torch.cuda.synchronize()
    check(y.cpu().numpy(), lse.cpu().numpy(), x, f"M{M} N{N} spread{spread} masked{masked}")


def test_pages_shape_4096_square(fa):
    """The shape the pages measure their kernels on: 4096 x 4096 fp32, every element checked."""
    x = make_rows(4096, 4096, seed=4096)
    y, lse = fa.softmax(torch.from_numpy(x).cuda())
    torch.cuda.synchronize()
    check(y.cpu().numpy(), lse.cpu().numpy(), x, "4096x4096")


def test_empty_and_single_rows(fa):
    x = make_rows(4, 64, seed=3)
    x[0, :] = -np.inf                      # nothing finite: y = 0, lse = -inf
    x[1, :] = -np.inf
    x[1, 17] = 2.5                         # one finite value: one-hot
    y, lse = fa.softmax(torch.from_numpy(x).cuda())
    torch.cuda.synchronize()
    y, lse = y.cpu().numpy(), lse.cpu().numpy()
    assert np.all(y[0] == 0) and lse[0] == -np.inf
    assert y[1, 17] == 1.0 and np.all(np.delete(y[1], 17) == 0) and abs(lse[1] - 2.5) <= 1e-6
    check(y[2:], lse[2:], x[2:], "rows beside the degenerate ones")


def test_in_place_and_unaligned(fa):
    x = make_rows(64, 2048, seed=9)
    xd = torch.from_numpy(x).cuda()
    fa.fa_softmax_rows(xd, xd, None, 64, 2048)  # y = x
    torch.cuda.synchronize()
    check(xd.cpu().numpy(), None, x, "in place")
    # 4-byte aligned but not 16-byte aligned rows take the two-sweep path
    base = torch.from_numpy(np.concatenate([[0.0], make_rows(8, 1000, seed=10).ravel()]).astype(np.float32)).cuda()
    xs = base[1:]
    out = torch.empty(8 * 1000 + 1, dtype=torch.float32, device="cuda")[1:]
    lse = torch.empty(8, dtype=torch.float32, device="cuda")
    fa.fa_softmax_rows(xs, out, lse, 8, 1000)
    torch.cuda.synchronize()
    check(out.cpu().numpy().reshape(8, 1000), lse.cpu().numpy(), xs.cpu().numpy().reshape(8, 1000), "unaligned")


def test_rejects_bad_arguments(fa):
    x = torch.zeros(4, 16, dtype=torch.float32, device="cuda")
    y = torch.empty_like(x)
    L = fa.lib()
    assert L.fa_softmax_rows(0, y.data_ptr(), 0, 4, 16, 0) == fa.FA_ERR_NULL_POINTER
    assert L.fa_softmax_rows(x.data_ptr(), y.data_ptr(), 0, 0, 16, 0) == fa.FA_ERR_SHAPE
    assert L.fa_softmax_rows(x.data_ptr() + 2, y.data_ptr(), 0, 4, 16, 0) == fa.FA_ERR_ALIGNMENT
    assert L.fa_softmax_rows(x.data_ptr() + 4, x.data_ptr(), 0, 4, 16, 0) == fa.FA_ERR_ALIAS
