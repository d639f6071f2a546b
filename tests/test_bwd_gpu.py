"""GPU parity of the backward pass (fa_bwd) against the fp64 CPU oracle.

The forward outputs the backward consumes (O in bf16, LSE in fp32) come from
the oracle's own forward, rounded to the kernel's storage types; the same
values go to the GPU backward and to the oracle backward, so no expected value
depends on the CUDA path.

Tolerance per element: |g - g_ref| <= 2^-8 (mag + |g_ref|) + 2^-16 max|g_ref| + 1e-6,
where mag is the oracle's sum of |term| over the element's contributions and
the max runs over the whole tensor.  Each gradient is a sum of products with
one bf16-rounded factor (P for dV, dS for dQ and dK: relative 2^-9 each)
accumulated in fp32, then rounded to bf16 (2^-9 of the result); the first term
doubles both.  dS = P (dP - D) also carries the fp32 accumulation error of dP
(d products) and of D, which does not shrink with the element's own terms when
dP and D nearly cancel; the second term (about 1.5e-5 of the tensor's largest
element) covers it.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from online_softmax_04_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


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


def make_case(B, H, N, d, causal, seed, dist="iid"):
    w = wl.Workload("bwd", B, H, N, d, causal, dist, seed)
    q, k, v = wl.make_inputs(w)
    rng = np.random.default_rng(seed + 1)
    dout = torch.from_numpy(rng.standard_normal((B, H, N, d), dtype=np.float32)).to(torch.bfloat16)
    o, lse = oracle.attention_three_pass(q, k, v, causal, w.scale)       # fp64, from the oracle
    o_bf = torch.from_numpy(o.reshape(B, H, N, d)).to(torch.bfloat16)      # what the forward stores
    lse_f = torch.from_numpy(lse.reshape(B, H, N)).to(torch.float32)
    return w, q, k, v, dout, o_bf, lse_f


def check(fa, B, H, N, d, causal, seed, q_rows=None, k_rows=None, label="", dist="iid"):
    w, q, k, v, dout, o_bf, lse_f = make_case(B, H, N, d, causal, seed, dist)
    dev = torch.device("cuda:0")
    dq, dk, dv = fa.attention_backward(*(t.to(dev) for t in (q, k, v, o_bf, lse_f, dout)), causal=causal)
    torch.cuda.synchronize()
    ref = oracle.attention_backward(q, k, v, o_bf, dout, lse_f, causal, w.scale, q_rows=q_rows, k_rows=k_rows)
    qr = np.arange(B * H * N) if q_rows is None else np.asarray(q_rows)
    kr = np.arange(B * H * N) if k_rows is None else np.asarray(k_rows)
    msg = [label]
    for name, got, rows in (("dq", dq, qr), ("dk", dk, kr), ("dv", dv, kr)):
        g = got.float().cpu().numpy().reshape(-1, d)[rows].astype(np.float64)
        r, mag = ref[name], ref["mag_" + name]
        excess = np.abs(g - r) - (2.0 ** -8 * (mag + np.abs(r)) + 2.0 ** -16 * np.abs(r).max() + 1e-6)
        rel = np.abs(g - r).max() / max(np.abs(r).max(), 1e-30)
        msg.append(f"{name}: max|d|={np.abs(g - r).max():.2e} (rel to max {rel:.2e})")
        assert np.all(np.isfinite(g)), name
        assert excess.max() <= 0, " ".join(msg) + f" worst excess {excess.max():.2e}"
    print(" ".join(msg))


SHAPES = [(1, 1, 1, 64, False), (1, 1, 1, 128, True), (1, 2, 130, 64, True), (2, 1, 257, 128, True),
          (1, 2, 300, 128, False), (1, 1, 1000, 64, True), (2, 2, 384, 64, False), (1, 1, 640, 128, True)]


@pytest.mark.parametrize("B,H,N,d,causal", SHAPES)
def test_backward_every_row(fa, B, H, N, d, causal):
    check(fa, B, H, N, d, causal, seed=N * 3 + d, label=f"B{B}H{H}N{N}d{d} causal={causal}")


@pytest.mark.parametrize("d,causal", [(128, True), (64, True), (64, False)])
def test_backward_late_max_rows_sampled(fa, d, causal):
    """Large, growing scores (the late-max distribution) at N = 2048, sampled rows: 16 query
    steps per key tile (up to 16 per query tile), many turns of every barrier's phase."""
    B, H, N = 1, 4, 2048
    rng = np.random.default_rng(5)
    rows = np.unique(np.concatenate([rng.integers(0, B * H * N, 200), [0, N - 1, B * H * N - 1]])).astype(np.int64)
    check(fa, B, H, N, d, causal, seed=77 + d, q_rows=rows, k_rows=rows[::-1].copy(),
          label=f"late N2048 d{d} causal={causal}", dist="late")


def test_zero_upstream_gradient_gives_zero(fa):
    B, H, N, d = 1, 2, 200, 64
    w, q, k, v, dout, o_bf, lse_f = make_case(B, H, N, d, True, 3)
    dev = torch.device("cuda:0")
    dq, dk, dv = fa.attention_backward(*(t.to(dev) for t in (q, k, v, o_bf, lse_f)), torch.zeros_like(dout).to(dev),
                                       causal=True)
    torch.cuda.synchronize()
    assert not dq.any() and not dk.any() and not dv.any()


def test_rejects_bad_arguments(fa):
    t = torch.zeros((1, 1, 128, 64), dtype=torch.bfloat16, device="cuda")
    o, dq, dk, dv = (torch.empty_like(t) for _ in range(4))
    lse = torch.zeros((1, 1, 128), dtype=torch.float32, device="cuda")
    ws = torch.empty(fa.fa_bwd_workspace_bytes(1, 1, 128, 64), dtype=torch.uint8, device="cuda")
    L = fa.lib()
    P = t.data_ptr()

    def call(**kw):
        a = dict(q=P, k=P, v=P, o=o.data_ptr(), do=P, lse=lse.data_ptr(), dq=dq.data_ptr(), dk=dk.data_ptr(),
                 dv=dv.data_ptr(), d=64, ws=ws.data_ptr(), wsb=ws.numel())
        a.update(kw)
        return L.fa_bwd(a["q"], a["k"], a["v"], a["o"], a["do"], a["lse"], a["dq"], a["dk"], a["dv"], 1, 1, 128,
                        a["d"], 1, 0.125, a["ws"], a["wsb"], 0)

    assert call(dq=0) == fa.FA_ERR_NULL_POINTER
    assert call(d=96) == fa.FA_ERR_HEAD_DIM
    assert call(wsb=ws.numel() - 4) == fa.FA_ERR_WORKSPACE
    assert call(dk=dq.data_ptr()) == fa.FA_ERR_ALIAS
    assert call(dv=P) == fa.FA_ERR_ALIAS
    assert call(q=P + 2) == fa.FA_ERR_ALIGNMENT
