"""fa_fwd_splitkv_noalloc: the split-KV forward for callers that cannot
allocate device memory when they run attention (their memory belongs to a
host framework or a fixed budget, or the path cannot afford cudaMalloc).  Its
partial states live in a static array inside the library instead of a
caller workspace.

Two calls in a row go through the C ABI and are checked against the
workspace entry point fa_fwd_splitkv on the same inputs; the second call is
smaller than the first, so it runs over whatever the first left behind.
"""
import ctypes

import pytest
import torch

from online_softmax_04_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

O_TOL = 2e-2
LSE_TOL = 1e-3


@pytest.fixture(scope="module")
def fa():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__

    __graft_entry__.build()
    import online_softmax_04_gb300 as m

    torch.cuda.set_device(0)
    m.fa_clear_device_status()
    yield m
    assert m.fa_get_device_status() == 0, "a kernel gave up on a barrier"


def noalloc_via_c_abi(fa, q, k, v, causal, scale, n_splits):
    B, H, N, d = q.shape
    o = torch.empty_like(q)
    lse = torch.empty((B, H, N), dtype=torch.float32, device=q.device)
    stream = torch.cuda.current_stream().cuda_stream
    rc = fa.lib().fa_fwd_splitkv_noalloc(
        ctypes.c_void_p(q.data_ptr()), ctypes.c_void_p(k.data_ptr()), ctypes.c_void_p(v.data_ptr()),
        ctypes.c_void_p(o.data_ptr()), ctypes.c_void_p(lse.data_ptr()), B, H, N, d, 1 if causal else 0,
        ctypes.c_float(scale), n_splits, ctypes.c_void_p(stream))
    return rc, o, lse


def test_noalloc_matches_workspace_entry_point_on_two_calls(fa):
    cases = [
        wl.Workload("noalloc-1", 1, 2, 2048, 128, True, "iid", 501),   # 4 splits: 4*4096*131*4 B = 8.6 MB
        wl.Workload("noalloc-2", 2, 1, 777, 64, False, "iid", 502),    # smaller, ragged: reuses a dirty scratch
    ]
    for w, n_splits in zip(cases, (4, 3)):
        q, k, v = (t.cuda() for t in wl.make_inputs(w))
        rc, o1, l1 = noalloc_via_c_abi(fa, q, k, v, w.causal, w.scale, n_splits)
        assert rc == fa.FA_OK, fa.fa_strerror(rc)
        o2, l2 = fa.attention_splitkv(q, k, v, causal=w.causal, scale=w.scale, n_splits=n_splits)
        torch.cuda.synchronize()
        assert torch.isfinite(o1.float()).all() and torch.isfinite(l1).all()
        assert (o1.float() - o2.float()).abs().max().item() <= O_TOL, w.name
        assert ((l1 - l2).abs() / l2.abs().clamp(min=1)).max().item() <= LSE_TOL, w.name


def test_noalloc_rejects_problems_larger_than_the_scratch(fa):
    B, H, N, d = 1, 8, 16384, 128  # 2 splits need 2*131072*131*4 B = 137 MB > 32 MiB
    q = torch.zeros((B, H, N, d), dtype=torch.bfloat16, device="cuda")
    o = torch.empty_like(q)
    lse = torch.full((B, H, N), 7.0, dtype=torch.float32, device="cuda")
    rc, _, _ = noalloc_via_c_abi(fa, q, q, q, True, 0.125, 2)
    assert rc == fa.FA_ERR_SCRATCH_LIMIT
    assert fa.fa_splitkv_workspace_bytes(B, H, N, d, 2) > fa.FA_NOALLOC_SCRATCH_BYTES
