"""fa_fwd_splitkv_noalloc: the split-KV forward for callers that cannot
allocate device memory when they run attention (their memory belongs to a
host framework or a fixed budget, or the path cannot afford cudaMalloc).  Its
partial states live in a static array inside the library instead of a
caller workspace.

Calls in a row go through the C ABI.  Each is checked against the workspace
entry point fa_fwd_splitkv on the same inputs and split count: both run the
same split kernel and merge, so the outputs must be identical bit for bit.
The second call runs over the partial states the first left in the shared
array: it is causal with more splits than the first query tiles have key
tiles, so its empty splits must overwrite stale finite states; that call is
also compared with the oracle, element by element, on every row.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
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
    o = torch.full_like(q, float("nan"))
    lse = torch.full((B, H, N), float("nan"), dtype=torch.float32, device=q.device)
    stream = torch.cuda.current_stream().cuda_stream
    rc = fa.lib().fa_fwd_splitkv_noalloc(
        ctypes.c_void_p(q.data_ptr()), ctypes.c_void_p(k.data_ptr()), ctypes.c_void_p(v.data_ptr()),
        ctypes.c_void_p(o.data_ptr()), ctypes.c_void_p(lse.data_ptr()), B, H, N, d, 1 if causal else 0,
        ctypes.c_float(scale), n_splits, ctypes.c_void_p(stream))
    return rc, o, lse


def check_against_workspace_entry_point(fa, w, n_splits):
    q, k, v = (t.cuda() for t in wl.make_inputs(w))
    rc, o1, l1 = noalloc_via_c_abi(fa, q, k, v, w.causal, w.scale, n_splits)
    assert rc == fa.FA_OK, fa.fa_strerror(rc)
    splits = n_splits or fa.fa_splitkv_auto_splits(w.B, w.H, w.N, w.d, w.causal)
    o2, l2 = fa.attention_splitkv(q, k, v, causal=w.causal, scale=w.scale, n_splits=splits)
    torch.cuda.synchronize()
    assert torch.isfinite(o1.float()).all() and torch.isfinite(l1).all(), w.name
    assert torch.equal(o1, o2), f"{w.name}: o differs from fa_fwd_splitkv"
    assert torch.equal(l1, l2), f"{w.name}: lse differs from fa_fwd_splitkv"
    return q, k, v, o1, l1


def test_noalloc_matches_workspace_entry_point_on_two_calls(fa):
    # 1: fills the array with finite partial states (4 splits: 4*4096*131*4 B = 8.6 MB)
    check_against_workspace_entry_point(fa, wl.Workload("noalloc-1", 1, 2, 2048, 128, True, "iid", 501), 4)
    # 2: causal, ragged, 7 key tiles in 5 splits: query tiles 0-3 leave splits empty,
    # which must replace the stale states of call 1 with empty ones
    w = wl.Workload("noalloc-2", 2, 1, 777, 64, True, "iid", 502)
    q, k, v, o, lse = check_against_workspace_entry_point(fa, w, 5)
    rows = np.arange(w.B * w.H * w.N, dtype=np.int64)
    ref_o, ref_lse = oracle.attention_three_pass(q.cpu(), k.cpu(), v.cpu(), True, w.scale, rows=rows)
    got_o = o.float().cpu().numpy().reshape(-1, w.d).astype(np.float64)
    got_l = lse.cpu().numpy().reshape(-1).astype(np.float64)
    assert np.abs(got_o - ref_o).max() <= O_TOL
    assert (np.abs(got_l - ref_lse) / np.maximum(1.0, np.abs(ref_lse))).max() <= LSE_TOL


def test_noalloc_automatic_split_count(fa):
    # n_splits = 0: the automatic count (4 on a 152-SM GB300 for 32 query tiles)
    w = wl.Workload("noalloc-auto", 1, 1, 4096, 128, False, "iid", 503)
    auto = fa.fa_splitkv_auto_splits(w.B, w.H, w.N, w.d, w.causal)
    assert auto > 1
    # the automatic count fills one wave, so its states take at most about
    # SMs * 128 rows * (d + 3) * 4 bytes: always inside the array on this device
    assert fa.fa_splitkv_workspace_bytes(w.B, w.H, w.N, w.d, auto) <= fa.FA_NOALLOC_SCRATCH_BYTES
    check_against_workspace_entry_point(fa, w, 0)


def test_noalloc_rejects_problems_larger_than_the_scratch(fa):
    B, H, N, d = 1, 8, 16384, 128  # 2 splits need 2*131072*131*4 B = 137 MB > 32 MiB
    q = torch.zeros((B, H, N, d), dtype=torch.bfloat16, device="cuda")
    rc, o, lse = noalloc_via_c_abi(fa, q, q, q, True, 0.125, 2)
    torch.cuda.synchronize()
    assert rc == fa.FA_ERR_SCRATCH_LIMIT
    assert fa.fa_splitkv_workspace_bytes(B, H, N, d, 2) > fa.FA_NOALLOC_SCRATCH_BYTES
    assert torch.isnan(lse).all()  # nothing was enqueued
