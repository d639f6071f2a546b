"""GPU parity of the split-KV forward (fa_fwd_splitkv + merge) against the
fp64 oracle, with the same tolerances as fa_fwd."""
import numpy as np
import pytest
import torch

from online_softmax_04_gb300 import workloads as wl
from tests.test_fa_gpu import all_rows, compare, fa  # noqa: F401  (fixture)

pytestmark = pytest.mark.gpu


def run_split(fa, q, k, v, causal, scale, n_splits):
    dev = torch.device("cuda:0")
    o, lse = fa.attention_splitkv(q.to(dev), k.to(dev), v.to(dev), causal=causal, scale=scale, n_splits=n_splits)
    torch.cuda.synchronize()
    return o.float().cpu().numpy(), lse.cpu().numpy()


@pytest.mark.parametrize("name", ["B1-H1-N256-d64-full", "B1-H1-N256-d64-full-sorted-strict",
                                  "B1-H1-N4096-d64-full"])
def test_small_workloads_auto_splits(fa, name):
    w = wl.WORKLOADS[name]
    q, k, v = wl.make_inputs(w)
    o, lse = run_split(fa, q, k, v, w.causal, w.scale, 0)
    compare(o, lse, q, k, v, w.causal, w.scale, wl.sample_rows(w), name + " split-KV auto")


@pytest.mark.parametrize("B,H,N,d,causal,splits", [
    (1, 1, 1000, 64, True, 5),    # early causal tiles get empty chunks
    (1, 2, 1000, 128, False, 3),
    (2, 1, 129, 128, True, 2),    # ragged tail
    (1, 1, 640, 64, False, 1),
    (1, 1, 640, 64, False, 64),   # more splits than key tiles
    (3, 2, 300, 128, True, 7),
])
def test_small_shapes_explicit_splits(fa, B, H, N, d, causal, splits):
    w = wl.Workload("split", B, H, N, d, causal, "iid", 300 + N + splits)
    q, k, v = wl.make_inputs(w)
    o, lse = run_split(fa, q, k, v, causal, w.scale, splits)
    compare(o, lse, q, k, v, causal, w.scale, all_rows(B, H, N), f"B{B} H{H} N{N} d{d} causal={causal} S={splits}")


def test_late_workload_two_splits_sampled(fa):
    w = wl.WORKLOADS["B1-H32-N16384-d128-causal-late"].with_(H=4, rows_per_head=128)
    q, k, v = wl.make_inputs(w)
    o, lse = run_split(fa, q, k, v, True, w.scale, 2)
    compare(o, lse, q, k, v, True, w.scale, wl.sample_rows(w), "late H4 split-KV S=2")


def test_split_matches_single_pass(fa):
    w = wl.Workload("cmp", 2, 2, 1500, 128, True, "iid", 9)
    q, k, v = (t.cuda() for t in wl.make_inputs(w))
    o1, l1 = fa.attention(q, k, v, causal=True)
    o2, l2 = fa.attention_splitkv(q, k, v, causal=True, n_splits=4)
    torch.cuda.synchronize()
    assert (o1.float() - o2.float()).abs().max().item() <= 2e-2
    assert ((l1 - l2).abs() / l1.abs().clamp(min=1)).max().item() <= 1e-3


def test_splitkv_workspace_too_small_is_rejected(fa):
    q = torch.zeros((1, 1, 256, 64), dtype=torch.bfloat16, device="cuda")
    o = torch.empty_like(q)
    lse = torch.empty((1, 1, 256), dtype=torch.float32, device="cuda")
    ws = torch.empty(16, dtype=torch.uint8, device="cuda")
    with pytest.raises(fa.FaError) as e:
        fa.fa_fwd_splitkv(q, q, q, o, lse, 1, 1, 256, 64, False, 0.125, 2, ws, 16)
    assert e.value.code == fa.FA_ERR_WORKSPACE
