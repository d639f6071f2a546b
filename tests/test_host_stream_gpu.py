"""fa_fwd_host: the forward on host-resident tensors, streamed through a three-slot
device workspace in chunks of heads.  The per-tile arithmetic is the one fa_fwd
runs, so the results must equal fa_fwd's bit for bit (fa_fwd itself is held to
the fp64 oracle in test_fa_gpu.py); every chunking, ragged last chunk, pinned
and pageable host memory, and back-to-back calls that reuse one workspace.
"""
import numpy as np
import pytest
import torch

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


def host_inputs(w, pinned):
    q, k, v = wl.make_inputs(w)
    if pinned:
        q, k, v = (t.pin_memory() for t in (q, k, v))
    return q, k, v


CASES = [  # (B, H, N, d, causal, heads_per_chunk, pinned)
    (2, 3, 200, 64, True, 2, True),      # chunks of 2 heads, ragged N
    (1, 5, 1000, 128, True, 0, True),    # automatic: ceil(5 / 8) = 1 head per chunk
    (2, 4, 384, 128, False, 3, False),   # pageable host memory; chunks 3, 3, 2
    (1, 2, 129, 64, False, 2, True),     # one chunk holds every head
    (1, 16, 2048, 128, True, 4, True),   # four chunks, several persistent rounds each
    (1, 7, 513, 64, True, 1, True),      # seven chunks: every one of the three slots reused
    (4, 16, 4096, 64, True, 0, True),    # d = 64, 64 heads: two tiles per CTA, also in every 8-head chunk
]


@pytest.mark.parametrize("B,H,N,d,causal,hpc,pinned", CASES)
def test_equals_device_forward(fa, B, H, N, d, causal, hpc, pinned):
    w = wl.Workload("host", B, H, N, d, causal, "iid", 31 + N)
    q, k, v = host_inputs(w, pinned)
    o, lse = fa.attention_host(q, k, v, causal=causal, heads_per_chunk=hpc)
    torch.cuda.synchronize()
    ro, rl = fa.attention(q.cuda(), k.cuda(), v.cuda(), causal=causal)
    torch.cuda.synchronize()
    assert torch.equal(o, ro.cpu()) and torch.equal(lse, rl.cpu())


def test_back_to_back_calls_share_a_workspace(fa):
    """Two calls on one stream with one workspace: the second call's copies into
    the slots wait for the first call's read-backs."""
    wa = wl.Workload("ha", 1, 6, 1500, 128, True, "iid", 41)
    wb = wl.Workload("hb", 1, 6, 1500, 128, True, "late", 42)
    qa, ka, va = host_inputs(wa, True)
    qb, kb, vb = host_inputs(wb, True)
    ws = torch.empty(fa.fa_fwd_host_workspace_bytes(1, 6, 1500, 128, 2), dtype=torch.uint8, device="cuda")
    oa, la = fa.attention_host(qa, ka, va, causal=True, heads_per_chunk=2, workspace=ws)
    ob, lb = fa.attention_host(qb, kb, vb, causal=True, heads_per_chunk=2, workspace=ws)
    torch.cuda.synchronize()
    for (o, l), (q, k, v) in (((oa, la), (qa, ka, va)), ((ob, lb), (qb, kb, vb))):
        ro, rl = fa.attention(q.cuda(), k.cuda(), v.cuda(), causal=True)
        torch.cuda.synchronize()
        assert torch.equal(o, ro.cpu()) and torch.equal(l, rl.cpu())


def test_stream_order_with_later_device_work(fa):
    """Work enqueued on the caller's stream after the call sees its outputs:
    a device copy of o made on the same stream equals the host result."""
    w = wl.Workload("hs", 1, 4, 700, 64, True, "iid", 43)
    q, k, v = host_inputs(w, True)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        o, lse = fa.attention_host(q, k, v, causal=True, heads_per_chunk=1, stream=s)
        dev = torch.empty(o.shape, dtype=o.dtype, device="cuda")
        dev.copy_(o, non_blocking=True)   # ordered after the read-back into o
    s.synchronize()
    assert torch.equal(dev.cpu(), o)
    assert np.isfinite(lse.numpy()).all()
