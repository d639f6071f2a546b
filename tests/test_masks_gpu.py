"""GPU parity of the masked forward (fa_fwd_masked: sliding windows and
document boundaries) against the fp64 CPU oracle's masked three-pass route,
element by element.  Tolerances as for the unmasked forward: max |dO| <= 2e-2,
|dLSE| / max(1, |LSE|) <= 1e-3.
"""
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

    m.fa_clear_device_status()
    yield m
    assert m.fa_get_device_status() == 0, "a kernel gave up on a barrier"


def doc_ids(B, N, seed, mean_len):
    """Seeded document ids: runs of random length (some of length 1), non-decreasing per sequence."""
    rng = np.random.default_rng(seed)
    out = np.zeros((B, N), dtype=np.int32)
    for b in range(B):
        pos, doc = 0, 0
        while pos < N:
            n = 1 if rng.random() < 0.15 else int(rng.integers(1, 2 * mean_len))
            out[b, pos:pos + n] = doc
            pos += n
            doc += 1
    return out


def check(fa, B, H, N, d, wl_, wr_, docs, seed, rows=None, label=""):
    w = wl.Workload("mask", B, H, N, d, False, "iid", seed)
    q, k, v = wl.make_inputs(w)
    dev = torch.device("cuda:0")
    doc_t = torch.from_numpy(docs).to(dev) if docs is not None else None
    o, lse = fa.attention_masked(q.to(dev), k.to(dev), v.to(dev), wl_, wr_, doc_t)
    torch.cuda.synchronize()
    if rows is None:
        rows = np.arange(B * H * N, dtype=np.int64)
    ref_o, ref_lse = oracle.attention_masked(q, k, v, w.scale, wl_, wr_, docs, rows=rows)
    got_o = o.float().cpu().numpy().reshape(-1, d)[rows].astype(np.float64)
    got_l = lse.cpu().numpy().reshape(-1)[rows].astype(np.float64)
    err_o = np.abs(got_o - ref_o).max()
    err_l = (np.abs(got_l - ref_lse) / np.maximum(1.0, np.abs(ref_lse))).max()
    msg = f"{label}: max|dO|={err_o:.3e} max rel dLSE={err_l:.3e} rows={len(rows)}"
    print(msg)
    assert np.all(np.isfinite(got_o)) and np.all(np.isfinite(got_l)), msg
    assert err_o <= O_TOL and err_l <= LSE_TOL, msg


WINDOWS = [  # (B, H, N, d, window_left, window_right)
    (1, 2, 1000, 128, 99, 0),     # causal sliding window of 100 keys
    (2, 2, 700, 64, 128, 128),    # bidirectional band of 257 keys, tile-aligned bounds
    (1, 1, 300, 64, 0, 0),        # the diagonal only
    (1, 2, 1500, 64, 300, -1),    # left window, unbounded right
    (1, 1, 513, 128, -1, 5),      # unbounded left, five keys ahead
    (1, 3, 2000, 128, 1023, 0),   # causal window spanning eight key tiles
]


@pytest.mark.parametrize("B,H,N,d,wl_,wr_", WINDOWS)
def test_windows_every_row(fa, B, H, N, d, wl_, wr_):
    check(fa, B, H, N, d, wl_, wr_, None, seed=N + d, label=f"window({wl_},{wr_}) B{B}H{H}N{N}d{d}")


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("B,H,N,d,mean_len", [(2, 2, 900, 64, 150), (1, 2, 1300, 128, 400), (3, 1, 257, 128, 20)])
def test_documents_every_row(fa, causal, B, H, N, d, mean_len):
    docs = doc_ids(B, N, seed=N, mean_len=mean_len)
    check(fa, B, H, N, d, -1, 0 if causal else -1, docs, seed=N + 1,
          label=f"docs(mean {mean_len}) causal={causal} B{B}H{H}N{N}d{d}")


def test_documents_and_window(fa):
    docs = doc_ids(2, 1100, seed=5, mean_len=300)
    check(fa, 2, 2, 1100, 128, 200, 0, docs, seed=6, label="docs + causal window 201")


def test_one_document_per_sequence_and_one_token_documents(fa):
    N = 400
    check(fa, 2, 1, N, 64, -1, 0, np.zeros((2, N), dtype=np.int32), seed=7, label="one document")
    check(fa, 1, 1, N, 64, -1, -1, np.arange(N, dtype=np.int32)[None, :], seed=8, label="one token per document")


def test_large_sliding_window_sampled_rows(fa):
    """Many query tiles through the persistent schedule: B1 H8 N8192 d128, causal window of 1024."""
    B, H, N, d = 1, 8, 8192, 128
    rng = np.random.default_rng(9)
    rows = np.unique(np.concatenate([rng.integers(0, B * H * N, 512),
                                     np.arange(0, B * H * N, N), np.arange(N - 1, B * H * N, N)]))
    check(fa, B, H, N, d, 1023, 0, None, seed=10, rows=rows.astype(np.int64), label="N8192 window 1024")


def test_documents_at_the_largest_batch(fa):
    """B = 65535 sequences, each with its own document ids (the per-batch doc
    offset at its largest), sampled rows including the last sequence."""
    B, H, N, d = 65535, 1, 65, 64
    docs = doc_ids(B, N, seed=21, mean_len=20)
    rng = np.random.default_rng(22)
    rows = np.unique(np.concatenate([rng.integers(0, B * H * N, 600), [0, B * H * N - 1]])).astype(np.int64)
    check(fa, B, H, N, d, -1, 0, docs, seed=23, rows=rows, label="documents, B = 65535")


def test_trivial_masks_equal_fa_fwd_bit_for_bit(fa):
    w = wl.Workload("eq", 1, 2, 777, 128, True, "iid", 12)
    q, k, v = (t.cuda() for t in wl.make_inputs(w))
    for causal, wr in ((True, 0), (False, -1)):
        o1, l1 = fa.attention(q, k, v, causal=causal)
        o2, l2 = fa.attention_masked(q, k, v, -1, wr, None)
        torch.cuda.synchronize()
        assert torch.equal(o1, o2) and torch.equal(l1, l2), causal


def test_rejects_bad_masks(fa):
    q = torch.zeros((1, 1, 128, 64), dtype=torch.bfloat16, device="cuda")
    o = torch.empty_like(q)
    lse = torch.empty((1, 1, 128), dtype=torch.float32, device="cuda")
    docs = torch.zeros((1, 129), dtype=torch.int32, device="cuda")
    L = fa.lib()
    p = q.data_ptr()
    assert L.fa_fwd_masked(p, p, p, o.data_ptr(), lse.data_ptr(), 1, 1, 128, 64, -2, 0, None, 0.1, 0) == fa.FA_ERR_MASK
    assert L.fa_fwd_masked(p, p, p, o.data_ptr(), lse.data_ptr(), 1, 1, 128, 64, 3, -5, None, 0.1, 0) == fa.FA_ERR_MASK
    assert L.fa_fwd_masked(p, p, p, o.data_ptr(), lse.data_ptr(), 1, 1, 128, 64, -1, 0, docs.data_ptr() + 2, 0.1,
                           0) == fa.FA_ERR_ALIGNMENT
    assert L.fa_fwd_masked(p, p, p, o.data_ptr(), lse.data_ptr(), 1, 1, 128, 64, -1, 0, o.data_ptr(), 0.1,
                           0) == fa.FA_ERR_ALIAS


@pytest.mark.parametrize("name", ["B1-H32-N16384-d128-window4096", "B4-H16-N4096-d128-docs"])
def test_masked_workloads_sampled_rows(fa, name):
    """The masked workloads bench.py measures, at full size, in the launch it times."""
    w = wl.WORKLOADS[name]
    q, k, v = wl.make_inputs(w)
    docs = wl.make_doc_ids(w)
    dev = torch.device("cuda:0")
    o, lse = fa.attention_masked(q.to(dev), k.to(dev), v.to(dev), w.window_left, w.window_right,
                                 torch.from_numpy(docs).to(dev) if docs is not None else None)
    torch.cuda.synchronize()
    rows = wl.sample_rows(w)
    ref_o, ref_lse = oracle.attention_masked(q, k, v, w.scale, w.window_left, w.window_right, docs, rows=rows)
    got_o = o.float().cpu().numpy().reshape(-1, w.d)[rows].astype(np.float64)
    got_l = lse.cpu().numpy().reshape(-1)[rows].astype(np.float64)
    err_o = np.abs(got_o - ref_o).max()
    err_l = (np.abs(got_l - ref_lse) / np.maximum(1.0, np.abs(ref_lse))).max()
    print(f"{name}: max|dO|={err_o:.3e} max rel dLSE={err_l:.3e} rows={len(rows)}")
    assert err_o <= O_TOL and err_l <= LSE_TOL
