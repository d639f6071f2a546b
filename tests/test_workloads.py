"""The seeded input generators: determinism, shapes and the stated structure."""
import numpy as np
import torch

from online_softmax_04_gb300 import workloads as wl


def test_deterministic_and_bf16():
    w = wl.Workload("t", 1, 2, 100, 64, False, "iid", 5)
    a = wl.make_inputs(w)
    b = wl.make_inputs(w)
    for x, y in zip(a, b):
        assert x.dtype == torch.bfloat16 and x.shape == (1, 2, 100, 64) and x.is_contiguous()
        assert torch.equal(x, y)
    assert not torch.equal(a[0], a[1])


def test_late_workload_key_norms_grow_linearly():
    w = wl.WORKLOADS["B1-H32-N16384-d128-causal-late"].with_(H=1, N=2048)
    q, k, v = wl.make_inputs(w)
    norms = k[0, 0].float().norm(dim=1).numpy()
    ramp = 0.25 + 3.75 * np.arange(2048) / 2047
    ratio = norms / (ramp * np.sqrt(128))
    assert abs(np.median(ratio) - 1) < 0.05
    assert np.corrcoef(norms, ramp)[0, 1] > 0.95
    assert abs(q.float().std().item() - 4.0) < 0.1


def test_strict_sorted_variant_has_every_max_in_last_tile():
    w = wl.WORKLOADS["B1-H1-N256-d64-full-sorted-strict"]
    q, k, _ = wl.make_inputs(w)
    s = q[0, 0].double() @ k[0, 0].double().T
    assert bool((s.argmax(dim=1) >= 128).all())


def test_sorted_variant_is_a_permutation_of_the_iid_draw():
    base = wl.make_inputs(wl.WORKLOADS["B1-H1-N256-d64-full"])
    srt = wl.make_inputs(wl.WORKLOADS["B1-H1-N256-d64-full-sorted"])
    assert torch.equal(base[0], srt[0])
    kb = {tuple(r) for r in base[1][0, 0].float().numpy().tolist()}
    ks = {tuple(r) for r in srt[1][0, 0].float().numpy().tolist()}
    assert kb == ks


def test_sample_rows():
    w = wl.WORKLOADS["B4-H16-N4096-d128-causal"]
    r = wl.sample_rows(w)
    assert len(r) == 64 * 256
    per = r.reshape(64, 256)
    assert np.all(per[:, 0] % 4096 == 0) and np.all(per[:, -1] % 4096 == 4095)
    assert all(len(set(row)) == 256 for row in per.tolist())
    assert np.array_equal(r, wl.sample_rows(w))
    assert len(wl.sample_rows(wl.WORKLOADS["B1-H1-N4096-d64-full"])) == 4096


def test_visible_pairs_match_a_brute_force_mask():
    """Masked workloads count 4 d FLOPs per visible (query, key) pair; the count
    must equal a mask built element by element."""
    for w in (wl.Workload("t", 2, 3, 300, 64, True, "iid", 5, window_left=40),
              wl.Workload("t", 2, 1, 257, 64, True, "iid", 6, doc_mean=30),
              wl.Workload("t", 1, 2, 200, 64, False, "iid", 7, doc_mean=50),
              wl.Workload("t", 1, 1, 150, 64, True, "iid", 8, window_left=9, doc_mean=20)):
        docs = wl.make_doc_ids(w)
        i = np.arange(w.N)[:, None]
        j = np.arange(w.N)[None, :]
        base = np.ones((w.N, w.N), dtype=bool)
        if w.causal:
            base &= j <= i
        if w.window_left >= 0:
            base &= j >= i - w.window_left
        total = 0
        for b in range(w.B):
            m = base if docs is None else base & (docs[b][:, None] == docs[b][None, :])
            total += int(m.sum()) * w.H
        assert wl.visible_pairs(w) == total
        rows = np.arange(w.B * w.H * w.N)
        assert int(wl.visible_per_row(w, rows).sum()) == total
