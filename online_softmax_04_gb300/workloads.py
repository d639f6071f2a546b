"""Seeded synthetic inputs shaped like the workloads the pages measure.

This module draws random numbers and arranges them; it holds none of the
attention arithmetic, so both the CUDA path and the CPU oracle can be fed
from it.  Every tensor is drawn in float32 with ``numpy.random.default_rng``
and rounded to bf16 (round-to-nearest-even) by torch.  Q, K and V are drawn
in that order from one generator.  Layout is ``[B][H][N][d]``.

Workloads (all with scale = 1/sqrt(d)):

* ``B1-H1-N256-d64-full`` -- one head, iid N(0,1), full attention; the
  variants ``...-sorted`` (key/value pairs reordered by increasing score
  against the mean query) and ``...-sorted-strict`` (every query row equal
  to the first one, keys sorted by their score against it, so every row's
  largest score sits in the last key tile).
* ``B1-H1-N4096-d64-full`` -- one head, iid N(0,1), full attention.
* ``B4-H16-N4096-d128-causal`` -- iid N(0,1), causal.
* ``B1-H32-N16384-d128-causal-late`` -- causal; Q = 4 N(0,1); key row j is
  N(0,1) scaled by 0.25 + 3.75 j/(N-1), so the norms of the keys grow
  linearly along the sequence and large scores arrive late; V iid N(0,1).
* ``B1-H8-N131072-d64-causal`` -- iid N(0,1), causal, long context.

Structured masks (the window / document-boundary skips of "Online Softmax:
Tiling Across a Reduction", causal section), run through ``fa_fwd_masked``:

* ``B1-H32-N16384-d128-window4096`` -- iid N(0,1), causal sliding window of
  4096 keys (window_left = 4095, window_right = 0).
* ``B4-H16-N4096-d128-docs`` -- iid N(0,1), causal within packed documents:
  seeded document lengths, uniform on [1, 2047] (mean 1024), per sequence.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, replace

import numpy as np


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    H: int
    N: int
    d: int
    causal: bool
    dist: str = "iid"            # iid | late | sorted | sorted-strict | zeros-q | onehot
    seed: int = 1000
    rows_per_head: int | None = None  # oracle rows checked per (b, h); None = every row
    window_left: int = -1         # masked workloads: keys i - window_left .. (-1 = unbounded)
    doc_mean: int = 0             # masked workloads: mean document length (0 = no documents)

    @property
    def masked(self) -> bool:
        return self.window_left >= 0 or self.doc_mean > 0

    @property
    def window_right(self) -> int:
        return 0 if self.causal else -1

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.d)

    def with_(self, **kw) -> "Workload":
        return replace(self, **kw)


WORKLOADS = {
    w.name: w
    for w in [
        Workload("B1-H1-N256-d64-full", 1, 1, 256, 64, False, "iid", 1000, None),
        Workload("B1-H1-N256-d64-full-sorted", 1, 1, 256, 64, False, "sorted", 1000, None),
        Workload("B1-H1-N256-d64-full-sorted-strict", 1, 1, 256, 64, False, "sorted-strict", 1000, None),
        Workload("B1-H1-N4096-d64-full", 1, 1, 4096, 64, False, "iid", 1001, None),
        Workload("B4-H16-N4096-d128-causal", 4, 16, 4096, 128, True, "iid", 1002, 256),
        Workload("B1-H32-N16384-d128-causal-late", 1, 32, 16384, 128, True, "late", 1003, 256),
        Workload("B1-H8-N131072-d64-causal", 1, 8, 131072, 64, True, "iid", 1004, 64),
        Workload("B1-H32-N16384-d128-window4096", 1, 32, 16384, 128, True, "iid", 1005, 64, window_left=4095),
        Workload("B4-H16-N4096-d128-docs", 4, 16, 4096, 128, True, "iid", 1006, 64, doc_mean=1024),
    ]
}

# The configuration the headline throughput is quoted on (d=128, causal, the
# late-arriving-maximum stress case).
HEADLINE = "B1-H32-N16384-d128-causal-late"


def _normal(rng: np.random.Generator, shape) -> np.ndarray:
    return rng.standard_normal(size=shape, dtype=np.float32)


def _to_bf16(a: np.ndarray):
    import torch

    return torch.from_numpy(np.ascontiguousarray(a)).to(torch.bfloat16)


def make_inputs(w: Workload):
    """Returns (q, k, v) as contiguous bf16 CPU torch tensors of shape [B, H, N, d]."""
    rng = np.random.default_rng(w.seed)
    shape = (w.B, w.H, w.N, w.d)
    if w.dist == "iid":
        q, k, v = _normal(rng, shape), _normal(rng, shape), _normal(rng, shape)
    elif w.dist == "late":
        q = 4.0 * _normal(rng, shape)
        z = _normal(rng, shape)
        denom = max(w.N - 1, 1)
        ramp = (0.25 + 3.75 * np.arange(w.N, dtype=np.float32) / np.float32(denom)).astype(np.float32)
        k = z * ramp[None, None, :, None]
        v = _normal(rng, shape)
    elif w.dist in ("sorted", "sorted-strict"):
        q, k, v = _normal(rng, shape), _normal(rng, shape), _normal(rng, shape)
        qb, kb, vb = (np.asarray(_to_bf16(t).float().numpy(), dtype=np.float64) for t in (q, k, v))
        if w.dist == "sorted-strict":
            qb = np.broadcast_to(qb[:, :, :1, :], qb.shape).copy()
        ref = qb.mean(axis=2) if w.dist == "sorted" else qb[:, :, 0, :]
        order = np.argsort(np.einsum("bhnd,bhd->bhn", kb, ref), axis=-1, kind="stable")
        kb = np.take_along_axis(kb, order[..., None], axis=2)
        vb = np.take_along_axis(vb, order[..., None], axis=2)
        q, k, v = qb.astype(np.float32), kb.astype(np.float32), vb.astype(np.float32)
    elif w.dist == "zeros-q":
        q = np.zeros(shape, dtype=np.float32)
        k, v = _normal(rng, shape), _normal(rng, shape)
    else:
        raise ValueError(f"unknown distribution {w.dist!r}")
    return _to_bf16(q), _to_bf16(k), _to_bf16(v)


def make_doc_ids(w: Workload):
    """int32 [B, N] document ids for a workload with documents (None otherwise):
    runs of seeded lengths uniform on [1, 2 doc_mean - 1], numbered 0, 1, ...
    along each sequence."""
    if w.doc_mean <= 0:
        return None
    rng = np.random.default_rng(w.seed + 31)
    out = np.zeros((w.B, w.N), dtype=np.int32)
    for b in range(w.B):
        pos, doc = 0, 0
        while pos < w.N:
            n = int(rng.integers(1, 2 * w.doc_mean))
            out[b, pos:pos + n] = doc
            pos += n
            doc += 1
    return out


def visible_pairs(w: Workload) -> int:
    """Number of (query, key) pairs the mask leaves visible, over all B*H heads."""
    N = w.N
    docs = make_doc_ids(w)
    total = 0
    for b in range(w.B):
        if docs is None:
            starts, ends = np.array([0]), np.array([N])
        else:
            change = np.flatnonzero(np.diff(docs[b])) + 1
            starts = np.concatenate([[0], change])
            ends = np.concatenate([change, [N]])
        for s0, e0 in zip(starts, ends):
            n = int(e0 - s0)
            i = np.arange(n, dtype=np.int64)
            hi = i if w.causal else np.full(n, n - 1, dtype=np.int64)
            lo = np.maximum(0, i - w.window_left) if w.window_left >= 0 else np.zeros(n, dtype=np.int64)
            total += int(np.sum(hi - lo + 1))
    return total * w.H


def visible_per_row(w: Workload, rows) -> np.ndarray:
    """Number of keys each given flat query row (bh * N + i) may see."""
    rows = np.asarray(rows, dtype=np.int64)
    N = w.N
    i = rows % N
    b = (rows // N) // w.H
    lo = np.maximum(0, i - w.window_left) if w.window_left >= 0 else np.zeros(len(i), dtype=np.int64)
    hi = i.copy() if w.causal else np.full(len(i), N - 1, dtype=np.int64)
    docs = make_doc_ids(w)
    if docs is not None:
        for bb in np.unique(b):
            sel = b == bb
            d = docs[bb]
            first = np.searchsorted(d, d[i[sel]], side="left")
            last = np.searchsorted(d, d[i[sel]], side="right") - 1
            lo[sel] = np.maximum(lo[sel], first)
            hi[sel] = np.minimum(hi[sel], last)
    return hi - lo + 1


def onehot_inputs(B: int, H: int, N: int, d: int, c: float, seed: int = 7):
    """q_i = k_i = c * e_i (needs N <= d); V iid N(0,1).  Returns bf16 tensors."""
    if N > d:
        raise ValueError("one-hot rows need N <= d")
    rng = np.random.default_rng(seed)
    q = np.zeros((B, H, N, d), dtype=np.float32)
    idx = np.arange(N)
    q[:, :, idx, idx] = c
    v = _normal(rng, (B, H, N, d))
    return _to_bf16(q), _to_bf16(q.copy()), _to_bf16(v)


def sample_rows(w: Workload, seed_offset: int = 17) -> np.ndarray:
    """Flat query-row indices checked against the oracle.

    Every row when ``rows_per_head`` is None; otherwise, per (b, h), rows 0 and
    N-1 plus distinct seeded rows in between.
    """
    BH, N = w.B * w.H, w.N
    if w.rows_per_head is None or w.rows_per_head >= N:
        return np.arange(BH * N, dtype=np.int64)
    rng = np.random.default_rng(w.seed + seed_offset)
    out = []
    k = w.rows_per_head
    for bh in range(BH):
        inner = rng.choice(np.arange(1, N - 1), size=k - 2, replace=False) if N > 2 else np.array([], dtype=np.int64)
        rows = np.concatenate([[0], np.sort(inner), [N - 1]]).astype(np.int64)
        out.append(bh * N + rows)
    return np.concatenate(out)
