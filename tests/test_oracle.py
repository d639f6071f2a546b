"""Pins for the CPU oracle: each test checks it against something other than
itself -- an identity, an invariant, a closed form, brute force or a library
routine -- so that a dropped term, a wrong sign, a transposed operand or a
wrong mask in the oracle fails at least one of them.  No GPU is involved.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from online_softmax_04_gb300 import workloads as wl
from tests.conftest import read_golden


def bf16(a):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(torch.bfloat16)


def as_f64(t):
    return t.float().numpy().astype(np.float64)


def rand_qkv(B, H, N, d, seed, std=1.0):
    rng = np.random.default_rng(seed)
    return tuple(bf16(std * rng.standard_normal((B, H, N, d))) for _ in range(3))


# --------------------------------------------------------------------------
# (a) online route == three-pass route (the rescaling identity is exact)
# --------------------------------------------------------------------------

@pytest.mark.parametrize("std", [1.0, 4.0])
def test_softmax_online_equals_three_pass(std):
    rng = np.random.default_rng(1)
    for n in [1, 2, 3, 5, 16, 127, 128, 129, 1000, 4096]:
        x = std * rng.standard_normal(n)
        y3 = oracle.softmax_three_pass(x)
        yo, m, d = oracle.softmax_online(x)
        assert np.max(np.abs(y3 - yo)) <= 1e-12
        assert m == np.max(x)
        assert abs(d - np.sum(np.exp(x - np.max(x)))) <= 1e-12 * d


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("tile", [1, 7, 64, 128, 300])
def test_attention_online_equals_three_pass(causal, tile):
    q, k, v = rand_qkv(2, 2, 300, 64, seed=2 + tile)
    scale = 1 / 8
    o3, l3 = oracle.attention_three_pass(q, k, v, causal, scale)
    oo, lo = oracle.attention_online(q, k, v, causal, scale, tile=tile)
    assert np.max(np.abs(o3 - oo)) <= 1e-12
    assert np.max(np.abs(l3 - lo)) <= 1e-12


def test_attention_online_equals_three_pass_large_scores():
    # N(0,16)-sized scores: the running max moves by large steps
    q, k, v = rand_qkv(1, 1, 513, 128, seed=9, std=2.0)
    scale = 1 / math.sqrt(128)
    o3, l3 = oracle.attention_three_pass(q, k, v, True, scale)
    oo, lo = oracle.attention_online(q, k, v, True, scale, tile=128)
    assert np.max(np.abs(o3 - oo)) <= 1e-12
    assert np.max(np.abs(l3 - lo) / np.maximum(1, np.abs(l3))) <= 1e-12


# --------------------------------------------------------------------------
# (b) the sixteen-element row in four tiles, largest value last
# --------------------------------------------------------------------------

def sixteen_case():
    g = read_golden("sixteen_row_four_tiles.txt")
    return np.array(g["x"]), int(g["tile"][0])


def test_sixteen_row_fixture_moves_max_in_last_tile():
    x, t = sixteen_case()
    tile_max = [x[i:i + t].max() for i in range(0, 16, t)]
    running = np.maximum.accumulate(tile_max)
    assert running[-1] > running[-2], "the maximum must still move in the last tile"
    assert np.argmax(x) == 15


def softmax_by_ratios(x):
    """Softmax fixed by its two defining invariants: y_i / y_j = e^(x_i - x_j), sum y = 1."""
    return np.array([1.0 / math.fsum(math.exp(xj - xi) for xj in x) for xi in x])


def test_sixteen_row_softmax_routes():
    x, _ = sixteen_case()
    want = softmax_by_ratios(x)
    y3 = oracle.softmax_three_pass(x)
    yo, m, d = oracle.softmax_online(x)
    assert np.max(np.abs(y3 - want)) <= 1e-15 * 16
    assert np.max(np.abs(yo - want)) <= 1e-15 * 16
    assert m == 6.5


def sixteen_attention():
    """q = e_0, k_j = 8 x_j e_0, v_j = e_j, d = 64, scale = 1/8: O_0[:16] = softmax(x)."""
    x, _ = sixteen_case()
    d = 64
    q = np.zeros((1, 1, 16, d), np.float32)
    q[0, 0, :, 0] = 1.0
    k = np.zeros((1, 1, 16, d), np.float32)
    k[0, 0, :, 0] = 8 * x
    v = np.zeros((1, 1, 16, d), np.float32)
    v[0, 0, np.arange(16), np.arange(16)] = 1.0
    q, k, v = bf16(q), bf16(k), bf16(v)
    assert np.array_equal(as_f64(k)[0, 0, :, 0], 8 * x), "fixture must be exact in bf16"
    return x, q, k, v


def test_sixteen_row_attention_equals_softmax():
    x, q, k, v = sixteen_attention()
    want = softmax_by_ratios(x)
    for tile in (1, 4, 16):
        o, lse = oracle.attention_online(q, k, v, False, 1 / 8, tile=tile, rows=[0])
        assert np.max(np.abs(o[0, :16] - want)) <= 1e-14
        assert np.all(o[0, 16:] == 0)
        assert abs(lse[0] - (6.5 + math.log(math.fsum(math.exp(t - 6.5) for t in x)))) <= 1e-14
    o, _ = oracle.attention_three_pass(q, k, v, False, 1 / 8, rows=[0])
    assert np.max(np.abs(o[0, :16] - want)) <= 1e-14


def test_mutant_without_rescale_fails_sixteen_row():
    x, q, k, v = sixteen_attention()
    want = softmax_by_ratios(x)
    o, _ = oracle.attention_online(q, k, v, False, 1 / 8, tile=4, rows=[0], mutation=oracle.MUT_NO_RESCALE)
    assert np.max(np.abs(o[0, :16] - want)) > 1e-3
    # the same mutant passes when the largest score lands in the first tile,
    # which is why the fixture puts it last
    o1, _ = oracle.attention_online(q, k, v, False, 1 / 8, tile=16, rows=[0], mutation=oracle.MUT_NO_RESCALE)
    assert np.max(np.abs(o1[0, :16] - want)) <= 1e-14


def test_mutant_normalising_per_tile_breaks_row_sum():
    x, q, k, v = sixteen_attention()
    o, _ = oracle.attention_online(q, k, v, False, 1 / 8, tile=4, rows=[0], mutation=oracle.MUT_NORMALISE_TILE)
    assert abs(o[0, :16].sum() - 1.0) > 1e-3


def test_mutant_sum_before_max_overflows():
    x, q, k, v = sixteen_attention()
    o, lse = oracle.attention_online(q, k, v, False, 1 / 8, tile=4, rows=[0], mutation=oracle.MUT_SUM_BEFORE_MAX)
    assert not np.all(np.isfinite(o)) or not np.isfinite(lse[0])


# --------------------------------------------------------------------------
# (c) rows sum to one; masked keys get zero weight; ratios and linearity
# --------------------------------------------------------------------------

@pytest.mark.parametrize("causal", [False, True])
def test_rows_sum_to_one(causal):
    q, k, _ = rand_qkv(1, 2, 200, 64, seed=4)
    v = bf16(np.ones((1, 2, 200, 64)))
    for fn in (oracle.attention_three_pass, oracle.attention_online):
        o, _ = fn(q, k, v, causal, 1 / 8)
        assert np.max(np.abs(o - 1.0)) <= 1e-12


@pytest.mark.parametrize("causal", [False, True])
def test_weights_ratios_mask_and_linearity(causal):
    """With v_j = e_j (N <= d) row i of O is the weight row W_i."""
    N, d = 48, 64
    q, k, vr = rand_qkv(1, 1, N, d, seed=5)
    eye = np.zeros((1, 1, N, d), np.float32)
    eye[0, 0, np.arange(N), np.arange(N)] = 1.0
    scale = 1 / 8
    for fn in (oracle.attention_three_pass, oracle.attention_online):
        W, _ = fn(q, k, bf16(eye), causal, scale)
        W = W[:, :N]
        qd, kd = as_f64(q)[0, 0], as_f64(k)[0, 0]
        x = scale * (qd @ kd.T)  # exact: products of bf16 values summed in double
        for i in range(N):
            vis = i + 1 if causal else N
            assert np.all(W[i, vis:] == 0)
            assert abs(W[i, :vis].sum() - 1) <= 1e-12
            # ratio invariant against key 0 (always visible)
            ratio = W[i, :vis] / W[i, 0]
            assert np.max(np.abs(ratio / np.exp(x[i, :vis] - x[i, 0]) - 1)) <= 1e-12
        # linearity in V: O(V) = W V
        o, _ = fn(q, k, vr, causal, scale)
        assert np.max(np.abs(o - W @ as_f64(vr)[0, 0])) <= 1e-12


# --------------------------------------------------------------------------
# (d) closed forms: a dominant one-hot key, and uniform attention
# --------------------------------------------------------------------------

@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("N,d,c", [(64, 64, 18.0), (128, 128, 22.0), (37, 64, 18.0)])
def test_onehot_dominant_key_closed_form(causal, N, d, c):
    q, k, v = wl.onehot_inputs(1, 1, N, d, c)
    scale = 1 / math.sqrt(d)
    s = scale * c * c
    assert s >= 40
    vd = as_f64(v)[0, 0]
    for fn in (oracle.attention_three_pass, oracle.attention_online):
        o, lse = fn(q, k, v, causal, scale)
        for i in range(N):
            n_vis = i + 1 if causal else N
            others = vd[:n_vis].sum(axis=0) - vd[i]
            want = (math.exp(s) * vd[i] + others) / (math.exp(s) + n_vis - 1)
            assert np.max(np.abs(o[i] - want)) <= 1e-12
            assert abs(lse[i] - math.log(math.exp(s) + n_vis - 1)) <= 1e-12
            # and the bound used for the GPU check: O_i = v_i within (n-1) e^-s max|v|
            assert np.max(np.abs(o[i] - vd[i])) <= (n_vis - 1) * math.exp(-s) * 2 * np.max(np.abs(vd)) + 1e-15


@pytest.mark.parametrize("causal", [False, True])
def test_uniform_attention_closed_form(causal):
    w = wl.Workload("t", 1, 2, 333, 64, causal, "zeros-q", 3)
    q, k, v = wl.make_inputs(w)
    vd = as_f64(v)
    for fn in (oracle.attention_three_pass, oracle.attention_online):
        o, lse = fn(q, k, v, causal, w.scale)
        o = o.reshape(2, 333, 64)
        lse = lse.reshape(2, 333)
        for h in range(2):
            if causal:
                want = np.cumsum(vd[0, h], axis=0) / np.arange(1, 334)[:, None]
                want_lse = np.log(np.arange(1, 334))
            else:
                want = np.broadcast_to(vd[0, h].mean(axis=0), (333, 64))
                want_lse = np.full(333, math.log(333))
            assert np.max(np.abs(o[h] - want)) <= 1e-12
            assert np.max(np.abs(lse[h] - want_lse)) <= 1e-12


# --------------------------------------------------------------------------
# (e) brute force on tiny inputs, and a library routine
# --------------------------------------------------------------------------

def brute_force_longdouble(q, k, v, causal, scale):
    qd, kd, vd = (as_f64(t).astype(np.longdouble) for t in (q, k, v))
    S = np.einsum("bhid,bhjd->bhij", qd, kd) * np.longdouble(scale)
    N = S.shape[-1]
    if causal:
        S = np.where(np.tri(N, dtype=bool), S, np.longdouble(-np.inf))
    m = S.max(axis=-1, keepdims=True)
    P = np.exp(S - m)
    l = P.sum(axis=-1, keepdims=True)
    O = np.einsum("bhij,bhjd->bhid", P / l, vd)
    return O, (m + np.log(l))[..., 0]


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("N,d", [(1, 64), (17, 64), (64, 64), (64, 128)])
def test_brute_force_tiny(causal, N, d):
    q, k, v = rand_qkv(2, 3, N, d, seed=N + d, std=1.5)
    scale = 1 / math.sqrt(d)
    O, L = brute_force_longdouble(q, k, v, causal, scale)
    O = O.reshape(-1, d).astype(np.float64)
    L = L.reshape(-1).astype(np.float64)
    for fn in (oracle.attention_three_pass, oracle.attention_online):
        o, lse = fn(q, k, v, causal, scale)
        assert np.max(np.abs(o - O)) <= 1e-12
        assert np.max(np.abs(lse - L)) <= 1e-12


@pytest.mark.parametrize("causal", [False, True])
def test_library_sdpa_float64(causal):
    B, H, N, d = 2, 2, 64, 64
    q, k, v = rand_qkv(B, H, N, d, seed=11)
    scale = 1 / 8
    ref = torch.nn.functional.scaled_dot_product_attention(
        q.double(), k.double(), v.double(), is_causal=causal, scale=scale).numpy().reshape(-1, d)
    o, _ = oracle.attention_three_pass(q, k, v, causal, scale)
    assert np.max(np.abs(o - ref)) <= 1e-12


# --------------------------------------------------------------------------
# merge: associativity, and the two-empty-states NaN trap
# --------------------------------------------------------------------------

def test_softmax_state_merge_any_order():
    rng = np.random.default_rng(12)
    x = 3 * rng.standard_normal(1000)
    _, m_full, d_full = oracle.softmax_online(x)
    for trial in range(20):
        cuts = np.sort(rng.choice(np.arange(1, 1000), size=rng.integers(1, 9), replace=False))
        parts = [oracle.softmax_online(seg)[1:] for seg in np.split(x, cuts)]
        while len(parts) > 1:  # merge a random adjacent pair until one is left
            i = rng.integers(0, len(parts) - 1)
            parts[i:i + 2] = [oracle.online_merge(*parts[i], *parts[i + 1])]
        m, d = parts[0]
        assert m == m_full
        assert abs(d - d_full) <= 1e-12 * d_full


def test_attention_state_merge_any_order():
    rng = np.random.default_rng(13)
    N, d = 777, 64
    q, k, v = rand_qkv(1, 1, N, d, seed=14, std=1.5)
    scale = 1 / 8
    o3, l3 = oracle.attention_three_pass(q, k, v, False, scale, rows=[5])
    for trial in range(10):
        cuts = [0] + sorted(rng.choice(np.arange(1, N), size=rng.integers(1, 7), replace=False).tolist()) + [N]
        parts = [oracle.row_online_state(q, k, v, 5, a, b, False, scale, tile=int(rng.integers(1, 200)))
                 for a, b in zip(cuts[:-1], cuts[1:])]
        while len(parts) > 1:
            i = rng.integers(0, len(parts) - 1)
            parts[i:i + 2] = [oracle.state_merge(parts[i], parts[i + 1])]
        m, l, acc = parts[0]
        assert np.max(np.abs(acc / l - o3[0])) <= 1e-12
        assert abs(m + math.log(l) - l3[0]) <= 1e-12


def test_merge_of_two_empty_states_is_not_nan():
    m, d = oracle.online_merge(-np.inf, 0.0, -np.inf, 0.0)
    assert m == -np.inf and d == 0.0
    m, l, acc = oracle.state_merge((-np.inf, 0.0, np.zeros(4)), (-np.inf, 0.0, np.zeros(4)))
    assert m == -np.inf and l == 0.0 and np.all(acc == 0)
    m, l, acc = oracle.state_merge((-np.inf, 0.0, np.zeros(4)), (1.5, 2.0, np.ones(4)))
    assert m == 1.5 and l == 2.0 and np.all(acc == 1)


def test_outputs_finite_with_large_scores():
    q, k, v = rand_qkv(1, 2, 300, 64, seed=15, std=6.0)  # scores of order +-300
    for causal in (False, True):
        for fn in (oracle.attention_three_pass, oracle.attention_online):
            o, lse = fn(q, k, v, causal, 1 / 8)
            assert np.all(np.isfinite(o)) and np.all(np.isfinite(lse))


def test_row_subset_matches_full_run():
    q, k, v = rand_qkv(2, 2, 100, 64, seed=16)
    o, lse = oracle.attention_three_pass(q, k, v, True, 1 / 8)
    rows = np.array([0, 99, 150, 399, 250])
    os_, ls_ = oracle.attention_three_pass(q, k, v, True, 1 / 8, rows=rows)
    assert np.array_equal(os_, o[rows]) and np.array_equal(ls_, lse[rows])


def test_lse_shift_by_common_key_component():
    """Adding u to every key adds scale*q.u to a row's scores: O unchanged, LSE shifted."""
    N, d = 90, 64
    rng = np.random.default_rng(18)
    q = np.zeros((1, 1, N, d), np.float32)
    q[..., :32] = np.round(rng.standard_normal((N, 32)) * 4) / 4
    k = np.zeros((1, 1, N, d), np.float32)
    k[..., :32] = np.round(rng.standard_normal((N, 32)) * 4) / 4
    v = rng.standard_normal((1, 1, N, d)).astype(np.float32)
    u = np.zeros(d, np.float32)
    u[:32] = 0.5
    k2 = k + u  # quarter-integers plus 0.5 stay exact in bf16 at these sizes
    q, k, v, k2 = bf16(q), bf16(k), bf16(v), bf16(k2)
    assert np.array_equal(as_f64(k2), as_f64(k) + u.astype(np.float64))
    for causal in (False, True):
        o1, l1 = oracle.attention_three_pass(q, k, v, causal, 1 / 8)
        o2, l2 = oracle.attention_three_pass(q, k2, v, causal, 1 / 8)
        shift = (as_f64(q)[0, 0] @ u.astype(np.float64)) / 8
        assert np.max(np.abs(o1 - o2)) <= 1e-12
        assert np.max(np.abs(l2 - l1 - shift)) <= 1e-12


# --------------------------------------------------------------------------
# structured masks: window and document boundaries ("Online Softmax: Tiling
# Across a Reduction", causal section, last paragraph)
# --------------------------------------------------------------------------

def doc_ids_from_lengths(B, N, lengths_per_batch):
    doc = np.zeros((B, N), dtype=np.int32)
    for b, lengths in enumerate(lengths_per_batch):
        assert sum(lengths) == N
        doc[b] = np.repeat(np.arange(len(lengths), dtype=np.int32), lengths)
    return doc


def test_masked_without_mask_is_full_and_right_window_zero_is_causal():
    q, k, v = rand_qkv(1, 2, 70, 64, seed=21)
    for causal, wr in ((False, -1), (True, 0)):
        o_ref, l_ref = oracle.attention_three_pass(q, k, v, causal, 0.125)
        o, lse = oracle.attention_masked(q, k, v, 0.125, window_left=-1, window_right=wr)
        assert np.max(np.abs(o - o_ref)) <= 1e-14 and np.max(np.abs(lse - l_ref)) <= 1e-14


@pytest.mark.parametrize("causal", [False, True])
def test_document_mask_equals_independent_documents(causal):
    """A document mask is attention run separately on each document's slice."""
    B, H, N, d = 2, 2, 96, 64
    q, k, v = rand_qkv(B, H, N, d, seed=22)
    lengths = [[30, 1, 65], [96]]
    doc = doc_ids_from_lengths(B, N, lengths)
    o, lse = oracle.attention_masked(q, k, v, 0.125, -1, 0 if causal else -1, doc)
    o = o.reshape(B, H, N, d)
    lse = lse.reshape(B, H, N)
    for b in range(B):
        start = 0
        for n in lengths[b]:
            sl = slice(start, start + n)
            qs, ks, vs = (t[b:b + 1, :, sl].contiguous() for t in (q, k, v))
            o_ref, l_ref = oracle.attention_three_pass(qs, ks, vs, causal, 0.125)
            assert np.max(np.abs(o[b, :, sl].reshape(-1, d) - o_ref)) <= 1e-13
            assert np.max(np.abs(lse[b, :, sl].reshape(-1) - l_ref)) <= 1e-13
            start += n


@pytest.mark.parametrize("wl,wr", [(0, 0), (5, 0), (16, 3), (40, -1), (-1, 7)])
def test_window_row_equals_attention_over_its_keys(wl, wr):
    """Row i under a window sees exactly keys [i - wl, i + wr] (clipped):
    plain attention of that query over the key slice."""
    B, H, N, d = 1, 1, 60, 64
    q, k, v = rand_qkv(B, H, N, d, seed=23)
    o, lse = oracle.attention_masked(q, k, v, 0.125, wl, wr)
    for i in (0, 1, 17, 30, 59):
        lo = 0 if wl < 0 else max(0, i - wl)
        hi = N - 1 if wr < 0 else min(N - 1, i + wr)
        ks, vs = k[:, :, lo:hi + 1].contiguous(), v[:, :, lo:hi + 1].contiguous()
        qs = q[:, :, i:i + 1].expand(1, 1, hi - lo + 1, d).contiguous()  # every row = query i, full attention
        o_ref, l_ref = oracle.attention_three_pass(qs, ks, vs, False, 0.125, rows=[0])
        assert np.max(np.abs(o[i] - o_ref[0])) <= 1e-13 and abs(lse[i] - l_ref[0]) <= 1e-13


def test_masks_brute_force_tiny():
    """Window and document masks built independently (tril/triu bands and an
    outer equality), softmax in long double."""
    B, H, N, d = 2, 2, 33, 64
    q, k, v = rand_qkv(B, H, N, d, seed=24, std=1.5)
    doc = doc_ids_from_lengths(B, N, [[10, 23], [5, 5, 5, 18]])
    qd, kd, vd = (as_f64(t).astype(np.longdouble) for t in (q, k, v))
    S = np.einsum("bhid,bhjd->bhij", qd, kd) * np.longdouble(0.125)
    for wl, wr, use_doc in ((4, 0, False), (3, 2, True), (-1, 0, True), (-1, -1, True)):
        band = np.ones((N, N), dtype=bool)
        if wl >= 0:
            band &= np.triu(band, k=-wl)
        if wr >= 0:
            band &= np.tril(band, k=wr)
        mask = np.broadcast_to(band, (B, H, N, N)).copy()
        if use_doc:
            mask &= (doc[:, None, :, None] == doc[:, None, None, :])
        Sm = np.where(mask, S, np.longdouble(-np.inf))
        m = Sm.max(axis=-1, keepdims=True)
        P = np.exp(Sm - m)
        l = P.sum(axis=-1, keepdims=True)
        O = np.einsum("bhij,bhjd->bhid", P / l, vd).reshape(-1, d).astype(np.float64)
        L = (m + np.log(l)).reshape(-1).astype(np.float64)
        o, lse = oracle.attention_masked(q, k, v, 0.125, wl, wr, doc if use_doc else None)
        assert np.max(np.abs(o - O)) <= 1e-12, (wl, wr, use_doc)
        assert np.max(np.abs(lse - L)) <= 1e-12, (wl, wr, use_doc)


# --------------------------------------------------------------------------
# backward pass: gradients of L = sum(O * dO), scores recomputed and
# normalised with the saved LSE ("Online Softmax: Tiling Across a Reduction",
# backward-pass section); pinned to automatic differentiation in float64
# --------------------------------------------------------------------------

def autograd_reference(q, k, v, dout, causal, scale):
    qd, kd, vd = (t.double().clone().requires_grad_(True) for t in (q, k, v))
    S = torch.einsum("bhid,bhjd->bhij", qd, kd) * scale
    N = S.shape[-1]
    if causal:
        S = S.masked_fill(~torch.ones(N, N, dtype=torch.bool).tril(), float("-inf"))
    lse = torch.logsumexp(S, dim=-1)
    O = torch.einsum("bhij,bhjd->bhid", torch.exp(S - lse[..., None]), vd)
    (O * dout.double()).sum().backward()
    return O.detach(), lse.detach(), qd.grad, kd.grad, vd.grad


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("B,H,N,d", [(1, 1, 1, 64), (2, 2, 50, 64), (1, 2, 130, 128)])
def test_backward_matches_autograd_float64(causal, B, H, N, d):
    q, k, v = rand_qkv(B, H, N, d, seed=N + d, std=1.3)
    dout = bf16(np.random.default_rng(N).standard_normal((B, H, N, d)))
    scale = 1 / math.sqrt(d)
    O, lse, gq, gk, gv = autograd_reference(q, k, v, dout, causal, scale)
    g = oracle.attention_backward(q, k, v, O, dout, lse, causal, scale)
    for name, ref in (("dq", gq), ("dk", gk), ("dv", gv)):
        ref = ref.numpy().reshape(-1, d)
        assert np.max(np.abs(g[name] - ref)) <= 1e-12 * max(1.0, np.max(np.abs(ref))), name
        assert np.all(g["mag_" + name] + 1e-15 >= np.abs(g[name])), name


@pytest.mark.parametrize("causal", [False, True])
def test_backward_dv_sums_to_dout_and_rows_agree(causal):
    """Each row's visible weights sum to one, so sum_j dV_j = sum_i dO_i; and a
    sample of rows equals the same rows of the full computation."""
    B, H, N, d = 1, 2, 90, 64
    q, k, v = rand_qkv(B, H, N, d, seed=3)
    dout = bf16(np.random.default_rng(4).standard_normal((B, H, N, d)))
    O, lse, *_ = autograd_reference(q, k, v, dout, causal, 0.125)
    g = oracle.attention_backward(q, k, v, O, dout, lse, causal, 0.125)
    dv = g["dv"].reshape(B, H, N, d).sum(axis=2)
    assert np.max(np.abs(dv - as_f64(dout).sum(axis=2))) <= 1e-11
    rows = np.array([0, 5, 89, 90, 133, 179])
    gs = oracle.attention_backward(q, k, v, O, dout, lse, causal, 0.125, q_rows=rows, k_rows=rows[::-1])
    assert np.array_equal(gs["dq"], g["dq"][rows])
    assert np.array_equal(gs["dk"], g["dk"][rows[::-1]]) and np.array_equal(gs["dv"], g["dv"][rows[::-1]])
