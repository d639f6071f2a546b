"""GPU parity: the CUDA path against the fp64 CPU oracle on the same seeded
inputs, element by element.

Tolerances (bf16 inputs, fp32 accumulation, bf16 output): max |O_gpu - O_ref|
<= 2e-2 over every checked element, and |LSE_gpu - LSE_ref| / max(1, |LSE_ref|)
<= 1e-3 per checked row.
"""
import contextlib
import math

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


@contextlib.contextmanager
def pairing(fa, mode):
    """Force the forward kernel for the block: one query tile per CTA (OFF), or pairs of
    adjacent query tiles (ON: CTA pairs at d = 128, two tiles in one CTA at d = 64)."""
    prev = fa.fa_set_fwd_pairing(mode)
    try:
        yield
    finally:
        fa.fa_set_fwd_pairing(prev)


AUTO, OFF, ON = 0, 1, 2  # FA_PAIR_AUTO, FA_PAIR_OFF, FA_PAIR_ON


def run_gpu(fa, q, k, v, causal, scale):
    dev = torch.device("cuda:0")
    o, lse = fa.attention(q.to(dev), k.to(dev), v.to(dev), causal=causal, scale=scale)
    torch.cuda.synchronize()
    return o.float().cpu().numpy(), lse.cpu().numpy()


def compare(o_gpu, lse_gpu, q, k, v, causal, scale, rows, label=""):
    B, H, N, d = q.shape
    ref_o, ref_lse = oracle.attention_three_pass(q, k, v, causal, scale, rows=rows)
    got_o = o_gpu.reshape(-1, d)[rows].astype(np.float64)
    got_lse = lse_gpu.reshape(-1)[rows].astype(np.float64)
    assert np.all(np.isfinite(got_o)) and np.all(np.isfinite(got_lse)), f"{label}: non-finite output"
    err_o = np.abs(got_o - ref_o)
    err_l = np.abs(got_lse - ref_lse) / np.maximum(1.0, np.abs(ref_lse))
    worst = int(np.argmax(err_o.max(axis=1)))
    msg = (f"{label}: max|dO|={err_o.max():.3e} (row {rows[worst]}) max rel dLSE={err_l.max():.3e} "
           f"rows={len(rows)}")
    print(msg)
    assert err_o.max() <= O_TOL, msg
    assert err_l.max() <= LSE_TOL, msg
    return err_o.max(), err_l.max()


def all_rows(B, H, N):
    return np.arange(B * H * N, dtype=np.int64)


# --------------------------------------------------------------------------
# small shapes: every row, ragged tails, both head dims, both mask modes
# --------------------------------------------------------------------------
SMALL = [
    (1, 1, 1, 64, False), (1, 1, 1, 128, True), (1, 2, 7, 64, True), (2, 1, 100, 128, False),
    (1, 1, 128, 64, False), (1, 1, 128, 128, True), (1, 1, 129, 128, True), (1, 1, 129, 64, False),
    (1, 1, 255, 64, True), (1, 2, 300, 128, True), (2, 2, 384, 64, False), (1, 1, 1000, 128, True),
    (1, 1, 1000, 64, False), (3, 5, 520, 64, True),
]


@pytest.mark.parametrize("B,H,N,d,causal", SMALL)
def test_small_shapes_every_row(fa, B, H, N, d, causal):
    w = wl.Workload("small", B, H, N, d, causal, "iid", 100 + N + d)
    q, k, v = wl.make_inputs(w)
    o, lse = run_gpu(fa, q, k, v, causal, w.scale)
    compare(o, lse, q, k, v, causal, w.scale, all_rows(B, H, N), f"B{B} H{H} N{N} d{d} causal={causal}")


def paired_kind(fa, d):
    return fa.FA_KERNEL_FWD_PAIR if d == 128 else fa.FA_KERNEL_FWD_TWO


@pytest.mark.parametrize("mode", [OFF, ON])
@pytest.mark.parametrize("B,H,N,d,causal", SMALL + [(1, 3, 640, 128, True), (2, 2, 383, 128, False),
                                                    (1, 3, 640, 64, True), (2, 2, 383, 64, False)])
def test_small_shapes_each_kernel(fa, mode, B, H, N, d, causal):
    """Both forward kernels of each head dim on every small shape, every row: one
    query tile per CTA, and pairs of adjacent tiles (CTA pairs at d = 128, two
    tiles per CTA at d = 64).  Odd tile counts leave the second tile of the last
    pair past N; causal pairs compute a fully masked key tile for the first."""
    w = wl.Workload("small", B, H, N, d, causal, "iid", 100 + N + d)
    q, k, v = wl.make_inputs(w)
    with pairing(fa, mode):
        assert fa.fa_fwd_kernel_for(B, H, N, d, causal) == (paired_kind(fa, d) if mode == ON else fa.FA_KERNEL_FWD)
        o, lse = run_gpu(fa, q, k, v, causal, w.scale)
    compare(o, lse, q, k, v, causal, w.scale, all_rows(B, H, N), f"mode {mode} B{B} H{H} N{N} causal={causal}")


@pytest.mark.parametrize("name", [
    "B1-H1-N256-d64-full", "B1-H1-N256-d64-full-sorted", "B1-H1-N256-d64-full-sorted-strict",
    "B1-H1-N4096-d64-full",
])
def test_small_workloads_every_row(fa, name):
    w = wl.WORKLOADS[name]
    q, k, v = wl.make_inputs(w)
    o, lse = run_gpu(fa, q, k, v, w.causal, w.scale)
    compare(o, lse, q, k, v, w.causal, w.scale, wl.sample_rows(w), name)


def test_random_shapes_both_d128_kernels(fa):
    """Twelve seeded random shapes (B, H, N with odd and even query-tile counts and
    ragged tails, causal or not), each through both d = 128 forward kernels and
    compared with the oracle on every row: the two kernels' per-row arithmetic is
    the same, so they must also agree with each other bit for bit."""
    rng = np.random.default_rng(20261202)
    for case in range(12):
        B, H = int(rng.integers(1, 3)), int(rng.integers(1, 4))
        N = int(rng.integers(1, 1400))
        causal = bool(rng.integers(0, 2))
        w = wl.Workload(f"rand{case}", B, H, N, 128, causal, "iid", 500 + case)
        q, k, v = wl.make_inputs(w)
        outs = []
        for mode in (OFF, ON):
            with pairing(fa, mode):
                outs.append(run_gpu(fa, q, k, v, causal, w.scale))
        assert np.array_equal(outs[0][0], outs[1][0]) and np.array_equal(outs[0][1], outs[1][1]), \
            f"B{B} H{H} N{N} causal={causal}: the two kernels differ"
        compare(outs[1][0], outs[1][1], q, k, v, causal, w.scale, all_rows(B, H, N),
                f"random B{B} H{H} N{N} causal={causal}")


def test_random_shapes_both_d64_kernels(fa):
    """Twelve seeded random d = 64 shapes (odd and even query-tile counts, ragged
    tails, causal or not), each through both d = 64 forward kernels and compared
    with the oracle on every row.  The two normalise O differently (the
    tensor-core sum of the rounded weights; the fp32 sum with each tile's
    largest-weight rounding), so they agree to rounding, not bit for bit."""
    rng = np.random.default_rng(20261203)
    for case in range(12):
        B, H = int(rng.integers(1, 3)), int(rng.integers(1, 4))
        N = int(rng.integers(1, 1400))
        causal = bool(rng.integers(0, 2))
        w = wl.Workload(f"rand64-{case}", B, H, N, 64, causal, "iid", 700 + case)
        q, k, v = wl.make_inputs(w)
        for mode in (OFF, ON):
            with pairing(fa, mode):
                o, lse = run_gpu(fa, q, k, v, causal, w.scale)
            compare(o, lse, q, k, v, causal, w.scale, all_rows(B, H, N),
                    f"random d64 mode {mode} B{B} H{H} N{N} causal={causal}")


@pytest.mark.parametrize("name,mode", [
    ("B4-H16-N4096-d128-causal", AUTO), ("B1-H32-N16384-d128-causal-late", AUTO), ("B1-H8-N131072-d64-causal", AUTO),
    ("B4-H16-N4096-d128-causal", ON), ("B1-H32-N16384-d128-causal-late", OFF), ("B1-H8-N131072-d64-causal", ON),
    ("B1-H8-N131072-d64-causal", OFF),
])
def test_large_workloads_sampled_rows(fa, name, mode):
    """The full-size configurations in the kernel the default policy picks (the
    headline in CTA pairs, B4-H16-N4096 one CTA per tile), and in the other one."""
    w = wl.WORKLOADS[name]
    q, k, v = wl.make_inputs(w)
    with pairing(fa, mode):
        o, lse = run_gpu(fa, q, k, v, w.causal, w.scale)
    compare(o, lse, q, k, v, w.causal, w.scale, wl.sample_rows(w), f"{name} mode {mode}")


@pytest.mark.parametrize("d,causal,mode", [(64, True, OFF), (64, False, OFF), (64, True, ON), (64, False, ON),
                                           (128, True, OFF), (128, True, ON), (128, False, AUTO)])
def test_reference_moves_often(fa, d, causal, mode):
    """Scores that grow steeply along the keys (q = 8 N(0,1), key norms ramping
    from 0.25 to 8.25 times N(0,1)): a row's running maximum outgrows its
    reference by more than the rescale threshold on ~13% of (row, key tile)
    steps, so O -- and at d = 64 the row sums kept beside O in tensor memory --
    is rescaled often.  Every row checked."""
    B, H, N = 1, 2, 2048
    rng = np.random.default_rng(4242 + d)
    ramp = (0.25 + 8.0 * np.arange(N) / (N - 1)).astype(np.float32)
    q = torch.from_numpy(rng.standard_normal((B, H, N, d), dtype=np.float32) * 8.0).to(torch.bfloat16)
    k = torch.from_numpy(rng.standard_normal((B, H, N, d), dtype=np.float32) * ramp[:, None]).to(torch.bfloat16)
    v = torch.from_numpy(rng.standard_normal((B, H, N, d), dtype=np.float32)).to(torch.bfloat16)
    scale = 1.0 / math.sqrt(d)
    with pairing(fa, mode):
        o, lse = run_gpu(fa, q, k, v, causal, scale)
    compare(o, lse, q, k, v, causal, scale, all_rows(B, H, N), f"moving reference d{d} causal={causal} mode {mode}")


# --------------------------------------------------------------------------
# closed forms that hold at any size
# --------------------------------------------------------------------------
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("N,d,c", [(64, 64, 18.0), (128, 128, 22.0)])
def test_onehot_dominant_key(fa, causal, N, d, c):
    q, k, v = wl.onehot_inputs(2, 3, N, d, c)
    scale = 1 / math.sqrt(d)
    s = scale * c * c
    o, lse = run_gpu(fa, q, k, v, causal, scale)
    vd = v.float().numpy().astype(np.float64)
    bound = (N - 1) * math.exp(-s) * 2 * np.abs(vd).max() + np.abs(vd).max() * 2.0 ** -8
    assert np.max(np.abs(o - vd)) <= bound
    n_vis = np.arange(1, N + 1) if causal else np.full(N, N)
    want_lse = s + np.log1p((n_vis - 1) * math.exp(-s))
    assert np.max(np.abs(lse - want_lse[None, None, :]) / np.maximum(1, want_lse)) <= LSE_TOL


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("N,d", [(8192, 64), (3000, 128)])
def test_uniform_attention_any_size(fa, causal, N, d):
    """q = 0: every visible key weighs the same, so O is a (prefix) mean of V and LSE = ln(#visible)."""
    w = wl.Workload("zeros", 1, 2, N, d, causal, "zeros-q", 77)
    q, k, v = wl.make_inputs(w)
    o, lse = run_gpu(fa, q, k, v, causal, w.scale)
    vd = v.float().numpy().astype(np.float64)[0]
    if causal:
        want = np.cumsum(vd, axis=1) / np.arange(1, N + 1)[None, :, None]
        want_lse = np.log(np.arange(1, N + 1))
    else:
        want = np.broadcast_to(vd.mean(axis=1, keepdims=True), vd.shape)
        want_lse = np.full(N, math.log(N))
    assert np.max(np.abs(o[0] - want)) <= O_TOL
    assert np.max(np.abs(lse[0] - want_lse[None]) / np.maximum(1, want_lse[None])) <= LSE_TOL


# --------------------------------------------------------------------------
# behaviour of the boundary
# --------------------------------------------------------------------------
def test_deterministic_and_stream(fa):
    w = wl.Workload("det", 2, 3, 700, 128, True, "iid", 5)
    q, k, v = (t.cuda() for t in wl.make_inputs(w))
    o1, l1 = fa.attention(q, k, v, causal=True)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        o2, l2 = fa.attention(q, k, v, causal=True, stream=s)
    s.synchronize()
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


@pytest.mark.parametrize("mode", [AUTO, ON])
def test_work_queue_across_calls_and_streams(fa, mode):
    """The persistent kernel takes tiles from a device work counter that every
    launch leaves at zero: back-to-back calls, and calls overlapping on two
    streams, must give exactly the results of the same calls run alone (every
    tile's arithmetic is independent of which CTA runs it).  ON: the d = 128
    calls run in CTA pairs (128 two-tile units: static rounds + dynamic tail),
    the d = 64 calls two tiles per CTA (48 units, one CTA each)."""
    with pairing(fa, mode):
        _work_queue_calls(fa)


def _work_queue_calls(fa):
    wa = wl.Workload("qa", 2, 8, 2048, 128, True, "iid", 11)   # 256 tiles: static pairs + dynamic tail
    wb = wl.Workload("qb", 1, 4, 3000, 64, True, "iid", 12)    # ragged N, d = 64
    qa, ka, va = (t.cuda() for t in wl.make_inputs(wa))
    qb, kb, vb = (t.cuda() for t in wl.make_inputs(wb))
    ref_a = fa.attention(qa, ka, va, causal=True)
    ref_b = fa.attention(qb, kb, vb, causal=True)
    torch.cuda.synchronize()
    for _ in range(20):  # back to back on one stream
        o, l = fa.attention(qa, ka, va, causal=True)
    torch.cuda.synchronize()
    assert torch.equal(o, ref_a[0]) and torch.equal(l, ref_a[1])
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    outs = []
    for _ in range(8):  # alternating streams, no synchronisation in between
        with torch.cuda.stream(s1):
            outs.append(("a", fa.attention(qa, ka, va, causal=True, stream=s1)))
        with torch.cuda.stream(s2):
            outs.append(("b", fa.attention(qb, kb, vb, causal=True, stream=s2)))
    torch.cuda.synchronize()
    for which, (o, l) in outs:
        ro, rl = ref_a if which == "a" else ref_b
        assert torch.equal(o, ro) and torch.equal(l, rl), which


@pytest.mark.parametrize("d,mode", [(64, OFF), (64, ON), (128, OFF), (128, ON)])
def test_output_alignment_and_bounds(fa, d, mode):
    """O at a 16-byte but not 32-byte aligned address, N ragged: the same values
    as an aligned output, and nothing written outside O (rows past N are not
    stored, by row stores or tensor stores)."""
    B, H, N = 2, 3, 200
    w = wl.Workload("al", B, H, N, d, True, "iid", 13)
    q, k, v = (t.cuda() for t in wl.make_inputs(w))
    with pairing(fa, mode):
        _aligned_and_bounded(fa, q, k, v, B, H, N, d)


def _aligned_and_bounded(fa, q, k, v, B, H, N, d):
    ref_o, ref_l = fa.attention(q, k, v, causal=True)
    n = B * H * N * d
    pad = 64                                    # elements of sentinel on each side
    buf = torch.full((n + 2 * pad + 8,), -7.0, dtype=torch.bfloat16, device="cuda")
    assert buf.data_ptr() % 32 == 0
    o = buf[pad + 8: pad + 8 + n]               # 16-byte aligned, 32-byte misaligned
    assert o.data_ptr() % 16 == 0 and o.data_ptr() % 32 == 16
    lse = torch.empty((B, H, N), dtype=torch.float32, device="cuda")
    rc = fa.lib().fa_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(), B, H, N, d, 1,
                         1.0 / math.sqrt(d), torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    assert rc == 0
    assert torch.equal(o.view(B, H, N, d), ref_o) and torch.equal(lse, ref_l)
    assert torch.all(buf[:pad + 8] == -7.0) and torch.all(buf[pad + 8 + n:] == -7.0)


@pytest.mark.parametrize("B,H,N,d,mode", [(1, 65535, 3, 64, OFF), (1, 65535, 3, 64, ON), (65535, 1, 40, 128, OFF),
                                         (65535, 1, 40, 128, ON)])
def test_largest_head_count(fa, B, H, N, d, mode):
    """B*H at the limit the boundary accepts (65535): every (head, query tile)
    unit runs through the persistent schedule's static rounds and dynamic tail;
    sampled rows across the whole range, including the last head."""
    w = wl.Workload("maxbh", B, H, N, d, True, "iid", 99)
    q, k, v = wl.make_inputs(w)
    with pairing(fa, mode):
        o, lse = run_gpu(fa, q, k, v, True, w.scale)
    rng = np.random.default_rng(100)
    total = B * H * N
    rows = np.unique(np.concatenate([rng.integers(0, total, 600), [0, N - 1, total - N, total - 1]])).astype(np.int64)
    compare(o, lse, q, k, v, True, w.scale, rows, f"B{B} H{H} N{N} d{d}")


def test_inputs_untouched(fa):
    w = wl.Workload("ro", 1, 2, 300, 64, False, "iid", 6)
    q, k, v = (t.cuda() for t in wl.make_inputs(w))
    qc, kc, vc = q.clone(), k.clone(), v.clone()
    fa.attention(q, k, v)
    torch.cuda.synchronize()
    assert torch.equal(q, qc) and torch.equal(k, kc) and torch.equal(v, vc)


def test_rejects_bad_arguments_on_device(fa):
    q = torch.zeros((1, 1, 128, 64), dtype=torch.bfloat16, device="cuda")
    o = torch.empty_like(q)
    lse = torch.empty((1, 1, 128), dtype=torch.float32, device="cuda")
    L = fa.lib()
    ptr = q.data_ptr()
    assert L.fa_fwd(ptr, ptr, ptr, o.data_ptr(), lse.data_ptr(), 1, 1, 128, 96, 0, 0.1, 0) == fa.FA_ERR_HEAD_DIM
    assert L.fa_fwd(ptr + 2, ptr, ptr, o.data_ptr(), lse.data_ptr(), 1, 1, 128, 64, 0, 0.1, 0) == fa.FA_ERR_ALIGNMENT
    assert L.fa_fwd(ptr, ptr, ptr, ptr, lse.data_ptr(), 1, 1, 128, 64, 0, 0.1, 0) == fa.FA_ERR_ALIAS
    assert L.fa_fwd(ptr, ptr, ptr, o.data_ptr(), lse.data_ptr(), 1, 1, 128, 64, 0, -1.0, 0) == fa.FA_ERR_SCALE
    with pytest.raises(ValueError):
        fa.attention(q.cpu(), q.cpu(), q.cpu())


def test_watchdog_ends_a_wait_nothing_completes(fa):
    st = fa.fa_watchdog_selftest(20_000_000)  # 20 ms limit on a barrier no one arrives on
    assert st & (1 << 8), f"status {st:#x}"
    fa.fa_clear_device_status()
    assert fa.fa_get_device_status() == 0
    # the context is still usable afterwards
    w = wl.Workload("after", 1, 1, 256, 64, True, "iid", 8)
    q, k, v = wl.make_inputs(w)
    o, lse = run_gpu(fa, q, k, v, True, w.scale)
    compare(o, lse, q, k, v, True, w.scale, all_rows(1, 1, 256), "after watchdog")
    # the device-side timeout flag as the boundary's int: set by the self-test, 0 once cleared
    assert fa.fa_watchdog_selftest(20_000_000) & (1 << 8)
    assert fa.fa_get_last_error() & (1 << 8)
    fa.fa_clear_device_status()
    assert fa.fa_get_last_error() == 0


@pytest.mark.parametrize("d,mode", [(64, OFF), (64, ON), (128, OFF), (128, ON)])
def test_watchdog_abort_leaves_nan_lse(fa, d, mode):
    """The forward kernel's own abort path: its S products withheld, the softmax
    warps' first wait runs out; the tile's lse rows read NaN, o is not written,
    and the context stays usable.  ON at d = 128: a CTA pair, both CTAs abort
    (the peer's query tile lies past N) and leave together; at d = 64 one CTA
    with two tiles, the second past N."""
    N = 100
    w = wl.Workload("abort", 1, 1, N, d, False, "iid", 31)
    q, k, v = (t.cuda() for t in wl.make_inputs(w))
    o = torch.full_like(q, 3.0)
    lse = torch.full((1, 1, N), 7.0, dtype=torch.float32, device="cuda")
    with pairing(fa, mode):
        st = fa.fa_watchdog_selftest_fwd(5_000_000, q, k, v, o, lse, N, d)
    # the first wait to run out names itself: the softmax's wait on S, or the P V issuer's wait on P
    assert st & ((1 << 5) | (1 << 3)), f"status {st:#x}"
    assert torch.isnan(lse).all()
    assert (o == 3.0).all()
    fa.fa_clear_device_status()
    assert fa.fa_get_last_error() == 0
    o2, lse2 = run_gpu(fa, q.cpu(), k.cpu(), v.cpu(), False, w.scale)
    compare(o2, lse2, q.cpu(), k.cpu(), v.cpu(), False, w.scale, all_rows(1, 1, N), "after abort")


@pytest.mark.parametrize("d", [64, 128])
def test_kernel_resources_report(fa, d):
    """The runtime's view of the kernels as launched: one CTA per SM, the whole
    tensor memory, no local memory (no spills), 384 threads."""
    sm = torch.cuda.get_device_properties(0).multi_processor_count
    assert sm >= 1
    kernels = [fa.FA_KERNEL_FWD, fa.FA_KERNEL_FWD_MASKED, fa.FA_KERNEL_FWD_SPLITKV, fa.FA_KERNEL_BWD_DQ,
               fa.FA_KERNEL_BWD_DKDV, paired_kind(fa, d)]
    with pytest.raises(fa.FaError):  # each paired kernel exists at one head dim only
        fa.fa_kernel_resources(d, fa.FA_KERNEL_FWD_PAIR if d == 64 else fa.FA_KERNEL_FWD_TWO)
    for kernel in kernels:
        r = fa.fa_kernel_resources(d, kernel)
        assert r["threads_per_cta"] == 384, r
        assert r["ctas_per_sm"] == 1, r
        assert r["tmem_columns"] == 512, r
        assert 0 < r["registers_per_thread"] <= 168, r
        assert r["local_bytes_per_thread"] == 0, r
        assert 150 * 1024 < r["dynamic_smem_bytes"] <= 227 * 1024, r


@pytest.mark.parametrize("heads,d,causal", [(None, 64, False), ("sm+1", 64, False), (None, 128, True),
                                           ("pairs", 128, True), ("pairs+1", 128, True), ("units", 64, True),
                                           ("units+1", 64, False)])
def test_one_tile_per_cta_boundary(fa, heads, d, causal):
    """N = 128, so each head is one query tile: as many heads as SMs gives each CTA
    its tile by index; one more head takes the persistent schedule with its work
    counter.  CTA pairs (N = 256, one two-tile unit per head): as many heads as
    pairs fit on the device (one per two SMs), and one more.  Two tiles per CTA
    (d = 64, N = 256): as many units as SMs, and one more.  Every row against
    the oracle."""
    sm = torch.cuda.get_device_properties(0).multi_processor_count
    H = {"sm+1": sm + 1, "pairs": sm // 2, "pairs+1": sm // 2 + 1, "units": sm, "units+1": sm + 1}.get(heads, sm)
    N = 256 if heads and heads.startswith(("pairs", "units")) else 128
    w = wl.Workload(f"tiles-{H}", 1, H, N, d, causal, "iid", 61 + H)
    q, k, v = wl.make_inputs(w)
    with pairing(fa, ON if N == 256 else OFF):
        o, lse = run_gpu(fa, q, k, v, causal, w.scale)
    compare(o, lse, q, k, v, causal, w.scale, all_rows(1, H, N), w.name)
