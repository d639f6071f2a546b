"""The C-ABI library: it loads, exports every function include/fa.h declares,
and rejects bad arguments on the host before any CUDA work (no GPU needed)."""
import ctypes
import re

import pytest
import torch

import __graft_entry__


@pytest.fixture(scope="module")
def fa():
    __graft_entry__.build()
    import online_softmax_04_gb300 as m

    return m


def declared_functions(path):
    text = open(path).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return re.findall(r"^\s*[A-Za-z_][\w\s\*]*?\b(fa_\w+)\s*\(", text, flags=re.M)


def test_exports_every_declared_symbol(fa):
    names = declared_functions(fa.HEADER_PATH)
    assert {"fa_fwd", "fa_strerror", "fa_get_last_error", "fa_get_device_status", "fa_clear_device_status",
            "fa_set_watchdog_ns", "fa_watchdog_selftest", "fa_watchdog_selftest_fwd", "fa_kernel_resources",
            "fa_set_fwd_pairing", "fa_fwd_kernel_for", "fa_version"} <= set(names)
    raw = ctypes.CDLL(fa.LIB_PATH)
    for n in names:
        assert hasattr(raw, n), n


def test_strerror_and_version(fa):
    assert fa.fa_version() >= 10000
    for code in range(-9, 1):
        assert fa.fa_strerror(code) and fa.fa_strerror(code) != "unknown error code"
    assert fa.fa_strerror(-1000) == "unknown error code"


def test_fwd_pairing_policy(fa):
    """Which forward kernel a call takes.  d = 128: CTA pairs for full attention and
    for causal attention from 96 query tiles on (the masked key tile a pair
    computes per two query tiles costs 1 / (tiles / 2 + 1)).  d = 64: two tiles
    per CTA once there are enough units to fill the SMs (not for one head of
    N = 4096, nor for many heads of two tiles, where the masked tile is a third
    of the work).  The override modes; host-only, no device touched."""
    F, P, T = fa.FA_KERNEL_FWD, fa.FA_KERNEL_FWD_PAIR, fa.FA_KERNEL_FWD_TWO
    prev = fa.fa_set_fwd_pairing(fa.FA_PAIR_AUTO)
    try:
        assert fa.fa_fwd_kernel_for(1, 32, 16384, 128, True) == P      # 128 tiles
        assert fa.fa_fwd_kernel_for(1, 1, 96 * 128, 128, True) == P    # 96 tiles
        assert fa.fa_fwd_kernel_for(1, 1, 95 * 128, 128, True) == F    # 95 tiles
        assert fa.fa_fwd_kernel_for(4, 16, 4096, 128, True) == F
        assert fa.fa_fwd_kernel_for(1, 1, 1, 128, False) == P
        assert fa.fa_fwd_kernel_for(4, 16, 4096, 128, False) == P
        assert fa.fa_fwd_kernel_for(1, 8, 131072, 64, True) == T
        assert fa.fa_fwd_kernel_for(4, 16, 4096, 64, True) == T
        assert fa.fa_fwd_kernel_for(2, 16, 8192, 64, False) == T
        assert fa.fa_fwd_kernel_for(1, 1, 4096, 64, False) == F      # 16 units on 152 SMs
        assert fa.fa_fwd_kernel_for(1, 4, 4096, 64, False) == F
        assert fa.fa_fwd_kernel_for(32, 32, 256, 64, True) == F     # two tiles a head
        assert fa.fa_fwd_kernel_for(1, 1, 256, 64, False) == F
        assert fa.fa_set_fwd_pairing(fa.FA_PAIR_OFF) == fa.FA_PAIR_AUTO
        assert fa.fa_fwd_kernel_for(1, 1, 4096, 128, False) == F
        assert fa.fa_fwd_kernel_for(1, 8, 131072, 64, True) == F
        assert fa.fa_set_fwd_pairing(fa.FA_PAIR_ON) == fa.FA_PAIR_OFF
        assert fa.fa_fwd_kernel_for(1, 1, 256, 128, True) == P
        assert fa.fa_fwd_kernel_for(1, 1, 256, 64, True) == T
        assert fa.lib().fa_fwd_kernel_for(1, 1, 256, 96, 0) == fa.FA_ERR_HEAD_DIM
        assert fa.lib().fa_fwd_kernel_for(0, 1, 256, 128, 0) == fa.FA_ERR_SHAPE
        assert fa.lib().fa_fwd_kernel_for(300, 300, 256, 128, 0) == fa.FA_ERR_SHAPE
        assert fa.lib().fa_set_fwd_pairing(7) == fa.FA_ERR_SHAPE
        assert fa.fa_set_fwd_pairing(fa.FA_PAIR_AUTO) == fa.FA_PAIR_ON  # the bad mode changed nothing
    finally:
        fa.fa_set_fwd_pairing(prev)


FAKE = 1 << 40  # never dereferenced: every case below fails validation first


def call(fa, q=FAKE, k=FAKE + (1 << 30), v=FAKE + (2 << 30), o=FAKE + (3 << 30), lse=FAKE + (4 << 30), B=1, H=1,
         N=128, d=64, causal=0, scale=0.125):
    return fa.lib().fa_fwd(q, k, v, o, lse, B, H, N, d, causal, scale, 0)


def test_host_validation(fa):
    assert call(fa, q=0) == fa.FA_ERR_NULL_POINTER
    assert call(fa, lse=0) == fa.FA_ERR_NULL_POINTER
    assert call(fa, d=96) == fa.FA_ERR_HEAD_DIM
    assert call(fa, d=256) == fa.FA_ERR_HEAD_DIM
    assert call(fa, N=0) == fa.FA_ERR_SHAPE
    assert call(fa, B=0) == fa.FA_ERR_SHAPE
    assert call(fa, B=300, H=300) == fa.FA_ERR_SHAPE
    assert call(fa, q=FAKE + 8) == fa.FA_ERR_ALIGNMENT
    assert call(fa, lse=FAKE + (4 << 30) + 2) == fa.FA_ERR_ALIGNMENT
    assert call(fa, scale=0.0) == fa.FA_ERR_SCALE
    assert call(fa, scale=-1.0) == fa.FA_ERR_SCALE
    assert call(fa, scale=float("nan")) == fa.FA_ERR_SCALE
    assert call(fa, scale=float("inf")) == fa.FA_ERR_SCALE
    assert call(fa, o=FAKE + 64) == fa.FA_ERR_ALIAS          # o overlaps q
    assert call(fa, lse=FAKE + (3 << 30) + 64) == fa.FA_ERR_ALIAS  # lse overlaps o


def test_masked_host_validation(fa):
    L = fa.lib()
    q, k, v, o, lse = FAKE, FAKE + (1 << 30), FAKE + (2 << 30), FAKE + (3 << 30), FAKE + (4 << 30)
    doc = FAKE + (5 << 30)

    def m(wl=-1, wr=0, d=doc, N=128):
        return L.fa_fwd_masked(q, k, v, o, lse, 1, 1, N, 64, wl, wr, d, 0.125, 0)

    assert m(wl=-2) == fa.FA_ERR_MASK
    assert m(wr=-7) == fa.FA_ERR_MASK
    assert m(d=doc + 2) == fa.FA_ERR_ALIGNMENT
    assert m(d=o + 64) == fa.FA_ERR_ALIAS            # ids inside o
    assert m(N=0) == fa.FA_ERR_SHAPE
    assert L.fa_fwd_masked(0, k, v, o, lse, 1, 1, 128, 64, -1, 0, None, 0.125, 0) == fa.FA_ERR_NULL_POINTER
    if not torch.cuda.is_available():
        assert m() in (fa.FA_ERR_CUDA, fa.FA_ERR_DEVICE)


def test_backward_host_validation(fa):
    L = fa.lib()
    q, k, v, o, do = (FAKE + (i << 30) for i in range(5))
    lse, dq, dk, dv, ws = (FAKE + (i << 30) for i in range(5, 10))
    nws = fa.fa_bwd_workspace_bytes(2, 3, 100, 64)
    assert nws == 2 * 3 * 100 * 4 and fa.fa_bwd_workspace_bytes(2, 3, 100, 96) == 0

    def b(**kw):
        a = dict(q=q, k=k, v=v, o=o, do=do, lse=lse, dq=dq, dk=dk, dv=dv, d=64, ws=ws, wsb=nws, scale=0.125)
        a.update(kw)
        return L.fa_bwd(a["q"], a["k"], a["v"], a["o"], a["do"], a["lse"], a["dq"], a["dk"], a["dv"], 2, 3, 100,
                        a["d"], 1, a["scale"], a["ws"], a["wsb"], 0)

    assert b(do=0) == fa.FA_ERR_NULL_POINTER
    assert b(ws=0) == fa.FA_ERR_NULL_POINTER
    assert b(d=256) == fa.FA_ERR_HEAD_DIM
    assert b(dk=dk + 8) == fa.FA_ERR_ALIGNMENT
    assert b(scale=0.0) == fa.FA_ERR_SCALE
    assert b(wsb=nws - 1) == fa.FA_ERR_WORKSPACE
    assert b(dq=o + 64) == fa.FA_ERR_ALIAS      # dq over o
    assert b(ws=dv + 64) == fa.FA_ERR_ALIAS     # workspace over dv
    if not torch.cuda.is_available():
        assert b() in (fa.FA_ERR_CUDA, fa.FA_ERR_DEVICE)


def test_softmax_rows_host_validation(fa):
    L = fa.lib()
    x, y, lse = FAKE, FAKE + (1 << 30), FAKE + (2 << 30)
    assert L.fa_softmax_rows(0, y, lse, 4, 16, 0) == fa.FA_ERR_NULL_POINTER
    assert L.fa_softmax_rows(x, 0, lse, 4, 16, 0) == fa.FA_ERR_NULL_POINTER
    assert L.fa_softmax_rows(x, y, lse, 0, 16, 0) == fa.FA_ERR_SHAPE
    assert L.fa_softmax_rows(x, y, lse, 4, 0, 0) == fa.FA_ERR_SHAPE
    assert L.fa_softmax_rows(x, y, lse, (1 << 40) + 1, 1, 0) == fa.FA_ERR_SHAPE
    assert L.fa_softmax_rows(x + 2, y, lse, 4, 16, 0) == fa.FA_ERR_ALIGNMENT
    assert L.fa_softmax_rows(x, y, lse + 1, 4, 16, 0) == fa.FA_ERR_ALIGNMENT
    assert L.fa_softmax_rows(x, x + 4, lse, 4, 16, 0) == fa.FA_ERR_ALIAS     # y shifted over x
    assert L.fa_softmax_rows(x, y, x + 8, 4, 16, 0) == fa.FA_ERR_ALIAS       # lse inside x
    if not torch.cuda.is_available():  # valid arguments, in place: no device to run on
        assert L.fa_softmax_rows(x, x, 0, 4, 16, 0) in (fa.FA_ERR_CUDA, fa.FA_ERR_DEVICE)


@pytest.mark.skipif(torch.cuda.is_available(), reason="valid arguments would launch on a real GPU")
def test_valid_arguments_without_a_gpu_fail_cleanly(fa):
    rc = call(fa)
    assert rc in (fa.FA_ERR_CUDA, fa.FA_ERR_DEVICE)


def test_binding_refuses_cpu_tensors(fa):
    q = torch.zeros((1, 1, 8, 64), dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        fa.attention(q, q, q)


def test_product_does_not_import_the_oracle():
    import os

    import online_softmax_04_gb300

    pkg = os.path.dirname(online_softmax_04_gb300.__file__)
    for name in os.listdir(pkg):
        if name.endswith((".py", ".cu", ".cuh")):
            src = open(os.path.join(pkg, name)).read()
            assert "import oracle" not in src and "from oracle" not in src and "liboracle" not in src, name
    for name in os.listdir(os.path.join(pkg, "csrc")):
        src = open(os.path.join(pkg, "csrc", name)).read()
        assert "oracle" not in src, name


def test_splitkv_host_validation(fa):
    L = fa.lib()
    W = FAKE + (5 << 30)

    def sk(n_splits=2, ws=W, wsb=1 << 30, **kw):
        a = dict(q=FAKE, k=FAKE + (1 << 30), v=FAKE + (2 << 30), o=FAKE + (3 << 30), lse=FAKE + (4 << 30), B=1, H=1,
                 N=128, d=64, causal=0, scale=0.125)
        a.update(kw)
        return L.fa_fwd_splitkv(a["q"], a["k"], a["v"], a["o"], a["lse"], a["B"], a["H"], a["N"], a["d"],
                                a["causal"], a["scale"], n_splits, ws, wsb, 0)

    assert sk(n_splits=65) == fa.FA_ERR_SPLITS
    assert sk(n_splits=-1) == fa.FA_ERR_SPLITS
    assert sk(ws=0) == fa.FA_ERR_NULL_POINTER
    assert sk(ws=W + 4) == fa.FA_ERR_ALIGNMENT
    assert sk(wsb=10) == fa.FA_ERR_WORKSPACE
    assert sk(ws=FAKE + 16) == fa.FA_ERR_ALIAS
    assert sk(d=96) == fa.FA_ERR_HEAD_DIM  # the fa_fwd checks come first


def test_splitkv_workspace_formula(fa):
    assert fa.fa_splitkv_workspace_bytes(1, 1, 4096, 64, 4) == 4 * 4096 * (64 + 3) * 4
    assert fa.fa_splitkv_workspace_bytes(2, 3, 100, 128, 7) == 7 * 6 * 100 * 131 * 4
    assert fa.fa_splitkv_workspace_bytes(1, 1, 128, 96, 2) == 0
    assert fa.fa_splitkv_workspace_bytes(1, 1, 128, 64, 65) == 0
    # automatic count: never more than the key tiles, 1 once the plain grid fills the GPU
    assert 1 <= fa.fa_splitkv_auto_splits(1, 1, 256, 64, 0) <= 2
    assert fa.fa_splitkv_auto_splits(1, 32, 16384, 128, 1) == 1


def test_host_streamed_validation(fa):
    """fa_fwd_host: argument checks that need no GPU, and the workspace size rule."""
    L = fa.lib()
    q, k, v, o, lse = FAKE, FAKE + (1 << 30), FAKE + (2 << 30), FAKE + (3 << 30), FAKE + (4 << 30)
    ws = FAKE + (5 << 30)
    B, H, N, d = 2, 3, 200, 64
    need = fa.fa_fwd_host_workspace_bytes(B, H, N, d, 2)
    # three slots of 2 heads: q, k, v, o (2*200*64*2 = 51200 B each, 256-aligned) and lse (1600 -> 1792 B)
    assert need == 3 * (4 * 51200 + 1792)
    assert fa.fa_fwd_host_workspace_bytes(B, H, N, d, 0) == 3 * (4 * 25600 + 1024)  # ceil(6 / 8) = 1 head
    assert fa.fa_fwd_host_workspace_bytes(B, H, N, d, 7) == 0
    assert fa.fa_fwd_host_workspace_bytes(B, H, N, 96, 1) == 0

    def call(hpc=2, w=ws, wb=need, **kw):
        a = dict(q=q, k=k, v=v, o=o, lse=lse, d=d)
        a.update(kw)
        return L.fa_fwd_host(a["q"], a["k"], a["v"], a["o"], a["lse"], B, H, N, a["d"], 1, 0.125, hpc, w, wb, 0)

    assert call(q=0) == fa.FA_ERR_NULL_POINTER
    assert call(d=96) == fa.FA_ERR_HEAD_DIM
    assert call(hpc=-1) == fa.FA_ERR_SHAPE
    assert call(hpc=B * H + 1) == fa.FA_ERR_SHAPE
    assert call(w=0) == fa.FA_ERR_NULL_POINTER
    assert call(w=ws + 128) == fa.FA_ERR_ALIGNMENT
    assert call(wb=need - 1) == fa.FA_ERR_WORKSPACE
    assert call(o=q + 64) == fa.FA_ERR_ALIAS


def test_kernel_resources_host_checks(fa):
    L = fa.lib()
    r = fa.KernelResources()
    assert L.fa_kernel_resources(64, 0, None) == fa.FA_ERR_NULL_POINTER
    assert L.fa_kernel_resources(96, 0, ctypes.byref(r)) == fa.FA_ERR_HEAD_DIM
    if not torch.cuda.is_available():
        assert L.fa_kernel_resources(64, 0, ctypes.byref(r)) in (fa.FA_ERR_CUDA, fa.FA_ERR_DEVICE)
