"""GB300 (sm_103a) fused attention forward -- Python binding of include/fa.h.

This module only marshals arguments: it turns tensors into device pointers
and streams into handles and calls the C ABI in ``libfa_gb300.so``.  Every
step of the computation runs in the CUDA kernels; there is no CPU or PyTorch
fallback, and a missing library is an error.

    fa_fwd(q, k, v, o, lse, B, H, N, d, causal, scale, stream)   # C ABI mirror
    o, lse = attention(q, k, v, causal=False, scale=None)         # allocates outputs
"""
from __future__ import annotations

import ctypes
import math
import os
import threading

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libfa_gb300.so")
HEADER_PATH = os.path.join(os.path.dirname(_HERE), "include", "fa.h")

FA_OK = 0
FA_ERR_NULL_POINTER = -1
FA_ERR_HEAD_DIM = -2
FA_ERR_SHAPE = -3
FA_ERR_ALIGNMENT = -4
FA_ERR_SCALE = -5
FA_ERR_ALIAS = -6
FA_ERR_TENSOR_MAP = -7
FA_ERR_CUDA = -8
FA_ERR_DEVICE = -9
FA_ERR_SPLITS = -10
FA_ERR_WORKSPACE = -11
FA_ERR_SCRATCH_LIMIT = -12
FA_ERR_MASK = -13
FA_NOALLOC_SCRATCH_BYTES = 32 * 1024 * 1024
(FA_KERNEL_FWD, FA_KERNEL_FWD_MASKED, FA_KERNEL_FWD_SPLITKV, FA_KERNEL_BWD_DQ, FA_KERNEL_BWD_DKDV, FA_KERNEL_FWD_PAIR,
 FA_KERNEL_FWD_TWO) = range(7)
FA_PAIR_AUTO, FA_PAIR_OFF, FA_PAIR_ON = range(3)


class KernelResources(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int) for n in ("registers_per_thread", "threads_per_cta", "dynamic_smem_bytes",
                                            "static_smem_bytes", "local_bytes_per_thread", "ctas_per_sm",
                                            "tmem_columns")]

_lock = threading.Lock()
_lib = None


class FaError(RuntimeError):
    def __init__(self, code: int, what: str):
        super().__init__(f"{what} (FA code {code})")
        self.code = code


def lib() -> ctypes.CDLL:
    """The loaded C library; raises if it has not been built."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(f"{LIB_PATH} is missing: build it first (python -c 'import __graft_entry__ as g; "
                                   "g.build()')")
            L = ctypes.CDLL(LIB_PATH)
            P, I, F = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
            L.fa_fwd.argtypes = [P, P, P, P, P, I, I, I, I, I, F, P]
            L.fa_fwd.restype = I
            L.fa_fwd_masked.argtypes = [P, P, P, P, P, I, I, I, I, I, I, P, F, P]
            L.fa_fwd_masked.restype = I
            L.fa_fwd_splitkv.argtypes = [P, P, P, P, P, I, I, I, I, I, F, I, P, ctypes.c_size_t, P]
            L.fa_fwd_splitkv.restype = I
            L.fa_fwd_splitkv_noalloc.argtypes = [P, P, P, P, P, I, I, I, I, I, F, I, P]
            L.fa_fwd_splitkv_noalloc.restype = I
            L.fa_splitkv_workspace_bytes.argtypes = [I, I, I, I, I]
            L.fa_splitkv_workspace_bytes.restype = ctypes.c_size_t
            L.fa_splitkv_auto_splits.argtypes = [I, I, I, I, I]
            L.fa_splitkv_auto_splits.restype = I
            L.fa_fwd_host.argtypes = [P, P, P, P, P, I, I, I, I, I, F, I, P, ctypes.c_size_t, P]
            L.fa_fwd_host.restype = I
            L.fa_fwd_host_workspace_bytes.argtypes = [I, I, I, I, I]
            L.fa_fwd_host_workspace_bytes.restype = ctypes.c_size_t
            L.fa_strerror.argtypes = [I]
            L.fa_strerror.restype = ctypes.c_char_p
            L.fa_get_device_status.argtypes = [ctypes.POINTER(ctypes.c_uint)]
            L.fa_get_device_status.restype = I
            L.fa_clear_device_status.argtypes = []
            L.fa_clear_device_status.restype = I
            L.fa_set_watchdog_ns.argtypes = [ctypes.c_uint64]
            L.fa_set_watchdog_ns.restype = ctypes.c_uint64
            L.fa_watchdog_selftest.argtypes = [ctypes.c_uint64, P, ctypes.POINTER(ctypes.c_uint)]
            L.fa_watchdog_selftest.restype = I
            L.fa_softmax_rows.argtypes = [P, P, P, ctypes.c_longlong, I, P]
            L.fa_softmax_rows.restype = I
            L.fa_bwd.argtypes = [P, P, P, P, P, P, P, P, P, I, I, I, I, I, F, P, ctypes.c_size_t, P]
            L.fa_bwd.restype = I
            L.fa_bwd_workspace_bytes.argtypes = [I, I, I, I]
            L.fa_bwd_workspace_bytes.restype = ctypes.c_size_t
            L.fa_get_last_error.argtypes = []
            L.fa_get_last_error.restype = I
            L.fa_watchdog_selftest_fwd.argtypes = [ctypes.c_uint64, P, P, P, P, P, I, I, P, ctypes.POINTER(ctypes.c_uint)]
            L.fa_watchdog_selftest_fwd.restype = I
            L.fa_kernel_resources.argtypes = [I, I, ctypes.POINTER(KernelResources)]
            L.fa_kernel_resources.restype = I
            L.fa_set_fwd_pairing.argtypes = [I]
            L.fa_set_fwd_pairing.restype = I
            L.fa_fwd_kernel_for.argtypes = [I, I, I, I, I]
            L.fa_fwd_kernel_for.restype = I
            L.fa_version.argtypes = []
            L.fa_version.restype = I
            _lib = L
    return _lib


def _ptr(x) -> int:
    if x is None:
        return 0
    if isinstance(x, int):
        return x
    if hasattr(x, "data_ptr"):
        if not x.is_cuda:
            raise ValueError("tensors must live on a CUDA device (no CPU path exists)")
        if not x.is_contiguous():
            raise ValueError("tensors must be contiguous")
        return x.data_ptr()
    raise TypeError(f"cannot take a device pointer from {type(x)!r}")


def _stream(stream) -> int:
    if stream is None:
        import torch

        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _host_ptr(x) -> int:
    """Address of a contiguous CPU tensor (the host side of fa_fwd_host)."""
    if isinstance(x, int):
        return x
    if hasattr(x, "data_ptr"):
        if x.is_cuda:
            raise ValueError("fa_fwd_host takes host (CPU) tensors")
        if not x.is_contiguous():
            raise ValueError("tensors must be contiguous")
        return x.data_ptr()
    raise TypeError(f"cannot take a host pointer from {type(x)!r}")


def fa_strerror(code: int) -> str:
    return lib().fa_strerror(int(code)).decode()


def fa_fwd(q, k, v, o, lse, B: int, H: int, N: int, d: int, causal: bool, scale: float, stream=None) -> None:
    """Enqueue the fused forward; raises FaError on a nonzero C return code."""
    rc = lib().fa_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), int(B), int(H), int(N), int(d),
                      1 if causal else 0, float(scale), _stream(stream))
    if rc != FA_OK:
        raise FaError(rc, fa_strerror(rc))


def attention(q, k, v, causal: bool = False, scale: float | None = None, stream=None):
    """q, k, v: CUDA bf16 [B, H, N, d].  Returns (o bf16 [B,H,N,d], lse fp32 [B,H,N])."""
    import torch

    if q.dtype != torch.bfloat16 or k.dtype != torch.bfloat16 or v.dtype != torch.bfloat16:
        raise ValueError("q, k and v must be bfloat16")
    if q.dim() != 4 or q.shape != k.shape or q.shape != v.shape:
        raise ValueError("q, k and v must share one [B, H, N, d] shape")
    B, H, N, d = q.shape
    o = torch.empty_like(q)
    lse = torch.empty((B, H, N), dtype=torch.float32, device=q.device)
    fa_fwd(q, k, v, o, lse, B, H, N, d, causal, (1.0 / math.sqrt(d)) if scale is None else scale, stream)
    return o, lse


def fa_fwd_masked(q, k, v, o, lse, B: int, H: int, N: int, d: int, window_left: int, window_right: int, doc_ids,
                  scale: float, stream=None) -> None:
    """Enqueue the masked forward (window and/or document ids); raises FaError on a nonzero C return code."""
    rc = lib().fa_fwd_masked(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), int(B), int(H), int(N), int(d),
                             int(window_left), int(window_right), _ptr(doc_ids), float(scale), _stream(stream))
    if rc != FA_OK:
        raise FaError(rc, fa_strerror(rc))


def attention_masked(q, k, v, window_left: int = -1, window_right: int = -1, doc_ids=None, scale: float | None = None,
                     stream=None):
    """q, k, v: CUDA bf16 [B, H, N, d]; doc_ids: CUDA int32 [B, N] or None.
    Returns (o bf16 [B,H,N,d], lse fp32 [B,H,N])."""
    import torch

    if q.dtype != torch.bfloat16 or k.dtype != torch.bfloat16 or v.dtype != torch.bfloat16:
        raise ValueError("q, k and v must be bfloat16")
    if q.dim() != 4 or q.shape != k.shape or q.shape != v.shape:
        raise ValueError("q, k and v must share one [B, H, N, d] shape")
    B, H, N, d = q.shape
    if doc_ids is not None and (doc_ids.dtype != torch.int32 or tuple(doc_ids.shape) != (B, N)):
        raise ValueError("doc_ids must be int32 [B, N]")
    o = torch.empty_like(q)
    lse = torch.empty((B, H, N), dtype=torch.float32, device=q.device)
    fa_fwd_masked(q, k, v, o, lse, B, H, N, d, window_left, window_right, doc_ids,
                  (1.0 / math.sqrt(d)) if scale is None else scale, stream)
    return o, lse


def fa_fwd_splitkv(q, k, v, o, lse, B: int, H: int, N: int, d: int, causal: bool, scale: float, n_splits: int,
                   workspace, workspace_bytes: int, stream=None) -> None:
    """Enqueue the split-KV forward and its merge; raises FaError on a nonzero C return code."""
    rc = lib().fa_fwd_splitkv(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), int(B), int(H), int(N), int(d),
                              1 if causal else 0, float(scale), int(n_splits), _ptr(workspace), int(workspace_bytes),
                              _stream(stream))
    if rc != FA_OK:
        raise FaError(rc, fa_strerror(rc))


def fa_fwd_splitkv_noalloc(q, k, v, o, lse, B: int, H: int, N: int, d: int, causal: bool, scale: float,
                           n_splits: int = 0, stream=None) -> None:
    """Split-KV forward for callers that cannot allocate device memory when they
    run attention: its partial states go to a static 32 MiB array inside the
    library, shared by every call.  Calls that may overlap on the GPU must be
    serialised by the caller; the first call on a device should come before any
    stream capture.  Raises FaError (FA_ERR_SCRATCH_LIMIT when the problem does
    not fit)."""
    rc = lib().fa_fwd_splitkv_noalloc(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), int(B), int(H), int(N), int(d),
                                      1 if causal else 0, float(scale), int(n_splits), _stream(stream))
    if rc != FA_OK:
        raise FaError(rc, fa_strerror(rc))


def fa_splitkv_workspace_bytes(B: int, H: int, N: int, d: int, n_splits: int) -> int:
    return int(lib().fa_splitkv_workspace_bytes(int(B), int(H), int(N), int(d), int(n_splits)))


def fa_splitkv_auto_splits(B: int, H: int, N: int, d: int, causal: bool) -> int:
    return int(lib().fa_splitkv_auto_splits(int(B), int(H), int(N), int(d), 1 if causal else 0))


def fa_fwd_host(q, k, v, o, lse, B: int, H: int, N: int, d: int, causal: bool, scale: float, heads_per_chunk: int,
                workspace, workspace_bytes: int, stream=None) -> None:
    """Enqueue the forward on host tensors (q, k, v, o, lse on the CPU, pinned for
    overlap), streamed through a device workspace; raises FaError on a nonzero C return code."""
    rc = lib().fa_fwd_host(_host_ptr(q), _host_ptr(k), _host_ptr(v), _host_ptr(o), _host_ptr(lse), int(B), int(H),
                           int(N), int(d), 1 if causal else 0, float(scale), int(heads_per_chunk), _ptr(workspace),
                           int(workspace_bytes), _stream(stream))
    if rc != FA_OK:
        raise FaError(rc, fa_strerror(rc))


def fa_fwd_host_workspace_bytes(B: int, H: int, N: int, d: int, heads_per_chunk: int = 0) -> int:
    return int(lib().fa_fwd_host_workspace_bytes(int(B), int(H), int(N), int(d), int(heads_per_chunk)))


def attention_host(q, k, v, causal: bool = False, scale: float | None = None, heads_per_chunk: int = 0,
                   workspace=None, out=None, stream=None):
    """Forward on CPU bf16 tensors [B, H, N, d]: returns CPU (o, lse), pinned.
    The call is asynchronous on `stream`; synchronise before reading the outputs.
    Allocates the device workspace with torch when none is given."""
    import torch

    if q.dtype != torch.bfloat16 or k.dtype != torch.bfloat16 or v.dtype != torch.bfloat16:
        raise ValueError("q, k and v must be bfloat16")
    if q.dim() != 4 or q.shape != k.shape or q.shape != v.shape:
        raise ValueError("q, k and v must share one [B, H, N, d] shape")
    B, H, N, d = q.shape
    need = fa_fwd_host_workspace_bytes(B, H, N, d, heads_per_chunk)
    if workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device="cuda")
    if out is None:
        out = (torch.empty(q.shape, dtype=torch.bfloat16, pin_memory=True),
               torch.empty((B, H, N), dtype=torch.float32, pin_memory=True))
    o, lse = out
    fa_fwd_host(q, k, v, o, lse, B, H, N, d, causal, (1.0 / math.sqrt(d)) if scale is None else scale,
                heads_per_chunk, workspace, workspace.numel() * workspace.element_size(), stream)
    return o, lse


def attention_splitkv(q, k, v, causal: bool = False, scale: float | None = None, n_splits: int = 0, workspace=None,
                      stream=None):
    """Split-KV forward; allocates the workspace with torch when none is given."""
    import torch

    B, H, N, d = q.shape
    if n_splits == 0:
        n_splits = fa_splitkv_auto_splits(B, H, N, d, causal)
    need = fa_splitkv_workspace_bytes(B, H, N, d, n_splits)
    if workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    o = torch.empty_like(q)
    lse = torch.empty((B, H, N), dtype=torch.float32, device=q.device)
    nbytes = workspace.numel() * workspace.element_size() if hasattr(workspace, "numel") else need
    fa_fwd_splitkv(q, k, v, o, lse, B, H, N, d, causal, (1.0 / math.sqrt(d)) if scale is None else scale, n_splits,
                   workspace, nbytes, stream)
    return o, lse


def fa_softmax_rows(x, y, lse, M: int, N: int, stream=None) -> None:
    """Enqueue the row softmax; raises FaError on a nonzero C return code."""
    rc = lib().fa_softmax_rows(_ptr(x), _ptr(y), _ptr(lse), int(M), int(N), _stream(stream))
    if rc != FA_OK:
        raise FaError(rc, fa_strerror(rc))


def softmax(x, stream=None, out=None, with_lse: bool = True):
    """x: CUDA fp32 [..., N].  Returns (y, lse) with lse None unless with_lse."""
    import torch

    if x.dtype != torch.float32:
        raise ValueError("x must be float32")
    N = x.shape[-1]
    M = x.numel() // N if N else 0
    y = torch.empty_like(x) if out is None else out
    lse = torch.empty(x.shape[:-1], dtype=torch.float32, device=x.device) if with_lse else None
    fa_softmax_rows(x, y, lse, M, N, stream)
    return y, lse


def fa_bwd(q, k, v, o, dout, lse, dq, dk, dv, B: int, H: int, N: int, d: int, causal: bool, scale: float, workspace,
           workspace_bytes: int, stream=None) -> None:
    """Enqueue the backward pass; raises FaError on a nonzero C return code."""
    rc = lib().fa_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(dout), _ptr(lse), _ptr(dq), _ptr(dk), _ptr(dv),
                      int(B), int(H), int(N), int(d), 1 if causal else 0, float(scale), _ptr(workspace),
                      int(workspace_bytes), _stream(stream))
    if rc != FA_OK:
        raise FaError(rc, fa_strerror(rc))


def fa_bwd_workspace_bytes(B: int, H: int, N: int, d: int) -> int:
    return int(lib().fa_bwd_workspace_bytes(int(B), int(H), int(N), int(d)))


def attention_backward(q, k, v, o, lse, dout, causal: bool = False, scale: float | None = None, stream=None):
    """Gradients (dq, dk, dv), bf16 like q, for the forward outputs o, lse and the gradient dout."""
    import torch

    B, H, N, d = q.shape
    ws = torch.empty(fa_bwd_workspace_bytes(B, H, N, d), dtype=torch.uint8, device=q.device)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    fa_bwd(q, k, v, o, dout, lse, dq, dk, dv, B, H, N, d, causal, (1.0 / math.sqrt(d)) if scale is None else scale,
           ws, ws.numel(), stream)
    return dq, dk, dv


def fa_get_device_status() -> int:
    st = ctypes.c_uint(0)
    rc = lib().fa_get_device_status(ctypes.byref(st))
    if rc != FA_OK:
        raise FaError(rc, fa_strerror(rc))
    return st.value


def fa_clear_device_status() -> None:
    rc = lib().fa_clear_device_status()
    if rc != FA_OK:
        raise FaError(rc, fa_strerror(rc))


def fa_set_watchdog_ns(ns: int) -> int:
    return int(lib().fa_set_watchdog_ns(int(ns)))


def fa_watchdog_selftest(ns: int, stream=None) -> int:
    st = ctypes.c_uint(0)
    rc = lib().fa_watchdog_selftest(int(ns), _stream(stream), ctypes.byref(st))
    if rc != FA_OK:
        raise FaError(rc, fa_strerror(rc))
    return st.value


def fa_get_last_error() -> int:
    """The device-side timeout flag: 0, the status word (> 0), or a negative FA code."""
    return int(lib().fa_get_last_error())


def fa_watchdog_selftest_fwd(ns: int, q, k, v, o, lse, N: int, d: int, stream=None) -> int:
    """fa_fwd on one tile with its S products withheld: the watchdog must end the
    softmax's wait; returns the device status word."""
    st = ctypes.c_uint(0)
    rc = lib().fa_watchdog_selftest_fwd(int(ns), _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), int(N), int(d),
                                        _stream(stream), ctypes.byref(st))
    if rc != FA_OK:
        raise FaError(rc, fa_strerror(rc))
    return st.value


def fa_kernel_resources(d: int, kernel: int = FA_KERNEL_FWD) -> dict:
    """Registers, shared memory, CTAs per SM and TMEM columns of one kernel, as the runtime reports them."""
    r = KernelResources()
    rc = lib().fa_kernel_resources(int(d), int(kernel), ctypes.byref(r))
    if rc != FA_OK:
        raise FaError(rc, fa_strerror(rc))
    return {name: getattr(r, name) for name, _ in KernelResources._fields_}


def fa_set_fwd_pairing(mode: int) -> int:
    """Choose the forward kernel: one query tile per CTA, or units of two tiles (CTA pairs at d = 128,
    two tiles per CTA at d = 64); FA_PAIR_AUTO / FA_PAIR_OFF / FA_PAIR_ON.  Returns the previous mode."""
    rc = int(lib().fa_set_fwd_pairing(int(mode)))
    if rc < 0:
        raise FaError(rc, fa_strerror(rc))
    return rc


def fa_fwd_kernel_for(B: int, H: int, N: int, d: int, causal: bool) -> int:
    """FA_KERNEL_FWD, FA_KERNEL_FWD_PAIR or FA_KERNEL_FWD_TWO: the kernel fa_fwd launches for these sizes."""
    rc = int(lib().fa_fwd_kernel_for(int(B), int(H), int(N), int(d), 1 if causal else 0))
    if rc < 0:
        raise FaError(rc, fa_strerror(rc))
    return rc


def fa_version() -> int:
    return int(lib().fa_version())
