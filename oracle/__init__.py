"""Double-precision CPU oracle for softmax attention -- TEST INFRASTRUCTURE.

Only the test-suite, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product path (the CUDA library and
its Python binding) never imports, links or calls it, and it imports nothing
from the product path.

The arithmetic lives in ``oracle.c`` (plain C, IEEE double); this module only
builds it with gcc on first use and marshals numpy arrays through ctypes.

Inputs are bf16 tensors passed as their uint16 bit patterns (numpy ``uint16``
arrays, layout ``[B][H][N][d]``), so the oracle sees exactly the rounded
values the GPU sees.  Query rows are named by their flat index
``(b*H + h)*N + i``.

Every function below cites the passage it follows:

* ``softmax_three_pass`` -- safe softmax in three passes (infra-guide page
  "5.2 CUDA Online Softmax", section 1.1).
* ``softmax_online`` -- the online normaliser recurrence (same page, sections
  2.1-2.2); ``online_merge`` -- the associative (m, d) merge (section 4.1).
* ``attention_three_pass`` -- softmax(Q K^T * scale) V one score row at a
  time, max / exp-sum / normalise ("LLM kernels 3: attention and online
  softmax", section "Two paths, one head, one reference").
* ``attention_online`` -- key tiles with running (m, l, O), each rescaled by
  exp(m_old - m_new), divided by l once at the end ("Online softmax, and the
  register that can't move", section "Online softmax").
* ``row_online_state`` / ``state_merge`` -- partial (m, l, acc) over a key
  range and their associative merge ("LLM kernels 3", Solution: the
  combining rule is associative).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

MUT_NONE = 0
MUT_NO_RESCALE = 1
MUT_NORMALISE_TILE = 2
MUT_SUM_BEFORE_MAX = 3


def build(force: bool = False) -> str:
    """Compile oracle.c into liboracle.so (gcc, -O2, IEEE double, pthreads)."""
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread", "-fno-fast-math",
               "-ffp-contract=off", "-o", tmp, _SRC, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            P = ctypes.c_void_p
            I64 = ctypes.c_int64
            D = ctypes.c_double
            lib.oracle_attention_three_pass.argtypes = [P, P, P, I64, I64, I64, I64, ctypes.c_int, D, P, I64, P, P,
                                                        ctypes.c_int]
            lib.oracle_attention_three_pass.restype = ctypes.c_int
            lib.oracle_attention_online.argtypes = [P, P, P, I64, I64, I64, I64, ctypes.c_int, D, I64, ctypes.c_int,
                                                    P, I64, P, P, ctypes.c_int]
            lib.oracle_attention_online.restype = ctypes.c_int
            lib.oracle_attention_masked.argtypes = [P, P, P, I64, I64, I64, I64, D, I64, I64, P, P, I64, P, P,
                                                    ctypes.c_int]
            lib.oracle_attention_masked.restype = ctypes.c_int
            lib.oracle_attention_backward.argtypes = [P, P, P, P, P, P, I64, I64, I64, I64, ctypes.c_int, D, P, I64,
                                                      P, I64, P, P, P, P, P, P, ctypes.c_int]
            lib.oracle_attention_backward.restype = ctypes.c_int
            lib.oracle_softmax_three_pass.argtypes = [P, I64, P]
            lib.oracle_softmax_three_pass.restype = None
            lib.oracle_softmax_online.argtypes = [P, I64, P, P, P]
            lib.oracle_softmax_online.restype = None
            lib.oracle_online_merge.argtypes = [D, D, D, D, P, P]
            lib.oracle_online_merge.restype = None
            lib.oracle_row_online_state.argtypes = [P, P, P, I64, I64, I64, I64, I64, D, ctypes.c_int, P, P, P]
            lib.oracle_row_online_state.restype = None
            lib.oracle_state_merge.argtypes = [D, D, P, D, D, P, I64, P, P, P]
            lib.oracle_state_merge.restype = None
            _lib = lib
    return _lib


def _ptr(a: np.ndarray) -> int:
    return a.ctypes.data


def _bits(t) -> np.ndarray:
    """Accept a numpy uint16 array of bf16 bits, or a torch bf16 tensor on CPU."""
    if isinstance(t, np.ndarray):
        assert t.dtype == np.uint16, "bf16 inputs are passed as uint16 bit patterns"
        return np.ascontiguousarray(t)
    import torch  # only to read the bits of a CPU tensor
    assert t.dtype == torch.bfloat16 and t.device.type == "cpu"
    return np.ascontiguousarray(t.contiguous().view(torch.int16).numpy().view(np.uint16))


def _rows_array(rows, total: int) -> np.ndarray:
    if rows is None:
        rows = np.arange(total, dtype=np.int64)
    return np.ascontiguousarray(np.asarray(rows, dtype=np.int64))


def attention_three_pass(q, k, v, causal: bool, scale: float, rows=None, n_threads: int = 0,
                         return_threads: bool = False):
    """O (n_rows, d) float64 and LSE (n_rows,) for the given flat query rows.

    With ``return_threads`` the number of host threads used is returned too.
    """
    q, k, v = _bits(q), _bits(k), _bits(v)
    B, H, N, d = q.shape
    r = _rows_array(rows, B * H * N)
    o = np.zeros((len(r), d), dtype=np.float64)
    lse = np.zeros(len(r), dtype=np.float64)
    used = _load().oracle_attention_three_pass(_ptr(q), _ptr(k), _ptr(v), B, H, N, d, int(bool(causal)),
                                               float(scale), _ptr(r), len(r), _ptr(o), _ptr(lse), int(n_threads))
    if used < 0:
        raise ValueError(f"oracle rejected the arguments (code {used})")
    return (o, lse, used) if return_threads else (o, lse)


def attention_masked(q, k, v, scale: float, window_left: int = -1, window_right: int = -1, doc_ids=None, rows=None,
                     n_threads: int = 0):
    """Three-pass attention where key j is visible to query i iff
    (window_left < 0 or j >= i - window_left) and (window_right < 0 or
    j <= i + window_right) and (doc_ids is None or doc_ids[b, i] == doc_ids[b, j]).
    doc_ids: int32 [B, N] or None.  Returns O (n_rows, d) float64 and LSE (n_rows,)."""
    q, k, v = _bits(q), _bits(k), _bits(v)
    B, H, N, d = q.shape
    r = _rows_array(rows, B * H * N)
    doc = None
    if doc_ids is not None:
        doc = np.ascontiguousarray(np.asarray(doc_ids), dtype=np.int32)
        if doc.shape != (B, N):
            raise ValueError("doc_ids must be [B, N]")
    o = np.zeros((len(r), d), dtype=np.float64)
    lse = np.zeros(len(r), dtype=np.float64)
    used = _load().oracle_attention_masked(_ptr(q), _ptr(k), _ptr(v), B, H, N, d, float(scale), int(window_left),
                                           int(window_right), _ptr(doc) if doc is not None else None, _ptr(r), len(r),
                                           _ptr(o), _ptr(lse), int(n_threads))
    if used < 0:
        raise ValueError(f"oracle rejected the arguments (code {used})")
    return o, lse


def attention_backward(q, k, v, o, dout, lse, causal: bool, scale: float, q_rows=None, k_rows=None,
                       n_threads: int = 0):
    """Gradients of L = sum(O * dO): dQ for the flat query rows q_rows, dK and dV
    for the flat key rows k_rows (None = every row).  q, k, v: bf16 tensors
    [B, H, N, d]; o, dout: the values the GPU sees, any float type, [B, H, N, d];
    lse: natural-log statistic [B, H, N].  Returns a dict with dq, dk, dv and
    their magnitudes mag_dq, mag_dk, mag_dv (sums of |term|), all float64."""
    qb, kb, vb = _bits(q), _bits(k), _bits(v)
    B, H, N, d = qb.shape
    def f64(t, shape):  # torch tensors of any float type, or numpy arrays, widened exactly
        a = t.detach().cpu().double().numpy() if hasattr(t, "detach") else np.asarray(t, dtype=np.float64)
        return np.ascontiguousarray(a, dtype=np.float64).reshape(shape)

    od, dod, ld = f64(o, (B, H, N, d)), f64(dout, (B, H, N, d)), f64(lse, (B, H, N))
    qr = _rows_array(q_rows, B * H * N)
    kr = _rows_array(k_rows, B * H * N)
    out = {n: np.zeros((len(qr), d)) for n in ("dq", "mag_dq")}
    out.update({n: np.zeros((len(kr), d)) for n in ("dk", "dv", "mag_dk", "mag_dv")})
    used = _load().oracle_attention_backward(
        _ptr(qb), _ptr(kb), _ptr(vb), _ptr(od), _ptr(dod), _ptr(ld), B, H, N, d, int(bool(causal)), float(scale),
        _ptr(qr), len(qr), _ptr(kr), len(kr), _ptr(out["dq"]), _ptr(out["dk"]), _ptr(out["dv"]),
        _ptr(out["mag_dq"]), _ptr(out["mag_dk"]), _ptr(out["mag_dv"]), int(n_threads))
    if used < 0:
        raise ValueError(f"oracle rejected the arguments (code {used})")
    return out


def attention_online(q, k, v, causal: bool, scale: float, tile: int = 128, rows=None, mutation: int = MUT_NONE,
                     n_threads: int = 0):
    """Tiled online route; ``tile=1`` is the scalar recurrence."""
    q, k, v = _bits(q), _bits(k), _bits(v)
    B, H, N, d = q.shape
    r = _rows_array(rows, B * H * N)
    o = np.zeros((len(r), d), dtype=np.float64)
    lse = np.zeros(len(r), dtype=np.float64)
    rc = _load().oracle_attention_online(_ptr(q), _ptr(k), _ptr(v), B, H, N, d, int(bool(causal)), float(scale),
                                         int(tile), int(mutation), _ptr(r), len(r), _ptr(o), _ptr(lse), int(n_threads))
    if rc < 0:
        raise ValueError(f"oracle rejected the arguments (code {rc})")
    return o, lse


def softmax_three_pass(x) -> np.ndarray:
    x = np.ascontiguousarray(x, dtype=np.float64)
    y = np.empty_like(x)
    _load().oracle_softmax_three_pass(_ptr(x), len(x), _ptr(y))
    return y


def softmax_online(x):
    """Returns (y, m, d): the normalised row and the final (max, exp-sum) state."""
    x = np.ascontiguousarray(x, dtype=np.float64)
    y = np.empty_like(x)
    m = ctypes.c_double()
    dd = ctypes.c_double()
    _load().oracle_softmax_online(_ptr(x), len(x), _ptr(y), ctypes.addressof(m), ctypes.addressof(dd))
    return y, m.value, dd.value


def online_merge(m1: float, d1: float, m2: float, d2: float):
    m = ctypes.c_double()
    dd = ctypes.c_double()
    _load().oracle_online_merge(float(m1), float(d1), float(m2), float(d2), ctypes.addressof(m), ctypes.addressof(dd))
    return m.value, dd.value


def row_online_state(q, k, v, flat_row: int, j0: int, j1: int, causal: bool, scale: float, tile: int = 128,
                     mutation: int = MUT_NONE):
    """Partial state (m, l, acc[d]) of one query row over keys [j0, j1)."""
    q, k, v = _bits(q), _bits(k), _bits(v)
    B, H, N, d = q.shape
    bh, i = divmod(int(flat_row), N)
    jvis = min(i + 1, N) if causal else N
    qf = q.reshape(-1, d)
    kh = np.ascontiguousarray(k.reshape(B * H, N, d)[bh])
    vh = np.ascontiguousarray(v.reshape(B * H, N, d)[bh])
    qrow = np.ascontiguousarray(qf[int(flat_row)])
    acc = np.zeros(d, dtype=np.float64)
    m = ctypes.c_double()
    l = ctypes.c_double()
    _load().oracle_row_online_state(_ptr(qrow), _ptr(kh), _ptr(vh), d, int(j0), int(j1), int(jvis), int(tile),
                                    float(scale), int(mutation), ctypes.addressof(m), ctypes.addressof(l), _ptr(acc))
    return m.value, l.value, acc


def state_merge(s1, s2):
    """Merge two (m, l, acc) partial states."""
    m1, l1, a1 = s1
    m2, l2, a2 = s2
    a1 = np.ascontiguousarray(a1, dtype=np.float64)
    a2 = np.ascontiguousarray(a2, dtype=np.float64)
    acc = np.zeros_like(a1)
    m = ctypes.c_double()
    l = ctypes.c_double()
    _load().oracle_state_merge(float(m1), float(l1), _ptr(a1), float(m2), float(l2), _ptr(a2), len(a1),
                               ctypes.addressof(m), ctypes.addressof(l), _ptr(acc))
    return m.value, l.value, acc
