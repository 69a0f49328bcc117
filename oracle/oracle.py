"""ctypes front end of the fp64 CPU oracle (``oracle.c``) -- TEST INFRASTRUCTURE ONLY.

Inputs are numpy arrays, either float64 or bfloat16 bit patterns held as uint16
(a bf16 value widens to fp64 exactly, inside ``oracle.c``).  All tensors are
``[BH, N, d]`` row-major, BH = batch * heads.  Outputs are float64.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

F64 = 0
BF16 = 1

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_HDR = os.path.join(_HERE, "oracle.h")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile ``oracle.c`` into ``liboracle.so`` next to it (plain gcc, -O2,
    no fast-math) and return the library path."""
    with _lock:
        stale = (not os.path.exists(_LIB)) or any(
            os.path.getmtime(p) > os.path.getmtime(_LIB) for p in (_SRC, _HDR)
        )
        if force or stale:
            tmp = _LIB + f".tmp{os.getpid()}"
            cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread",
                   "-fno-fast-math", _SRC, "-o", tmp, "-lm"]
            subprocess.run(cmd, check=True)
            os.replace(tmp, _LIB)
    return _LIB


def _bind(path: str):
    """Load an oracle shared library and declare its C signatures."""
    lib = ctypes.CDLL(path)
    vp, i64p, dp = ctypes.c_void_p, ctypes.POINTER(ctypes.c_int64), ctypes.POINTER(ctypes.c_double)
    L, I, D = ctypes.c_long, ctypes.c_int, ctypes.c_double
    lib.oracle_online_row.argtypes = [dp, dp, L, L, L, dp, dp, dp]
    lib.oracle_fwd.argtypes = [vp, vp, vp, I, L, L, L, D, I, i64p, L, dp, dp, I]
    lib.oracle_fwd_rows.argtypes = [vp, vp, vp, I, L, L, L, D, I, i64p, L, dp, dp, I]
    lib.oracle_fwd_blockwise.argtypes = [vp, vp, vp, I, L, L, L, D, I, L, L, dp, dp, I]
    lib.oracle_bwd.argtypes = [vp, vp, vp, vp, I, L, L, L, D, I, i64p, L, dp, dp, dp, dp, dp, I]
    lib.oracle_bwd_rows.argtypes = [vp, vp, vp, vp, I, L, L, L, D, I, i64p, L, i64p, L,
                                    dp, dp, dp, I]
    lib.oracle_default_threads.argtypes = []
    for f in ("oracle_online_row", "oracle_fwd", "oracle_fwd_rows",
              "oracle_fwd_blockwise", "oracle_bwd", "oracle_bwd_rows", "oracle_default_threads"):
        getattr(lib, f).restype = ctypes.c_int
    return lib


def _load():
    global _lib
    if _lib is None:
        _lib = _bind(build())
    return _lib


def compile_variant(src_text: str, out_path: str) -> str:
    """Compile an edited copy of ``oracle.c`` (used by the tests that plant a
    mistake in the oracle to show that a pin catches it) and return its path."""
    import shutil
    import tempfile
    with tempfile.TemporaryDirectory() as td:
        shutil.copy(_HDR, os.path.join(td, "oracle.h"))
        src = os.path.join(td, "oracle.c")
        with open(src, "w") as f:
            f.write(src_text)
        subprocess.run(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread",
                        src, "-o", out_path, "-lm"], check=True)
    return out_path


_active = threading.local()


class use_library:
    """Context manager: route this thread's oracle calls to another compiled
    oracle library (a planted-mistake variant) for the duration of a test."""

    def __init__(self, path: str):
        self.lib = _bind(path)

    def __enter__(self):
        self.prev = getattr(_active, "lib", None)
        _active.lib = self.lib
        return self

    def __exit__(self, *exc):
        _active.lib = self.prev
        return False


def _cur():
    lib = getattr(_active, "lib", None)
    return lib if lib is not None else _load()


def default_threads() -> int:
    return int(_cur().oracle_default_threads())


def _dp(a):
    if a is None:
        return None
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def _i64p(a):
    if a is None:
        return None
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_int64))


def _prep(*arrays):
    """Return (contiguous arrays, dtype code, BH, N, d) for [BH,N,d] inputs."""
    out = []
    dt = None
    for a in arrays:
        a = np.ascontiguousarray(a)
        if a.dtype == np.float64:
            code = F64
        elif a.dtype == np.uint16:
            code = BF16
        else:
            raise TypeError(f"oracle inputs must be float64 or bf16 bits (uint16), got {a.dtype}")
        if dt is None:
            dt = code
        elif dt != code:
            raise TypeError("all oracle inputs must share one dtype")
        if a.ndim != 3:
            raise ValueError("oracle inputs are [BH, N, d]")
        out.append(a)
    shape = out[0].shape
    for a in out:
        if a.shape != shape:
            raise ValueError("oracle inputs must share one shape")
    return out, dt, shape[0], shape[1], shape[2]


def _check(rc, what):
    if rc != 0:
        raise RuntimeError(f"{what} failed with code {rc}")


def online_row(scores, values=None, block: int = 1):
    """Online softmax over one row of scores in key blocks of ``block``.
    Returns (m, l, u) with u = sum_j exp(s_j - m) values[j] (None without values)."""
    s = np.ascontiguousarray(scores, dtype=np.float64).reshape(-1)
    n = s.shape[0]
    if values is None:
        v, dv, u = None, 0, None
    else:
        v = np.ascontiguousarray(values, dtype=np.float64).reshape(n, -1)
        dv = v.shape[1]
        u = np.zeros(dv, dtype=np.float64)
    m = ctypes.c_double()
    l = ctypes.c_double()
    rc = _cur().oracle_online_row(_dp(s), _dp(v), n, dv, int(block),
                                   ctypes.byref(m), ctypes.byref(l), _dp(u))
    _check(rc, "oracle_online_row")
    return m.value, l.value, u


def fwd(q, k, v, scale: float, causal: bool, heads=None, nthreads: int = 0):
    """Forward by the definition.  Returns (o [n,N,d], lse [n,N]) for the heads
    listed (all heads when ``heads`` is None)."""
    (q, k, v), dt, BH, N, d = _prep(q, k, v)
    hl = None if heads is None else np.ascontiguousarray(heads, dtype=np.int64)
    n = BH if hl is None else hl.shape[0]
    o = np.empty((n, N, d), dtype=np.float64)
    lse = np.empty((n, N), dtype=np.float64)
    rc = _cur().oracle_fwd(q.ctypes.data, k.ctypes.data, v.ctypes.data, dt, BH, N, d,
                            float(scale), int(bool(causal)), _i64p(hl), n,
                            _dp(o), _dp(lse), int(nthreads))
    _check(rc, "oracle_fwd")
    return o, lse


def fwd_rows(q, k, v, scale: float, causal: bool, rows, nthreads: int = 0):
    """Forward for selected query rows: rows is [BH, R].  Returns (o [BH,R,d], lse [BH,R])."""
    (q, k, v), dt, BH, N, d = _prep(q, k, v)
    r = np.ascontiguousarray(rows, dtype=np.int64)
    if r.ndim != 2 or r.shape[0] != BH:
        raise ValueError("rows must be [BH, R]")
    R = r.shape[1]
    o = np.empty((BH, R, d), dtype=np.float64)
    lse = np.empty((BH, R), dtype=np.float64)
    rc = _cur().oracle_fwd_rows(q.ctypes.data, k.ctypes.data, v.ctypes.data, dt, BH, N, d,
                                 float(scale), int(bool(causal)), _i64p(r), R,
                                 _dp(o), _dp(lse), int(nthreads))
    _check(rc, "oracle_fwd_rows")
    return o, lse


def fwd_blockwise(q, k, v, scale: float, causal: bool, block_q: int, block_k: int,
                  nthreads: int = 0):
    """Forward in the tiled order with the online recurrence."""
    (q, k, v), dt, BH, N, d = _prep(q, k, v)
    o = np.empty((BH, N, d), dtype=np.float64)
    lse = np.empty((BH, N), dtype=np.float64)
    rc = _cur().oracle_fwd_blockwise(q.ctypes.data, k.ctypes.data, v.ctypes.data, dt, BH, N, d,
                                      float(scale), int(bool(causal)), int(block_q), int(block_k),
                                      _dp(o), _dp(lse), int(nthreads))
    _check(rc, "oracle_fwd_blockwise")
    return o, lse


def bwd(q, k, v, dout, scale: float, causal: bool, heads=None, nthreads: int = 0):
    """Backward by the derived formulas.  Returns (dq, dk, dv, o, lse) for the heads
    listed (all heads when ``heads`` is None); o/lse are the oracle's own forward."""
    (q, k, v, dout), dt, BH, N, d = _prep(q, k, v, dout)
    hl = None if heads is None else np.ascontiguousarray(heads, dtype=np.int64)
    n = BH if hl is None else hl.shape[0]
    dq = np.empty((n, N, d), dtype=np.float64)
    dk = np.empty((n, N, d), dtype=np.float64)
    dv = np.empty((n, N, d), dtype=np.float64)
    o = np.empty((n, N, d), dtype=np.float64)
    lse = np.empty((n, N), dtype=np.float64)
    rc = _cur().oracle_bwd(q.ctypes.data, k.ctypes.data, v.ctypes.data, dout.ctypes.data, dt,
                            BH, N, d, float(scale), int(bool(causal)), _i64p(hl), n,
                            _dp(dq), _dp(dk), _dp(dv), _dp(o), _dp(lse), int(nthreads))
    _check(rc, "oracle_bwd")
    return dq, dk, dv, o, lse


def bwd_rows(q, k, v, dout, scale: float, causal: bool, qrows=None, krows=None,
             nthreads: int = 0):
    """Backward for selected rows: qrows [BH, R] query rows whose dQ rows are
    wanted, krows [BH, Rk] key rows whose dK and dV rows are wanted (either may
    be None).  Returns (dq [BH,R,d] or None, dk [BH,Rk,d] or None, dv or None)."""
    (q, k, v, dout), dt, BH, N, d = _prep(q, k, v, dout)

    def rows_of(r):
        if r is None:
            return None, 0
        r = np.ascontiguousarray(r, dtype=np.int64)
        if r.ndim != 2 or r.shape[0] != BH:
            raise ValueError("row lists must be [BH, R]")
        return r, r.shape[1]

    qr, nq = rows_of(qrows)
    kr, nk = rows_of(krows)
    dq = np.empty((BH, nq, d)) if nq else None
    dk = np.empty((BH, nk, d)) if nk else None
    dv = np.empty((BH, nk, d)) if nk else None
    rc = _cur().oracle_bwd_rows(q.ctypes.data, k.ctypes.data, v.ctypes.data, dout.ctypes.data, dt,
                                 BH, N, d, float(scale), int(bool(causal)), _i64p(qr), nq,
                                 _i64p(kr), nk, _dp(dq), _dp(dk), _dp(dv), int(nthreads))
    _check(rc, "oracle_bwd_rows")
    return dq, dk, dv
