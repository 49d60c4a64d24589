"""fp64 CPU attention oracle -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product path (the CUDA library and
its Python binding) never calls it and shares no code with it.

The arithmetic lives in ``attention_oracle.c`` (plain row-streamed loops in
double precision, one attention head per call, threaded over rows or columns).
This module only marshals numpy arrays to it.  ``tiled.py`` restates the pages'
tiled online-softmax algorithm in fp64 so that its exactness can be checked
against the plain definition.

Definitions and citations are in the header of ``attention_oracle.c``.
Every function here is pinned by tests/test_oracle_pins.py to closed forms,
invariants, finite differences and an independent library routine.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "attention_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

TILE = 128  # tile edge of the block mask ("BLOCK_SIZE_Q = BLOCK_SIZE_K = 128" in the pages' listing)


def build(force: bool = False) -> str:
    """Compile attention_oracle.c into liboracle.so with gcc (plain C11, -O2)."""
    if not force and os.path.exists(_LIB_PATH) and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-std=c11", "-O2", "-fPIC", "-shared", "-pthread", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def bind(lib):
    """Declare the C signatures on a loaded oracle library and return it."""
    f64p = ctypes.POINTER(ctypes.c_double)
    u8p = ctypes.POINTER(ctypes.c_uint8)
    i32p = ctypes.POINTER(ctypes.c_int32)
    i = ctypes.c_int
    lib.oracle_rows.argtypes = [f64p, f64p, f64p, f64p, i, i, ctypes.c_double, i, i, u8p, i,
                                i32p, i, f64p, f64p, f64p, f64p, f64p, f64p, i]
    lib.oracle_rows.restype = i
    lib.oracle_cols.argtypes = [f64p, f64p, f64p, f64p, i, i, ctypes.c_double, i, i, u8p, i,
                                f64p, f64p, f64p, i32p, i, f64p, f64p, i]
    lib.oracle_cols.restype = i
    lib.oracle_default_threads.argtypes = []
    lib.oracle_default_threads.restype = i
    return lib


def _load():
    global _lib
    with _lock:
        if _lib is None:
            _lib = bind(ctypes.CDLL(build()))
        return _lib


def default_threads() -> int:
    return int(_load().oracle_default_threads())


def _ptr(a, ctype):
    if a is None:
        return None
    return a.ctypes.data_as(ctypes.POINTER(ctype))


def _f64(a):
    return np.ascontiguousarray(a, dtype=np.float64)


def _mask_arg(block_mask):
    if block_mask is None:
        return None
    return np.ascontiguousarray(block_mask, dtype=np.uint8)


def head_rows(q, k, v, dout, scale, *, causal=False, kv_len=None, block_mask=None,
              tile=TILE, rows=None, nthreads=0):
    """Row pass of one head ([N, d] arrays).  Returns dict o, lse, m, l, D[, dq]."""
    lib = _load()
    qh, kh, vh = _f64(q), _f64(k), _f64(v)
    dh = _f64(dout) if dout is not None else None
    n, d = qh.shape
    kl = -1 if kv_len is None else min(max(int(kv_len), 0), n)  # -1: no key padding
    rows = np.arange(n, dtype=np.int32) if rows is None else np.ascontiguousarray(rows, dtype=np.int32)
    nr = rows.shape[0]
    o = np.empty((nr, d), np.float64)
    lse = np.empty(nr, np.float64)
    m = np.empty(nr, np.float64)
    l = np.empty(nr, np.float64)
    D = np.empty(nr, np.float64)
    dq = np.empty((nr, d), np.float64) if dh is not None else None
    bm = _mask_arg(block_mask)
    f64 = ctypes.c_double
    rc = lib.oracle_rows(_ptr(qh, f64), _ptr(kh, f64), _ptr(vh, f64), _ptr(dh, f64), n, d, float(scale),
                         int(bool(causal)), kl, _ptr(bm, ctypes.c_uint8), int(tile),
                         _ptr(rows, ctypes.c_int32), nr, _ptr(o, f64), _ptr(lse, f64), _ptr(m, f64),
                         _ptr(l, f64), _ptr(D, f64), _ptr(dq, f64), int(nthreads))
    if rc != 0:
        raise ValueError("oracle_rows rejected its arguments")
    out = {"o": o, "lse": lse, "m": m, "l": l, "D": D}
    if dq is not None:
        out["dq"] = dq
    return out


def head_cols(q, k, v, dout, scale, m, l, D, *, causal=False, kv_len=None, block_mask=None,
              tile=TILE, cols=None, nthreads=0):
    """Column pass of one head: dK, dV for keys `cols` given full-length row statistics."""
    lib = _load()
    qh, kh, vh, dh = _f64(q), _f64(k), _f64(v), _f64(dout)
    n, d = qh.shape
    kl = -1 if kv_len is None else min(max(int(kv_len), 0), n)  # -1: no key padding
    cols = np.arange(n, dtype=np.int32) if cols is None else np.ascontiguousarray(cols, dtype=np.int32)
    nc = cols.shape[0]
    m = np.ascontiguousarray(m, np.float64)
    l = np.ascontiguousarray(l, np.float64)
    D = np.ascontiguousarray(D, np.float64)
    dk = np.empty((nc, d), np.float64)
    dv = np.empty((nc, d), np.float64)
    bm = _mask_arg(block_mask)
    f64 = ctypes.c_double
    rc = lib.oracle_cols(_ptr(qh, f64), _ptr(kh, f64), _ptr(vh, f64), _ptr(dh, f64), n, d, float(scale),
                         int(bool(causal)), kl, _ptr(bm, ctypes.c_uint8), int(tile),
                         _ptr(m, f64), _ptr(l, f64), _ptr(D, f64), _ptr(cols, ctypes.c_int32), nc,
                         _ptr(dk, f64), _ptr(dv, f64), int(nthreads))
    if rc != 0:
        raise ValueError("oracle_cols rejected its arguments")
    return {"dk": dk, "dv": dv}


def attention_forward(q, k, v, scale, *, causal=False, kv_len=None, block_mask=None, tile=TILE,
                      heads=None, nthreads=0):
    """O [B,H,N,d] and LSE [B,H,N] (float64) for [B,H,N,d] inputs.

    heads: optional list of (b, h) pairs; other heads are left as NaN."""
    B, H, N, d = q.shape
    o = np.full((B, H, N, d), np.nan)
    lse = np.full((B, H, N), np.nan)
    for b, h in (heads if heads is not None else [(b, h) for b in range(B) for h in range(H)]):
        kl = None if kv_len is None else int(kv_len[b])
        r = head_rows(q[b, h], k[b, h], v[b, h], None, scale, causal=causal, kv_len=kl,
                      block_mask=block_mask, tile=tile, nthreads=nthreads)
        o[b, h], lse[b, h] = r["o"], r["lse"]
    return o, lse


def attention_backward(q, k, v, dout, scale, *, causal=False, kv_len=None, block_mask=None, tile=TILE,
                       heads=None, nthreads=0):
    """Full forward + backward.  Returns dict of float64 arrays o, lse, dq, dk, dv."""
    B, H, N, d = q.shape
    out = {name: np.full((B, H, N, d), np.nan) for name in ("o", "dq", "dk", "dv")}
    out["lse"] = np.full((B, H, N), np.nan)
    for b, h in (heads if heads is not None else [(b, h) for b in range(B) for h in range(H)]):
        kl = None if kv_len is None else int(kv_len[b])
        kw = dict(causal=causal, kv_len=kl, block_mask=block_mask, tile=tile, nthreads=nthreads)
        r = head_rows(q[b, h], k[b, h], v[b, h], dout[b, h], scale, **kw)
        c = head_cols(q[b, h], k[b, h], v[b, h], dout[b, h], scale, r["m"], r["l"], r["D"], **kw)
        out["o"][b, h], out["lse"][b, h], out["dq"][b, h] = r["o"], r["lse"], r["dq"]
        out["dk"][b, h], out["dv"][b, h] = c["dk"], c["dv"]
    return out
