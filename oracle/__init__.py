"""fp64 CPU oracle for the fused attention forward -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The CUDA library and its Python binding
never import, link or execute anything here, and this package imports nothing
from them: the two sides share only the seeded input generators, which hold
none of the method's arithmetic.

The arithmetic lives in ``oracle.c`` (plain C, fp64, two-pass softmax, no
tiling).  This module only builds that file with gcc and marshals numpy
arrays into it through ctypes.  Inputs are numpy arrays holding either bf16
bit patterns (``uint16``) or ``float64`` values; outputs are ``float64``.

The definition it implements is the one stated in
"b200-flash-attention4-planner", section E step 1 (math semantics) and
section A1 (the streamed result equals O / row_sum, i.e. masked softmax
attention); the readings of open points (layout, GQA mapping, bottom-right
causal alignment, empty rows, LSE units) are spelled out in ``oracle.c``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from concurrent.futures import ThreadPoolExecutor

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_libs = {}


def build(force: bool = False) -> str:
    """Compile oracle.c into liboracle.so with gcc (no fast-math)."""
    up_to_date = (os.path.exists(_LIB)
                  and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC))
    if force or not up_to_date:
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-std=c99", "-fPIC", "-shared",
                               "-fno-fast-math", "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def _load(lib_path=None):
    """Load liboracle.so (built on first use), or another build of oracle.c."""
    with _lock:
        key = lib_path or _LIB
        if key not in _libs:
            if lib_path is None:
                build()
            lib = ctypes.CDLL(key)
            i64, dbl, vp = ctypes.c_int64, ctypes.c_double, ctypes.c_void_p
            for name in ("oracle_attention_fwd_bf16", "oracle_attention_fwd_f64"):
                fn = getattr(lib, name)
                fn.restype = ctypes.c_int
                fn.argtypes = [vp, vp, vp, i64, i64, i64, i64, i64, i64, vp,
                               dbl, ctypes.c_int, vp, i64, vp, vp]
            ex = lib.oracle_attention_fwd_ex
            ex.restype = ctypes.c_int
            ex.argtypes = [vp, vp, vp, ctypes.c_int, i64, i64, i64, i64, i64, i64, vp,
                           dbl, ctypes.c_int, i64, vp, vp, i64, vp, vp]
            _libs[key] = lib
    return _libs[key]


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def attention_fwd(q, k, v, *, scale, causal=False, seqlens_k=None, rows=None,
                  threads=1, lib_path=None, window=0, sinks=None):
    """Masked softmax attention with per-row LSE, in fp64.

    q: [B, Hq, Sq, d]; k, v: [B, Hkv, Sk, d].  All three are either ``uint16``
    (bf16 bit patterns) or ``float64``.  ``seqlens_k``: optional int sequence of
    length B (valid key count per batch entry).  ``rows``: optional flattened
    row indices ``(b*Hq + h)*Sq + i``; default all rows.

    Returns ``(o, lse)``: with ``rows`` given, o is [n_rows, d] and lse
    [n_rows]; otherwise o is [B, Hq, Sq, d] and lse [B, Hq, Sq].
    ``threads`` > 1 splits the rows over that many concurrent calls of the
    same single-threaded C routine (each call computes disjoint rows).
    ``lib_path`` loads a different build of ``oracle.c`` (the oracle's own
    mutation test uses it to check that its pins catch planted mistakes).
    ``window`` > 0 keeps, for row i, only keys j > i + (L - Sq) - window;
    ``sinks``: optional Hq sink logits (units of the scaled score) that join
    each row's softmax normaliser without a value (see oracle.c).
    """
    lib = _load(lib_path)
    q = np.ascontiguousarray(q)
    k = np.ascontiguousarray(k)
    v = np.ascontiguousarray(v)
    if not (q.dtype == k.dtype == v.dtype):
        raise TypeError("q, k, v must share one dtype")
    if q.dtype == np.uint16:
        fn, kind = lib.oracle_attention_fwd_bf16, 0
    elif q.dtype == np.float64:
        fn, kind = lib.oracle_attention_fwd_f64, 1
    else:
        raise TypeError(f"unsupported dtype {q.dtype}")
    B, Hq, Sq, d = q.shape
    Bk, Hkv, Sk, dk = k.shape
    if v.shape != k.shape or Bk != B or dk != d:
        raise ValueError("shape mismatch")
    sl = None
    if seqlens_k is not None:
        sl = np.ascontiguousarray(np.asarray(seqlens_k, dtype=np.int32))
        if sl.shape != (B,):
            raise ValueError("seqlens_k must have B entries")
    sk_arr = None
    if sinks is not None:
        sk_arr = np.ascontiguousarray(np.asarray(sinks, dtype=np.float64))
        if sk_arr.shape != (q.shape[1],):
            raise ValueError("sinks must have Hq entries")
    extended = int(window) > 0 or sk_arr is not None
    full = rows is None
    if full:
        rows = np.arange(B * Hq * Sq, dtype=np.int64)
    rows = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
    n = rows.shape[0]
    o = np.zeros((n, d), dtype=np.float64)
    lse = np.zeros((n,), dtype=np.float64)

    def run(lo, hi):
        if hi <= lo:
            return 0
        r = rows[lo:hi]
        o_part = o[lo:hi]
        l_part = lse[lo:hi]
        if extended:
            return lib.oracle_attention_fwd_ex(
                _ptr(q), _ptr(k), _ptr(v), kind, B, Hq, Hkv, Sq, Sk, d, _ptr(sl),
                float(scale), int(bool(causal)), int(window), _ptr(sk_arr), _ptr(r),
                hi - lo, _ptr(o_part), _ptr(l_part))
        return fn(_ptr(q), _ptr(k), _ptr(v), B, Hq, Hkv, Sq, Sk, d, _ptr(sl),
                  float(scale), int(bool(causal)), _ptr(r), hi - lo,
                  _ptr(o_part), _ptr(l_part))

    threads = max(1, min(int(threads), n))
    if threads == 1:
        rc = [run(0, n)]
    else:
        bounds = np.linspace(0, n, threads + 1).astype(np.int64)
        with ThreadPoolExecutor(max_workers=threads) as ex:
            rc = list(ex.map(lambda t: run(int(bounds[t]), int(bounds[t + 1])),
                             range(threads)))
    if any(c != 0 for c in rc):
        raise RuntimeError(f"oracle returned {rc}")
    if full:
        return o.reshape(B, Hq, Sq, d), lse.reshape(B, Hq, Sq)
    return o, lse
