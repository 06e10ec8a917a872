"""CPU oracle for the LFM2 gated short convolution -- TEST INFRASTRUCTURE.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package. The product library never calls it.

This module compiles ``shortconv_oracle.c`` with gcc (on first use, or when
the source is newer than the build) and exposes its functions on numpy arrays.
Storage conventions, matching the product's C ABI:

* ``"f32"`` arrays are ``np.float32``; ``"bf16"`` arrays are ``np.uint16``
  holding bf16 bit patterns; ``"f64"`` (oracle-only, no rounding) is
  ``np.float64``.
* ``bcx`` is ``[T, 3H]`` with columns ``B | C | x``; ``w`` is ``[H, K]``;
  the state pool is ``[n_slots, H, K]`` with tap ``K-1`` the newest value.

The arithmetic and its sources are described in ``shortconv_oracle.c``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "shortconv_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liboracle_shortconv.so")

DTYPES = {"f32": (0, np.float32), "bf16": (1, np.uint16), "f64": (2, np.float64)}
OK, EINVAL, EDATA = 0, 1, 4

_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle with gcc into ``oracle/_build``; return the .so path.

    ``-ffp-contract=off`` keeps every double multiply and add a separate
    rounding step, as written in the source.
    """
    os.makedirs(_BUILD_DIR, exist_ok=True)
    stale = (not os.path.exists(_LIB_PATH)) or (
        os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC))
    if force or stale:
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        cmd = ["gcc", "-std=c11", "-O2", "-ffp-contract=off", "-fno-fast-math",
               "-fPIC", "-shared", "-Wall", "-Wextra", "-o", tmp, _SRC, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            # A test may point this at a deliberately broken copy of the oracle
            # to check that the pins catch the mistake.
            lib = ctypes.CDLL(os.environ.get("SHORTCONV_ORACLE_LIB") or build())
            p, i32, i64 = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64
            lib.orc_prefill.argtypes = [i32, i32, i32, p, i64, p, p, p, i32, p, p, i32, p]
            lib.orc_decode.argtypes = [i32, i32, i32, p, i32, p, p, p, p, i32, p]
            lib.orc_verify.argtypes = [i32, i32, i32, p, i32, i32, p, p, p, p, i32, p, p]
            lib.orc_rollback.argtypes = [i32, i32, i32, i32, i32, p, p, p, p, i32]
            lib.orc_backward.argtypes = [i32, i32, i32, p, i64, p, p, p, p, p, p]
            lib.orc_backward_varlen.argtypes = [i32, i32, i32, p, i64, p, p, p, i32, p, p, p, p,
                                                p, p, p]
            for f in (lib.orc_prefill, lib.orc_decode, lib.orc_verify,
                      lib.orc_rollback, lib.orc_backward, lib.orc_backward_varlen):
                f.restype = i32
            lib.orc_double_to_bf16.argtypes = [ctypes.c_double]
            lib.orc_double_to_bf16.restype = ctypes.c_uint16
            lib.orc_bf16_to_double.argtypes = [ctypes.c_uint16]
            lib.orc_bf16_to_double.restype = ctypes.c_double
            lib.orc_round_bf16_array.argtypes = [ctypes.c_void_p, ctypes.c_void_p,
                                                 ctypes.c_int64]
            lib.orc_round_bf16_array.restype = None
            _lib = lib
    return _lib


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def _arr(a, npdt) -> np.ndarray:
    a = np.ascontiguousarray(a)
    if a.dtype != npdt:
        raise TypeError(f"expected {np.dtype(npdt)}, got {a.dtype}")
    return a


def _idx(a) -> np.ndarray:
    """int32 index array (lists and wider integer arrays are converted)."""
    a = np.asarray(a)
    if a.dtype.kind not in "iu":
        raise TypeError(f"index array must be integer, got {a.dtype}")
    out = np.ascontiguousarray(a, dtype=np.int32)
    if not np.array_equal(out, a):
        raise ValueError("index values do not fit in int32")
    return out


def _opt(a, npdt, shape, name):
    """Pointer of an optional array (None: NULL)."""
    if a is None:
        return None, None
    a = _arr(a, npdt)
    if a.shape != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}")
    return a, _ptr(a)


def _code(dtype: str):
    if dtype not in DTYPES:
        raise ValueError(f"dtype must be one of {sorted(DTYPES)}")
    return DTYPES[dtype]


def round_bf16(values) -> np.ndarray:
    """Round doubles to bf16 bit patterns (ties to even) with the oracle's routine."""
    v = np.ascontiguousarray(values, dtype=np.float64)
    out = np.empty(v.shape, dtype=np.uint16)
    _load().orc_round_bf16_array(_ptr(v), _ptr(out), v.size)
    return out.reshape(np.shape(values))


def bf16_to_f64(bits) -> np.ndarray:
    """Exact widening of bf16 bit patterns to float64."""
    b = np.asarray(bits, dtype=np.uint16)
    return (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def to_f64(dtype: str, a: np.ndarray) -> np.ndarray:
    """Exact widening of stored values of ``dtype`` to float64."""
    return bf16_to_f64(a) if dtype == "bf16" else np.asarray(a, dtype=np.float64)


def prefill(dtype, bcx, w, cu_seqlens, slot_ids, pool, y=None, bias=None):
    """Varlen prefill. ``pool`` is updated in place; returns ``(status, y)``.

    ``bias`` is an optional ``[H]`` array of ``dtype`` added to the conv output.
    """
    code, npdt = _code(dtype)
    bcx, w, pool = _arr(bcx, npdt), _arr(w, npdt), pool
    if pool.dtype != npdt or not pool.flags.c_contiguous:
        raise TypeError("pool must be a C-contiguous array of the call's dtype")
    cu = _idx(cu_seqlens)
    slots = _idx(slot_ids)
    if cu.shape != (len(slots) + 1,):
        raise ValueError("cu_seqlens must hold len(slot_ids) + 1 entries")
    T, H3 = bcx.shape
    H = H3 // 3
    K = w.shape[1]
    if y is None:
        y = np.zeros((T, H), dtype=npdt)
    bias, bp = _opt(bias, npdt, (H,), "bias")
    st = _load().orc_prefill(code, H, K, _ptr(bcx), T, _ptr(w), bp, _ptr(cu),
                             len(slots), _ptr(slots), _ptr(pool), pool.shape[0], _ptr(y))
    return st, y


def decode(dtype, bcx, w, slot_ids, pool, y=None, bias=None):
    """One token per sequence (row i of ``bcx`` for sequence i), pool in place."""
    code, npdt = _code(dtype)
    bcx, w = _arr(bcx, npdt), _arr(w, npdt)
    if pool.dtype != npdt or not pool.flags.c_contiguous:
        raise TypeError("pool must be a C-contiguous array of the call's dtype")
    slots = _idx(slot_ids)
    N, H3 = bcx.shape
    H = H3 // 3
    K = w.shape[1]
    if y is None:
        y = np.zeros((N, H), dtype=npdt)
    bias, bp = _opt(bias, npdt, (H,), "bias")
    st = _load().orc_decode(code, H, K, _ptr(bcx), N, _ptr(w), bp, _ptr(slots),
                            _ptr(pool), pool.shape[0], _ptr(y))
    return st, y


def verify(dtype, bcx, w, slot_ids, pool, D, win=None, y=None, bias=None):
    """Speculative verify over ``[N*D, 3H]`` draft rows; returns ``(status, win, y)``."""
    code, npdt = _code(dtype)
    bcx, w, pool = _arr(bcx, npdt), _arr(w, npdt), _arr(pool, npdt)
    slots = _idx(slot_ids)
    N = len(slots)
    H = bcx.shape[1] // 3
    K = w.shape[1]
    if win is None:
        win = np.zeros((N, D, H, K), dtype=npdt)
    if y is None:
        y = np.zeros((N * D, H), dtype=npdt)
    bias, bp = _opt(bias, npdt, (H,), "bias")
    st = _load().orc_verify(code, H, K, _ptr(bcx), N, D, _ptr(w), bp, _ptr(slots),
                            _ptr(pool), pool.shape[0], _ptr(win), _ptr(y))
    return st, win, y


def rollback(dtype, win, accepted, slot_ids, pool):
    """Restore each slot at its accepted length; ``pool`` in place; returns status."""
    code, npdt = _code(dtype)
    win = _arr(win, npdt)
    if pool.dtype != npdt or not pool.flags.c_contiguous:
        raise TypeError("pool must be a C-contiguous array of the call's dtype")
    acc = _idx(accepted)
    slots = _idx(slot_ids)
    N, D, H, K = win.shape
    return _load().orc_rollback(code, H, K, N, D, _ptr(win), _ptr(acc), _ptr(slots),
                                _ptr(pool), pool.shape[0])


def backward(dtype, bcx, w, dy, bias=None, with_dbias=False):
    """Single-sequence backward from a zero state; returns ``(status, dbcx, dw)``,
    or ``(status, dbcx, dw, dbias)`` when ``with_dbias``.

    ``dbcx`` has the ``[T, 3H]`` layout ``dB | dC | dx`` in ``dtype``; ``dw``
    is ``[H, K]`` float64; ``dbias`` is ``[H]`` float64.
    """
    code, npdt = _code(dtype)
    bcx, w, dy = _arr(bcx, npdt), _arr(w, npdt), _arr(dy, npdt)
    T, H3 = bcx.shape
    H = H3 // 3
    K = w.shape[1]
    dbcx = np.zeros((T, 3 * H), dtype=npdt)
    dw = np.zeros((H, K), dtype=np.float64)
    dbias = np.zeros((H,), dtype=np.float64)
    bias, bp = _opt(bias, npdt, (H,), "bias")
    st = _load().orc_backward(code, H, K, _ptr(bcx), T, _ptr(w), bp, _ptr(dy),
                              _ptr(dbcx), _ptr(dw), _ptr(dbias) if with_dbias else None)
    return (st, dbcx, dw, dbias) if with_dbias else (st, dbcx, dw)


def backward_varlen(dtype, bcx, w, cu_seqlens, dy, init=None, d_final=None, bias=None,
                    with_dbias=False):
    """Packed varlen backward with initial states; returns ``(status, dbcx, dw, d_init)``,
    or ``(status, dbcx, dw, d_init, dbias)`` when ``with_dbias``.

    ``init`` is ``[N, H, K]`` in ``dtype`` (None: zeros); ``d_final`` is
    ``[N, H, K]`` float64 (None: zeros); ``dw`` and ``d_init`` are float64.
    """
    code, npdt = _code(dtype)
    bcx, w, dy = _arr(bcx, npdt), _arr(w, npdt), _arr(dy, npdt)
    cu = _idx(cu_seqlens)
    N = len(cu) - 1
    T, H3 = bcx.shape
    H = H3 // 3
    K = w.shape[1]
    if init is not None:
        init = _arr(init, npdt)
        if init.shape != (N, H, K):
            raise ValueError("init must be [N, H, K]")
    if d_final is not None:
        d_final = _arr(d_final, np.float64)
        if d_final.shape != (N, H, K):
            raise ValueError("d_final must be [N, H, K]")
    dbcx = np.zeros((T, 3 * H), dtype=npdt)
    dw = np.zeros((H, K), dtype=np.float64)
    d_init = np.zeros((N, H, K), dtype=np.float64)
    dbias = np.zeros((H,), dtype=np.float64)
    bias, bp = _opt(bias, npdt, (H,), "bias")
    st = _load().orc_backward_varlen(
        code, H, K, _ptr(bcx), T, _ptr(w), bp, _ptr(cu), N,
        _ptr(init) if init is not None else None, _ptr(dy),
        _ptr(d_final) if d_final is not None else None, _ptr(dbcx), _ptr(dw),
        _ptr(dbias) if with_dbias else None, _ptr(d_init))
    return (st, dbcx, dw, d_init, dbias) if with_dbias else (st, dbcx, dw, d_init)

