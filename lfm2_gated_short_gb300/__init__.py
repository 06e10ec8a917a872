"""LFM2 gated short convolution (ShortConv) on GB300 (sm_103a).

A thin ctypes binding over ``libshortconv.so`` (see ``include/shortconv.h``).
Every function here only checks and marshals arguments: torch CUDA tensors
become device pointers plus sizes, the current torch stream becomes the
``cudaStream_t``, and all the work runs in the library's CUDA kernels. There
is no CPU or PyTorch fallback: if the library is not built, or a call fails,
an exception is raised.

Layouts (row-major, contiguous, one dtype per call: torch.bfloat16 or
torch.float32): ``bcx [T, 3H]`` (B | C | x), ``w [H, K]``, state pool
``[n_slots, H, K]`` (tap K-1 newest), ``y [T, H]``; index arrays are int32.
Every forward and backward call takes an optional conv ``bias [H]`` (the data
dtype; None for none), added to the conv output before the C gate.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
# SHORTCONV_LIBRARY selects another build of this library (the tests use it to
# load the bounds-checked build, _build/bounds/libshortconv.so).
LIB_PATH = os.environ.get("SHORTCONV_LIBRARY") or os.path.join(_HERE, "_build", "libshortconv.so")
DEV_OUT_OF_BOUNDS = 0x20

SC_OK, SC_EINVAL, SC_EUNSUPPORTED, SC_ECUDA, SC_EDEVICE = 0, 1, 2, 3, 4
SC_F32, SC_BF16 = 0, 1
DEV_BAD_SLOT, DEV_BAD_SEQLENS, DEV_BAD_ACCEPTED, DEV_TIMEOUT, DEV_NO_SLOT = 0x1, 0x2, 0x4, 0x8, 0x10

_lock = threading.Lock()
_lib = None


class ShortConvError(RuntimeError):
    """A library call returned a status other than SC_OK."""

    def __init__(self, fn: str, status: int, message: str):
        super().__init__(f"{fn}: {message} (status {status})")
        self.status = status


def lib() -> ctypes.CDLL:
    """The loaded C library (argument types declared). Raises if it is not built."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(
                    f"{LIB_PATH} is missing: build it with "
                    "`python -m lfm2_gated_short_gb300.build` (nvcc, sm_103a)")
            L = ctypes.CDLL(LIB_PATH)
            p, i32, i64 = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64
            L.shortconv_prefill.argtypes = [i32, i32, i32, p, i64, p, p, p, i32, p, p, i32, p, p]
            L.shortconv_prefill_tiled.argtypes = [i32, i32, i32, p, i64, p, p, p, i32, p, p,
                                                  i32, p, i32, p]
            L.shortconv_decode.argtypes = [i32, i32, i32, p, i32, p, p, p, p, i32, p, p]
            L.shortconv_verify.argtypes = [i32, i32, i32, p, i32, i32, p, p, p, p, i32, p, p,
                                           p]
            L.shortconv_rollback.argtypes = [i32, i32, i32, i32, i32, p, p, p, p, i32, p]
            L.shortconv_rollback_layers.argtypes = [i32, i32, i32, i32, i32, i32, p, p, p, p,
                                                    i32, p]
            L.shortconv_backward_workspace_bytes.argtypes = [i32, i32, i64]
            L.shortconv_backward_workspace_bytes.restype = ctypes.c_size_t
            L.shortconv_backward.argtypes = [i32, i32, i32, p, i64, p, p, p, p, p, p, p,
                                             ctypes.c_size_t, p]
            L.shortconv_backward_varlen.argtypes = [i32, i32, i32, p, i64, p, p, p, i32, p, p,
                                                    p, p, p, p, p, p, ctypes.c_size_t, p]
            L.shortconv_in_proj_workspace_bytes.argtypes = [i32, i32, i32]
            L.shortconv_in_proj_workspace_bytes.restype = ctypes.c_size_t
            L.shortconv_in_proj_prefill.argtypes = [i32, i32, i32, i32, p, i64, p, p, p, p, i32,
                                                    p, p, i32, p, p, ctypes.c_size_t, p]
            L.shortconv_out_proj.argtypes = [i32, i32, i32, p, i64, p, p, p]
            L.shortconv_in_proj_decode.argtypes = [i32, i32, i32, i32, p, i32, p, p, p, p, p,
                                                   i32, p, p]
            L.shortconv_slots_claim.argtypes = [p, i32, i32, p, i32, i32, i32, p, p]
            L.shortconv_slots_release.argtypes = [p, i32, p, i32, p]
            L.shortconv_pool_copy.argtypes = [i32, i32, i32, p, i32, p, p, i32, p]
            L.shortconv_get_error.argtypes = [p, ctypes.POINTER(ctypes.c_int)]
            L.shortconv_check_wait_limit.argtypes = [p]
            L.shortconv_bounds_checked.argtypes = []
            L.shortconv_bounds_checked.restype = i32
            L.shortconv_bounds_trim_next.argtypes = [i32, ctypes.c_uint64]
            L.shortconv_bounds_take_first_bad.argtypes = [p, ctypes.POINTER(ctypes.c_uint64)]
            L.shortconv_status_string.argtypes = [i32]
            L.shortconv_status_string.restype = ctypes.c_char_p
            for f in ("prefill", "prefill_tiled", "decode", "verify", "rollback",
                      "rollback_layers", "backward",
                      "backward_varlen", "in_proj_prefill", "in_proj_decode", "out_proj",
                      "slots_claim",
                      "slots_release", "pool_copy", "get_error", "check_wait_limit",
                      "bounds_trim_next", "bounds_take_first_bad"):
                getattr(L, "shortconv_" + f).restype = i32
            _lib = L
    return _lib


def _raise_on(fn: str, status: int) -> None:
    if status != SC_OK:
        msg = lib().shortconv_status_string(status).decode()
        raise ShortConvError(fn, status, msg)


def _dcode(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return SC_BF16
    if t.dtype == torch.float32:
        return SC_F32
    raise TypeError(f"unsupported dtype {t.dtype}: use torch.bfloat16 or torch.float32")


def _dev(t: torch.Tensor, name: str, dtype=None, shape=None) -> int:
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.device.type != "cuda":
        raise ValueError(f"{name} must be a CUDA tensor, got {t.device}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")
    return t.data_ptr()


def _stream(stream, device) -> int:
    s = stream if stream is not None else torch.cuda.current_stream(device)
    return s.cuda_stream


def _bias(bias, dt, H):
    return None if bias is None else _dev(bias, "bias", dt, (H,))


def prefill(bcx, w, cu_seqlens, slot_ids, pool, y=None, rows_per_thread=0, stream=None,
            bias=None):
    """Packed varlen prefill; updates ``pool`` in place and returns ``y [T, H]``."""
    dt = bcx.dtype
    T, H3 = bcx.shape
    H, K = w.shape
    if H3 != 3 * H:
        raise ValueError("bcx must be [T, 3H] for w [H, K]")
    N = slot_ids.shape[0]
    if y is None:
        y = torch.empty((T, H), dtype=dt, device=bcx.device)
    args = (_dcode(bcx), H, K, _dev(bcx, "bcx", dt), T, _dev(w, "w", dt), _bias(bias, dt, H),
            _dev(cu_seqlens, "cu_seqlens", torch.int32, (N + 1,)), N,
            _dev(slot_ids, "slot_ids", torch.int32, (N,)),
            _dev(pool, "pool", dt, (pool.shape[0], H, K)), pool.shape[0],
            _dev(y, "y", dt, (T, H)))
    st = _stream(stream, bcx.device)
    if rows_per_thread:
        _raise_on("shortconv_prefill_tiled",
                  lib().shortconv_prefill_tiled(*args, rows_per_thread, st))
    else:
        _raise_on("shortconv_prefill", lib().shortconv_prefill(*args, st))
    return y


def decode(bcx, w, slot_ids, pool, y=None, stream=None, bias=None):
    """One token per sequence; updates ``pool`` in place and returns ``y [N, H]``."""
    dt = bcx.dtype
    N, H3 = bcx.shape
    H, K = w.shape
    if H3 != 3 * H:
        raise ValueError("bcx must be [N, 3H] for w [H, K]")
    if y is None:
        y = torch.empty((N, H), dtype=dt, device=bcx.device)
    _raise_on("shortconv_decode", lib().shortconv_decode(
        _dcode(bcx), H, K, _dev(bcx, "bcx", dt), N, _dev(w, "w", dt), _bias(bias, dt, H),
        _dev(slot_ids, "slot_ids", torch.int32, (N,)),
        _dev(pool, "pool", dt, (pool.shape[0], H, K)), pool.shape[0],
        _dev(y, "y", dt, (N, H)), _stream(stream, bcx.device)))
    return y


def verify(bcx, w, slot_ids, pool, D, win=None, y=None, stream=None, bias=None):
    """Speculative verify of ``D`` drafts per sequence; returns ``(win, y)``. Pool is read only."""
    dt = bcx.dtype
    H, K = w.shape
    N = slot_ids.shape[0]
    if tuple(bcx.shape) != (N * D, 3 * H):
        raise ValueError(f"bcx must be [N*D, 3H] = {(N * D, 3 * H)}")
    if win is None:
        win = torch.empty((N, D, H, K), dtype=dt, device=bcx.device)
    if y is None:
        y = torch.empty((N * D, H), dtype=dt, device=bcx.device)
    _raise_on("shortconv_verify", lib().shortconv_verify(
        _dcode(bcx), H, K, _dev(bcx, "bcx", dt), N, D, _dev(w, "w", dt), _bias(bias, dt, H),
        _dev(slot_ids, "slot_ids", torch.int32, (N,)),
        _dev(pool, "pool", dt, (pool.shape[0], H, K)), pool.shape[0],
        _dev(win, "win", dt, (N, D, H, K)), _dev(y, "y", dt, (N * D, H)),
        _stream(stream, bcx.device)))
    return win, y


def rollback(win, accepted, slot_ids, pool, stream=None):
    """Commit each sequence's accepted prefix into its slot (in place on ``pool``)."""
    dt = win.dtype
    N, D, H, K = win.shape
    _raise_on("shortconv_rollback", lib().shortconv_rollback(
        _dcode(win), H, K, N, D, _dev(win, "win", dt),
        _dev(accepted, "accepted", torch.int32, (N,)),
        _dev(slot_ids, "slot_ids", torch.int32, (N,)),
        _dev(pool, "pool", dt, (pool.shape[0], H, K)), pool.shape[0],
        _stream(stream, win.device)))


def rollback_layers(win, accepted, slot_ids, pool, stream=None):
    """Roll back L layers at once: ``win [L, N, D, H, K]`` (stacked verify tapes),
    ``pool [L, n_slots, H, K]`` (stacked pools, in place)."""
    dt = win.dtype
    L, N, D, H, K = win.shape
    if pool.dim() != 4 or pool.shape[0] != L:
        raise ValueError("pool must be [L, n_slots, H, K] for win [L, N, D, H, K]")
    _raise_on("shortconv_rollback_layers", lib().shortconv_rollback_layers(
        _dcode(win), H, K, L, N, D, _dev(win, "win", dt),
        _dev(accepted, "accepted", torch.int32, (N,)),
        _dev(slot_ids, "slot_ids", torch.int32, (N,)),
        _dev(pool, "pool", dt, (L, pool.shape[1], H, K)), pool.shape[1],
        _stream(stream, win.device)))


def backward_workspace_bytes(H: int, K: int, T: int) -> int:
    return int(lib().shortconv_backward_workspace_bytes(H, K, T))


def backward(bcx, w, dy, dbcx=None, dw=None, workspace=None, stream=None, bias=None,
             with_dbias=False, dbias=None):
    """Backward from a zero state; returns ``(dbcx [T, 3H], dw [H, K] fp32)``,
    plus ``dbias [H] fp32`` when ``with_dbias``."""
    dt = bcx.dtype
    T, H3 = bcx.shape
    H, K = w.shape
    if H3 != 3 * H:
        raise ValueError("bcx must be [T, 3H] for w [H, K]")
    need = backward_workspace_bytes(H, K, T)
    if dbcx is None:
        dbcx = torch.empty_like(bcx)
    if dw is None:
        dw = torch.empty((H, K), dtype=torch.float32, device=bcx.device)
    if with_dbias and dbias is None:
        dbias = torch.empty((H,), dtype=torch.float32, device=bcx.device)
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=bcx.device)
    if workspace.dtype != torch.uint8 or workspace.numel() < need:
        raise ValueError(f"workspace must be a uint8 tensor of at least {need} bytes")
    db_p = _dev(dbias, "dbias", torch.float32, (H,)) if with_dbias else None
    _raise_on("shortconv_backward", lib().shortconv_backward(
        _dcode(bcx), H, K, _dev(bcx, "bcx", dt), T, _dev(w, "w", dt), _bias(bias, dt, H),
        _dev(dy, "dy", dt, (T, H)), _dev(dbcx, "dbcx", dt, (T, 3 * H)),
        _dev(dw, "dw", torch.float32, (H, K)), db_p, _dev(workspace, "workspace"),
        workspace.numel(), _stream(stream, bcx.device)))
    return (dbcx, dw, dbias) if with_dbias else (dbcx, dw)


def backward_varlen(bcx, w, cu_seqlens, dy, init_states=None, d_final=None, dbcx=None,
                    dw=None, d_init=None, workspace=None, want_d_init=True, stream=None,
                    bias=None, with_dbias=False, dbias=None):
    """Packed varlen backward with initial states; returns ``(dbcx, dw, d_init)``,
    plus ``dbias [H] fp32`` when ``with_dbias``.

    ``init_states`` is ``[N, H, K]`` (the data dtype; None: zeros);
    ``d_final`` is ``[N, H, K]`` float32 (None: zeros); ``d_init`` is
    ``[N, H, K]`` float32 (None when ``want_d_init`` is False).
    """
    dt = bcx.dtype
    T, H3 = bcx.shape
    H, K = w.shape
    if H3 != 3 * H:
        raise ValueError("bcx must be [T, 3H] for w [H, K]")
    N = cu_seqlens.shape[0] - 1
    need = backward_workspace_bytes(H, K, T)
    if dbcx is None:
        dbcx = torch.empty_like(bcx)
    if dw is None:
        dw = torch.empty((H, K), dtype=torch.float32, device=bcx.device)
    if want_d_init and d_init is None:
        d_init = torch.empty((N, H, K), dtype=torch.float32, device=bcx.device)
    if with_dbias and dbias is None:
        dbias = torch.empty((H,), dtype=torch.float32, device=bcx.device)
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=bcx.device)
    if workspace.dtype != torch.uint8 or workspace.numel() < need:
        raise ValueError(f"workspace must be a uint8 tensor of at least {need} bytes")
    init_p = _dev(init_states, "init_states", dt, (N, H, K)) if init_states is not None else None
    dfin_p = _dev(d_final, "d_final", torch.float32, (N, H, K)) if d_final is not None else None
    dini_p = _dev(d_init, "d_init", torch.float32, (N, H, K)) if d_init is not None else None
    db_p = _dev(dbias, "dbias", torch.float32, (H,)) if with_dbias else None
    _raise_on("shortconv_backward_varlen", lib().shortconv_backward_varlen(
        _dcode(bcx), H, K, _dev(bcx, "bcx", dt), T, _dev(w, "w", dt), _bias(bias, dt, H),
        _dev(cu_seqlens, "cu_seqlens", torch.int32, (N + 1,)), N, init_p,
        _dev(dy, "dy", dt, (T, H)), dfin_p, _dev(dbcx, "dbcx", dt, (T, 3 * H)),
        _dev(dw, "dw", torch.float32, (H, K)), db_p, dini_p, _dev(workspace, "workspace"),
        workspace.numel(), _stream(stream, bcx.device)))
    return (dbcx, dw, d_init, dbias) if with_dbias else (dbcx, dw, d_init)


def in_proj_workspace_bytes(H: int, K: int, N: int) -> int:
    return int(lib().shortconv_in_proj_workspace_bytes(H, K, N))


def in_proj_prefill(hidden, w_in, w, cu_seqlens, slot_ids, pool, y=None, bias=None,
                    workspace=None, stream=None):
    """in_proj fused with the packed varlen prefill (bf16); updates ``pool`` and
    returns ``y [T, H]``. ``hidden [T, D]``, ``w_in [3H, D]`` (rows b | c | xv)."""
    dt = torch.bfloat16
    T, D = hidden.shape
    H, K = w.shape
    N = slot_ids.shape[0]
    need = in_proj_workspace_bytes(H, K, N)
    if y is None:
        y = torch.empty((T, H), dtype=dt, device=hidden.device)
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=hidden.device)
    if workspace.dtype != torch.uint8 or workspace.numel() < need:
        raise ValueError(f"workspace must be a uint8 tensor of at least {need} bytes")
    _raise_on("shortconv_in_proj_prefill", lib().shortconv_in_proj_prefill(
        _dcode(hidden), D, H, K, _dev(hidden, "hidden", dt), T,
        _dev(w_in, "w_in", dt, (3 * H, D)), _dev(w, "w", dt), _bias(bias, dt, H),
        _dev(cu_seqlens, "cu_seqlens", torch.int32, (N + 1,)), N,
        _dev(slot_ids, "slot_ids", torch.int32, (N,)),
        _dev(pool, "pool", dt, (pool.shape[0], H, K)), pool.shape[0], _dev(y, "y", dt, (T, H)),
        _dev(workspace, "workspace"), workspace.numel(), _stream(stream, hidden.device)))
    return y


def in_proj_decode(hidden, w_in, w, slot_ids, pool, y=None, bias=None, stream=None):
    """in_proj fused with the decode of one token per sequence (bf16): row i of
    ``hidden [N, D]`` is sequence i; updates ``pool`` and returns ``y [N, H]``."""
    dt = torch.bfloat16
    N, D = hidden.shape
    H, K = w.shape
    if y is None:
        y = torch.empty((N, H), dtype=dt, device=hidden.device)
    _raise_on("shortconv_in_proj_decode", lib().shortconv_in_proj_decode(
        _dcode(hidden), D, H, K, _dev(hidden, "hidden", dt), N,
        _dev(w_in, "w_in", dt, (3 * H, D)), _dev(w, "w", dt), _bias(bias, dt, H),
        _dev(slot_ids, "slot_ids", torch.int32, (N,)),
        _dev(pool, "pool", dt, (pool.shape[0], H, K)), pool.shape[0], _dev(y, "y", dt, (N, H)),
        _stream(stream, hidden.device)))
    return y


def out_proj(y, w_out, out=None, stream=None):
    """out = y w_out^T (bf16, fp32 accumulation): ``y [T, H]``, ``w_out [D, H]``."""
    dt = torch.bfloat16
    T, H = y.shape
    D = w_out.shape[0]
    if out is None:
        out = torch.empty((T, D), dtype=dt, device=y.device)
    _raise_on("shortconv_out_proj", lib().shortconv_out_proj(
        _dcode(y), H, D, _dev(y, "y", dt), T, _dev(w_out, "w_out", dt, (D, H)),
        _dev(out, "out", dt, (T, D)), _stream(stream, y.device)))
    return out


def slot_bitmap(n_slots: int, device="cuda") -> torch.Tensor:
    """An all-free in-use bitmap for ``n_slots`` slots (int32 words, bit per slot)."""
    return torch.zeros(((n_slots + 31) // 32,), dtype=torch.int32, device=device)


def slots_claim(in_use, n_slots, n_claim, pool=None, slots_out=None, stream=None):
    """Claim ``n_claim`` free slots (lowest first, all-or-nothing); zero their
    states in ``pool`` if given. Returns the int32 slot ids (-1s if none)."""
    if slots_out is None:
        slots_out = torch.empty((n_claim,), dtype=torch.int32, device=in_use.device)
    dt, H, K, pp = SC_BF16, 8, 1, None
    if pool is not None:
        dt, H, K = _dcode(pool), pool.shape[1], pool.shape[2]
        pp = _dev(pool, "pool", pool.dtype, (n_slots, H, K))
    _raise_on("shortconv_slots_claim", lib().shortconv_slots_claim(
        _dev(in_use, "in_use", torch.int32, ((n_slots + 31) // 32,)), n_slots, n_claim,
        _dev(slots_out, "slots_out", torch.int32, (n_claim,)), dt, H, K, pp,
        _stream(stream, in_use.device)))
    return slots_out


def slots_release(in_use, n_slots, slot_ids, stream=None):
    """Mark ``slot_ids`` free."""
    n = slot_ids.shape[0]
    _raise_on("shortconv_slots_release", lib().shortconv_slots_release(
        _dev(in_use, "in_use", torch.int32, ((n_slots + 31) // 32,)), n_slots,
        _dev(slot_ids, "slot_ids", torch.int32, (n,)), n, _stream(stream, in_use.device)))


def pool_copy(pool, src_slots, dst_slots, stream=None):
    """``pool[dst[i]] = pool[src[i]]`` (destinations distinct, not among sources)."""
    n_slots, H, K = pool.shape
    n = src_slots.shape[0]
    _raise_on("shortconv_pool_copy", lib().shortconv_pool_copy(
        _dcode(pool), H, K, _dev(pool, "pool", pool.dtype, (n_slots, H, K)), n_slots,
        _dev(src_slots, "src_slots", torch.int32, (n,)),
        _dev(dst_slots, "dst_slots", torch.int32, (n,)), n, _stream(stream, pool.device)))


def check_wait_limit(stream=None, device=None) -> None:
    """Enqueue the device-side timeout check: a kernel whose bounded wait runs
    out (about 2 s) and sets DEV_TIMEOUT, which get_error() then returns."""
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else device
    _raise_on("shortconv_check_wait_limit", lib().shortconv_check_wait_limit(_stream(stream, dev)))


def get_error(stream=None, device=None) -> int:
    """Synchronize the stream, return and clear the device error word (SC_DEV_* bits)."""
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else device
    code = ctypes.c_int(0)
    st = lib().shortconv_get_error(_stream(stream, dev), ctypes.byref(code))
    if st not in (SC_OK, SC_EDEVICE):
        _raise_on("shortconv_get_error", st)
    return code.value


def bounds_checked() -> bool:
    """True when the loaded library is the bounds-checked build."""
    return bool(lib().shortconv_bounds_checked())


def bounds_trim_next(region: int, nbytes: int) -> None:
    """Bounds-checked build: shorten buffer ``region`` of the next call's record."""
    _raise_on("shortconv_bounds_trim_next", lib().shortconv_bounds_trim_next(region, nbytes))


def bounds_take_first_bad(stream=None, device=None) -> int:
    """Bounds-checked build: the first refused device address since the last take (0: none)."""
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else device
    addr = ctypes.c_uint64(0)
    _raise_on("shortconv_bounds_take_first_bad",
              lib().shortconv_bounds_take_first_bad(_stream(stream, dev), ctypes.byref(addr)))
    return addr.value
