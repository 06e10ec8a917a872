"""The C ABI without a GPU: the library loads, exports what the header declares,
and host-side argument validation answers before any CUDA call is made."""
import ctypes
import os
import re

import pytest

from lfm2_gated_short_gb300 import build as sc_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER_DIR = os.path.join(ROOT, "include")

SC_OK, SC_EINVAL, SC_EUNSUPPORTED = 0, 1, 2
BF16, F32 = 1, 0


def declared_functions():
    names = []
    for fn in sorted(os.listdir(HEADER_DIR)):
        if fn.endswith(".h"):
            text = open(os.path.join(HEADER_DIR, fn)).read()
            text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
            names += re.findall(r"\b(shortconv_\w+)\s*\(", text)
    return sorted(set(names))


@pytest.fixture(scope="module")
def L():
    path = sc_build.build()
    lib = ctypes.CDLL(path)
    p, i32, i64 = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64
    lib.shortconv_prefill.argtypes = [i32, i32, i32, p, i64, p, p, p, i32, p, p, i32, p, p]
    lib.shortconv_prefill_tiled.argtypes = [i32, i32, i32, p, i64, p, p, p, i32, p, p, i32, p,
                                            i32, p]
    lib.shortconv_decode.argtypes = [i32, i32, i32, p, i32, p, p, p, p, i32, p, p]
    lib.shortconv_verify.argtypes = [i32, i32, i32, p, i32, i32, p, p, p, p, i32, p, p, p]
    lib.shortconv_rollback.argtypes = [i32, i32, i32, i32, i32, p, p, p, p, i32, p]
    lib.shortconv_rollback_layers.argtypes = [i32, i32, i32, i32, i32, i32, p, p, p, p, i32, p]
    lib.shortconv_backward_workspace_bytes.argtypes = [i32, i32, i64]
    lib.shortconv_backward_workspace_bytes.restype = ctypes.c_size_t
    lib.shortconv_backward.argtypes = [i32, i32, i32, p, i64, p, p, p, p, p, p, p,
                                       ctypes.c_size_t, p]
    lib.shortconv_backward_varlen.argtypes = [i32, i32, i32, p, i64, p, p, p, i32, p, p, p, p,
                                              p, p, p, p, ctypes.c_size_t, p]
    lib.shortconv_in_proj_workspace_bytes.argtypes = [i32, i32, i32]
    lib.shortconv_in_proj_workspace_bytes.restype = ctypes.c_size_t
    lib.shortconv_in_proj_prefill.argtypes = [i32, i32, i32, i32, p, i64, p, p, p, p, i32, p, p,
                                              i32, p, p, ctypes.c_size_t, p]
    lib.shortconv_out_proj.argtypes = [i32, i32, i32, p, i64, p, p, p]
    lib.shortconv_get_error.argtypes = [p, p]
    lib.shortconv_status_string.argtypes = [i32]
    lib.shortconv_status_string.restype = ctypes.c_char_p
    return lib


def test_header_declares_the_hot_path_calls():
    names = declared_functions()
    for must in ("shortconv_prefill", "shortconv_decode", "shortconv_verify",
                 "shortconv_rollback", "shortconv_backward",
                 "shortconv_backward_workspace_bytes", "shortconv_get_error",
                 "shortconv_status_string"):
        assert must in names


def test_library_exports_every_declared_function(L):
    for name in declared_functions():
        assert hasattr(L, name), f"{name} declared in include/ but not exported"


# Fake, 256-byte aligned, non-overlapping "device" addresses: validation must
# reject the call before anything touches them.
BASE = 1 << 40
A, Bp, Cp, Dp, Ep, Fp, Gp = (BASE + i * (1 << 32) for i in range(7))


def prefill(L, dtype=BF16, H=256, K=3, bcx=A, T=64, w=Bp, bias=None, cu=Cp, N=1, slots=Dp,
            pool=Ep, n_slots=4, y=Fp):
    return L.shortconv_prefill(dtype, H, K, bcx, T, w, bias, cu, N, slots, pool, n_slots, y,
                               None)


@pytest.mark.parametrize("kw,status", [
    (dict(dtype=7), SC_EUNSUPPORTED),
    (dict(H=12), SC_EUNSUPPORTED),
    (dict(K=5), SC_EUNSUPPORTED),
    (dict(K=0), SC_EINVAL),
    (dict(H=0), SC_EINVAL),
    (dict(T=-1), SC_EINVAL),
    (dict(T=1 << 31), SC_EINVAL),
    (dict(N=-1), SC_EINVAL),
    (dict(N=0), SC_EINVAL),                 # T > 0 with no sequences
    (dict(n_slots=0), SC_EINVAL),
    (dict(bcx=A + 8), SC_EINVAL),           # not 16-byte aligned
    (dict(y=0), SC_EINVAL),                 # NULL output with rows
    (dict(cu=Cp + 2), SC_EINVAL),           # int32 array not 4-byte aligned
    (dict(y=A + 64), SC_EINVAL),            # y overlaps bcx
    (dict(pool=Bp), SC_EINVAL),             # pool overlaps w
    (dict(bias=Gp + 8), SC_EINVAL),         # bias not 16-byte aligned
    (dict(bias=Fp + 64), SC_EINVAL),        # bias overlaps y
    (dict(bias=Ep), SC_EINVAL),             # bias overlaps pool
])
def test_prefill_argument_errors(L, kw, status):
    assert prefill(L, **kw) == status


def test_prefill_empty_call_is_ok_without_a_device(L):
    assert prefill(L, T=0, N=0, bcx=0, y=0, cu=Cp, slots=0) == SC_OK


def test_prefill_tiled_rejects_unbuilt_tiles(L):
    st = L.shortconv_prefill_tiled(BF16, 256, 3, A, 64, Bp, None, Cp, 1, Dp, Ep, 4, Fp, 12, None)
    assert st == SC_EINVAL


def test_decode_verify_rollback_argument_errors(L):
    assert L.shortconv_decode(BF16, 256, 3, A, 4, Bp, None, Dp, Ep, 4, A + 16, None) == SC_EINVAL
    assert L.shortconv_decode(BF16, 256, 3, A, 4, Bp, None, Dp, Ep, 0, Fp, None) == SC_EINVAL
    assert L.shortconv_decode(BF16, 256, 3, A, 4, Bp, Gp + 4, Dp, Ep, 4, Fp, None) == SC_EINVAL
    assert L.shortconv_decode(BF16, 256, 3, A, 4, Bp, Fp + 64, Dp, Ep, 4, Fp, None) == SC_EINVAL
    assert L.shortconv_decode(BF16, 256, 3, A, 0, Bp, None, 0, Ep, 4, 0, None) == SC_OK
    assert L.shortconv_verify(BF16, 256, 3, A, 4, 0, Bp, None, Dp, Ep, 4, Fp, Gp,
                              None) == SC_EINVAL
    assert L.shortconv_verify(BF16, 256, 3, A, 4, 2, Bp, None, Dp, Ep, 4, Fp, Fp,
                              None) == SC_EINVAL
    assert L.shortconv_verify(BF16, 256, 3, A, 4, 2, Bp, Gp, Dp, Ep, 4, Fp, Gp,
                              None) == SC_EINVAL                       # y aliases bias
    assert L.shortconv_rollback(BF16, 256, 3, 4, 2, Fp, Cp, Dp, Fp, 4, None) == SC_EINVAL
    assert L.shortconv_rollback(F32, 256, 3, 0, 2, 0, 0, 0, Ep, 4, None) == SC_OK


def test_rollback_layers_argument_errors(L):
    # (dtype, H, K, L, N, D, win, accepted, slots, pool, n_slots, stream)
    f = L.shortconv_rollback_layers
    assert f(BF16, 256, 3, 0, 4, 2, Fp, Cp, Dp, Ep, 4, None) == SC_EINVAL       # no layers
    assert f(BF16, 256, 3, 2, 4, 2, Fp, Cp, Dp, Fp + 64, 4, None) == SC_EINVAL  # pool in the tape
    assert f(BF16, 256, 3, 2, 4, 2, Fp, Ep + 16, Dp, Ep, 4, None) == SC_EINVAL  # accepted in pool
    assert f(BF16, 256, 3, 2, 4, 2, Fp, Cp, Ep + 32, Ep, 4, None) == SC_EINVAL  # slots in pool
    assert f(BF16, 256, 3, 2, 4, 2, Fp + 8, Cp, Dp, Ep, 4, None) == SC_EINVAL   # misaligned tape
    assert f(BF16, 256, 3, 2, 0, 2, Fp, Cp, Dp, Ep, 4, None) == SC_OK           # nothing to do


def test_backward_workspace_and_errors(L):
    ws = L.shortconv_backward_workspace_bytes(2048, 3, 65536)
    assert ws > 0 and ws % 16 == 0
    assert ws < 64 * 1024 * 1024        # a few MB of fp32 partials, not a T-sized buffer
    assert L.shortconv_backward_workspace_bytes(12, 3, 100) == 0
    assert L.shortconv_backward_workspace_bytes(2048, 3, -1) == 0
    need = L.shortconv_backward_workspace_bytes(256, 3, 64)
    assert need == 4 * 256 * 4 * 4      # 4 row ranges x (dW 3 + dbias 1) x H fp32

    def bwd(bias=None, dbcx=Dp, dw=Ep, dbias=None, ws=Fp, wsb=need):
        return L.shortconv_backward(BF16, 256, 3, A, 64, Bp, bias, Cp, dbcx, dw, dbias, ws, wsb,
                                    None)
    assert bwd(wsb=need - 1) == SC_EINVAL
    assert bwd(dbcx=A) == SC_EINVAL                  # dbcx aliases bcx
    assert bwd(bias=Gp + 8) == SC_EINVAL             # misaligned bias
    assert bwd(dbias=Gp + 2) == SC_EINVAL            # misaligned dbias
    assert bwd(dbias=Ep + 64) == SC_EINVAL           # dbias overlaps dw
    assert bwd(bias=Gp, dbias=Gp) == SC_EINVAL       # dbias aliases bias
    assert bwd(dbias=Fp + 16) == SC_EINVAL           # dbias inside the workspace


def test_backward_varlen_argument_errors(L):
    need = L.shortconv_backward_workspace_bytes(256, 3, 64)
    ok = dict(dtype=BF16, H=256, K=3, bcx=A, T=64, w=Bp, bias=None, cu=Cp, N=2, init=None,
              dy=Dp, dfin=None, dbcx=Ep, dw=Fp, dbias=None, dinit=None, ws=Gp, wsb=need)

    def call(**kw):
        a = dict(ok, **kw)
        return L.shortconv_backward_varlen(a["dtype"], a["H"], a["K"], a["bcx"], a["T"], a["w"],
                                           a["bias"], a["cu"], a["N"], a["init"], a["dy"],
                                           a["dfin"], a["dbcx"], a["dw"], a["dbias"], a["dinit"],
                                           a["ws"], a["wsb"], None)
    assert call(N=0) == SC_EINVAL                 # rows but no sequences
    assert call(wsb=need - 1) == SC_EINVAL
    assert call(dbcx=A) == SC_EINVAL              # output aliases bcx
    assert call(dinit=Bp) == SC_EINVAL            # d_init aliases w
    assert call(K=5) == SC_EUNSUPPORTED
    assert call(bias=Fp + 4) == SC_EINVAL         # misaligned bias
    assert call(dbias=Bp) == SC_EINVAL            # dbias aliases w
    assert call(dbias=Fp + 8) == SC_EINVAL        # dbias overlaps dw


def test_in_proj_prefill_argument_errors(L):
    need = L.shortconv_in_proj_workspace_bytes(128, 3, 2)
    assert need == 2 * 128 * 3 * 2
    assert L.shortconv_in_proj_workspace_bytes(100, 3, 2) == 0
    ok = dict(dtype=BF16, D=256, H=128, K=3, hid=A, T=64, w_in=Bp, w=Cp, bias=None, cu=Dp, N=2,
              slots=Dp + 4096, pool=Ep, n_slots=4, y=Fp, ws=Gp, wsb=need)

    def call(**kw):
        a = dict(ok, **kw)
        return L.shortconv_in_proj_prefill(a["dtype"], a["D"], a["H"], a["K"], a["hid"], a["T"],
                                           a["w_in"], a["w"], a["bias"], a["cu"], a["N"],
                                           a["slots"], a["pool"], a["n_slots"], a["y"], a["ws"],
                                           a["wsb"], None)
    assert call(dtype=F32) == SC_EUNSUPPORTED      # bf16 only
    assert call(D=100) == SC_EUNSUPPORTED          # D % 64
    assert call(H=72) == SC_EUNSUPPORTED           # H % 64
    assert call(K=5) == SC_EUNSUPPORTED
    assert call(K=0) == SC_EINVAL
    assert call(N=0) == SC_EINVAL                  # rows but no sequences
    assert call(wsb=need - 1) == SC_EINVAL
    assert call(hid=A + 8) == SC_EINVAL            # not 16-byte aligned
    assert call(y=A) == SC_EINVAL                  # y aliases hidden
    assert call(pool=Bp) == SC_EINVAL              # pool overlaps w_in
    assert call(ws=Fp + 64) == SC_EINVAL           # workspace overlaps y
    assert call(bias=Fp + 32) == SC_EINVAL         # y overlaps bias
    assert call(T=0, N=0, hid=0, y=0) == SC_OK     # nothing to do


def test_out_proj_argument_errors(L):
    def call(dtype=BF16, H=128, D=512, y=A, T=64, wo=Bp, out=Cp):
        return L.shortconv_out_proj(dtype, H, D, y, T, wo, out, None)
    assert call(dtype=F32) == SC_EUNSUPPORTED
    assert call(D=300) == SC_EUNSUPPORTED          # D % 256
    assert call(H=100) == SC_EUNSUPPORTED          # H % 64
    assert call(T=-1) == SC_EINVAL
    assert call(out=A + 1024) == SC_EINVAL         # out overlaps y
    assert call(wo=Bp + 8) == SC_EINVAL            # misaligned


def test_status_strings_and_get_error_null(L):
    for s in range(6):
        assert L.shortconv_status_string(s)
    assert L.shortconv_get_error(None, None) == SC_EINVAL


def test_standard_build_has_no_bounds_checks(L):
    L.shortconv_bounds_checked.restype = ctypes.c_int
    L.shortconv_bounds_trim_next.argtypes = [ctypes.c_int, ctypes.c_uint64]
    assert L.shortconv_bounds_checked() == 0
    assert L.shortconv_bounds_trim_next(6, 16) == SC_EUNSUPPORTED
    addr = ctypes.c_uint64(0)
    L.shortconv_bounds_take_first_bad.argtypes = [ctypes.c_void_p, ctypes.c_void_p]
    assert L.shortconv_bounds_take_first_bad(None, ctypes.byref(addr)) == SC_EUNSUPPORTED


def test_bounds_checked_build_loads_and_exports_every_declared_function():
    B = ctypes.CDLL(sc_build.build(bounds_check=True))
    for name in declared_functions():
        assert hasattr(B, name), f"{name} declared in include/ but not exported"
    B.shortconv_bounds_checked.restype = ctypes.c_int
    B.shortconv_bounds_trim_next.argtypes = [ctypes.c_int, ctypes.c_uint64]
    assert B.shortconv_bounds_checked() == 1
    assert B.shortconv_bounds_trim_next(16, 1) == SC_EINVAL
    assert B.shortconv_bounds_trim_next(-1, 1) == SC_EINVAL
    # host validation answers before any record is installed or CUDA call made
    p, i32, i64 = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64
    B.shortconv_prefill.argtypes = [i32, i32, i32, p, i64, p, p, p, i32, p, p, i32, p, p]
    assert B.shortconv_prefill(7, 256, 3, A, 64, Bp, None, Cp, 1, Dp, Ep, 4, Fp,
                               None) == SC_EUNSUPPORTED


def test_in_proj_decode_argument_errors(L):
    p, i32 = ctypes.c_void_p, ctypes.c_int
    f = L.shortconv_in_proj_decode
    f.argtypes = [i32, i32, i32, i32, p, i32, p, p, p, p, p, i32, p, p]
    ok = dict(dtype=BF16, D=128, H=64, K=3, hidden=A, N=4, w_in=Bp, w=Cp, bias=None, slots=Dp,
              pool=Ep, n_slots=8, y=Fp)

    def call(**kw):
        a = dict(ok, **kw)
        return f(a["dtype"], a["D"], a["H"], a["K"], a["hidden"], a["N"], a["w_in"], a["w"],
                 a["bias"], a["slots"], a["pool"], a["n_slots"], a["y"], None)

    assert call(dtype=F32) == SC_EUNSUPPORTED
    assert call(D=96) == SC_EUNSUPPORTED
    assert call(H=96) == SC_EUNSUPPORTED
    assert call(K=5) == SC_EUNSUPPORTED
    assert call(N=-1) == SC_EINVAL
    assert call(n_slots=0) == SC_EINVAL
    assert call(hidden=A + 8) == SC_EINVAL        # not 16-byte aligned
    assert call(y=A + 64) == SC_EINVAL            # y overlaps hidden
    assert call(pool=Bp) == SC_EINVAL             # pool overlaps w_in
    assert call(slots=Dp + 2) == SC_EINVAL        # int32 array not 4-byte aligned
    assert call(N=0, hidden=0, y=0) == SC_OK      # nothing to do, no device needed
