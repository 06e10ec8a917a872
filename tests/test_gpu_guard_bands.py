"""Guard bands around every buffer a call writes.

Each output (and each in-place buffer: pools, bitmaps, workspaces) is placed
inside a larger allocation, with 4 KB bands of a fill pattern directly before
and after it. After the call the bands must hold the pattern bit for bit: a
kernel that writes one element before or past any buffer, or an asynchronous
copy or store with a wrong byte count, changes a band. Workspaces are given
exactly the size the library asks for, so a write past that size shows too.
Inputs that are only read are not banded (the bounds-checked build covers
reads). Every call also runs against the oracle, so the calls did their work.

The shapes are the ragged ones: channel counts that leave partial warps and
a partly used 512-channel slice (H = 8, 40, 520), row counts that are not a
multiple of any tile, empty sequences and sequences shorter than the window.
A packed call must also write nothing outside its own rows and slots: the
untouched slots of every pool hold a sentinel that must survive.
"""
import numpy as np
import pytest
import torch

import oracle
from oracle import layer
from oracle import slots as slot_model
import lfm2_gated_short_gb300 as sc
from lfm2_gated_short_gb300 import workloads as wl
from gpu_util import assert_bits, assert_close, assert_dw_close, dev, host

pytestmark = pytest.mark.gpu

BAND = 4096   # bytes of fill before and after each banded buffer
FILL = 0xA5   # fill byte


class Banded:
    """A device tensor of ``shape`` and ``dtype`` with BAND fill bytes on each side."""

    def __init__(self, shape, dtype, init=None):
        elem = torch.empty((), dtype=dtype).element_size()
        self.n = int(np.prod(shape, dtype=np.int64)) * elem
        self.raw = torch.full((BAND + self.n + BAND,), FILL, dtype=torch.uint8, device="cuda")
        self.t = self.raw[BAND:BAND + self.n].view(dtype).view(tuple(shape))
        if init is not None:
            self.t.copy_(init)

    def check(self, what):
        torch.cuda.synchronize()
        lo = int((self.raw[:BAND] != FILL).sum())
        hi = int((self.raw[BAND + self.n:] != FILL).sum())
        assert lo == 0 and hi == 0, f"{what}: {lo} band bytes changed before, {hi} after"


TORCH_DT = {"bf16": torch.bfloat16, "f32": torch.float32}


def banded_from(a, dtype):
    """A banded device copy of the host array ``a`` (storage dtype ``dtype``)."""
    t = dev(a, dtype)
    return Banded(t.shape, t.dtype, t)


def banded_empty(shape, dtype):
    return Banded(shape, TORCH_DT.get(dtype, dtype))


# ------------------------------------------------------------- forward

LENGTHS = [0, 1, 2, 37, 0, 3, 130, 5]


@pytest.mark.parametrize("H,K", [(8, 3), (40, 4), (520, 3), (40, 1)])
@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("tile", [0, 8])
def test_prefill_decode_verify_rollback(dtype, H, K, tile):
    p = wl.varlen_prefill(H=H, K=K, n_slots=13, seed=1200 + H + K, dtype=dtype,
                          lengths=LENGTHS)
    N = p.N
    pool = banded_from(p.pool, dtype)
    y = banded_empty((p.T, H), dtype)
    sc.prefill(dev(p.bcx, dtype), dev(p.w, dtype), dev(p.cu_seqlens, "i32"),
               dev(p.slot_ids, "i32"), pool.t, y=y.t, rows_per_thread=tile)
    ref = p.pool.copy()
    st, y_ref = oracle.prefill(dtype, p.bcx, p.w, p.cu_seqlens, p.slot_ids, ref)
    assert st == oracle.OK
    pool.check("prefill pool")
    y.check("prefill y")
    assert_close(dtype, host(y.t), y_ref, "prefill y")
    assert_bits(host(pool.t), ref, "prefill pool")

    rng = np.random.default_rng(1300 + H)
    bcx1 = wl.normal(rng, (N, 3 * H), 1.0, dtype)
    yd = banded_empty((N, H), dtype)
    sc.decode(dev(bcx1, dtype), dev(p.w, dtype), dev(p.slot_ids, "i32"), pool.t, y=yd.t)
    st, yd_ref = oracle.decode(dtype, bcx1, p.w, p.slot_ids, ref)
    assert st == oracle.OK
    pool.check("decode pool")
    yd.check("decode y")
    assert_close(dtype, host(yd.t), yd_ref, "decode y")
    assert_bits(host(pool.t), ref, "decode pool")

    D = 5
    bcxv = wl.normal(rng, (N * D, 3 * H), 1.0, dtype)
    win = banded_empty((N, D, H, K), dtype)
    yv = banded_empty((N * D, H), dtype)
    sc.verify(dev(bcxv, dtype), dev(p.w, dtype), dev(p.slot_ids, "i32"), pool.t, D, win=win.t,
              y=yv.t)
    st, win_ref, yv_ref = oracle.verify(dtype, bcxv, p.w, p.slot_ids, ref, D)
    assert st == oracle.OK
    for b, what in ((pool, "verify pool"), (win, "verify win"), (yv, "verify y")):
        b.check(what)
    assert_bits(host(pool.t), ref, "verify leaves the pool alone")
    assert_bits(host(win.t), win_ref, "verify windows")
    assert_close(dtype, host(yv.t), yv_ref, "verify y")

    accepted = rng.integers(0, D, size=N, endpoint=True).astype(np.int32)
    sc.rollback(win.t, dev(accepted, "i32"), dev(p.slot_ids, "i32"), pool.t)
    assert oracle.rollback(dtype, win_ref, accepted, p.slot_ids, ref) == oracle.OK
    pool.check("rollback pool")
    win.check("rollback win")
    assert_bits(host(pool.t), ref, "rollback pool")
    assert sc.get_error() == 0


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_rollback_layers(dtype):
    L, N, D, H, K, S = 3, 6, 4, 40, 3, 11
    s = wl.verify_serving(layers=L, batch=N, D=D, H=H, K=K, n_slots=S, seed=1400, dtype=dtype)
    pools = banded_from(s.pools, dtype)
    win = banded_empty((L, N, D, H, K), dtype)
    refs = s.pools.copy()
    win_refs = []
    for l in range(L):
        sc.verify(dev(s.bcx[l], dtype), dev(s.w[l], dtype), dev(s.slot_ids, "i32"), pools.t[l],
                  D, win=win.t[l])
        st, win_ref, _ = oracle.verify(dtype, s.bcx[l], s.w[l], s.slot_ids, refs[l], D)
        assert st == oracle.OK
        win_refs.append(win_ref)
    sc.rollback_layers(win.t, dev(s.accepted, "i32"), dev(s.slot_ids, "i32"), pools.t)
    for l in range(L):
        assert oracle.rollback(dtype, win_refs[l], s.accepted, s.slot_ids, refs[l]) == oracle.OK
    pools.check("stacked pools")
    win.check("stacked windows")
    assert_bits(host(pools.t), refs, "pools after the stacked rollback")
    assert sc.get_error() == 0


# ------------------------------------------------------------- backward

@pytest.mark.parametrize("H,K,T", [(8, 3, 301), (40, 4, 4099), (520, 3, 77), (40, 1, 5),
                                   (520, 2, 0)])
@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("with_bias", [False, True])
def test_backward(dtype, H, K, T, with_bias):
    t = wl.training(T=T, H=H, K=K, seed=1500 + H + T, dtype=dtype)
    rng = np.random.default_rng(1501)
    b = wl.normal(rng, (H,), 0.5, dtype) if with_bias else None
    need = sc.backward_workspace_bytes(H, K, T)
    dbcx = banded_empty((T, 3 * H), dtype)
    dw = banded_empty((H, K), torch.float32)
    dbias = banded_empty((H,), torch.float32)
    ws = banded_empty((need,), torch.uint8)
    sc.backward(dev(t.bcx, dtype), dev(t.w, dtype), dev(t.dy, dtype), dbcx=dbcx.t, dw=dw.t,
                workspace=ws.t, bias=None if b is None else dev(b, dtype),
                with_dbias=with_bias, dbias=dbias.t if with_bias else None)
    for x, what in ((dbcx, "dbcx"), (dw, "dW"), (dbias, "dbias"), (ws, "workspace")):
        x.check(what)
    st, d_ref, dw_ref, db_ref = oracle.backward(dtype, t.bcx, t.w, t.dy, bias=b, with_dbias=True)
    assert st == oracle.OK
    assert_close(dtype, host(dbcx.t), d_ref, "dB|dC|dx")
    assert_dw_close(host(dw.t), dw_ref)
    if with_bias:
        assert_dw_close(host(dbias.t), db_ref, "dbias")
    assert sc.get_error() == 0


@pytest.mark.parametrize("H,K", [(8, 3), (40, 4), (520, 3)])
@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_backward_varlen(dtype, H, K):
    rng = np.random.default_rng(1600 + H + K)
    cu = np.r_[0, np.cumsum(LENGTHS)].astype(np.int32)
    T, N = int(cu[-1]), len(LENGTHS)
    bcx = wl.normal(rng, (T, 3 * H), 1.0, dtype)
    w = wl.normal(rng, (H, K), wl.WEIGHT_STD, dtype)
    dy = wl.normal(rng, (T, H), 1.0, dtype)
    b = wl.normal(rng, (H,), 0.5, dtype)
    init = wl.normal(rng, (N, H, K), 1.0, dtype)
    dfin = rng.standard_normal((N, H, K)).astype(np.float32)
    need = sc.backward_workspace_bytes(H, K, T)
    dbcx = banded_empty((T, 3 * H), dtype)
    dw = banded_empty((H, K), torch.float32)
    dbias = banded_empty((H,), torch.float32)
    d_init = banded_empty((N, H, K), torch.float32)
    ws = banded_empty((need,), torch.uint8)
    sc.backward_varlen(dev(bcx, dtype), dev(w, dtype), dev(cu, "i32"), dev(dy, dtype),
                       init_states=dev(init, dtype), d_final=dev(dfin, "f32"), dbcx=dbcx.t,
                       dw=dw.t, d_init=d_init.t, workspace=ws.t, bias=dev(b, dtype),
                       with_dbias=True, dbias=dbias.t)
    for x, what in ((dbcx, "dbcx"), (dw, "dW"), (dbias, "dbias"), (d_init, "d_init"),
                    (ws, "workspace")):
        x.check(what)
    st, d_ref, dw_ref, di_ref, db_ref = oracle.backward_varlen(
        dtype, bcx, w, cu, dy, init, dfin.astype(np.float64), bias=b, with_dbias=True)
    assert st == oracle.OK
    assert_close(dtype, host(dbcx.t), d_ref, "dB|dC|dx")
    assert_dw_close(host(dw.t), dw_ref)
    assert_dw_close(host(d_init.t), di_ref, "d_init")
    assert_dw_close(host(dbias.t), db_ref, "dbias")
    assert sc.get_error() == 0


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_backward_noalloc(dtype):
    import ctypes
    H, K, T = 40, 3, 301
    t = wl.training(T=T, H=H, K=K, seed=1700, dtype=dtype)
    bcx, w, dy = dev(t.bcx, dtype), dev(t.w, dtype), dev(t.dy, dtype)
    dbcx = banded_empty((T, 3 * H), dtype)
    dw = banded_empty((H, K), torch.float32)
    f = sc.lib().shortconv_backward_noalloc
    p, i32, i64 = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64
    f.argtypes = [i32, i32, i32, p, i64, p, p, p, p, p]
    f.restype = i32
    code = sc.SC_BF16 if dtype == "bf16" else sc.SC_F32
    st = f(code, H, K, bcx.data_ptr(), T, w.data_ptr(), dy.data_ptr(), dbcx.t.data_ptr(),
           dw.t.data_ptr(), torch.cuda.current_stream().cuda_stream)
    assert st == sc.SC_OK
    dbcx.check("dbcx")
    dw.check("dW")
    st, d_ref, dw_ref = oracle.backward(dtype, t.bcx, t.w, t.dy)
    assert st == oracle.OK
    assert_close(dtype, host(dbcx.t), d_ref, "dB|dC|dx")
    assert_dw_close(host(dw.t), dw_ref)
    assert sc.get_error() == 0


# ---------------------------------------------------------- projections

def _dyadic(rng, shape, lim, exp):
    return oracle.round_bf16(rng.integers(-lim, lim, size=shape, endpoint=True) * 2.0 ** exp)


@pytest.mark.parametrize("D,H,K", [(64, 64, 3), (128, 192, 4)])
def test_in_proj_prefill_and_out_proj(D, H, K):
    rng = np.random.default_rng(1800 + D + H)
    lengths = [0, 1, 130, 2, 0, 257, 3]
    cu = np.r_[0, np.cumsum(lengths)].astype(np.int32)
    T, N = int(cu[-1]), len(lengths)
    hidden = _dyadic(rng, (T, D), 8, -3)
    w_in = _dyadic(rng, (3 * H, D), 8, -6)
    w = oracle.round_bf16(rng.standard_normal((H, K)) * np.sqrt(1 / 3))
    n_slots = N + 4
    slots = rng.permutation(n_slots)[:N].astype(np.int32)
    pool0 = np.full((n_slots, H, K), 0xDEAD, np.uint16)
    for s in slots:
        pool0[s] = oracle.round_bf16(rng.standard_normal((H, K)))
    pool = banded_from(pool0, "bf16")
    y = banded_empty((T, H), "bf16")
    ws = banded_empty((sc.in_proj_workspace_bytes(H, K, N),), torch.uint8)
    sc.in_proj_prefill(dev(hidden, "bf16"), dev(w_in, "bf16"), dev(w, "bf16"), dev(cu, "i32"),
                       dev(slots, "i32"), pool.t, y=y.t, workspace=ws.t)
    for x, what in ((pool, "pool"), (y, "y"), (ws, "workspace")):
        x.check(what)
    ref = pool0.copy()
    st, y_ref = layer.in_proj_prefill("bf16", hidden, w_in, w, cu, slots, ref)
    assert st == oracle.OK
    assert_close("bf16", host(y.t), y_ref, "y")
    assert_bits(host(pool.t), ref, "pool")

    Dout = 256  # out_proj's output width is a multiple of 256
    w_out = _dyadic(rng, (Dout, H), 8, -6)
    yin = _dyadic(rng, (T, H), 8, -3)
    out = banded_empty((T, Dout), "bf16")
    sc.out_proj(dev(yin, "bf16"), dev(w_out, "bf16"), out=out.t)
    out.check("out_proj out")
    assert_bits(host(out.t), layer.out_proj("bf16", yin, w_out), "out_proj")
    assert sc.get_error() == 0


@pytest.mark.parametrize("T,H", [(20000, 192), (200, 192)])
def test_in_proj_prefill_one_sequence(T, H):
    """One sequence: the fused call writes the new state itself, and its CTAs'
    last tiles store y through TMA boxes (the upper half of the last
    128-channel tile lies past H = 192 and must be clipped). Nothing outside
    y and the slot's state changes."""
    rng = np.random.default_rng(1870 + T)
    D, K = 64, 3
    hidden = _dyadic(rng, (T, D), 8, -3)
    w_in = _dyadic(rng, (3 * H, D), 8, -6)
    w = oracle.round_bf16(rng.standard_normal((H, K)) * np.sqrt(1 / 3))
    n_slots = 4
    slots = np.array([2], np.int32)
    pool0 = np.full((n_slots, H, K), 0xDEAD, np.uint16)
    pool0[2] = oracle.round_bf16(rng.standard_normal((H, K)))
    pool = banded_from(pool0, "bf16")
    y = banded_empty((T, H), "bf16")
    cu = np.array([0, T], np.int32)
    sc.in_proj_prefill(dev(hidden, "bf16"), dev(w_in, "bf16"), dev(w, "bf16"), dev(cu, "i32"),
                       dev(slots, "i32"), pool.t, y=y.t)
    for x, what in ((pool, "pool"), (y, "y")):
        x.check(what)
    ref = pool0.copy()
    st, y_ref = layer.in_proj_prefill("bf16", hidden, w_in, w, cu, slots, ref)
    assert st == oracle.OK
    assert sc.get_error() == 0
    assert_bits(host(pool.t), ref, "pool")
    assert_close("bf16", host(y.t), y_ref, "y")


@pytest.mark.parametrize("N,D,H,K", [(1, 64, 64, 3), (130, 64, 192, 4), (300, 128, 64, 1)])
def test_in_proj_decode(N, D, H, K):
    rng = np.random.default_rng(1850 + N)
    hidden = _dyadic(rng, (N, D), 8, -3)
    w_in = _dyadic(rng, (3 * H, D), 8, -6)
    w = oracle.round_bf16(rng.standard_normal((H, K)) * np.sqrt(1 / 3))
    n_slots = N + 5
    slots = rng.permutation(n_slots)[:N].astype(np.int32)
    pool0 = np.full((n_slots, H, K), 0xDEAD, np.uint16)
    for s_ in slots:
        pool0[s_] = oracle.round_bf16(rng.standard_normal((H, K)))
    pool = banded_from(pool0, "bf16")
    y = banded_empty((N, H), "bf16")
    sc.in_proj_decode(dev(hidden, "bf16"), dev(w_in, "bf16"), dev(w, "bf16"), dev(slots, "i32"),
                      pool.t, y=y.t)
    pool.check("pool")
    y.check("y")
    ref = pool0.copy()
    st, y_ref = layer.in_proj_decode("bf16", hidden, w_in, w, slots, ref)
    assert st == oracle.OK
    assert_close("bf16", host(y.t), y_ref, "y")
    assert_bits(host(pool.t), ref, "pool")
    assert sc.get_error() == 0


# ------------------------------------------------------------ slot pool

def test_slots_claim_release_copy():
    rng = np.random.default_rng(1900)
    n_slots, H, K = 77, 40, 3
    bm0 = np.zeros(slot_model.words(n_slots), np.uint32)
    for s in rng.choice(n_slots, 30, replace=False):
        bm0[s // 32] |= np.uint32(1 << (int(s) % 32))
    pool0 = wl.normal(rng, (n_slots, H, K), 1.0, "bf16")
    bm = banded_from(bm0.view(np.int32), "i32")
    pool = banded_from(pool0, "bf16")
    out = banded_empty((9,), torch.int32)
    sc.slots_claim(bm.t, n_slots, 9, pool=pool.t, slots_out=out.t)
    for x, what in ((bm, "bitmap"), (pool, "pool"), (out, "claimed ids")):
        x.check(what)
    bm_ref, pool_ref = bm0.copy(), pool0.copy()
    err, ids = slot_model.claim(bm_ref, n_slots, 9, pool_ref)
    assert err == slot_model.OK
    assert_bits(host(out.t), ids, "claimed ids")
    assert_bits(host(bm.t).view(np.uint32), bm_ref, "bitmap after claim")
    assert_bits(host(pool.t), pool_ref, "pool after claim")

    rel = ids[::2].copy()
    sc.slots_release(bm.t, n_slots, dev(rel, "i32"))
    bm.check("bitmap after release")
    assert slot_model.release(bm_ref, n_slots, rel) == slot_model.OK
    assert_bits(host(bm.t).view(np.uint32), bm_ref, "bitmap after release")

    src, dst = ids[:3].copy(), ids[5:8].copy()
    sc.pool_copy(pool.t, dev(src, "i32"), dev(dst, "i32"))
    pool.check("pool after copy")
    assert slot_model.copy(pool_ref, src, dst) == slot_model.OK
    assert_bits(host(pool.t), pool_ref, "pool after copy")
    assert sc.get_error() == 0


# ----------------------------------- the bounds-checked build at work
#
# These run only when the loaded library is the bounds-checked build (the
# test in test_gpu_bounds_build.py runs this whole file that way). A record
# is shortened with shortconv_bounds_trim_next, so the kernels' own, valid
# accesses to the cut-off bytes count as outside the call: they must be
# refused, reported with their address, and leave those bytes alone, while
# everything else is computed as usual and no wait runs out.

def _bounds_build_only():
    if not sc.bounds_checked():
        pytest.skip("the standard build has no bounds checks to show")


@pytest.mark.parametrize("tile", [0, 8])
@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_bounds_build_refuses_stores_past_a_shortened_output(dtype, tile):
    _bounds_build_only()
    H, K = 40, 3
    es = 2 if dtype == "bf16" else 4
    p = wl.varlen_prefill(H=H, K=K, n_slots=13, seed=1950, dtype=dtype, lengths=LENGTHS)
    ref = p.pool.copy()
    st, y_ref = oracle.prefill(dtype, p.bcx, p.w, p.cu_seqlens, p.slot_ids, ref)
    assert st == oracle.OK
    pool = banded_from(p.pool, dtype)
    y = banded_empty((p.T, H), dtype)
    sc.bounds_trim_next(6, H * es)  # y's record loses its last row
    sc.prefill(dev(p.bcx, dtype), dev(p.w, dtype), dev(p.cu_seqlens, "i32"),
               dev(p.slot_ids, "i32"), pool.t, y=y.t, rows_per_thread=tile)
    assert sc.get_error() == sc.DEV_OUT_OF_BOUNDS
    last = y.t.data_ptr() + (p.T - 1) * H * es
    assert last <= sc.bounds_take_first_bad() < last + H * es
    y.check("y")
    got = host(y.t)
    assert_close(dtype, got[:-1], y_ref[:-1], "rows inside the record")
    assert np.all(got[-1].view(np.uint8) == FILL), "the refused row was written"
    assert_bits(host(pool.t), ref, "pool")


@pytest.mark.parametrize("tile", [0, 8])
def test_bounds_build_refuses_loads_past_a_shortened_input(tile):
    _bounds_build_only()
    H, K, dtype = 40, 3, "bf16"
    p = wl.varlen_prefill(H=H, K=K, n_slots=13, seed=1951, dtype=dtype, lengths=LENGTHS)
    bcx = dev(p.bcx, dtype)
    sc.bounds_trim_next(0, 3 * H * 2)  # bcx's record loses its last row
    sc.prefill(bcx, dev(p.w, dtype), dev(p.cu_seqlens, "i32"), dev(p.slot_ids, "i32"),
               dev(p.pool, dtype), rows_per_thread=tile)
    # refused loads are reported; the refused bulk copies still complete their
    # barriers, so no wait runs out (no SC_DEV_TIMEOUT bit)
    assert sc.get_error() == sc.DEV_OUT_OF_BOUNDS
    last = bcx.data_ptr() + (p.T - 1) * 3 * H * 2
    assert last <= sc.bounds_take_first_bad() < last + 3 * H * 2


def test_bounds_build_refuses_the_last_dw_entry_when_cut_off():
    _bounds_build_only()
    H, K, T = 40, 3, 301
    t = wl.training(T=T, H=H, K=K, seed=1952)
    dw = banded_empty((H, K), torch.float32)
    dw.t.fill_(float("nan"))
    sc.bounds_trim_next(5, 4)  # dW's record loses its last entry
    sc.backward(dev(t.bcx, "bf16"), dev(t.w, "bf16"), dev(t.dy, "bf16"), dw=dw.t)
    assert sc.get_error() == sc.DEV_OUT_OF_BOUNDS
    assert sc.bounds_take_first_bad() == dw.t.data_ptr() + (H * K - 1) * 4
    dw.check("dW")
    st, _, dw_ref = oracle.backward("bf16", t.bcx, t.w, t.dy)
    got = host(dw.t).reshape(-1)
    assert np.isnan(got[-1])
    assert_dw_close(got[:-1], dw_ref.reshape(-1)[:-1])
