"""The optional per-channel conv bias on the GPU, against the CPU oracle.

The bias enters after the K-tap chain and before the C gate (z + b, then
y = C z); the backward gives dbias[h] = sum_t dz_t next to dW. Every kernel
path is covered: the streamed and the register-tiled prefill, decode,
verify, the single-sequence and the packed varlen backward. Passing no bias
must give what the bias-free calls give.
"""
import numpy as np
import pytest
import torch

import oracle
import lfm2_gated_short_gb300 as sc
from lfm2_gated_short_gb300 import workloads as wl
from gpu_util import assert_bits, assert_close, assert_dw_close, dev, host

pytestmark = pytest.mark.gpu

TILES = [0, 4, 8, 16, 32]
BIAS_STD = 0.5


def bias_for(H, dtype, seed):
    return wl.normal(np.random.default_rng(seed), (H,), BIAS_STD, dtype)


def same_values(dtype, a, b, what):
    """Equal as numbers (+0 and -0 count as equal)."""
    np.testing.assert_array_equal(oracle.to_f64(dtype, a), oracle.to_f64(dtype, b), what)


# ------------------------------------------------------------------ prefill

def _prefill(p, bias, tile=0):
    pool = dev(p.pool, p.dtype)
    y = sc.prefill(dev(p.bcx, p.dtype), dev(p.w, p.dtype), dev(p.cu_seqlens, "i32"),
                   dev(p.slot_ids, "i32"), pool, rows_per_thread=tile,
                   bias=None if bias is None else dev(bias, p.dtype))
    torch.cuda.synchronize()
    return host(y), host(pool)


def _oracle_prefill(p, bias):
    pool = p.pool.copy()
    st, y = oracle.prefill(p.dtype, p.bcx, p.w, p.cu_seqlens, p.slot_ids, pool, bias=bias)
    assert st == oracle.OK
    return y, pool


@pytest.mark.parametrize("K", [1, 2, 3, 4])
@pytest.mark.parametrize("tile", TILES)
@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_prefill_varlen_with_bias(dtype, tile, K):
    p = wl.varlen_prefill(H=256, K=K, n_slots=40, seed=400 + K, dtype=dtype,
                          lengths=[5, 0, 1, 2, 3, 40, 0, 7, 130, 2])
    b = bias_for(256, dtype, 401)
    y, pool = _prefill(p, b, tile)
    y_ref, pool_ref = _oracle_prefill(p, b)
    assert_close(dtype, y, y_ref, "y")
    assert_bits(pool, pool_ref, "state")           # the bias never enters the state


def test_prefill_bias_same_bits_on_every_kernel():
    p = wl.varlen_prefill(H=1024, K=3, n_slots=64, seed=402, lengths=[700, 3, 0, 1500, 64])
    b = bias_for(1024, "bf16", 403)
    y0, s0 = _prefill(p, b, 0)
    for tile in TILES[1:]:
        y, s = _prefill(p, b, tile)
        assert_bits(y, y0, f"y tile {tile}")
        assert_bits(s, s0, f"state tile {tile}")


def test_prefill_zero_bias_equals_no_bias():
    p = wl.single_prefill(T=999, H=512, K=3, seed=404)
    y_none, s_none = _prefill(p, None)
    y_zero, s_zero = _prefill(p, np.zeros(512, np.uint16))
    same_values("bf16", y_zero, y_none, "y")
    assert_bits(s_zero, s_none, "state")


def test_prefill_T4096_H2048_with_bias_sampled_channels():
    """The single-sequence prefill shape with a bias; oracle on 64 channels."""
    p = wl.single_prefill()
    b = bias_for(p.H, "bf16", 405)
    y, pool = _prefill(p, b)
    rng = np.random.default_rng(406)
    ch = np.sort(np.concatenate([[0, 7, 8, 511, 512, 2047],
                                 rng.choice(np.arange(9, 2040), 58, replace=False)]))
    cols = np.concatenate([ch, p.H + ch, 2 * p.H + ch])
    pool_ref = np.ascontiguousarray(p.pool[:, ch])
    st, y_ref = oracle.prefill("bf16", np.ascontiguousarray(p.bcx[:, cols]),
                               np.ascontiguousarray(p.w[ch]), p.cu_seqlens, p.slot_ids,
                               pool_ref, bias=np.ascontiguousarray(b[ch]))
    assert st == oracle.OK
    assert_close("bf16", y[:, ch], y_ref, "y")
    assert_bits(pool[:, ch], pool_ref, "state")


# ---------------------------------------------------------- decode / verify

@pytest.mark.parametrize("K", [1, 3, 4])
@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_decode_with_bias(dtype, K):
    s = wl.decode_serving(layers=1, steps=3, batch=37, H=512, K=K, n_slots=64,
                          seed=410 + K, dtype=dtype)
    b = bias_for(512, dtype, 411)
    pool = dev(s.pools[0], dtype)
    pool_ref = s.pools[0].copy()
    w, slots, bd = dev(s.w[0], dtype), dev(s.slot_ids, "i32"), dev(b, dtype)
    for step in range(3):
        y = sc.decode(dev(s.bcx[0, step], dtype), w, slots, pool, bias=bd)
        st, y_ref = oracle.decode(dtype, s.bcx[0, step], s.w[0], s.slot_ids, pool_ref, bias=b)
        assert st == oracle.OK
        assert_close(dtype, host(y), y_ref, f"y step {step}")
    assert_bits(host(pool), pool_ref, "pool")


@pytest.mark.parametrize("K", [2, 3])
@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_verify_and_rollback_with_bias(dtype, K):
    s = wl.verify_serving(layers=1, batch=19, D=5, H=256, K=K, n_slots=32, seed=420 + K,
                          dtype=dtype)
    b = bias_for(256, dtype, 421)
    pool = dev(s.pools[0], dtype)
    win, y = sc.verify(dev(s.bcx[0], dtype), dev(s.w[0], dtype), dev(s.slot_ids, "i32"), pool,
                       s.D, bias=dev(b, dtype))
    st, win_ref, y_ref = oracle.verify(dtype, s.bcx[0], s.w[0], s.slot_ids, s.pools[0], s.D,
                                       bias=b)
    assert st == oracle.OK
    assert_bits(host(win), win_ref, "win")
    assert_close(dtype, host(y), y_ref, "y")


def test_decode_and_verify_bias_agree_with_prefill():
    """One token by decode, by verify (D=1) and by a one-row prefill: same bits."""
    s = wl.decode_serving(layers=1, steps=1, batch=1, H=512, K=3, n_slots=4, seed=430)
    b = dev(bias_for(512, "bf16", 431), "bf16")
    w, slot = dev(s.w[0], "bf16"), dev(s.slot_ids, "i32")
    row = dev(s.bcx[0, 0], "bf16")
    p1, p2 = dev(s.pools[0], "bf16"), dev(s.pools[0], "bf16")
    yd = sc.decode(row, w, slot, p1, bias=b)
    _, yv = sc.verify(row, w, slot, dev(s.pools[0], "bf16"), 1, bias=b)
    yp = sc.prefill(row, w, dev(np.array([0, 1]), "i32"), slot, p2, bias=b)
    assert_bits(host(yv), host(yd), "verify vs decode")
    assert_bits(host(yp), host(yd), "prefill vs decode")
    assert_bits(host(p2), host(p1), "state")


# ----------------------------------------------------------------- backward

def _check_bwd(p, b, out, channels=None):
    dbcx, dw, dbias = (host(t) for t in out)
    H = p.H
    ch = np.arange(H) if channels is None else np.asarray(channels)
    cols = np.concatenate([ch, H + ch, 2 * H + ch])
    st, d_ref, dw_ref, db_ref = oracle.backward(
        p.dtype, np.ascontiguousarray(p.bcx[:, cols]), np.ascontiguousarray(p.w[ch]),
        np.ascontiguousarray(p.dy[:, ch]),
        bias=None if b is None else np.ascontiguousarray(b[ch]), with_dbias=True)
    assert st == oracle.OK
    assert_close(p.dtype, dbcx[:, cols], d_ref, "dB|dC|dx")
    assert_dw_close(dw[ch], dw_ref)
    assert_dw_close(dbias[ch], db_ref, "dbias")


@pytest.mark.parametrize("K", [1, 2, 3, 4])
@pytest.mark.parametrize("T", [0, 1, 5, 301, 4099])
@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_backward_with_bias(dtype, T, K):
    p = wl.training(T=T, H=256, K=K, seed=440 + T + K, dtype=dtype)
    b = bias_for(256, dtype, 441)
    out = sc.backward(dev(p.bcx, dtype), dev(p.w, dtype), dev(p.dy, dtype),
                      bias=dev(b, dtype), with_dbias=True)
    torch.cuda.synchronize()
    _check_bwd(p, b, out)
    if T == 0:
        assert np.all(host(out[2]) == 0.0)


def test_backward_dbias_without_bias():
    """dbias does not depend on the bias: it is sum_t dy_t C_t either way."""
    p = wl.training(T=2000, H=512, K=3, seed=450)
    out = sc.backward(dev(p.bcx, "bf16"), dev(p.w, "bf16"), dev(p.dy, "bf16"),
                      with_dbias=True)
    torch.cuda.synchronize()
    _check_bwd(p, None, out)
    d_nb, w_nb = sc.backward(dev(p.bcx, "bf16"), dev(p.w, "bf16"), dev(p.dy, "bf16"))
    assert_bits(host(out[0]), host(d_nb), "dbcx with and without dbias")
    np.testing.assert_array_equal(host(out[1]), host(w_nb))


def test_backward_bias_is_deterministic():
    p = wl.training(T=5000, H=512, K=3, seed=451)
    args = (dev(p.bcx, "bf16"), dev(p.w, "bf16"), dev(p.dy, "bf16"))
    b = dev(bias_for(512, "bf16", 452), "bf16")
    ws = torch.full((sc.backward_workspace_bytes(512, 3, 5000),), 0xFF, dtype=torch.uint8,
                    device="cuda")
    r1 = [host(t) for t in sc.backward(*args, bias=b, with_dbias=True, workspace=ws)]
    r2 = [host(t) for t in sc.backward(*args, bias=b, with_dbias=True, workspace=ws)]
    for a, c, what in zip(r1, r2, ("dbcx", "dw", "dbias")):
        assert_bits(a, c, what)


def test_backward_T65536_H2048_with_bias_sampled_channels():
    p = wl.training()
    b = bias_for(p.H, "bf16", 453)
    out = sc.backward(dev(p.bcx, "bf16"), dev(p.w, "bf16"), dev(p.dy, "bf16"),
                      bias=dev(b, "bf16"), with_dbias=True)
    torch.cuda.synchronize()
    rng = np.random.default_rng(454)
    ch = np.sort(np.concatenate([[0, 7, 8, 511, 512, 2047],
                                 rng.choice(np.arange(9, 2040), 58, replace=False)]))
    _check_bwd(p, b, out, ch)


@pytest.mark.parametrize("K", [1, 3, 4])
@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_backward_varlen_with_bias(dtype, K):
    rng = np.random.default_rng(460 + K)
    lengths = np.array([5, 0, 1, 2, 3, 40, 0, 7, 64, 1, 130, 2])
    cu = np.r_[0, np.cumsum(lengths)].astype(np.int32)
    T, N, H = int(cu[-1]), len(lengths), 256
    bcx = wl.normal(rng, (T, 3 * H), 1.0, dtype)
    w = wl.normal(rng, (H, K), wl.WEIGHT_STD, dtype)
    dy = wl.normal(rng, (T, H), 1.0, dtype)
    init = wl.normal(rng, (N, H, K), 1.0, dtype)
    dfin = rng.standard_normal((N, H, K)).astype(np.float32)
    b = bias_for(H, dtype, 461)
    dbcx, dw, dinit, dbias = sc.backward_varlen(
        dev(bcx, dtype), dev(w, dtype), dev(cu, "i32"), dev(dy, dtype),
        init_states=dev(init, dtype), d_final=dev(dfin, "f32"), bias=dev(b, dtype),
        with_dbias=True)
    torch.cuda.synchronize()
    st, d_ref, dw_ref, di_ref, db_ref = oracle.backward_varlen(
        dtype, bcx, w, cu, dy, init, dfin.astype(np.float64), bias=b, with_dbias=True)
    assert st == oracle.OK
    assert_close(dtype, host(dbcx), d_ref, "dB|dC|dx")
    assert_dw_close(host(dw), dw_ref)
    assert_dw_close(host(dinit), di_ref, "d_init")
    assert_dw_close(host(dbias), db_ref, "dbias")


def test_backward_varlen_one_sequence_bias_matches_single_sequence_kernel():
    p = wl.training(T=3001, H=512, K=3, seed=470)
    b = dev(bias_for(512, "bf16", 471), "bf16")
    args = (dev(p.bcx, "bf16"), dev(p.w, "bf16"))
    d1, w1, _, b1 = sc.backward_varlen(*args, dev(np.array([0, 3001]), "i32"),
                                       dev(p.dy, "bf16"), bias=b, with_dbias=True)
    d2, w2, b2 = sc.backward(*args, dev(p.dy, "bf16"), bias=b, with_dbias=True)
    assert_bits(host(d1), host(d2), "dbcx")
    np.testing.assert_array_equal(host(w1), host(w2))
    np.testing.assert_array_equal(host(b1), host(b2))


def test_backward_varlen_bad_seqlens_zero_dbias():
    rng = np.random.default_rng(480)
    H = 64
    bcx = wl.normal(rng, (15, 3 * H), 1.0, "bf16")
    w = wl.normal(rng, (H, 3), wl.WEIGHT_STD, "bf16")
    dy = wl.normal(rng, (15, H), 1.0, "bf16")
    bad = np.array([0, 9, 4, 15], np.int32)                   # not non-decreasing
    dbias = torch.full((H,), 5.0, device="cuda")
    _, dw, _, db = sc.backward_varlen(dev(bcx, "bf16"), dev(w, "bf16"), dev(bad, "i32"),
                                      dev(dy, "bf16"), with_dbias=True, dbias=dbias)
    assert sc.get_error() == sc.DEV_BAD_SEQLENS
    assert np.all(host(dw) == 0.0)
    assert np.all(host(db) == 0.0)
