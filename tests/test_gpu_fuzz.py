"""Seeded random sweeps of every conv call against the oracle.

Each case draws its shape (H a multiple of 8 up to 1536, K in 1..4, dtype,
optional bias) and its sequence structure (counts, lengths including empty
and shorter-than-K sequences, slot choice) from a seeded generator, then
checks the GPU against the oracle on the same inputs: states and windows bit
for bit, outputs within the tolerances in gpu_util.
"""
import numpy as np
import pytest

import oracle
import lfm2_gated_short_gb300 as sc
from lfm2_gated_short_gb300 import workloads as wl
from gpu_util import assert_bits, assert_close, assert_dw_close, dev, host

pytestmark = pytest.mark.gpu

CASES = 40


def draw(seed):
    rng = np.random.default_rng(seed)
    H = 8 * int(rng.integers(1, 193))
    K = int(rng.integers(1, 5))
    dtype = "bf16" if rng.random() < 0.7 else "f32"
    n = int(rng.integers(1, 9))
    short = rng.integers(0, 3 * K + 1, size=n)  # empty, shorter than K, a few windows
    long = rng.integers(K, 400, size=n)
    lengths = np.where(rng.random(n) < 0.5, long, short)
    bias = rng.random() < 0.3
    return rng, H, K, dtype, [int(v) for v in lengths], bias


def bias_of(rng, H, dtype, on):
    return wl.normal(rng, (H,), 0.5, dtype) if on else None


@pytest.mark.parametrize("seed", range(CASES))
def test_prefill_then_decode_and_verify(seed):
    rng, H, K, dtype, lengths, with_bias = draw(5000 + seed)
    n_slots = len(lengths) + 3
    p = wl.varlen_prefill(H=H, K=K, n_slots=n_slots, seed=6000 + seed, dtype=dtype,
                          lengths=lengths)
    b = bias_of(rng, H, dtype, with_bias)
    bd = None if b is None else dev(b, dtype)
    tile = [0, 4, 8, 16, 32][seed % 5]
    pool = dev(p.pool, dtype)
    y = sc.prefill(dev(p.bcx, dtype), dev(p.w, dtype), dev(p.cu_seqlens, "i32"),
                   dev(p.slot_ids, "i32"), pool, rows_per_thread=tile, bias=bd)
    ref = p.pool.copy()
    st, y_ref = oracle.prefill(dtype, p.bcx, p.w, p.cu_seqlens, p.slot_ids, ref, bias=b)
    assert st == oracle.OK
    assert_close(dtype, host(y), y_ref, f"prefill y (tile {tile})")
    assert_bits(host(pool), ref, "prefill pool")
    # one decode step on every sequence, then a verify of D drafts from the result
    N = len(lengths)
    bcx1 = wl.normal(rng, (N, 3 * H), 1.0, dtype)
    y = sc.decode(dev(bcx1, dtype), dev(p.w, dtype), dev(p.slot_ids, "i32"), pool, bias=bd)
    st, y_ref = oracle.decode(dtype, bcx1, p.w, p.slot_ids, ref, bias=b)
    assert st == oracle.OK
    assert_close(dtype, host(y), y_ref, "decode y")
    assert_bits(host(pool), ref, "decode pool")
    D = int(rng.integers(1, 13))  # past 8: more drafts than a thread holds at once
    bcxd = wl.normal(rng, (N * D, 3 * H), 1.0, dtype)
    win, y = sc.verify(dev(bcxd, dtype), dev(p.w, dtype), dev(p.slot_ids, "i32"), pool, D,
                       bias=bd)
    st, win_ref, y_ref = oracle.verify(dtype, bcxd, p.w, p.slot_ids, ref, D, bias=b)
    assert st == oracle.OK
    assert_close(dtype, host(y), y_ref, "verify y")
    assert_bits(host(win), win_ref, "verify windows")
    acc = rng.integers(0, D, size=N, endpoint=True).astype(np.int32)
    sc.rollback(win, dev(acc, "i32"), dev(p.slot_ids, "i32"), pool)
    assert oracle.rollback(dtype, win_ref, acc, p.slot_ids, ref) == oracle.OK
    assert_bits(host(pool), ref, "pool after rollback")
    assert sc.get_error() == 0


@pytest.mark.parametrize("seed", range(CASES))
def test_backward_and_varlen_backward(seed):
    rng, H, K, dtype, lengths, with_bias = draw(7000 + seed)
    cu = np.r_[0, np.cumsum(lengths)].astype(np.int32)
    T, N = int(cu[-1]), len(lengths)
    bcx = wl.normal(rng, (T, 3 * H), 1.0, dtype)
    w = wl.normal(rng, (H, K), wl.WEIGHT_STD, dtype)
    dy = wl.normal(rng, (T, H), 1.0, dtype)
    b = bias_of(rng, H, dtype, with_bias)
    bd = None if b is None else dev(b, dtype)
    out = sc.backward(dev(bcx, dtype), dev(w, dtype), dev(dy, dtype), bias=bd, with_dbias=True)
    st, d_ref, dw_ref, db_ref = oracle.backward(dtype, bcx, w, dy, bias=b, with_dbias=True)
    assert st == oracle.OK
    assert_close(dtype, host(out[0]), d_ref, "dB|dC|dx")
    assert_dw_close(host(out[1]), dw_ref)
    assert_dw_close(host(out[2]), db_ref, "dbias")
    init = wl.normal(rng, (N, H, K), 1.0, dtype)
    dfin = rng.standard_normal((N, H, K)).astype(np.float32)
    out = sc.backward_varlen(dev(bcx, dtype), dev(w, dtype), dev(cu, "i32"), dev(dy, dtype),
                             init_states=dev(init, dtype), d_final=dev(dfin, "f32"), bias=bd,
                             with_dbias=True)
    st, d_ref, dw_ref, di_ref, db_ref = oracle.backward_varlen(
        dtype, bcx, w, cu, dy, init, dfin.astype(np.float64), bias=b, with_dbias=True)
    assert st == oracle.OK
    assert_close(dtype, host(out[0]), d_ref, "varlen dB|dC|dx")
    assert_dw_close(host(out[1]), dw_ref, "varlen dW")
    assert_dw_close(host(out[2]), di_ref, "d_init")
    assert_dw_close(host(out[3]), db_ref, "varlen dbias")
    assert sc.get_error() == 0
