"""The narrowest channel counts the ABI accepts (H a multiple of 8).

The kernels split H into groups of 2, 4 or 8 channels a thread and into
512-channel slices; H = 8, 24 and 40 leave partial warps and a single,
partly used slice. Every call runs against the oracle in bf16 and fp32.
"""
import numpy as np
import pytest

import oracle
import lfm2_gated_short_gb300 as sc
from lfm2_gated_short_gb300 import workloads as wl
from gpu_util import assert_bits, assert_close, assert_dw_close, dev, host

pytestmark = pytest.mark.gpu

HS = [8, 24, 40]


@pytest.mark.parametrize("H", HS)
@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_prefill_and_decode(dtype, H):
    p = wl.varlen_prefill(n_seqs=5, lo=1, hi=30, H=H, K=3, n_slots=9, seed=900 + H, dtype=dtype)
    for tile in (0, 8):
        pool = dev(p.pool, dtype)
        y = sc.prefill(dev(p.bcx, dtype), dev(p.w, dtype), dev(p.cu_seqlens, "i32"),
                       dev(p.slot_ids, "i32"), pool, rows_per_thread=tile)
        ref = p.pool.copy()
        st, y_ref = oracle.prefill(dtype, p.bcx, p.w, p.cu_seqlens, p.slot_ids, ref)
        assert st == oracle.OK
        assert_close(dtype, host(y), y_ref, f"prefill y, tile {tile}")
        assert_bits(host(pool), ref, f"prefill pool, tile {tile}")
    rng = np.random.default_rng(910 + H)
    bcx1 = wl.normal(rng, (len(p.slot_ids), 3 * H), 1.0, dtype)
    y = sc.decode(dev(bcx1, dtype), dev(p.w, dtype), dev(p.slot_ids, "i32"), pool)
    st, y_ref = oracle.decode(dtype, bcx1, p.w, p.slot_ids, ref)
    assert st == oracle.OK
    assert_close(dtype, host(y), y_ref, "decode y")
    assert_bits(host(pool), ref, "decode pool")
    assert sc.get_error() == 0


@pytest.mark.parametrize("H", HS)
@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_verify_and_rollback(dtype, H):
    s = wl.verify_serving(layers=1, batch=7, D=5, H=H, K=3, n_slots=11, seed=920 + H,
                          dtype=dtype)
    pool = dev(s.pools[0], dtype)
    win, y = sc.verify(dev(s.bcx[0], dtype), dev(s.w[0], dtype), dev(s.slot_ids, "i32"), pool,
                       s.D)
    st, win_ref, y_ref = oracle.verify(dtype, s.bcx[0], s.w[0], s.slot_ids, s.pools[0], s.D)
    assert st == oracle.OK
    assert_close(dtype, host(y), y_ref, "verify y")
    assert_bits(host(win), win_ref, "verify windows")
    sc.rollback(win, dev(s.accepted, "i32"), dev(s.slot_ids, "i32"), pool)
    ref = s.pools[0].copy()
    assert oracle.rollback(dtype, win_ref, s.accepted, s.slot_ids, ref) == oracle.OK
    assert_bits(host(pool), ref, "pool after rollback")
    assert sc.get_error() == 0


@pytest.mark.parametrize("H", HS)
@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_backward(dtype, H):
    t = wl.training(T=301, H=H, K=3, seed=930 + H, dtype=dtype)
    d, dw = sc.backward(dev(t.bcx, dtype), dev(t.w, dtype), dev(t.dy, dtype))
    st, d_ref, dw_ref = oracle.backward(dtype, t.bcx, t.w, t.dy)
    assert st == oracle.OK
    assert_close(dtype, host(d), d_ref, "dB|dC|dx")
    assert_dw_close(host(dw), dw_ref)
    assert sc.get_error() == 0
