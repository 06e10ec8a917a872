"""Device-resident data errors: the kernels flag them in the error word and skip
the bad unit; nothing traps. Invalid data is planted on the host and every
index the kernels compute stays inside the buffers passed."""
import numpy as np
import pytest
import torch

import oracle
import lfm2_gated_short_gb300 as sc
from lfm2_gated_short_gb300 import workloads as wl
from gpu_util import assert_bits, assert_close, dev, host

pytestmark = pytest.mark.gpu

FILL = 0x1234  # bf16 bit pattern pre-filled into outputs to see what was written


def filled(shape):
    return dev(np.full(shape, FILL, np.uint16), "bf16")


def test_error_word_starts_clear():
    assert sc.get_error() == 0


def test_prefill_bad_slot_skips_only_that_sequence():
    p = wl.varlen_prefill(n_seqs=4, H=64, K=3, n_slots=6, seed=100, lengths=[5, 9, 3, 7])
    slots = p.slot_ids.copy()
    slots[1] = 6                       # == n_slots
    pool = dev(p.pool, "bf16")
    y = filled((p.T, p.H))
    sc.prefill(dev(p.bcx, "bf16"), dev(p.w, "bf16"), dev(p.cu_seqlens, "i32"),
               dev(slots, "i32"), pool, y=y)
    assert sc.get_error() == sc.DEV_BAD_SLOT
    assert sc.get_error() == 0         # cleared by the read
    ref_pool = p.pool.copy()
    y_ref = np.full((p.T, p.H), FILL, np.uint16)
    st, y_ref = oracle.prefill("bf16", p.bcx, p.w, p.cu_seqlens, slots, ref_pool, y_ref)
    assert st == oracle.EDATA
    got = host(y)
    assert np.all(got[5:14] == FILL)
    keep = np.r_[0:5, 14:p.T]
    assert_close("bf16", got[keep], y_ref[keep], "other sequences")
    assert_bits(host(pool), ref_pool, "pool")


@pytest.mark.parametrize("cu", [[0, 3, 2, 9], [1, 3, 5, 9], [0, 3, 5, 8], [0, 3, 5, 10]])
def test_prefill_bad_seqlens_write_nothing(cu):
    p = wl.varlen_prefill(n_seqs=3, H=64, K=3, n_slots=4, seed=101, lengths=[3, 2, 4])
    pool = dev(p.pool, "bf16")
    y = filled((p.T, p.H))
    sc.prefill(dev(p.bcx, "bf16"), dev(p.w, "bf16"), dev(np.array(cu), "i32"),
               dev(p.slot_ids, "i32"), pool, y=y)
    assert sc.get_error() == sc.DEV_BAD_SEQLENS
    assert np.all(host(y) == FILL)
    assert_bits(host(pool), p.pool, "pool")


def test_decode_and_verify_bad_slot():
    s = wl.verify_serving(layers=1, batch=4, D=2, H=64, K=3, n_slots=5, seed=102)
    slots = s.slot_ids.copy()
    slots[2] = -1
    pool = dev(s.pools[0], "bf16")
    y = filled((4, 64))
    sc.decode(dev(s.bcx[0][:4], "bf16"), dev(s.w[0], "bf16"), dev(slots, "i32"), pool, y=y)
    assert sc.get_error() == sc.DEV_BAD_SLOT
    assert np.all(host(y)[2] == FILL) and not np.all(host(y)[1] == FILL)
    win = filled((4, 2, 64, 3))
    yv = filled((8, 64))
    sc.verify(dev(s.bcx[0], "bf16"), dev(s.w[0], "bf16"), dev(slots, "i32"), pool, 2, win, yv)
    assert sc.get_error() == sc.DEV_BAD_SLOT
    assert np.all(host(win)[2] == FILL) and np.all(host(yv)[4:6] == FILL)


def test_rollback_bad_accepted_and_slot():
    s = wl.verify_serving(layers=1, batch=4, D=3, H=64, K=3, n_slots=6, seed=103)
    pool = dev(s.pools[0], "bf16")
    win, _ = sc.verify(dev(s.bcx[0], "bf16"), dev(s.w[0], "bf16"), dev(s.slot_ids, "i32"),
                       pool, 3)
    slots = s.slot_ids.copy()
    slots[3] = 99
    acc = np.array([4, 2, -1, 1], np.int32)
    sc.rollback(win, dev(acc, "i32"), dev(slots, "i32"), pool)
    assert sc.get_error() == sc.DEV_BAD_ACCEPTED | sc.DEV_BAD_SLOT
    got = host(pool)
    w = host(win)
    assert_bits(got[s.slot_ids[1]], w[1, 1], "accepted sequence")
    for i in (0, 2, 3):
        assert_bits(got[s.slot_ids[i]], s.pools[0][s.slot_ids[i]], f"skipped sequence {i}")


def test_bounded_wait_gives_up_reports_a_timeout_and_leaves_the_device_usable():
    """The device-side timeout path, without any copy failing: a kernel waits,
    with the bounded wait every waiting kernel uses, on a barrier that
    nothing completes. It must give up after about the wait limit (2 s), set
    DEV_TIMEOUT, and leave the device computing correctly afterwards."""
    import time
    assert sc.get_error() == 0
    t0 = time.perf_counter()
    sc.check_wait_limit()
    code = sc.get_error()
    elapsed = time.perf_counter() - t0
    assert code == sc.DEV_TIMEOUT
    assert 1.5 < elapsed < 60, elapsed
    assert sc.get_error() == 0
    p = wl.varlen_prefill(n_seqs=3, H=64, K=3, n_slots=4, seed=102, lengths=[7, 1, 12])
    pool = dev(p.pool, "bf16")
    y = sc.prefill(dev(p.bcx, "bf16"), dev(p.w, "bf16"), dev(p.cu_seqlens, "i32"),
                   dev(p.slot_ids, "i32"), pool)
    ref = p.pool.copy()
    st, y_ref = oracle.prefill("bf16", p.bcx, p.w, p.cu_seqlens, p.slot_ids, ref)
    assert st == oracle.OK
    assert_close("bf16", host(y), y_ref, "prefill after the timeout check")
    assert_bits(host(pool), ref, "pool after the timeout check")
    assert sc.get_error() == 0
