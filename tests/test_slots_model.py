"""Pins for the slot-pool reference model (oracle/slots.py): properties that
any correct allocator of the MAX ConvStateCache kind must have."""
import numpy as np

from oracle import slots as model


def _random_bitmap(rng, n_slots, frac):
    used = rng.random(n_slots) < frac
    bm = np.zeros(model.words(n_slots), np.uint32)
    for s in np.nonzero(used)[0]:
        bm[s // 32] |= np.uint32(1 << (int(s) % 32))
    return bm, used


def test_claim_takes_the_lowest_free_slots_and_marks_them():
    rng = np.random.default_rng(1)
    for n_slots in (1, 31, 32, 33, 100, 1024):
        bm, used = _random_bitmap(rng, n_slots, 0.4)
        free = np.nonzero(~used)[0]
        k = len(free) // 2
        before = bm.copy()
        err, got = model.claim(bm, n_slots, k)
        assert err == model.OK
        np.testing.assert_array_equal(got, free[:k])
        now = model.in_use(bm, n_slots)
        assert now[got].all() and len(set(got.tolist())) == k
        untouched = np.setdiff1d(np.arange(n_slots), got)
        np.testing.assert_array_equal(now[untouched], model.in_use(before, n_slots)[untouched])


def test_claim_is_all_or_nothing():
    rng = np.random.default_rng(2)
    bm, used = _random_bitmap(rng, 70, 0.7)
    before = bm.copy()
    err, got = model.claim(bm, 70, int((~used).sum()) + 1)
    assert err == model.NO_SLOT and np.all(got == -1)
    np.testing.assert_array_equal(bm, before)


def test_claim_zeroes_only_the_claimed_states():
    rng = np.random.default_rng(3)
    pool = rng.standard_normal((40, 8, 3))
    bm, _ = _random_bitmap(rng, 40, 0.5)
    ref = pool.copy()
    err, got = model.claim(bm, 40, 5, pool)
    assert err == model.OK
    assert np.all(pool[got] == 0)
    rest = np.setdiff1d(np.arange(40), got)
    np.testing.assert_array_equal(pool[rest], ref[rest])


def test_claim_then_release_restores_the_bitmap():
    rng = np.random.default_rng(4)
    bm, _ = _random_bitmap(rng, 200, 0.3)
    before = bm.copy()
    err, got = model.claim(bm, 200, 50)
    assert err == model.OK
    assert model.release(bm, 200, got[::-1]) == model.OK
    np.testing.assert_array_equal(bm, before)


def test_release_flags_free_and_out_of_range_slots_but_releases_the_rest():
    bm = np.zeros(model.words(64), np.uint32)
    err, got = model.claim(bm, 64, 4)
    assert got.tolist() == [0, 1, 2, 3]
    err = model.release(bm, 64, [1, 1, 64, -1, 3])
    assert err == model.BAD_SLOT
    assert model.in_use(bm, 64)[:5].tolist() == [True, False, True, False, False]


def test_copy_reads_the_states_before_the_call():
    rng = np.random.default_rng(5)
    pool = rng.standard_normal((6, 4, 3))
    ref = pool.copy()
    assert model.copy(pool, [0, 1], [1, 2]) == model.OK     # 1 gets old 0, 2 gets old 1
    np.testing.assert_array_equal(pool[1], ref[0])
    np.testing.assert_array_equal(pool[2], ref[1])
    assert model.copy(pool, [0, 9], [5, 4]) == model.BAD_SLOT
    np.testing.assert_array_equal(pool[5], ref[0])
    np.testing.assert_array_equal(pool[4], ref[4])
