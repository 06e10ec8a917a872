"""Device slot pool (claim, release, copy) against the reference model."""
import numpy as np
import pytest
import torch

import lfm2_gated_short_gb300 as sc
from lfm2_gated_short_gb300 import workloads as wl
from oracle import slots as model
from gpu_util import assert_bits, dev, host

pytestmark = pytest.mark.gpu


def bitmap_dev(bm):
    return torch.from_numpy(bm.view(np.int32).copy()).cuda()


def bitmap_host(t):
    return host(t).view(np.uint32)


def random_bitmap(rng, n_slots, frac):
    bm = np.zeros(model.words(n_slots), np.uint32)
    for s in np.nonzero(rng.random(n_slots) < frac)[0]:
        bm[s // 32] |= np.uint32(1 << (int(s) % 32))
    if n_slots % 32:  # bits past n_slots are ignored and must be kept
        bm[-1] |= np.uint32(0xFFFFFFFF << (n_slots % 32) & 0xFFFFFFFF)
    return bm


@pytest.mark.parametrize("n_slots,frac", [(1, 0.0), (33, 0.5), (1024, 0.3), (1000, 0.9),
                                          (100003, 0.5)])
def test_claim_matches_the_model(n_slots, frac):
    rng = np.random.default_rng(n_slots)
    bm = random_bitmap(rng, n_slots, frac)
    n_free = int((~model.in_use(bm, n_slots)).sum())
    k = max(0, n_free // 3)
    pool = wl.normal(rng, (n_slots, 8, 3), 1.0, "bf16")
    d_bm, d_pool = bitmap_dev(bm), dev(pool, "bf16")
    got = sc.slots_claim(d_bm, n_slots, k, pool=d_pool)
    err, ref = model.claim(bm, n_slots, k, pool)
    assert err == model.OK and sc.get_error() == 0
    assert_bits(host(got), ref, "slots")
    assert_bits(bitmap_host(d_bm), bm, "bitmap")
    assert_bits(host(d_pool), pool, "pool")


def test_claim_more_than_free_claims_nothing():
    rng = np.random.default_rng(5)
    bm = random_bitmap(rng, 300, 0.8)
    n_free = int((~model.in_use(bm, 300)).sum())
    d_bm = bitmap_dev(bm)
    got = sc.slots_claim(d_bm, 300, n_free + 1)
    assert sc.get_error() == sc.DEV_NO_SLOT
    assert np.all(host(got) == -1)
    assert_bits(bitmap_host(d_bm), bm, "bitmap unchanged")


def test_release_matches_the_model_and_flags_bad_ids():
    rng = np.random.default_rng(6)
    bm = random_bitmap(rng, 500, 0.5)
    used = np.nonzero(model.in_use(bm, 500))[0]
    rel = np.r_[rng.choice(used, 40, replace=False), [500, -3]].astype(np.int32)
    free_one = int(np.nonzero(~model.in_use(bm, 500))[0][0])
    rel = np.r_[rel, free_one].astype(np.int32)
    d_bm = bitmap_dev(bm)
    sc.slots_release(d_bm, 500, dev(rel, "i32"))
    err = model.release(bm, 500, rel)
    assert err == model.BAD_SLOT
    assert sc.get_error() == sc.DEV_BAD_SLOT
    assert_bits(bitmap_host(d_bm), bm, "bitmap")


def test_pool_copy_matches_the_model():
    rng = np.random.default_rng(7)
    pool = wl.normal(rng, (64, 128, 3), 1.0, "bf16")
    perm = rng.permutation(64)
    src, dst = perm[:10].astype(np.int32), perm[10:20].astype(np.int32)
    d_pool = dev(pool, "bf16")
    sc.pool_copy(d_pool, dev(src, "i32"), dev(dst, "i32"))
    assert model.copy(pool, src, dst) == model.OK
    assert sc.get_error() == 0
    assert_bits(host(d_pool), pool, "pool")


def test_serving_cycle_reclaims_zeroed_slots():
    """Claim slots, prefill and decode on them, release, claim again: the same
    slots come back and start from zero states."""
    rng = np.random.default_rng(8)
    n_slots, H, K = 96, 256, 3
    d_bm = sc.slot_bitmap(n_slots)
    pool = torch.zeros((n_slots, H, K), dtype=torch.bfloat16, device="cuda")
    slots = sc.slots_claim(d_bm, n_slots, 5, pool=pool)
    assert host(slots).tolist() == [0, 1, 2, 3, 4]
    p = wl.varlen_prefill(n_seqs=5, lo=3, hi=40, H=H, K=K, n_slots=n_slots, seed=9)
    sc.prefill(dev(p.bcx, "bf16"), dev(p.w, "bf16"), dev(p.cu_seqlens, "i32"), slots, pool)
    sc.decode(dev(p.bcx[:5], "bf16"), dev(p.w, "bf16"), slots, pool)
    assert host(pool)[:5].any()
    sc.slots_release(d_bm, n_slots, slots[1:4].contiguous())
    again = sc.slots_claim(d_bm, n_slots, 4, pool=pool)
    assert host(again).tolist() == [1, 2, 3, 5]
    assert not host(pool)[[1, 2, 3, 5]].any()
    assert host(pool)[[0, 4]].any()
    assert sc.get_error() == 0
