"""Reference model of the conv-state slot pool -- TEST INFRASTRUCTURE.

Only tests may import this module. It restates, in plain Python, the
slot-pool life cycle of the MAX LFM2 article ("MAX Pipelines 的 LFM2 架构支持",
section "推理状态管理：ConvStateCache 与卷积状态生命周期"): a request claims a
free slot (an error when none is free), the slot starts from a zero state,
the request releases it when done; and a slot's state can be copied to
another slot (a snapshot, for reusing a shared prefix's state).

Readings where the article leaves the rule open:
* claims are all-or-nothing: a request for more slots than are free claims
  none, sets every output to -1 and reports the error;
* the k requested slots are the k lowest-numbered free slots, in increasing
  order (one deterministic choice among the valid ones);
* releasing a slot that is out of range or not in use is an error and
  changes nothing for that entry; the other entries are still released;
* a copy whose source or destination is out of range is skipped (error).

The in-use set is a bitmap of (n_slots + 31) // 32 uint32 words, bit j of
word s // 32 set when slot s is in use; bits past n_slots are ignored.
"""
from __future__ import annotations

import numpy as np

OK, BAD_SLOT, NO_SLOT = 0, 0x1, 0x10


def words(n_slots: int) -> int:
    return (n_slots + 31) // 32


def in_use(bitmap: np.ndarray, n_slots: int) -> np.ndarray:
    """Boolean [n_slots] view of the bitmap."""
    b = np.asarray(bitmap, dtype=np.uint32)
    return np.array([(int(b[s // 32]) >> (s % 32)) & 1 == 1 for s in range(n_slots)], bool)


def claim(bitmap: np.ndarray, n_slots: int, n_claim: int, pool=None):
    """Claim n_claim slots in place; returns (error bits, slots int32 [n_claim])."""
    used = in_use(bitmap, n_slots)
    free = [s for s in range(n_slots) if not used[s]]
    if len(free) < n_claim:
        return NO_SLOT, np.full(n_claim, -1, np.int32)
    got = np.array(free[:n_claim], np.int32)
    for s in got:
        bitmap[s // 32] = np.uint32(int(bitmap[s // 32]) | (1 << (int(s) % 32)))
        if pool is not None:
            pool[s] = 0
    return OK, got


def release(bitmap: np.ndarray, n_slots: int, slot_ids) -> int:
    """Release slots in place; returns the error bits."""
    err = OK
    for s in np.asarray(slot_ids, np.int64):
        if s < 0 or s >= n_slots or not (int(bitmap[s // 32]) >> (int(s) % 32)) & 1:
            err |= BAD_SLOT
            continue
        bitmap[s // 32] = np.uint32(int(bitmap[s // 32]) & ~(1 << (int(s) % 32)) & 0xFFFFFFFF)
    return err


def copy(pool: np.ndarray, src, dst) -> int:
    """pool[dst[i]] = pool[src[i]] (values as before the call); returns the error bits."""
    n_slots = pool.shape[0]
    before = pool.copy()
    err = OK
    for s, d in zip(np.asarray(src, np.int64), np.asarray(dst, np.int64)):
        if not (0 <= s < n_slots and 0 <= d < n_slots):
            err |= BAD_SLOT
            continue
        pool[d] = before[s]
    return err
