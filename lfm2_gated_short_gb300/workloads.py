"""Seeded synthetic inputs for the ShortConv workloads.

This module only draws random numbers and lays them out; it holds none of
the convolution's arithmetic. The same arrays feed the CUDA path and the CPU
oracle. Storage conventions match the C ABI:

* ``"bf16"`` arrays are ``np.uint16`` bit patterns, drawn in float32 and
  cast to bfloat16 (round to nearest even) by torch's CPU cast;
* ``"f32"`` arrays are ``np.float32``;
* ``bcx`` is the in_proj output ``[T, 3H]`` laid out ``B | C | x`` per token;
  ``w`` is the depthwise conv weight ``[H, K]``; pools are ``[slots, H, K]``.

Shapes and distributions follow LFM2-1.2B's ShortConv layers (hidden 2048,
conv_L_cache 3, 10 conv layers): the LFM2-1.2B model card on the
inference-research site, and the conv weight layout ``[hidden, 1, K]`` of
the MAX LFM2 article's section on LFM2ShortConv.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

SENTINEL_BF16 = 0xDEAD          # bit pattern of never-touched pool slots (bf16)
SENTINEL_F32 = 0xDEADBEEF       # bit pattern of never-touched pool slots (f32)

WEIGHT_STD = (1.0 / 3.0) ** 0.5  # conv weight ~ N(0, 1/3): variance 1/3


def _cast(a32: np.ndarray, dtype: str) -> np.ndarray:
    if dtype == "f32":
        return np.ascontiguousarray(a32, dtype=np.float32)
    if dtype == "bf16":
        import torch  # the float32 -> bfloat16 cast only
        t = torch.from_numpy(np.ascontiguousarray(a32, dtype=np.float32))
        return t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16).copy()
    raise ValueError(f"unsupported dtype {dtype!r}")


def normal(rng: np.random.Generator, shape, std: float = 1.0, dtype: str = "bf16"):
    """Draw N(0, std^2) in float32 and store it as ``dtype``."""
    a = rng.standard_normal(size=shape, dtype=np.float32)
    if std != 1.0:
        a *= np.float32(std)
    return _cast(a, dtype)


def zeros(shape, dtype: str):
    return np.zeros(shape, dtype=np.uint16 if dtype == "bf16" else np.float32)


def sentinel(shape, dtype: str):
    if dtype == "bf16":
        return np.full(shape, SENTINEL_BF16, dtype=np.uint16)
    return np.full(shape, SENTINEL_F32, dtype=np.uint32).view(np.float32)


@dataclass
class PrefillProblem:
    dtype: str
    H: int
    K: int
    bcx: np.ndarray          # [T, 3H]
    w: np.ndarray            # [H, K]
    cu_seqlens: np.ndarray   # int32 [N + 1]
    slot_ids: np.ndarray     # int32 [N]
    pool: np.ndarray         # [n_slots, H, K]
    decode_bcx: np.ndarray | None = None   # [steps, N, 3H] follow-up decode rows

    @property
    def T(self) -> int:
        return int(self.bcx.shape[0])

    @property
    def N(self) -> int:
        return int(self.slot_ids.shape[0])


@dataclass
class ServingProblem:
    """Several conv layers sharing one slot mapping (decode or verify)."""
    dtype: str
    H: int
    K: int
    w: np.ndarray            # [layers, H, K]
    pools: np.ndarray        # [layers, n_slots, H, K]
    slot_ids: np.ndarray     # int32 [N]
    bcx: np.ndarray          # decode: [layers, steps, N, 3H]; verify: [layers, N*D, 3H]
    D: int = 1
    accepted: np.ndarray | None = None     # verify: int32 [N] in 0..D
    extra: dict = field(default_factory=dict)


@dataclass
class TrainingProblem:
    dtype: str
    H: int
    K: int
    bcx: np.ndarray          # [T, 3H]
    w: np.ndarray            # [H, K]
    dy: np.ndarray           # [T, H]


def tiny_fp32(seed: int = 1, H: int = 64, K: int = 3, T: int = 16,
              decode_steps: int = 4) -> PrefillProblem:
    """One fp32 sequence, H=64, K=3, T=16, zero state, then 4 decode tokens."""
    rng = np.random.default_rng(seed)
    bcx = normal(rng, (T, 3 * H), 1.0, "f32")
    w = normal(rng, (H, K), WEIGHT_STD, "f32")
    dec = normal(rng, (decode_steps, 1, 3 * H), 1.0, "f32")
    return PrefillProblem("f32", H, K, bcx, w, np.array([0, T], np.int32),
                          np.array([0], np.int32), zeros((1, H, K), "f32"), dec)


def single_prefill(T: int = 4096, H: int = 2048, K: int = 3, seed: int = 2,
                   dtype: str = "bf16") -> PrefillProblem:
    """One sequence of T tokens from a zero state written to slot 0 of a 1-slot pool."""
    rng = np.random.default_rng(seed)
    bcx = normal(rng, (T, 3 * H), 1.0, dtype)
    w = normal(rng, (H, K), WEIGHT_STD, dtype)
    return PrefillProblem(dtype, H, K, bcx, w, np.array([0, T], np.int32),
                          np.array([0], np.int32), zeros((1, H, K), dtype))


def varlen_prefill(n_seqs: int = 16, lo: int = 64, hi: int = 2048, H: int = 2048,
                   K: int = 3, n_slots: int = 1024, seed: int = 3,
                   dtype: str = "bf16", lengths=None) -> PrefillProblem:
    """Packed sequences with integer lengths uniform in [lo, hi] (inclusive).

    Each sequence gets a distinct random slot. Half of them (chosen at random)
    continue from an N(0, 1) state, the rest start from zeros; every other
    slot holds a sentinel bit pattern so that stray writes are visible.
    """
    rng = np.random.default_rng(seed)
    if lengths is None:
        lengths = rng.integers(lo, hi, size=n_seqs, endpoint=True)
    lengths = np.asarray(lengths, dtype=np.int64)
    n_seqs = len(lengths)
    cu = np.zeros(n_seqs + 1, np.int32)
    cu[1:] = np.cumsum(lengths)
    slots = rng.permutation(n_slots)[:n_seqs].astype(np.int32)
    pool = sentinel((n_slots, H, K), dtype)
    warm = rng.permutation(n_seqs)[: n_seqs // 2]
    for i in range(n_seqs):
        pool[slots[i]] = zeros((H, K), dtype)
    for i in warm:
        pool[slots[i]] = normal(rng, (H, K), 1.0, dtype)
    bcx = normal(rng, (int(cu[-1]), 3 * H), 1.0, dtype)
    w = normal(rng, (H, K), WEIGHT_STD, dtype)
    return PrefillProblem(dtype, H, K, bcx, w, cu, slots, pool)


def decode_serving(layers: int = 10, steps: int = 64, batch: int = 256,
                   H: int = 2048, K: int = 3, n_slots: int = 1024, seed: int = 4,
                   dtype: str = "bf16") -> ServingProblem:
    """Decode: ``batch`` sequences, one token each per step, per-layer pools ~ N(0, 1)."""
    rng = np.random.default_rng(seed)
    slots = rng.permutation(n_slots)[:batch].astype(np.int32)
    w = normal(rng, (layers, H, K), WEIGHT_STD, dtype)
    pools = normal(rng, (layers, n_slots, H, K), 1.0, dtype)
    bcx = normal(rng, (layers, steps, batch, 3 * H), 1.0, dtype)
    return ServingProblem(dtype, H, K, w, pools, slots, bcx)


def verify_serving(layers: int = 10, batch: int = 64, D: int = 8, H: int = 2048,
                   K: int = 3, n_slots: int = 1024, seed: int = 5,
                   dtype: str = "bf16") -> ServingProblem:
    """Speculative verify: ``batch`` sequences x ``D`` drafts, accepted ~ U{0..D}."""
    rng = np.random.default_rng(seed)
    slots = rng.permutation(n_slots)[:batch].astype(np.int32)
    w = normal(rng, (layers, H, K), WEIGHT_STD, dtype)
    pools = normal(rng, (layers, n_slots, H, K), 1.0, dtype)
    bcx = normal(rng, (layers, batch * D, 3 * H), 1.0, dtype)
    accepted = rng.integers(0, D, size=batch, endpoint=True).astype(np.int32)
    return ServingProblem(dtype, H, K, w, pools, slots, bcx, D=D, accepted=accepted)


def training(T: int = 65536, H: int = 2048, K: int = 3, seed: int = 6,
             dtype: str = "bf16") -> TrainingProblem:
    """One long sequence from a zero state with an upstream gradient dy ~ N(0, 1)."""
    rng = np.random.default_rng(seed)
    bcx = normal(rng, (T, 3 * H), 1.0, dtype)
    w = normal(rng, (H, K), WEIGHT_STD, dtype)
    dy = normal(rng, (T, H), 1.0, dtype)
    return TrainingProblem(dtype, H, K, bcx, w, dy)
