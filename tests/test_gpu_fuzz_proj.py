"""Seeded random sweeps of the projection calls against the layer oracle.

Each case draws D and H (multiples of 64; H % 128 == 64 leaves the fused
call's last 128-channel tile half full), K in 1..4, an optional conv bias and
a sequence structure: 1-12 sequences mixing empty, shorter-than-K and long
ones, each continued from a random state in a random slot of a pool whose
other slots hold a sentinel. Inputs are dyadic (small integers times powers of
two), so every projection sum is exact in fp32 whatever the order of
accumulation. The fused in_proj + ShortConv must then give the slots' new
states bit for bit and y within the bf16 tolerance; out_proj (output width a
multiple of 256) must give the oracle's bits; the fused decode step is checked
like the fused prefill, one token per sequence.
"""
import numpy as np
import pytest

import oracle
from oracle import layer
import lfm2_gated_short_gb300 as sc
from gpu_util import assert_bits, assert_close, dev, host

pytestmark = pytest.mark.gpu

CASES = 24
SENTINEL = 0xDEAD  # slots no call names keep this pattern


def dyadic(rng, shape, lim, exp):
    """Integers in [-lim, lim] times 2**exp, as bf16 bits (exact): with the
    scales below, every product is a multiple of 2**-9 and every sum of up to
    4096 of them is exact in fp32."""
    return oracle.round_bf16(rng.integers(-lim, lim, size=shape, endpoint=True) * 2.0 ** exp)


def draw(seed):
    rng = np.random.default_rng(5000 + seed)
    D = 64 * int(rng.integers(1, 17))
    H = 64 * int(rng.integers(1, 13))
    K = int(rng.integers(1, 5))
    n = int(rng.integers(1, 13))
    short = rng.integers(0, 3 * K + 1, size=n)  # empty, shorter than K, a few windows
    long = rng.integers(K, 700, size=n)
    lengths = [int(v) for v in np.where(rng.random(n) < 0.5, long, short)]
    bias = oracle.round_bf16(rng.standard_normal(H) * 0.5) if rng.random() < 0.3 else None
    return rng, D, H, K, lengths, bias


def pool_with_states(rng, n_slots, slots, H, K):
    pool = np.full((n_slots, H, K), SENTINEL, np.uint16)
    for s in slots:
        pool[s] = oracle.round_bf16(rng.standard_normal((H, K)))
    return pool


def taps(rng, H, K):
    return oracle.round_bf16(rng.standard_normal((H, K)) * np.sqrt(1 / 3))


@pytest.mark.parametrize("seed", range(CASES))
def test_in_proj_prefill_then_out_proj(seed):
    rng, D, H, K, lengths, bias = draw(seed)
    cu = np.r_[0, np.cumsum(lengths)].astype(np.int32)
    T, N = int(cu[-1]), len(lengths)
    hidden = dyadic(rng, (T, D), 8, -3)
    w_in = dyadic(rng, (3 * H, D), 8, -6)
    w = taps(rng, H, K)
    n_slots = N + int(rng.integers(0, 6))
    slots = rng.permutation(n_slots)[:N].astype(np.int32)
    pool0 = pool_with_states(rng, n_slots, slots, H, K)

    pool = dev(pool0, "bf16")
    y = sc.in_proj_prefill(dev(hidden, "bf16"), dev(w_in, "bf16"), dev(w, "bf16"),
                           dev(cu, "i32"), dev(slots, "i32"), pool,
                           bias=None if bias is None else dev(bias, "bf16"))
    ref = pool0.copy()
    st, y_ref = layer.in_proj_prefill("bf16", hidden, w_in, w, cu, slots, ref, bias=bias)
    assert st == oracle.OK
    assert sc.get_error() == 0
    case = f"seed {seed}: D={D} H={H} K={K} lengths={lengths} bias={bias is not None}"
    assert_bits(host(pool), ref, f"pool, {case}")
    assert_close("bf16", host(y), y_ref, f"y, {case}")

    if T == 0:
        return
    Dout = 256 * int(rng.integers(1, 5))
    y_in = dyadic(rng, (T, H), 8, -3)
    w_out = dyadic(rng, (Dout, H), 8, -6)
    out = sc.out_proj(dev(y_in, "bf16"), dev(w_out, "bf16"))
    assert_bits(host(out), layer.out_proj("bf16", y_in, w_out), f"out_proj D={Dout}, {case}")
    assert sc.get_error() == 0


@pytest.mark.parametrize("seed", range(CASES))
def test_in_proj_decode(seed):
    rng, D, H, K, _, bias = draw(100 + seed)
    N = int(rng.integers(1, 300))
    hidden = dyadic(rng, (N, D), 8, -3)
    w_in = dyadic(rng, (3 * H, D), 8, -6)
    w = taps(rng, H, K)
    n_slots = N + int(rng.integers(0, 6))
    slots = rng.permutation(n_slots)[:N].astype(np.int32)
    pool0 = pool_with_states(rng, n_slots, slots, H, K)

    pool = dev(pool0, "bf16")
    y = sc.in_proj_decode(dev(hidden, "bf16"), dev(w_in, "bf16"), dev(w, "bf16"),
                          dev(slots, "i32"), pool,
                          bias=None if bias is None else dev(bias, "bf16"))
    ref = pool0.copy()
    st, y_ref = layer.in_proj_decode("bf16", hidden, w_in, w, slots, ref, bias=bias)
    assert st == oracle.OK
    assert sc.get_error() == 0
    case = f"seed {seed}: N={N} D={D} H={H} K={K} bias={bias is not None}"
    assert_bits(host(pool), ref, f"pool, {case}")
    assert_close("bf16", host(y), y_ref, f"y, {case}")
