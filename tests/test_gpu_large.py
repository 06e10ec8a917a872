"""Inputs past 32-bit element offsets, checked against the oracle.

T = 400,000 tokens at H = 2048 puts 2.46e9 elements (4.9 GB of bf16) in
``bcx``, past what a 32-bit element index reaches. The kernels compute row
and slot offsets in 64 bits, and these tests cover them at those offsets.

The oracle only runs where it is cheap. Channels are independent in the
ShortConv, so for prefill, decode and backward it runs on a subset of
channels over every row. The subset is the first 32 channels and the last
64, which sit at the highest addresses. The projections mix channels, so for
them the oracle runs on rows: the first rows of a sequence, which start from
its slot state, and the last rows with K-1 rows of history before them.

Inputs are drawn on the device by torch's seeded generator and copied to the
host for the oracle.
"""
import numpy as np
import pytest
import torch

import oracle
from oracle import layer
import lfm2_gated_short_gb300 as sc
from gpu_util import assert_bits, assert_close, assert_dw_close, host

pytestmark = pytest.mark.gpu

T_BIG, H, K = 400_000, 2048, 3
CH = np.r_[0:32, H - 64:H]
CU = np.array([0, 150_000, T_BIG], np.int32)  # two sequences; the second ends at T_BIG


def gen(shape, seed, std=1.0):
    g = torch.Generator(device="cuda").manual_seed(seed)
    return (torch.randn(shape, generator=g, device="cuda") * std).to(torch.bfloat16)


def dyadic(shape, seed, lim, exp):
    """Integers in [-lim, lim] times 2**exp in bf16 (exact), on the device."""
    g = torch.Generator(device="cuda").manual_seed(seed)
    v = torch.randint(-lim, lim + 1, shape, generator=g, device="cuda", dtype=torch.int32)
    return (v.to(torch.float32) * 2.0 ** exp).to(torch.bfloat16)


def i32(a):
    return torch.as_tensor(np.asarray(a, np.int32), device="cuda")


def bcx_cols(bcx, ch):
    """B|C|x columns of the channels ``ch``, on the host: [rows, 3 len(ch)]."""
    idx = torch.as_tensor(np.r_[ch, H + ch, 2 * H + ch], device=bcx.device)
    return host(bcx.index_select(1, idx))


def chan(t, ch, dim=1):
    return host(t.index_select(dim, torch.as_tensor(ch, device=t.device)))


@pytest.fixture(scope="module")
def big():
    assert T_BIG * 3 * H > 2 ** 31
    bcx = gen((T_BIG, 3 * H), 1)
    w = gen((H, K), 2, std=np.sqrt(1 / 3))
    return bcx, w


@pytest.mark.parametrize("tile", [0, 8])
def test_prefill_past_32bit_offsets(big, tile):
    bcx, w = big
    slots = np.array([3, 1], np.int32)
    pool0 = gen((5, H, K), 3)
    pool = pool0.clone()
    y = sc.prefill(bcx, w, i32(CU), i32(slots), pool, rows_per_thread=tile)
    ref_pool = np.ascontiguousarray(chan(pool0, CH))
    st, y_ref = oracle.prefill("bf16", bcx_cols(bcx, CH), chan(w, CH, 0), CU, slots, ref_pool)
    assert st == oracle.OK
    assert sc.get_error() == 0
    assert_close("bf16", chan(y, CH), y_ref, "y")
    assert_bits(chan(pool, CH), ref_pool, "pool")
    del y, pool


def test_backward_past_32bit_offsets(big):
    bcx, w = big
    dy = gen((T_BIG, H), 4)
    dbcx, dw = sc.backward(bcx, w, dy)
    cols = np.r_[CH, H + CH, 2 * H + CH]
    st, d_ref, dw_ref = oracle.backward("bf16", bcx_cols(bcx, CH), chan(w, CH, 0), chan(dy, CH))
    assert st == oracle.OK
    assert sc.get_error() == 0
    assert_close("bf16", chan(dbcx, cols), d_ref, "dB|dC|dx")
    assert_dw_close(host(dw)[CH], dw_ref)
    del dbcx, dy


def test_backward_varlen_past_32bit_offsets(big):
    bcx, w = big
    dy = gen((T_BIG, H), 5)
    init = gen((2, H, K), 6)
    g = torch.Generator(device="cuda").manual_seed(7)
    dfin = torch.randn((2, H, K), generator=g, device="cuda")
    dbcx, dw, dinit = sc.backward_varlen(bcx, w, i32(CU), dy, init_states=init, d_final=dfin)
    cols = np.r_[CH, H + CH, 2 * H + CH]
    st, d_ref, dw_ref, di_ref = oracle.backward_varlen(
        "bf16", bcx_cols(bcx, CH), chan(w, CH, 0), CU, chan(dy, CH),
        np.ascontiguousarray(chan(init, CH)), chan(dfin, CH).astype(np.float64))
    assert st == oracle.OK
    assert sc.get_error() == 0
    assert_close("bf16", chan(dbcx, cols), d_ref, "dB|dC|dx")
    assert_dw_close(host(dw)[CH], dw_ref)
    assert_dw_close(chan(dinit, CH), di_ref, "d_init")
    del dbcx, dy


def test_decode_with_pool_offsets_past_32_bits():
    """400,000 sequences in a 400,000-slot pool: slot offsets reach 2.46e9 elements."""
    n = T_BIG
    rng = np.random.default_rng(11)
    slots = rng.permutation(n).astype(np.int32)
    bcx = gen((n, 3 * H), 12)
    w = gen((H, K), 13, std=np.sqrt(1 / 3))
    pool = gen((n, H, K), 14)
    ref_pool = np.ascontiguousarray(chan(pool, CH))
    y = sc.decode(bcx, w, i32(slots), pool)
    st, y_ref = oracle.decode("bf16", bcx_cols(bcx, CH), chan(w, CH, 0), slots, ref_pool)
    assert st == oracle.OK
    assert sc.get_error() == 0
    assert_close("bf16", chan(y, CH), y_ref, "y")
    assert_bits(chan(pool, CH), ref_pool, "pool")
    del bcx, pool, y


def test_in_proj_prefill_and_out_proj_past_32bit_offsets():
    """The fused in_proj + ShortConv and out_proj at T = 400,000, D = H = 2048.

    Dyadic inputs keep the projection exact in any summation order (see the
    projection tests), so states match bit for bit. The oracle runs on the
    second sequence's first rows (from its slot state) and on its last rows
    (with K-1 rows of history, from a zero state: those rows' windows lie
    inside the slice)."""
    D, R = 2048, 130
    hidden = dyadic((T_BIG, D), 21, 8, -3)
    w_in = dyadic((3 * H, D), 22, 8, -6)
    w = gen((H, K), 23, std=np.sqrt(1 / 3))
    slots = np.array([2, 0], np.int32)
    pool0 = gen((3, H, K), 24)
    pool = pool0.clone()
    y = sc.in_proj_prefill(hidden, w_in, w, i32(CU), i32(slots), pool)
    assert sc.get_error() == 0
    h_w_in, h_w = host(w_in), host(w)
    s0 = int(CU[1])
    # first rows of sequence 1, from its slot state (the pool before the call)
    st_pool = np.ascontiguousarray(host(pool0)[slots[1]][None])
    st, y_ref = layer.in_proj_prefill("bf16", host(hidden[s0:s0 + R]), h_w_in, h_w, [0, R],
                                      [0], st_pool)
    assert st == oracle.OK
    assert_close("bf16", host(y[s0:s0 + R]), y_ref, "y, first rows of sequence 1")
    # last rows, with K-1 rows of history; the slice's final state is the sequence's
    a = T_BIG - R - (K - 1)
    z_pool = np.zeros((1, H, K), np.uint16)
    st, y_ref = layer.in_proj_prefill("bf16", host(hidden[a:]), h_w_in, h_w, [0, T_BIG - a],
                                      [0], z_pool)
    assert st == oracle.OK
    assert_close("bf16", host(y[T_BIG - R:]), y_ref[K - 1:], "y, last rows")
    assert_bits(host(pool)[slots[1]], z_pool[0], "final state of sequence 1")
    del y
    # out_proj over the same rows (dyadic input, so exact): the last R rows
    w_out = dyadic((D, H), 25, 8, -6)
    out = sc.out_proj(hidden, w_out)
    assert sc.get_error() == 0
    assert_bits(host(out[T_BIG - R:]), layer.out_proj("bf16", host(hidden[T_BIG - R:]),
                                                      host(w_out)), "out_proj, last rows")
    del out, hidden
