"""Degenerate calls on the GPU: zero rows, zero sequences, only empty sequences.

An empty sequence extends its slot's window by nothing, so its final state
is the state it started from. A backward over zero rows has dW = 0 and
dbias = 0, the empty sums. With only empty sequences, each initial state
passes straight through to the final state, so d_init = d_final. Calls with
nothing to do succeed and write nothing. The outputs that are
written (dW, dbias, d_init) start as NaN here, so a missing write shows.
Where the oracle defines the result it is run on the same inputs.
"""
import numpy as np
import pytest
import torch

import oracle
from oracle import layer
import lfm2_gated_short_gb300 as sc
from gpu_util import assert_bits, assert_dw_close, dev, host

pytestmark = pytest.mark.gpu

H, K = 128, 3


def rand_bf16(rng, shape):
    return oracle.round_bf16(rng.standard_normal(shape))


@pytest.mark.parametrize("tile", [0, 8])
def test_prefill_with_only_empty_sequences_keeps_every_state(tile):
    rng = np.random.default_rng(50)
    pool0 = rand_bf16(rng, (5, H, K))
    w = rand_bf16(rng, (H, K))
    cu, slots = np.zeros(4, np.int32), np.array([2, 0, 4], np.int32)
    bcx = np.zeros((0, 3 * H), np.uint16)
    ref = pool0.copy()
    st, y_ref = oracle.prefill("bf16", bcx, w, cu, slots, ref)
    assert st == oracle.OK and y_ref.shape == (0, H)
    assert_bits(ref, pool0, "oracle: states unchanged")
    pool = dev(pool0, "bf16")
    y = sc.prefill(dev(bcx, "bf16"), dev(w, "bf16"), dev(cu, "i32"), dev(slots, "i32"), pool,
                   rows_per_thread=tile)
    assert tuple(y.shape) == (0, H)
    assert sc.get_error() == 0
    assert_bits(host(pool), pool0, "states")


def test_in_proj_prefill_with_only_empty_sequences_keeps_every_state():
    rng = np.random.default_rng(51)
    D = 128
    pool0 = rand_bf16(rng, (3, H, K))
    w = rand_bf16(rng, (H, K))
    w_in = rand_bf16(rng, (3 * H, D))
    cu, slots = np.zeros(3, np.int32), np.array([1, 2], np.int32)
    hidden = np.zeros((0, D), np.uint16)
    ref = pool0.copy()
    st, y_ref = layer.in_proj_prefill("bf16", hidden, w_in, w, cu, slots, ref)
    assert st == oracle.OK and y_ref.shape == (0, H)
    pool = dev(pool0, "bf16")
    y = sc.in_proj_prefill(dev(hidden, "bf16"), dev(w_in, "bf16"), dev(w, "bf16"),
                           dev(cu, "i32"), dev(slots, "i32"), pool)
    assert tuple(y.shape) == (0, H)
    assert sc.get_error() == 0
    assert_bits(host(pool), pool0, "states")


def test_out_proj_of_zero_rows():
    w_out = torch.zeros((256, H), dtype=torch.bfloat16, device="cuda")
    out = sc.out_proj(torch.zeros((0, H), dtype=torch.bfloat16, device="cuda"), w_out)
    assert tuple(out.shape) == (0, 256)
    assert sc.get_error() == 0


def test_decode_verify_rollback_with_no_sequences():
    rng = np.random.default_rng(52)
    pool0 = rand_bf16(rng, (4, H, K))
    pool = dev(pool0, "bf16")
    w = dev(rand_bf16(rng, (H, K)), "bf16")
    none = torch.zeros((0,), dtype=torch.int32, device="cuda")
    rows = torch.zeros((0, 3 * H), dtype=torch.bfloat16, device="cuda")
    y = sc.decode(rows, w, none, pool)
    assert tuple(y.shape) == (0, H)
    win, y = sc.verify(rows, w, none, pool, 4)
    assert tuple(win.shape) == (0, 4, H, K) and tuple(y.shape) == (0, H)
    sc.rollback(win, none, none, pool)
    assert sc.get_error() == 0
    assert_bits(host(pool), pool0, "states")


def test_backward_of_zero_rows_writes_zero_weight_and_bias_gradients():
    rng = np.random.default_rng(53)
    w = rand_bf16(rng, (H, K))
    empty = np.zeros((0, 3 * H), np.uint16)
    st, d_ref, dw_ref = oracle.backward("bf16", empty, w, np.zeros((0, H), np.uint16))
    assert st == oracle.OK and not dw_ref.any()
    nan = float("nan")
    dw = torch.full((H, K), nan, device="cuda")
    db = torch.full((H,), nan, device="cuda")
    dbcx, dw, db = sc.backward(dev(empty, "bf16"), dev(w, "bf16"),
                               torch.zeros((0, H), dtype=torch.bfloat16, device="cuda"),
                               dw=dw, with_dbias=True, dbias=db)
    assert tuple(dbcx.shape) == (0, 3 * H)
    assert sc.get_error() == 0
    assert_dw_close(host(dw), dw_ref)
    assert not host(db).any()


def test_backward_varlen_with_only_empty_sequences_passes_d_final_through():
    rng = np.random.default_rng(54)
    N = 3
    w = rand_bf16(rng, (H, K))
    init = rand_bf16(rng, (N, H, K))
    dfin = rng.standard_normal((N, H, K)).astype(np.float32)
    cu = np.zeros(N + 1, np.int32)
    empty = np.zeros((0, 3 * H), np.uint16)
    st, _, dw_ref, di_ref = oracle.backward_varlen("bf16", empty, w, cu,
                                                   np.zeros((0, H), np.uint16), init,
                                                   dfin.astype(np.float64))
    assert st == oracle.OK
    assert np.array_equal(di_ref, dfin.astype(np.float64)) and not dw_ref.any()
    nan = float("nan")
    dbcx, dw, dinit = sc.backward_varlen(
        dev(empty, "bf16"), dev(w, "bf16"), dev(cu, "i32"),
        torch.zeros((0, H), dtype=torch.bfloat16, device="cuda"),
        init_states=dev(init, "bf16"), d_final=dev(dfin, "f32"),
        dw=torch.full((H, K), nan, device="cuda"),
        d_init=torch.full((N, H, K), nan, device="cuda"))
    assert sc.get_error() == 0
    assert_dw_close(host(dw), dw_ref)
    assert_bits(host(dinit), dfin, "d_init = d_final")
