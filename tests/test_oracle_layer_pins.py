"""Pins of the layer oracle (``oracle/layer.py``): the in_proj / out_proj
projections and their composition with the conv, checked against exact
integer brute force, closed forms and a single-rounding case."""
import numpy as np
import pytest

import oracle
from oracle import layer


def _dyadic(rng, shape, lo, hi, scale_exp):
    """Integers in [lo, hi] times 2**scale_exp: exact in bf16 and float64."""
    ints = rng.integers(lo, hi, size=shape, endpoint=True)
    return ints, ints.astype(np.float64) * 2.0 ** scale_exp


def test_linear_matches_exact_integer_brute_force():
    """inp @ weight^T on non-square shapes, element by element in Python integers."""
    rng = np.random.default_rng(700)
    T, n, m = 5, 7, 4
    ai, a = _dyadic(rng, (T, n), -9, 9, -3)
    wi, w = _dyadic(rng, (m, n), -9, 9, -5)
    got = layer.linear("f64", a, w)
    assert got.shape == (T, m)
    for t in range(T):
        for j in range(m):
            exact = sum(int(ai[t, k]) * int(wi[j, k]) for k in range(n))  # units of 2^-8
            assert got[t, j] == exact * 2.0 ** -8


def test_linear_rounds_the_exact_sum_once():
    """1 + 2^-8 + 2^-30 lies just above the bf16 tie between 1 and 1 + 2^-7, so
    one rounding gives 1 + 2^-7. A float32 sum first would drop 2^-30, land on
    the tie and round to 1."""
    inp = oracle.round_bf16([[1.0, 2.0 ** -8, 2.0 ** -30]])
    wt = oracle.round_bf16([[1.0, 1.0, 1.0]])
    got = layer.linear("bf16", inp, wt)
    assert oracle.bf16_to_f64(got)[0, 0] == 1.0 + 2.0 ** -7
    assert layer.linear("f32", oracle.bf16_to_f64(inp).astype(np.float32),
                        np.ones((1, 3), np.float32))[0, 0] == np.float32(1.0 + 2.0 ** -8)


def test_in_proj_column_blocks_are_b_c_xv():
    """w_in rows [0, H) make b, [H, 2H) c and [2H, 3H) xv: with selection rows
    the projection returns the selected hidden columns in that order."""
    rng = np.random.default_rng(701)
    T, H = 6, 4
    D = 3 * H + 2
    hidden = oracle.round_bf16(rng.standard_normal((T, D)))
    w_in = np.zeros((3 * H, D))
    pick = rng.permutation(D)[:3 * H]
    w_in[np.arange(3 * H), pick] = 1.0
    got = layer.in_proj("bf16", hidden, oracle.round_bf16(w_in))
    np.testing.assert_array_equal(got, hidden[:, pick])


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_in_proj_prefill_k1_closed_form(dtype):
    """K = 1, unit weight, selection in_proj: y = round(c * round(b * xv))."""
    rng = np.random.default_rng(702 + (dtype == "f32"))
    T, H, D = 9, 8, 24
    if dtype == "bf16":
        hidden = oracle.round_bf16(rng.standard_normal((T, D)))
        one = oracle.round_bf16(np.ones((H, 1)))
    else:
        hidden = rng.standard_normal((T, D)).astype(np.float32)
        one = np.ones((H, 1), np.float32)
    sel = np.zeros((3 * H, D))
    sel[np.arange(3 * H), np.arange(3 * H)] = 1.0
    w_in = oracle.round_bf16(sel) if dtype == "bf16" else sel.astype(np.float32)
    pool = np.zeros((1, H, 1), hidden.dtype)
    st, y = layer.in_proj_prefill(dtype, hidden, w_in, one, [0, T], [0], pool)
    assert st == oracle.OK
    h = oracle.to_f64(dtype, hidden)
    b, c, x = h[:, :H], h[:, H:2 * H], h[:, 2 * H:3 * H]
    u = oracle.to_f64(dtype, layer.round_to(dtype, b * x))
    np.testing.assert_array_equal(y, layer.round_to(dtype, c * u))
    np.testing.assert_array_equal(pool[0, :, 0], layer.round_to(dtype, b[-1] * x[-1]))


def test_in_proj_prefill_is_in_proj_then_prefill_and_splits():
    """The layer prefill equals prefill of the projected rows, and two
    continued calls over a split equal one call."""
    rng = np.random.default_rng(704)
    T, H, D, K = 20, 8, 16, 3
    hidden = oracle.round_bf16(rng.standard_normal((T, D)))
    w_in = oracle.round_bf16(rng.standard_normal((3 * H, D)) / 4)
    w = oracle.round_bf16(rng.standard_normal((H, K)) / 2)
    p1 = np.zeros((1, H, K), np.uint16)
    st, y1 = layer.in_proj_prefill("bf16", hidden, w_in, w, [0, T], [0], p1)
    assert st == oracle.OK
    p2 = np.zeros((1, H, K), np.uint16)
    ya = layer.in_proj_prefill("bf16", hidden[:7], w_in, w, [0, 7], [0], p2)[1]
    yb = layer.in_proj_prefill("bf16", hidden[7:], w_in, w, [0, T - 7], [0], p2)[1]
    np.testing.assert_array_equal(np.concatenate([ya, yb]), y1)
    np.testing.assert_array_equal(p2, p1)


def test_out_proj_matches_brute_force_and_orientation():
    rng = np.random.default_rng(705)
    T, H, D = 4, 6, 5
    yi, y = _dyadic(rng, (T, H), -7, 7, -2)
    wi, w = _dyadic(rng, (D, H), -7, 7, -4)
    got = layer.out_proj("f64", y, w)
    assert got.shape == (T, D)
    exact = (yi.astype(object) @ wi.T.astype(object)).astype(np.float64) * 2.0 ** -6
    np.testing.assert_array_equal(got, exact)


def test_in_proj_decode_is_the_layer_prefill_of_one_token_sequences():
    """Decoding N one-token sequences equals the layer prefill of N sequences
    of length one (the per-token step of the page's definition); token by
    token it continues a longer prefill exactly."""
    rng = np.random.default_rng(706)
    N, H, D, K = 9, 8, 16, 3
    hidden = oracle.round_bf16(rng.standard_normal((N, D)))
    w_in = oracle.round_bf16(rng.standard_normal((3 * H, D)) / 4)
    w = oracle.round_bf16(rng.standard_normal((H, K)) / 2)
    b = oracle.round_bf16(rng.standard_normal(H) / 2)
    slots = rng.permutation(12)[:N].astype(np.int32)
    pool0 = oracle.round_bf16(rng.standard_normal((12, H, K)))
    p1 = pool0.copy()
    st, y1 = layer.in_proj_decode("bf16", hidden, w_in, w, slots, p1, bias=b)
    assert st == oracle.OK
    p2 = pool0.copy()
    st, y2 = layer.in_proj_prefill("bf16", hidden, w_in, w, np.arange(N + 1), slots, p2, bias=b)
    assert st == oracle.OK
    np.testing.assert_array_equal(y1, y2)
    np.testing.assert_array_equal(p1, p2)
    # one sequence, token by token, continues a prefill of its first rows
    T = 6
    hs = oracle.round_bf16(rng.standard_normal((T, D)))
    pa = np.zeros((1, H, K), np.uint16)
    ya = layer.in_proj_prefill("bf16", hs, w_in, w, [0, T], [0], pa)[1]
    pb = np.zeros((1, H, K), np.uint16)
    yb = [layer.in_proj_prefill("bf16", hs[:2], w_in, w, [0, 2], [0], pb)[1]]
    for t in range(2, T):
        yb.append(layer.in_proj_decode("bf16", hs[t:t + 1], w_in, w, [0], pb)[1])
    np.testing.assert_array_equal(np.concatenate(yb), ya)
    np.testing.assert_array_equal(pb, pa)
