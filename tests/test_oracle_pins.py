"""Pins for the CPU oracle: each test checks it against something other than itself.

The pages print no ShortConv input/output values, so the oracle is pinned by
library routines (torch ``conv1d`` and autograd in float64, numpy matrix
products, torch's float32->bfloat16 cast), textbook IEEE rounding cases,
brute force on tiny inputs and the invariants the pages state:

* full prefill equals prefill followed by token-by-token decode
  ("feat(model): support LFM2-1.2B", section "支持平台与测试结果": the tiny
  F32 "Full vs Prefill+Decode" check);
* packed sequences share no history (same page, "供审阅者关注的事项");
* the verify tape holds the window after each draft step and rollback
  restores the state at the accepted boundary (SGLang PR #31041,
  "实现拆解 2").
"""
import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
from lfm2_gated_short_gb300 import workloads as wl

RNG = np.random.default_rng(12345)


# ----------------------------------------------------------------- helpers

def _rand(shape, dtype, rng, std=1.0):
    return wl.normal(rng, shape, std, dtype)


def _f64(dtype, a):
    return oracle.to_f64(dtype, a)


def lib_forward_f64(bcx64, w64, state64):
    """y and final state from torch.conv1d over [state[1:], u] (float64, no rounding)."""
    T, H3 = bcx64.shape
    H = H3 // 3
    K = w64.shape[1]
    B, C, X = bcx64[:, :H], bcx64[:, H:2 * H], bcx64[:, 2 * H:]
    u = B * X
    ext = np.concatenate([state64[:, 1:], u.T], axis=1)            # [H, K-1+T]
    z = F.conv1d(torch.from_numpy(ext)[None], torch.from_numpy(w64)[:, None, :],
                 groups=H)[0].numpy()                              # [H, T]
    y = C * z.T
    full = np.concatenate([state64, u.T], axis=1)
    return y, full[:, -K:], z.T


def torch_bf16_bits(t32: torch.Tensor) -> np.ndarray:
    return t32.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


# --------------------------------------------------------- rounding (bf16)

def test_bf16_rounding_textbook_ties():
    # spacing of bf16 values in [1, 2) is 2^-7; midpoints go to the even neighbour
    cases = {
        1.0: 0x3F80,
        1.0 + 2.0 ** -8: 0x3F80,              # tie between 1 and 1+2^-7 -> even (1)
        1.0 + 3 * 2.0 ** -8: 0x3F82,          # tie between 1+2^-7 (odd) and 1+2^-6
        1.0 + 2.0 ** -8 + 2.0 ** -40: 0x3F81,  # just above the tie -> up
        -(1.0 + 2.0 ** -8): 0xBF80,
        2.0 ** -133: 0x0001,                  # smallest subnormal
        2.0 ** -134: 0x0000,                  # half of it: tie -> even (0)
        3 * 2.0 ** -134: 0x0002,              # 1.5 units: tie -> even (2)
        255.0 * 2.0 ** 120: 0x7F7F,           # largest finite bf16
        255.5 * 2.0 ** 120: 0x7F80,           # tie above the largest -> inf
        float("inf"): 0x7F80,
        -0.0: 0x8000,
    }
    got = oracle.round_bf16(list(cases))
    assert [int(g) for g in got] == list(cases.values())


def test_bf16_rounding_is_one_step_from_double():
    # float(d) lands exactly on a bf16 tie and would round down to even; the
    # correctly rounded bf16 of d itself is the upper neighbour.
    d = 1.0 + 2.0 ** -8 + 2.0 ** -40
    assert float(np.float32(d)) == 1.0 + 2.0 ** -8
    assert int(oracle.round_bf16([d])[0]) == 0x3F81


def test_bf16_rounding_matches_torch_cast_on_float32_inputs():
    rng = np.random.default_rng(7)
    mant = rng.standard_normal(20000).astype(np.float32)
    scale = np.ldexp(np.float32(1), rng.integers(-140, 127, size=20000))
    vals = (mant * scale.astype(np.float32)).astype(np.float32)
    vals = vals[np.isfinite(vals)]
    got = oracle.round_bf16(vals.astype(np.float64))
    ref = torch_bf16_bits(torch.from_numpy(vals))
    np.testing.assert_array_equal(got, ref)


# ---------------------------------------------------- forward vs libraries

@pytest.mark.parametrize("K", [1, 2, 3, 4])
@pytest.mark.parametrize("T", [1, 2, 3, 7, 33])
def test_forward_f64_matches_torch_conv1d(K, T):
    rng = np.random.default_rng(100 * K + T)
    H = 5
    bcx = rng.standard_normal((T, 3 * H))
    w = rng.standard_normal((H, K))
    state = rng.standard_normal((1, H, K))
    pool = state.copy()
    st, y = oracle.prefill("f64", bcx, w, [0, T], [0], pool)
    assert st == oracle.OK
    y_ref, s_ref, _ = lib_forward_f64(bcx, w, state[0])
    np.testing.assert_allclose(y, y_ref, rtol=1e-13, atol=1e-13)
    np.testing.assert_array_equal(pool[0], s_ref)


@pytest.mark.parametrize("K", [1, 2, 3, 4])
def test_forward_f64_matches_dense_toeplitz(K):
    """Brute force: y = C * (M @ ext) with an explicit [T, T+K-1] band matrix."""
    rng = np.random.default_rng(K)
    H, T = 3, 9
    bcx = rng.standard_normal((T, 3 * H))
    w = rng.standard_normal((H, K))
    state = rng.standard_normal((1, H, K))
    pool = state.copy()
    st, y = oracle.prefill("f64", bcx, w, [0, T], [0], pool)
    assert st == oracle.OK
    for h in range(H):
        u = bcx[:, h] * bcx[:, 2 * H + h]
        ext = np.concatenate([state[0, h, 1:], u])  # positions -(K-1) .. T-1
        M = np.zeros((T, T + K - 1))
        for t in range(T):
            for j in range(K):                      # j steps back from t
                M[t, t + (K - 1) - j] = w[h, K - 1 - j]
        y_ref = bcx[:, H + h] * (M @ ext)
        np.testing.assert_allclose(y[:, h], y_ref, rtol=1e-13, atol=1e-13)


def test_forward_f32_rounding_matches_library_casts():
    rng = np.random.default_rng(3)
    H, K, T = 16, 3, 40
    bcx = _rand((T, 3 * H), "f32", rng)
    w = _rand((H, K), "f32", rng, wl.WEIGHT_STD)
    state = _rand((1, H, K), "f32", rng)
    pool = state.copy()
    st, y = oracle.prefill("f32", bcx, w, [0, T], [0], pool)
    assert st == oracle.OK
    b64 = bcx.astype(np.float64)
    u32 = (b64[:, :H] * b64[:, 2 * H:]).astype(np.float32)  # exact product, one rounding
    ext = np.concatenate([state[0].astype(np.float64)[:, 1:], u32.T.astype(np.float64)], 1)
    z = F.conv1d(torch.from_numpy(ext)[None],
                 torch.from_numpy(w.astype(np.float64))[:, None, :], groups=H)[0].numpy().T
    y_ref = (b64[:, H:2 * H] * z).astype(np.float32)
    np.testing.assert_array_equal(y, y_ref)
    np.testing.assert_array_equal(pool[0], np.concatenate([state[0], u32.T], 1)[:, -K:])


def test_forward_bf16_rounding_matches_library_casts():
    rng = np.random.default_rng(4)
    H, K, T = 16, 3, 64
    bcx = _rand((T, 3 * H), "bf16", rng)
    w = _rand((H, K), "bf16", rng, wl.WEIGHT_STD)
    state = _rand((1, H, K), "bf16", rng)
    pool = state.copy()
    st, y = oracle.prefill("bf16", bcx, w, [0, T], [0], pool)
    assert st == oracle.OK
    b64 = _f64("bf16", bcx)
    prod = torch.from_numpy((b64[:, :H] * b64[:, 2 * H:]).astype(np.float32))  # exact
    u_bits = torch_bf16_bits(prod)
    u64 = _f64("bf16", u_bits)
    ext = np.concatenate([_f64("bf16", state[0])[:, 1:], u64.T], 1)
    z = F.conv1d(torch.from_numpy(ext)[None],
                 torch.from_numpy(_f64("bf16", w))[:, None, :], groups=H)[0].numpy().T
    yz = b64[:, H:2 * H] * z
    y32 = yz.astype(np.float32)
    ref = torch_bf16_bits(torch.from_numpy(y32))
    # torch reaches bf16 through float32 (two roundings); they can differ from one
    # correct rounding only where the float32 value sits exactly on a bf16 tie.
    at_tie = (y32.view(np.uint32) & 0xFFFF) == 0x8000
    assert np.all((y == ref) | at_tie)
    np.testing.assert_array_equal(pool[0], np.concatenate([state[0], u_bits.T], 1)[:, -K:])


# ------------------------------------------------- closed-form special cases

def test_k1_unit_weight_is_elementwise_bcx():
    rng = np.random.default_rng(5)
    H, T = 24, 11
    bcx = _rand((T, 3 * H), "bf16", rng)
    w = np.full((H, 1), 0x3F80, np.uint16)  # 1.0
    pool = _rand((1, H, 1), "bf16", rng)
    st, y = oracle.prefill("bf16", bcx, w, [0, T], [0], pool)
    assert st == oracle.OK
    b = torch.from_numpy(_f64("bf16", bcx).astype(np.float32))
    u = (b[:, :H] * b[:, 2 * H:]).to(torch.bfloat16).float()
    ref = torch_bf16_bits(b[:, H:2 * H] * u)  # C*u exact in float32, one rounding
    np.testing.assert_array_equal(y, ref)
    np.testing.assert_array_equal(pool[0, :, 0],
                                  torch_bf16_bits(b[-1:, :H] * b[-1:, 2 * H:])[0])


@pytest.mark.parametrize("tap", [0, 2])
def test_unit_tap_shifts_the_gated_input(tap):
    """w = e_{K-1} gives y_t = C_t u_t; w = e_0 gives y_t = C_t u_{t-K+1} (history from the state)."""
    rng = np.random.default_rng(6 + tap)
    H, K, T = 8, 3, 10
    bcx = _rand((T, 3 * H), "bf16", rng)
    w = np.zeros((H, K), np.uint16)
    w[:, tap] = 0x3F80
    state = _rand((1, H, K), "bf16", rng)
    pool = state.copy()
    st, y = oracle.prefill("bf16", bcx, w, [0, T], [0], pool)
    assert st == oracle.OK
    b = torch.from_numpy(_f64("bf16", bcx).astype(np.float32))
    u = (b[:, :H] * b[:, 2 * H:]).to(torch.bfloat16).float()                 # [T, H]
    hist = torch.from_numpy(_f64("bf16", state[0]).astype(np.float32)).T      # [K, H]
    ext = torch.cat([hist[1:], u], 0)                                          # rows -(K-1)..T-1
    shift = (K - 1) - tap
    src = ext[(K - 1) - shift:(K - 1) - shift + T]
    np.testing.assert_array_equal(y, torch_bf16_bits(b[:, H:2 * H] * src))


@pytest.mark.parametrize("length", [0, 1, 2])
def test_short_sequence_state_mixes_old_state_and_new_inputs(length):
    rng = np.random.default_rng(20 + length)
    H, K = 4, 3
    bcx = rng.standard_normal((length, 3 * H))
    w = rng.standard_normal((H, K))
    state = rng.standard_normal((1, H, K))
    pool = state.copy()
    st, _ = oracle.prefill("f64", bcx, w, [0, length], [0], pool)
    assert st == oracle.OK
    u = (bcx[:, :H] * bcx[:, 2 * H:]).T                  # [H, length]
    expect = np.concatenate([state[0, :, length:], u], 1)
    np.testing.assert_array_equal(pool[0], expect)


# ------------------------------------------------------------- invariants

@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_prefill_equals_prefill_plus_decode_for_every_split(dtype):
    rng = np.random.default_rng(30)
    H, K, T = 16, 3, 12
    bcx = _rand((T, 3 * H), dtype, rng)
    w = _rand((H, K), dtype, rng, wl.WEIGHT_STD)
    state = _rand((1, H, K), dtype, rng)
    full_pool = state.copy()
    _, y_full = oracle.prefill(dtype, bcx, w, [0, T], [0], full_pool)
    for t1 in range(T + 1):
        pool = state.copy()
        _, y1 = oracle.prefill(dtype, bcx[:t1], w, [0, t1], [0], pool)
        ys = [y1]
        for t in range(t1, T):
            _, yd = oracle.decode(dtype, bcx[t:t + 1], w, [0], pool)
            ys.append(yd)
        np.testing.assert_array_equal(np.concatenate(ys, 0), y_full)
        np.testing.assert_array_equal(pool, full_pool)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_chunked_prefill_equals_full_prefill(dtype):
    rng = np.random.default_rng(31)
    H, K, T = 16, 4, 50
    bcx = _rand((T, 3 * H), dtype, rng)
    w = _rand((H, K), dtype, rng, wl.WEIGHT_STD)
    state = _rand((1, H, K), dtype, rng)
    full_pool = state.copy()
    _, y_full = oracle.prefill(dtype, bcx, w, [0, T], [0], full_pool)
    cuts = [0, 1, 3, 4, 17, 18, 41, T]
    pool = state.copy()
    ys = []
    for a, b in zip(cuts[:-1], cuts[1:]):
        _, yc = oracle.prefill(dtype, bcx[a:b], w, [0, b - a], [0], pool)
        ys.append(yc)
    np.testing.assert_array_equal(np.concatenate(ys), y_full)
    np.testing.assert_array_equal(pool, full_pool)


def test_varlen_equals_per_sequence_calls_and_leaves_other_slots():
    p = wl.varlen_prefill(n_seqs=7, H=16, K=3, n_slots=20, seed=32,
                          lengths=[5, 0, 1, 2, 9, 3, 4])
    pool = p.pool.copy()
    st, y = oracle.prefill(p.dtype, p.bcx, p.w, p.cu_seqlens, p.slot_ids, pool)
    assert st == oracle.OK
    for i in range(p.N):
        a, b = int(p.cu_seqlens[i]), int(p.cu_seqlens[i + 1])
        one = p.pool[p.slot_ids[i]][None].copy()
        _, yi = oracle.prefill(p.dtype, p.bcx[a:b], p.w, [0, b - a], [0], one)
        np.testing.assert_array_equal(y[a:b], yi)
        np.testing.assert_array_equal(pool[p.slot_ids[i]], one[0])
    others = np.setdiff1d(np.arange(20), p.slot_ids)
    np.testing.assert_array_equal(pool[others], p.pool[others])


def test_verify_tape_and_rollback_equal_decoding_the_accepted_prefix():
    s = wl.verify_serving(layers=1, batch=5, D=4, H=16, K=3, n_slots=9, seed=33)
    pool0 = s.pools[0]
    st, win, y = oracle.verify(s.dtype, s.bcx[0], s.w[0], s.slot_ids, pool0, s.D)
    assert st == oracle.OK
    for i in range(5):
        p = pool0.copy()
        for j in range(s.D):
            row = s.bcx[0][i * s.D + j:i * s.D + j + 1]
            _, yd = oracle.decode(s.dtype, row, s.w[0], [s.slot_ids[i]], p)
            np.testing.assert_array_equal(y[i * s.D + j], yd[0])
            np.testing.assert_array_equal(win[i, j], p[s.slot_ids[i]])
    for acc in ([0, 1, 2, 3, 4], [4, 0, 3, 0, 1]):
        pool = pool0.copy()
        assert oracle.rollback(s.dtype, win, acc, s.slot_ids, pool) == oracle.OK
        for i in range(5):
            p = pool0.copy()
            for j in range(acc[i]):
                row = s.bcx[0][i * s.D + j:i * s.D + j + 1]
                oracle.decode(s.dtype, row, s.w[0], [s.slot_ids[i]], p)
            np.testing.assert_array_equal(pool[s.slot_ids[i]], p[s.slot_ids[i]])
        others = np.setdiff1d(np.arange(9), s.slot_ids)
        np.testing.assert_array_equal(pool[others], pool0[others])


# --------------------------------------------------------------- backward

def _torch_grads(bcx64, w64, dy64, round_u=None):
    """Gradients of <dy, y> from torch autograd, forward written with conv1d."""
    T, H3 = bcx64.shape
    H = H3 // 3
    K = w64.shape[1]
    bcx = torch.tensor(bcx64, requires_grad=True)
    w = torch.tensor(w64, requires_grad=True)
    B, C, X = bcx[:, :H], bcx[:, H:2 * H], bcx[:, 2 * H:]
    u = B * X
    if round_u is not None:  # straight-through: forward uses the rounded value
        u = u + (round_u(u.detach()) - u.detach())
    z = F.conv1d(F.pad(u.T[None], (K - 1, 0)), w[:, None, :], groups=H)[0].T
    y = C * z
    (y * torch.from_numpy(dy64)).sum().backward()
    return bcx.grad.numpy(), w.grad.numpy()


@pytest.mark.parametrize("K", [1, 2, 3, 4])
@pytest.mark.parametrize("T", [1, 2, 5, 31])
def test_backward_f64_matches_torch_autograd(K, T):
    rng = np.random.default_rng(40 + K * 7 + T)
    H = 6
    bcx = rng.standard_normal((T, 3 * H))
    w = rng.standard_normal((H, K))
    dy = rng.standard_normal((T, H))
    st, dbcx, dw = oracle.backward("f64", bcx, w, dy)
    assert st == oracle.OK
    g_bcx, g_w = _torch_grads(bcx, w, dy)
    np.testing.assert_allclose(dbcx, g_bcx, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(dw, g_w, rtol=1e-12, atol=1e-12)


def test_backward_f64_central_differences():
    rng = np.random.default_rng(50)
    H, K, T = 3, 3, 6
    bcx = rng.standard_normal((T, 3 * H))
    w = rng.standard_normal((H, K))
    dy = rng.standard_normal((T, H))

    def loss(bcx_, w_):
        _, y = oracle.prefill("f64", bcx_, w_, [0, T], [0], np.zeros((1, H, K)))
        return float((y * dy).sum())

    _, dbcx, dw = oracle.backward("f64", bcx, w, dy)
    h = 1e-6
    for idx in np.ndindex(bcx.shape):
        a, b = bcx.copy(), bcx.copy()
        a[idx] += h
        b[idx] -= h
        assert abs((loss(a, w) - loss(b, w)) / (2 * h) - dbcx[idx]) < 1e-7
    for idx in np.ndindex(w.shape):
        a, b = w.copy(), w.copy()
        a[idx] += h
        b[idx] -= h
        assert abs((loss(bcx, a) - loss(bcx, b)) / (2 * h) - dw[idx]) < 1e-7


def _fwd64(bcx, w):
    """The oracle's float64 forward from a zero state: y [T, H]."""
    T, H, K = bcx.shape[0], w.shape[0], w.shape[1]
    st, y = oracle.prefill("f64", bcx, w, [0, T], [0], np.zeros((1, H, K)))
    assert st == oracle.OK
    return y


@pytest.mark.parametrize("K", [1, 3, 4])
def test_backward_f64_adjoint_identity(K):
    """<dy, J v> = <J^T dy, v> for a random direction v = (vB, vC, vx).

    y = C * conv(w, B * x) is linear in C and bilinear in (B, x), so the
    directional derivative is a sum of three forward calls:
    J v = F(B, vC, x) + F(vB, C, x) + F(B, C, vx). The right side is the
    backward's dB|dC|dx dotted with v."""
    rng = np.random.default_rng(60 + K)
    H, T = 5, 23
    bcx, v = rng.standard_normal((T, 3 * H)), rng.standard_normal((T, 3 * H))
    w, dy = rng.standard_normal((H, K)), rng.standard_normal((T, H))
    B, C, X = np.split(bcx, 3, axis=1)
    vB, vC, vX = np.split(v, 3, axis=1)
    jv = (_fwd64(np.hstack([B, vC, X]), w) + _fwd64(np.hstack([vB, C, X]), w)
          + _fwd64(np.hstack([B, C, vX]), w))
    st, dbcx, _ = oracle.backward("f64", bcx, w, dy)
    assert st == oracle.OK
    lhs, rhs = float((dy * jv).sum()), float((dbcx * v).sum())
    assert abs(lhs - rhs) <= 1e-12 * max(1.0, abs(lhs))


@pytest.mark.parametrize("K", [2, 3, 4])
def test_backward_f64_weight_gradient_by_linearity_in_w(K):
    """The forward is linear in w: y(w) = sum_k w_k y(e_k), per channel, where
    e_k is the weight with tap k = 1 in every channel. So
    dW[h, k] = sum_t dy[t, h] y(e_k)[t, h]."""
    rng = np.random.default_rng(70 + K)
    H, T = 4, 19
    bcx, w, dy = (rng.standard_normal((T, 3 * H)), rng.standard_normal((H, K)),
                  rng.standard_normal((T, H)))
    basis = [_fwd64(bcx, np.eye(K)[None, k].repeat(H, 0)) for k in range(K)]
    y = _fwd64(bcx, w)
    np.testing.assert_allclose(y, sum(w[:, k] * basis[k] for k in range(K)),
                               rtol=1e-12, atol=1e-12)
    st, _, dw = oracle.backward("f64", bcx, w, dy)
    assert st == oracle.OK
    closed = np.stack([(dy * basis[k]).sum(axis=0) for k in range(K)], axis=1)
    np.testing.assert_allclose(dw, closed, rtol=1e-12, atol=1e-12)


def test_backward_bf16_matches_autograd_with_straight_through_rounding():
    rng = np.random.default_rng(51)
    H, K, T = 16, 3, 40
    bcx = _rand((T, 3 * H), "bf16", rng)
    w = _rand((H, K), "bf16", rng, wl.WEIGHT_STD)
    dy = _rand((T, H), "bf16", rng)
    st, dbcx, dw = oracle.backward("bf16", bcx, w, dy)
    assert st == oracle.OK
    rnd = lambda u: u.float().to(torch.bfloat16).double()  # u is an exact float32 product
    g_bcx, g_w = _torch_grads(_f64("bf16", bcx), _f64("bf16", w), _f64("bf16", dy), rnd)
    np.testing.assert_allclose(dw, g_w, rtol=1e-12, atol=1e-12)
    g32 = g_bcx.astype(np.float32)
    ref = torch_bf16_bits(torch.from_numpy(g32))
    at_tie = (g32.view(np.uint32) & 0xFFFF) == 0x8000
    assert np.all((dbcx == ref) | at_tie)


# ------------------------------------------------------------ bad inputs

def test_out_of_range_slot_skips_only_that_sequence():
    p = wl.varlen_prefill(n_seqs=3, H=8, K=3, n_slots=4, seed=60, lengths=[3, 4, 2])
    slots = p.slot_ids.copy()
    slots[1] = 4                                         # == n_slots: out of range
    pool = p.pool.copy()
    y = np.full((p.T, p.H), 0x1234, np.uint16)
    st, y = oracle.prefill(p.dtype, p.bcx, p.w, p.cu_seqlens, slots, pool, y)
    assert st == oracle.EDATA
    assert np.all(y[3:7] == 0x1234)
    assert not np.all(y[:3] == 0x1234) and not np.all(y[7:] == 0x1234)


@pytest.mark.parametrize("cu", [[0, 3, 2, 9], [1, 3, 5, 9], [0, 3, 5, 8]])
def test_bad_cu_seqlens_touch_nothing(cu):
    p = wl.varlen_prefill(n_seqs=3, H=8, K=3, n_slots=4, seed=61, lengths=[3, 2, 4])
    pool = p.pool.copy()
    y = np.full((p.T, p.H), 0x1234, np.uint16)
    st, y = oracle.prefill(p.dtype, p.bcx, p.w, cu, p.slot_ids, pool, y)
    assert st == oracle.EDATA
    assert np.all(y == 0x1234)
    np.testing.assert_array_equal(pool, p.pool)


def test_rollback_rejects_accepted_out_of_range():
    s = wl.verify_serving(layers=1, batch=3, D=2, H=8, K=3, n_slots=5, seed=62)
    _, win, _ = oracle.verify(s.dtype, s.bcx[0], s.w[0], s.slot_ids, s.pools[0], s.D)
    pool = s.pools[0].copy()
    st = oracle.rollback(s.dtype, win, [3, -1, 2], s.slot_ids, pool)
    assert st == oracle.EDATA
    np.testing.assert_array_equal(pool[s.slot_ids[:2]], s.pools[0][s.slot_ids[:2]])
    np.testing.assert_array_equal(pool[s.slot_ids[2]], win[2, 1])


# ------------------------------------------------------- tiny fp32 config

def test_tiny_fp32_config_prefill_then_decode_matches_conv1d():
    """H=64, K=3, T=16 prefill, then 4 decode tokens, against conv1d over all 20 tokens."""
    p = wl.tiny_fp32()
    pool = p.pool.copy()
    st, y = oracle.prefill("f32", p.bcx, p.w, p.cu_seqlens, p.slot_ids, pool)
    assert st == oracle.OK
    ys = [y]
    for step in range(p.decode_bcx.shape[0]):
        st, yd = oracle.decode("f32", p.decode_bcx[step], p.w, [0], pool)
        assert st == oracle.OK
        ys.append(yd)
    allrows = np.concatenate([p.bcx, p.decode_bcx[:, 0]], 0).astype(np.float64)
    H = p.H
    u32 = (allrows[:, :H] * allrows[:, 2 * H:]).astype(np.float32).astype(np.float64)
    z = F.conv1d(F.pad(torch.from_numpy(u32.T)[None], (p.K - 1, 0)),
                 torch.from_numpy(p.w.astype(np.float64))[:, None, :], groups=H)[0].numpy().T
    y_ref = (allrows[:, H:2 * H] * z).astype(np.float32)
    np.testing.assert_array_equal(np.concatenate(ys, 0), y_ref)
    np.testing.assert_array_equal(pool[0], u32[-p.K:].T.astype(np.float32))


# ------------------------------------------- varlen backward with states

def _torch_varlen_grads(bcx64, w64, cu, dy64, init64, dfin64, round_u=None):
    """<dy, y> + <d_final, final state> differentiated by torch autograd (float64)."""
    T, H3 = bcx64.shape
    H = H3 // 3
    K = w64.shape[1]
    bcx = torch.tensor(bcx64, requires_grad=True)
    w = torch.tensor(w64, requires_grad=True)
    init = torch.tensor(init64, requires_grad=True)
    loss = torch.zeros((), dtype=torch.float64)
    for i in range(len(cu) - 1):
        a, b = int(cu[i]), int(cu[i + 1])
        B, C, X = bcx[a:b, :H], bcx[a:b, H:2 * H], bcx[a:b, 2 * H:]
        u = B * X
        if round_u is not None:
            u = u + (round_u(u.detach()) - u.detach())
        ext = torch.cat([init[i], u.T], dim=1)                    # [H, K + len]
        if b > a:
            z = F.conv1d(ext[None, :, 1:], w[:, None, :], groups=H)[0].T
            loss = loss + (C * z * torch.from_numpy(dy64[a:b])).sum()
        loss = loss + (ext[:, -K:] * torch.from_numpy(dfin64[i])).sum()
    loss.backward()
    return bcx.grad.numpy(), w.grad.numpy(), init.grad.numpy()


@pytest.mark.parametrize("K", [1, 2, 3, 4])
def test_backward_varlen_f64_matches_torch_autograd(K):
    rng = np.random.default_rng(70 + K)
    H, lengths = 4, [3, 0, 1, 2, 7, 5]
    cu = np.r_[0, np.cumsum(lengths)].astype(np.int32)
    T, N = int(cu[-1]), len(lengths)
    bcx = rng.standard_normal((T, 3 * H))
    w = rng.standard_normal((H, K))
    dy = rng.standard_normal((T, H))
    init = rng.standard_normal((N, H, K))
    dfin = rng.standard_normal((N, H, K))
    st, dbcx, dw, dinit = oracle.backward_varlen("f64", bcx, w, cu, dy, init, dfin)
    assert st == oracle.OK
    g_bcx, g_w, g_init = _torch_varlen_grads(bcx, w, cu, dy, init, dfin)
    np.testing.assert_allclose(dbcx, g_bcx, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(dw, g_w, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(dinit, g_init, rtol=1e-12, atol=1e-12)


def test_backward_varlen_reduces_to_the_single_sequence_backward():
    rng = np.random.default_rng(75)
    H, K, T = 6, 3, 40
    bcx = rng.standard_normal((T, 3 * H))
    w = rng.standard_normal((H, K))
    dy = rng.standard_normal((T, H))
    st, dbcx, dw, dinit = oracle.backward_varlen("f64", bcx, w, [0, T], dy)
    st2, dbcx2, dw2 = oracle.backward("f64", bcx, w, dy)
    assert st == st2 == oracle.OK
    np.testing.assert_allclose(dbcx, dbcx2, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(dw, dw2, rtol=1e-12, atol=1e-12)


def test_backward_varlen_equals_per_sequence_calls():
    rng = np.random.default_rng(76)
    H, K, lengths = 8, 4, [5, 1, 0, 9, 2]
    cu = np.r_[0, np.cumsum(lengths)].astype(np.int32)
    T, N = int(cu[-1]), len(lengths)
    bcx = _rand((T, 3 * H), "bf16", rng)
    w = _rand((H, K), "bf16", rng, wl.WEIGHT_STD)
    dy = _rand((T, H), "bf16", rng)
    init = _rand((N, H, K), "bf16", rng)
    dfin = rng.standard_normal((N, H, K))
    st, dbcx, dw, dinit = oracle.backward_varlen("bf16", bcx, w, cu, dy, init, dfin)
    assert st == oracle.OK
    dw_sum = np.zeros_like(dw)
    for i in range(N):
        a, b = int(cu[i]), int(cu[i + 1])
        st, d1, w1, i1 = oracle.backward_varlen("bf16", bcx[a:b], w, [0, b - a], dy[a:b],
                                                init[i:i + 1], dfin[i:i + 1])
        assert st == oracle.OK
        np.testing.assert_array_equal(dbcx[a:b], d1)
        np.testing.assert_array_equal(dinit[i], i1[0])
        dw_sum += w1
    np.testing.assert_allclose(dw, dw_sum, rtol=1e-12, atol=1e-12)


def test_backward_varlen_bf16_matches_autograd_with_straight_through_rounding():
    rng = np.random.default_rng(77)
    H, K, lengths = 16, 3, [7, 2, 12]
    cu = np.r_[0, np.cumsum(lengths)].astype(np.int32)
    T, N = int(cu[-1]), len(lengths)
    bcx = _rand((T, 3 * H), "bf16", rng)
    w = _rand((H, K), "bf16", rng, wl.WEIGHT_STD)
    dy = _rand((T, H), "bf16", rng)
    init = _rand((N, H, K), "bf16", rng)
    dfin = rng.standard_normal((N, H, K))
    st, dbcx, dw, dinit = oracle.backward_varlen("bf16", bcx, w, cu, dy, init, dfin)
    assert st == oracle.OK
    rnd = lambda u: u.float().to(torch.bfloat16).double()
    g_bcx, g_w, g_init = _torch_varlen_grads(_f64("bf16", bcx), _f64("bf16", w), cu,
                                             _f64("bf16", dy), _f64("bf16", init), dfin, rnd)
    np.testing.assert_allclose(dw, g_w, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(dinit, g_init, rtol=1e-12, atol=1e-12)
    g32 = g_bcx.astype(np.float32)
    ref = torch_bf16_bits(torch.from_numpy(g32))
    at_tie = (g32.view(np.uint32) & 0xFFFF) == 0x8000
    assert np.all((dbcx == ref) | at_tie)


def test_backward_varlen_rejects_bad_cu_seqlens():
    rng = np.random.default_rng(78)
    bcx = rng.standard_normal((6, 12))
    st, *_ = oracle.backward_varlen("f64", bcx, rng.standard_normal((4, 3)), [0, 4, 3, 6],
                                    rng.standard_normal((6, 4)))
    assert st == oracle.EDATA


# ----------------------------------------------------------- conv bias

@pytest.mark.parametrize("K", [1, 3, 4])
def test_forward_bias_f64_matches_torch_conv1d_with_bias(K):
    rng = np.random.default_rng(80 + K)
    H, T = 5, 13
    bcx = rng.standard_normal((T, 3 * H))
    w = rng.standard_normal((H, K))
    b = rng.standard_normal(H)
    state = rng.standard_normal((1, H, K))
    pool = state.copy()
    st, y = oracle.prefill("f64", bcx, w, [0, T], [0], pool, bias=b)
    assert st == oracle.OK
    u = bcx[:, :H] * bcx[:, 2 * H:]
    ext = np.concatenate([state[0, :, 1:], u.T], axis=1)
    z = F.conv1d(torch.from_numpy(ext)[None], torch.from_numpy(w)[:, None, :],
                 bias=torch.from_numpy(b), groups=H)[0].numpy().T
    np.testing.assert_allclose(y, bcx[:, H:2 * H] * z, rtol=1e-13, atol=1e-13)
    # the state keeps u, so the bias never reaches it
    np.testing.assert_array_equal(pool[0], np.concatenate([state[0], u.T], 1)[:, -K:])


def test_forward_bias_bf16_matches_library_casts():
    rng = np.random.default_rng(85)
    H, K, T = 16, 3, 50
    bcx = _rand((T, 3 * H), "bf16", rng)
    w = _rand((H, K), "bf16", rng, wl.WEIGHT_STD)
    b = _rand((H,), "bf16", rng)
    pool = np.zeros((1, H, K), np.uint16)
    st, y = oracle.prefill("bf16", bcx, w, [0, T], [0], pool, bias=b)
    assert st == oracle.OK
    b64 = _f64("bf16", bcx)
    u64 = _f64("bf16", torch_bf16_bits(torch.from_numpy((b64[:, :H] * b64[:, 2 * H:]).astype(np.float32))))
    z = F.conv1d(F.pad(torch.from_numpy(u64.T)[None], (K - 1, 0)),
                 torch.from_numpy(_f64("bf16", w))[:, None, :],
                 bias=torch.from_numpy(_f64("bf16", b)), groups=H)[0].numpy().T
    y32 = (b64[:, H:2 * H] * z).astype(np.float32)
    ref = torch_bf16_bits(torch.from_numpy(y32))
    at_tie = (y32.view(np.uint32) & 0xFFFF) == 0x8000
    assert np.all((y == ref) | at_tie)


def test_bias_keeps_prefill_equal_to_prefill_plus_decode_and_verify_windows():
    rng = np.random.default_rng(86)
    H, K, T = 8, 3, 9
    bcx = _rand((T, 3 * H), "bf16", rng)
    w = _rand((H, K), "bf16", rng, wl.WEIGHT_STD)
    b = _rand((H,), "bf16", rng)
    state = _rand((1, H, K), "bf16", rng)
    full = state.copy()
    _, y_full = oracle.prefill("bf16", bcx, w, [0, T], [0], full, bias=b)
    pool = state.copy()
    _, y1 = oracle.prefill("bf16", bcx[:4], w, [0, 4], [0], pool, bias=b)
    ys = [y1] + [oracle.decode("bf16", bcx[t:t + 1], w, [0], pool, bias=b)[1] for t in range(4, T)]
    np.testing.assert_array_equal(np.concatenate(ys), y_full)
    np.testing.assert_array_equal(pool, full)
    st, win_b, yv = oracle.verify("bf16", bcx, w, [0], state, T, bias=b)
    st, win_0, _ = oracle.verify("bf16", bcx, w, [0], state, T)
    np.testing.assert_array_equal(win_b, win_0)       # the tape holds u: no bias in it
    np.testing.assert_array_equal(yv, y_full)


def _torch_bias_grads(bcx64, w64, b64, dy64):
    T, H3 = bcx64.shape
    H = H3 // 3
    K = w64.shape[1]
    bcx = torch.tensor(bcx64, requires_grad=True)
    w = torch.tensor(w64, requires_grad=True)
    b = torch.tensor(b64, requires_grad=True)
    u = bcx[:, :H] * bcx[:, 2 * H:]
    z = F.conv1d(F.pad(u.T[None], (K - 1, 0)), w[:, None, :], bias=b, groups=H)[0].T
    ((bcx[:, H:2 * H] * z) * torch.from_numpy(dy64)).sum().backward()
    return bcx.grad.numpy(), w.grad.numpy(), b.grad.numpy()


@pytest.mark.parametrize("K", [1, 3, 4])
def test_backward_bias_f64_matches_torch_autograd(K):
    rng = np.random.default_rng(87 + K)
    H, T = 6, 21
    bcx = rng.standard_normal((T, 3 * H))
    w = rng.standard_normal((H, K))
    b = rng.standard_normal(H)
    dy = rng.standard_normal((T, H))
    st, dbcx, dw, db = oracle.backward("f64", bcx, w, dy, bias=b, with_dbias=True)
    assert st == oracle.OK
    g_bcx, g_w, g_b = _torch_bias_grads(bcx, w, b, dy)
    np.testing.assert_allclose(dbcx, g_bcx, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(dw, g_w, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(db, g_b, rtol=1e-12, atol=1e-12)


def test_backward_varlen_bias_matches_per_sequence_sums():
    rng = np.random.default_rng(90)
    H, K, lengths = 6, 3, [4, 0, 9, 2]
    cu = np.r_[0, np.cumsum(lengths)].astype(np.int32)
    T, N = int(cu[-1]), len(lengths)
    bcx = rng.standard_normal((T, 3 * H))
    w = rng.standard_normal((H, K))
    b = rng.standard_normal(H)
    dy = rng.standard_normal((T, H))
    st, dbcx, dw, di, db = oracle.backward_varlen("f64", bcx, w, cu, dy, bias=b, with_dbias=True)
    assert st == oracle.OK
    g_b = np.zeros(H)
    for i in range(N):
        a, e = int(cu[i]), int(cu[i + 1])
        if e > a:
            s2, d1, w1, b1 = oracle.backward("f64", bcx[a:e], w, dy[a:e], bias=b, with_dbias=True)
            np.testing.assert_allclose(dbcx[a:e], d1, rtol=1e-12, atol=1e-12)
            g_b += b1
    np.testing.assert_allclose(db, g_b, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(db, _torch_bias_grads(bcx, w, b, dy)[2] * 0 + g_b, rtol=1e-12)
