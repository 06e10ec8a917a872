"""The layer's projections on the GPU (tensor cores) against the layer oracle.

shortconv_in_proj_prefill computes in_proj (fp32 accumulation on the tensor
cores), rounds the projection to bf16 and runs the ShortConv in the GEMM's
epilogue. With dyadic inputs (small integers times powers of two, bounded so
that every partial sum of the projection is exact in fp32), the projection is
exact in any accumulation order. Then its bf16 rounding is the oracle's, the
states must match bit for bit and y must meet the bf16 tolerance. With
normal inputs the projection is exact only up to fp32 accumulation error: a
projection value within that error of a bf16 rounding boundary may round
either way, and outputs that use such a value are excluded (they are
counted, and rare).
"""
import numpy as np
import pytest
import torch

import oracle
from oracle import layer
import lfm2_gated_short_gb300 as sc
from gpu_util import assert_bits, assert_close, dev, host

pytestmark = pytest.mark.gpu


def dyadic(rng, shape, lim, exp):
    """Integers in [-lim, lim] times 2**exp, as bf16 bits (exact)."""
    return oracle.round_bf16(rng.integers(-lim, lim, size=shape, endpoint=True) * 2.0 ** exp)


def make_case(rng, lengths, D, H, K, extra_slots=5, exact=True, state=True):
    lengths = np.asarray(lengths, np.int64)
    cu = np.r_[0, np.cumsum(lengths)].astype(np.int32)
    T, N = int(cu[-1]), len(lengths)
    if exact:  # products are multiples of 2^-9 below 2^-3, sums of D <= 4096 are exact
        hidden = dyadic(rng, (T, D), 8, -3)
        w_in = dyadic(rng, (3 * H, D), 8, -6)
    else:
        hidden = oracle.round_bf16(rng.standard_normal((T, D)))
        w_in = oracle.round_bf16(rng.standard_normal((3 * H, D)) / np.sqrt(D))
    w = oracle.round_bf16(rng.standard_normal((H, K)) * np.sqrt(1 / 3))
    n_slots = N + extra_slots
    slots = rng.permutation(n_slots)[:N].astype(np.int32)
    pool = np.full((n_slots, H, K), 0xDEAD, np.uint16)  # untouched slots keep this
    for s in slots:
        pool[s] = oracle.round_bf16(rng.standard_normal((H, K))) if state else 0
    return dict(hidden=hidden, w_in=w_in, w=w, cu=cu, slots=slots, pool=pool, D=D, H=H, K=K)


def run_gpu(c, bias=None):
    pool = dev(c["pool"], "bf16")
    y = sc.in_proj_prefill(dev(c["hidden"], "bf16"), dev(c["w_in"], "bf16"), dev(c["w"], "bf16"),
                           dev(c["cu"], "i32"), dev(c["slots"], "i32"), pool,
                           bias=None if bias is None else dev(bias, "bf16"))
    torch.cuda.synchronize()
    return host(y), host(pool)


def run_oracle(c, bias=None):
    pool = c["pool"].copy()
    st, y = layer.in_proj_prefill("bf16", c["hidden"], c["w_in"], c["w"], c["cu"], c["slots"],
                                  pool, bias=bias)
    assert st == oracle.OK
    return y, pool


def test_tiny_single_tile():
    c = make_case(np.random.default_rng(800), [50], 64, 64, 3, state=False)
    y, pool = run_gpu(c)
    y_ref, pool_ref = run_oracle(c)
    assert sc.get_error() == 0
    assert_close("bf16", y, y_ref, "y")
    assert_bits(pool, pool_ref, "pool")


TILE_EDGE_LENGTHS = [1, 2, 0, 130, 5, 126, 127, 128, 3, 260, 0, 4]


@pytest.mark.parametrize("K", [1, 2, 3, 4])
def test_varlen_exact_inputs(K):
    c = make_case(np.random.default_rng(810 + K), TILE_EDGE_LENGTHS, 128, 128, K)
    y, pool = run_gpu(c)
    y_ref, pool_ref = run_oracle(c)
    assert sc.get_error() == 0
    assert_close("bf16", y, y_ref, "y")
    assert_bits(pool, pool_ref, "pool (states bit-exact, untouched slots unchanged)")


def test_varlen_exact_inputs_with_bias():
    rng = np.random.default_rng(820)
    c = make_case(rng, TILE_EDGE_LENGTHS, 192, 256, 3)
    b = oracle.round_bf16(rng.standard_normal(256) * 0.5)
    y, pool = run_gpu(c, b)
    y_ref, pool_ref = run_oracle(c, b)
    assert_close("bf16", y, y_ref, "y")
    assert_bits(pool, pool_ref, "pool")


def test_fused_equals_the_conv_kernel_on_the_same_projection():
    """With an exact projection, the fused epilogue gives the bits of the
    streamed prefill kernel run on the projection (same operation order)."""
    c = make_case(np.random.default_rng(830), TILE_EDGE_LENGTHS, 128, 192, 3)
    y, pool = run_gpu(c)
    bcx = layer.in_proj("bf16", c["hidden"], c["w_in"])
    pool2 = dev(c["pool"], "bf16")
    y2 = sc.prefill(dev(bcx, "bf16"), dev(c["w"], "bf16"), dev(c["cu"], "i32"),
                    dev(c["slots"], "i32"), pool2)
    torch.cuda.synchronize()
    assert_bits(y, host(y2), "y")
    assert_bits(pool, host(pool2), "pool")


def test_one_token_per_sequence_equals_decode():
    rng = np.random.default_rng(840)
    c = make_case(rng, [1] * 37, 128, 128, 3)
    y, pool = run_gpu(c)
    bcx = layer.in_proj("bf16", c["hidden"], c["w_in"])
    pool2 = dev(c["pool"], "bf16")
    y2 = sc.decode(dev(bcx, "bf16"), dev(c["w"], "bf16"), dev(c["slots"], "i32"), pool2)
    torch.cuda.synchronize()
    assert_bits(y, host(y2), "y")
    assert_bits(pool, host(pool2), "pool")


def test_lfm2_shape_T4096_D2048_H2048_sampled_channels():
    """One 4096-token sequence at LFM2-1.2B's width; oracle on 64 channels."""
    rng = np.random.default_rng(850)
    D = H = 2048
    c = make_case(rng, [4096], D, H, 3, extra_slots=0, state=False)
    y, pool = run_gpu(c)
    ch = np.sort(np.concatenate([[0, 63, 64, 1023, 1024, 2047],
                                 rng.choice(np.arange(65, 2040), 58, replace=False)]))
    rows = np.concatenate([ch, H + ch, 2 * H + ch])
    sub = dict(c, w_in=c["w_in"][rows], w=np.ascontiguousarray(c["w"][ch]),
               pool=np.ascontiguousarray(c["pool"][:, ch]))
    y_ref, pool_ref = run_oracle(sub)
    assert_close("bf16", y[:, ch], y_ref, "y")
    assert_bits(pool[:, ch], pool_ref, "pool")


# One sequence per call: when the tile groups allow it (every column's first
# and last row-tile pairs in one cluster, on the 76 pairs of this device), the
# fused kernel writes the new state itself after its cluster's last tile and
# no commit pass runs; otherwise the workspace and the commit pass do it.
# (T, D, H, K): one row tile; two row tiles on the two CTAs of one pair;
# T < K; T = K; two pairs and one column (too few groups: commit pass); many
# pairs of one column; of two columns, the second half full; LFM2's width.
SINGLE_CASES = [(50, 64, 64, 3), (200, 128, 128, 3), (1, 64, 128, 3), (2, 64, 64, 4),
                (3, 64, 64, 3), (300, 64, 128, 3), (20000, 64, 128, 3), (12000, 128, 192, 2),
                (12000, 64, 192, 1), (9000, 64, 128, 4), (4096, 2048, 2048, 3)]


@pytest.mark.parametrize("T,D,H,K", SINGLE_CASES)
def test_single_sequence_from_a_random_state(T, D, H, K):
    rng = np.random.default_rng(860 + T + D + H + K)
    c = make_case(rng, [T], D, H, K, extra_slots=3)
    bias = oracle.round_bf16(rng.standard_normal(H) * 0.5) if T % 2 == 0 else None
    y, pool = run_gpu(c, bias)
    assert sc.get_error() == 0
    if H > 256:  # the oracle on 64 channels (channels are independent)
        ch = np.sort(np.concatenate([[0, 127, 128, H - 1], rng.choice(np.arange(1, H - 1), 60,
                                                                      replace=False)]))
        rows = np.concatenate([ch, H + ch, 2 * H + ch])
        sub = dict(c, w_in=c["w_in"][rows], w=np.ascontiguousarray(c["w"][ch]),
                   pool=np.ascontiguousarray(c["pool"][:, ch]), H=len(ch))
        y_ref, pool_ref = run_oracle(sub, None if bias is None else bias[ch])
        y, pool = y[:, ch], pool[:, ch]
    else:
        y_ref, pool_ref = run_oracle(c, bias)
    assert_bits(pool, pool_ref, "pool (new state bit-exact, other slots unchanged)")
    assert_close("bf16", y, y_ref, "y")


@pytest.mark.parametrize("H,splits", [(128, [7000, 1, 2, 13000]), (192, [5000, 11000])])
def test_single_sequence_continued_over_calls(H, splits):
    """A sequence prefilled in pieces, one call per piece (each call carries
    its state to the next through the slot), equals the oracle on the whole
    sequence: y piece by piece, and the final state."""
    rng = np.random.default_rng(870 + H)
    D, K = 64, 3
    T = sum(splits)
    c = make_case(rng, [T], D, H, K, extra_slots=2)
    pool = dev(c["pool"], "bf16")
    w_in, w, slot = dev(c["w_in"], "bf16"), dev(c["w"], "bf16"), dev(c["slots"], "i32")
    ys, t0 = [], 0
    for n in splits:
        cu = dev(np.array([0, n], np.int32), "i32")
        ys.append(host(sc.in_proj_prefill(dev(c["hidden"][t0:t0 + n], "bf16"), w_in, w, cu,
                                          slot, pool)))
        t0 += n
    torch.cuda.synchronize()
    assert sc.get_error() == 0
    y_ref, pool_ref = run_oracle(c)
    assert_bits(host(pool), pool_ref, "pool after the last piece")
    assert_close("bf16", np.concatenate(ys), y_ref, "y")


@pytest.mark.parametrize("T", [50, 20000])
def test_single_sequence_errors_write_nothing(T):
    """One-sequence calls (with and without the reordered walk): lengths that
    do not cover the rows, or a slot id out of range, report the error and
    leave y and the whole pool as they were."""
    rng = np.random.default_rng(880 + T)
    D, H, K = 64, 128, 3
    c = make_case(rng, [T], D, H, K, extra_slots=3)
    for cu, slots, code in ((np.array([0, T - 1], np.int32), c["slots"], sc.DEV_BAD_SEQLENS),
                            (c["cu"], np.array([10 ** 6], np.int32), sc.DEV_BAD_SLOT)):
        pool = dev(c["pool"], "bf16")
        y = torch.full((T, H), 3.0, dtype=torch.bfloat16, device="cuda")
        sc.in_proj_prefill(dev(c["hidden"], "bf16"), dev(c["w_in"], "bf16"), dev(c["w"], "bf16"),
                           dev(cu, "i32"), dev(slots, "i32"), pool, y=y)
        assert sc.get_error() == code
        assert np.all(host(y) == np.uint16(0x4040)), "y written"
        assert_bits(host(pool), c["pool"], "pool")


def test_single_sequence_calls_in_a_cuda_graph():
    """Two single-sequence fused prefills of one slot, captured in a CUDA
    graph and replayed twice, give the bits of the same calls made eagerly."""
    rng = np.random.default_rng(875)
    D, H, K = 64, 128, 3
    c1 = make_case(rng, [20000], D, H, K, extra_slots=1)
    h2 = dyadic(rng, (9000, D), 8, -3)

    def run(graph: bool):
        pool = dev(c1["pool"], "bf16")
        w_in, w, slot = dev(c1["w_in"], "bf16"), dev(c1["w"], "bf16"), dev(c1["slots"], "i32")
        hs = [dev(c1["hidden"], "bf16"), dev(h2, "bf16")]
        cus = [dev(np.array([0, len(h)], np.int32), "i32") for h in (c1["hidden"], h2)]
        ys = [torch.empty((h.shape[0], H), dtype=torch.bfloat16, device="cuda") for h in hs]
        ws = torch.empty(max(16, sc.in_proj_workspace_bytes(H, K, 1)), dtype=torch.uint8,
                         device="cuda")

        def body():
            for h, cu, y in zip(hs, cus, ys):
                sc.in_proj_prefill(h, w_in, w, cu, slot, pool, y=y, workspace=ws)

        if graph:
            side = torch.cuda.Stream()
            side.wait_stream(torch.cuda.current_stream())
            g = torch.cuda.CUDAGraph()
            with torch.cuda.stream(side):
                with torch.cuda.graph(g, stream=side):
                    body()
            g.replay()
            g.replay()
        else:
            body()
            body()
        torch.cuda.synchronize()
        return [host(y) for y in ys], host(pool)

    ys_e, pool_e = run(False)
    ys_g, pool_g = run(True)
    for a, b in zip(ys_g, ys_e):
        assert_bits(a, b, "y")
    assert_bits(pool_g, pool_e, "pool")
    assert sc.get_error() == 0


def _ambiguous(exact, bound):
    """True where [exact - bound, exact + bound] holds a bf16 rounding boundary
    (rounding is monotone, so exactly where its two ends round apart)."""
    return oracle.round_bf16(exact - bound) != oracle.round_bf16(exact + bound)


def _check_unambiguous(c, y, pool, ch=None, min_keep=0.5):
    """Outputs whose projection values all lie farther than the accumulation
    bound from a bf16 rounding boundary meet the tolerance, and their states
    match bit for bit; on the channel subset ``ch`` (all when None). Returns
    the share of outputs kept."""
    D, H, K = c["D"], c["H"], c["K"]
    ch = np.arange(H) if ch is None else np.asarray(ch)
    rows = np.concatenate([ch, H + ch, 2 * H + ch])
    sub = dict(c, w_in=c["w_in"][rows], w=np.ascontiguousarray(c["w"][ch]),
               pool=np.ascontiguousarray(c["pool"][:, ch]), H=len(ch))
    y_ref, pool_ref = run_oracle(sub)
    y, pool = y[:, ch], pool[:, ch]
    Hs = len(ch)
    h = oracle.bf16_to_f64(c["hidden"])
    wi = oracle.bf16_to_f64(sub["w_in"])
    exact = h @ wi.T
    # fp32 accumulation of D products: |error| <= lam sqrt(D) 2^-24 sum|terms| except
    # with probability below 2 exp(-lam^2 / 2) (Higham and Mary's probabilistic
    # rounding-error bound); lam = 8 puts that below 1e-13 per sum. The worst-case
    # bound (D in place of lam sqrt(D)) spans a quarter of a bf16 step at D = 128
    # and would exclude nearly every output. The ambiguous share grows with D.
    bound = 8 * np.sqrt(D) * 2.0 ** -24 * (np.abs(h) @ np.abs(wi).T)
    amb = _ambiguous(exact, bound)
    amb_b, amb_c, amb_x = amb[:, :Hs], amb[:, Hs:2 * Hs], amb[:, 2 * Hs:]
    u_amb = amb_b | amb_x
    T = y.shape[0]
    bad_in = np.zeros((T, Hs), bool)  # output (t, h) uses C_t and u of rows t-K+1 .. t
    for k in range(K):
        bad_in[k:] |= u_amb[:T - k] if k else u_amb
    bad_in |= amb_c
    keep = ~bad_in
    assert keep.mean() > min_keep, keep.mean()  # each output uses 2K + 1 projection values
    g, r = oracle.bf16_to_f64(y), oracle.bf16_to_f64(y_ref)
    ok = np.abs(g - r) <= 1e-2 + 2.0 ** -7 * np.abs(r)
    assert ok[keep].all(), f"{int((~ok[keep]).sum())} unambiguous outputs out of tolerance"
    # states: the last K u of each sequence, where unambiguous
    cu = c["cu"]
    for i, s in enumerate(c["slots"]):
        n = cu[i + 1] - cu[i]
        for m in range(K):
            t = cu[i + 1] - K + m
            if n + m < K or t < cu[i]:
                continue
            sel = ~u_amb[t]
            np.testing.assert_array_equal(pool[s, sel, m], pool_ref[s, sel, m])
    return float(keep.mean())


def test_normal_inputs_outside_rounding_ambiguity():
    """Normal inputs at D = 128, every channel."""
    rng = np.random.default_rng(860)
    c = make_case(rng, [200, 0, 3, 333, 64], 128, 128, 3, exact=False)
    y, pool = run_gpu(c)
    _check_unambiguous(c, y, pool)


def _check_intervals(c, y, pool, ch):
    """Every output against the range the fp32 accumulation allows.

    Each projection value the GPU rounds is within the accumulation bound of
    the exact value (Higham-Mary, lam = 8, as above), and bf16 rounding is
    monotone, so the GPU's bf16 value is round(exact - bound) or
    round(exact + bound). Carried through u = round(B x), the K-tap window and
    y = C z by interval arithmetic, this gives for every output a range that
    holds the GPU's value up to its own fp32 rounding; y must lie within the
    usual tolerance of that range, and every state value within its range
    (bit-exact where the range is one value). No output is excluded."""
    D, H, K = c["D"], c["H"], c["K"]
    ch = np.asarray(ch)
    Hs = len(ch)
    rows = np.concatenate([ch, H + ch, 2 * H + ch])
    h = oracle.bf16_to_f64(c["hidden"])
    wi = oracle.bf16_to_f64(c["w_in"][rows])
    exact = h @ wi.T
    bound = 8 * np.sqrt(D) * 2.0 ** -24 * (np.abs(h) @ np.abs(wi).T)
    lo = oracle.bf16_to_f64(oracle.round_bf16(exact - bound))
    hi = oracle.bf16_to_f64(oracle.round_bf16(exact + bound))
    B, C, X = [(lo[:, j * Hs:(j + 1) * Hs], hi[:, j * Hs:(j + 1) * Hs]) for j in range(3)]
    uc = [oracle.bf16_to_f64(oracle.round_bf16(b * x)) for b in B for x in X]
    u_lo, u_hi = np.minimum.reduce(uc), np.maximum.reduce(uc)
    w = oracle.bf16_to_f64(c["w"][ch])  # [Hs, K]
    g = oracle.bf16_to_f64(y[:, ch])
    gp = oracle.bf16_to_f64(pool[:, ch])
    cu = c["cu"]
    for i, slot in enumerate(c["slots"]):
        s0, s1 = int(cu[i]), int(cu[i + 1])
        n = s1 - s0
        st = oracle.bf16_to_f64(c["pool"][slot][ch]).T  # [K, Hs]
        e_lo = np.concatenate([st, u_lo[s0:s1]])       # [state; u] of the sequence
        e_hi = np.concatenate([st, u_hi[s0:s1]])
        z_lo = np.zeros((n, Hs))
        z_hi = np.zeros((n, Hs))
        for k in range(K):  # row j's window is ext[j + 1 .. j + K]
            a, b = w[:, k] * e_lo[1 + k:1 + k + n], w[:, k] * e_hi[1 + k:1 + k + n]
            z_lo += np.minimum(a, b)
            z_hi += np.maximum(a, b)
        yc = [cc[s0:s1] * z for cc in C for z in (z_lo, z_hi)]
        y_lo, y_hi = np.minimum.reduce(yc), np.maximum.reduce(yc)
        tol = lambda v: 1e-2 + 2.0 ** -7 * np.abs(v)  # noqa: E731
        gi = g[s0:s1]
        ok = (gi >= y_lo - tol(y_lo)) & (gi <= y_hi + tol(y_hi))
        assert ok.all(), f"sequence {i}: {int((~ok).sum())} outputs outside their range"
        f_lo, f_hi = e_lo[n:n + K].T, e_hi[n:n + K].T   # final state [Hs, K]
        gs = gp[slot]
        assert np.all((gs >= f_lo) & (gs <= f_hi)), f"sequence {i}: state outside its range"
        one = f_lo == f_hi
        np.testing.assert_array_equal(gs[one], f_lo[one])
    untouched = np.setdiff1d(np.arange(c["pool"].shape[0]), c["slots"])
    assert_bits(pool[untouched], c["pool"][untouched], "untouched slots")


def test_normal_inputs_within_accumulation_ranges_lfm2_width():
    """Normal inputs at LFM2-1.2B's width (D = H = 2048): four sequences that
    continue from N(0, 1) states, 4,099 rows, oracle ranges on 64 sampled
    channels, every row. At this depth the accumulation bound puts about 46%
    of the projection values within reach of a bf16 rounding boundary, so
    excluding the outputs that touch one (as at D = 128) would keep only 1.3%
    of them; the ranges keep all."""
    rng = np.random.default_rng(861)
    c = make_case(rng, [1000, 7, 2048, 1044], 2048, 2048, 3, exact=False)
    y, pool = run_gpu(c)
    ch = np.sort(np.concatenate([[0, 63, 64, 127, 128, 1023, 1024, 2047],
                                 rng.choice(np.arange(129, 2040), 56, replace=False)]))
    _check_intervals(c, y, pool, ch)


def test_normal_inputs_within_accumulation_ranges_small():
    rng = np.random.default_rng(862)
    c = make_case(rng, [200, 0, 3, 333, 64, 1, 2], 128, 192, 4, exact=False)
    y, pool = run_gpu(c)
    _check_intervals(c, y, pool, np.arange(192))


def test_errors_write_nothing():
    rng = np.random.default_rng(870)
    c = make_case(rng, [5, 9, 4], 64, 64, 3)
    bad = c["cu"].copy()
    bad[1], bad[2] = 9, 5  # not non-decreasing
    pool = dev(c["pool"], "bf16")
    y0 = torch.full((18, 64), 3.0, dtype=torch.bfloat16, device="cuda")
    sc.in_proj_prefill(dev(c["hidden"], "bf16"), dev(c["w_in"], "bf16"), dev(c["w"], "bf16"),
                       dev(bad, "i32"), dev(c["slots"], "i32"), pool, y=y0)
    assert sc.get_error() == sc.DEV_BAD_SEQLENS
    assert np.all(host(y0) == np.uint16(0x4040))
    assert_bits(host(pool), c["pool"], "pool")
    # a bad slot skips that sequence only
    slots = c["slots"].copy()
    slots[1] = 10 ** 6
    y1 = torch.full((18, 64), 3.0, dtype=torch.bfloat16, device="cuda")
    pool = dev(c["pool"], "bf16")
    sc.in_proj_prefill(dev(c["hidden"], "bf16"), dev(c["w_in"], "bf16"), dev(c["w"], "bf16"),
                       dev(c["cu"], "i32"), dev(slots, "i32"), pool, y=y1)
    assert sc.get_error() == sc.DEV_BAD_SLOT
    yh = host(y1)
    assert np.all(yh[5:14] == np.uint16(0x4040))
    pool_ref = c["pool"].copy()
    cut = dict(c, cu=np.array([0, 5], np.int32), slots=c["slots"][:1], hidden=c["hidden"][:5])
    y_ref, p_ref = run_oracle(dict(cut, pool=pool_ref))
    assert_close("bf16", yh[:5], y_ref, "y of the good sequence")


def test_no_rows_with_sequences():
    c = make_case(np.random.default_rng(880), [0, 0, 0], 64, 64, 3)
    y, pool = run_gpu(c)
    assert y.shape == (0, 64)
    assert_bits(pool, c["pool"], "pool")
    assert sc.get_error() == 0


# ----------------------------------------------------------------- out_proj

@pytest.mark.parametrize("T", [1, 127, 300])
def test_out_proj_exact_inputs(T):
    rng = np.random.default_rng(890 + T)
    H, D = 192, 512
    y = dyadic(rng, (T, H), 8, -3)
    wo = dyadic(rng, (D, H), 8, -6)
    out = sc.out_proj(dev(y, "bf16"), dev(wo, "bf16"))
    torch.cuda.synchronize()
    assert_bits(host(out), layer.out_proj("bf16", y, wo), "out")


def test_out_proj_lfm2_shape_sampled_columns():
    rng = np.random.default_rng(895)
    T, H, D = 4096, 2048, 2048
    y = dyadic(rng, (T, H), 8, -3)
    wo = dyadic(rng, (D, H), 8, -6)
    out = host(sc.out_proj(dev(y, "bf16"), dev(wo, "bf16")))
    cols = np.sort(rng.choice(D, 48, replace=False))
    assert_bits(out[:, cols], layer.out_proj("bf16", y, wo[cols]), "out")


@pytest.mark.parametrize("T,H,D", [(1000, 64, 768), (513, 128, 256), (4133, 2048, 2048)])
def test_out_proj_every_column_on_sampled_rows(T, H, D):
    """Every output column, on sampled rows including the first and the last
    ones."""
    rng = np.random.default_rng(896 + T)
    y = dyadic(rng, (T, H), 8, -3)
    wo = dyadic(rng, (D, H), 8, -6)
    out = host(sc.out_proj(dev(y, "bf16"), dev(wo, "bf16")))
    rows = np.unique(np.concatenate([[0, 1, 127, 128, 255, 256, T - 2, T - 1],
                                     rng.choice(T, min(T, 56), replace=False)]))
    assert_bits(out[rows], layer.out_proj("bf16", y[rows], wo), "out")


def test_layer_chain_against_the_oracle():
    """in_proj + conv, then out_proj: the whole ShortConv layer."""
    rng = np.random.default_rng(899)
    c = make_case(rng, [70, 1, 190], 256, 128, 3)
    wo = dyadic(rng, (256, 128), 8, -6)
    pool = dev(c["pool"], "bf16")
    y = sc.in_proj_prefill(dev(c["hidden"], "bf16"), dev(c["w_in"], "bf16"), dev(c["w"], "bf16"),
                           dev(c["cu"], "i32"), dev(c["slots"], "i32"), pool)
    out = host(sc.out_proj(y, dev(wo, "bf16")))
    y_ref, _ = run_oracle(c)
    out_ref = layer.out_proj("bf16", y_ref, wo)
    # y may differ from the oracle's by one bf16 rounding; out inherits that
    assert_close("bf16", out, out_ref, "out")


def test_graph_captured_projections_match_eager_calls():
    """Two continued in_proj-fused prefills and an out_proj each, captured in one
    CUDA graph (tensor maps are encoded on the host at capture time), give the
    bits of eager calls."""
    rng = np.random.default_rng(905)
    c1 = make_case(rng, [100, 37], 128, 128, 3)
    c2 = make_case(rng, [60, 5], 128, 128, 3)
    wo = dyadic(rng, (256, 128), 8, -6)

    def run(graph: bool):
        pool = dev(c1["pool"], "bf16")
        args = []
        for c in (c1, c2):
            args.append((dev(c["hidden"], "bf16"), dev(c1["w_in"], "bf16"), dev(c1["w"], "bf16"),
                         dev(c["cu"], "i32"), dev(c1["slots"], "i32")))
        ys = [torch.empty((a[0].shape[0], 128), dtype=torch.bfloat16, device="cuda") for a in args]
        outs = [torch.empty((a[0].shape[0], 256), dtype=torch.bfloat16, device="cuda") for a in args]
        ws = [torch.empty(sc.in_proj_workspace_bytes(128, 3, 2), dtype=torch.uint8, device="cuda")
              for _ in args]
        w_out = dev(wo, "bf16")

        def body():
            for a, y, o, wsp in zip(args, ys, outs, ws):
                sc.in_proj_prefill(*a, pool, y=y, workspace=wsp)
                sc.out_proj(y, w_out, out=o)

        if graph:
            side = torch.cuda.Stream()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.stream(side):
                with torch.cuda.graph(g, stream=side):
                    body()
            g.replay()
        else:
            body()
        torch.cuda.synchronize()
        return [host(t) for t in ys + outs + [pool]]

    eager, graphed = run(False), run(True)
    for a, b in zip(eager, graphed):
        assert_bits(b, a, "graph vs eager")
    assert sc.get_error() == 0


def test_graph_captured_decode_steps_match_eager_calls():
    """Three fused decode steps (in_proj + decode, one token per sequence)
    captured in one CUDA graph give the bits of eager calls."""
    rng = np.random.default_rng(906)
    c = make_decode_case(rng, 200, 256, 128, 3)
    tokens = [dyadic(rng, (200, 256), 8, -3) for _ in range(3)]

    def run(graph: bool):
        pool = dev(c["pool"], "bf16")
        w_in, w, slots = dev(c["w_in"], "bf16"), dev(c["w"], "bf16"), dev(c["slots"], "i32")
        hs = [dev(t, "bf16") for t in tokens]
        ys = [torch.empty((200, 128), dtype=torch.bfloat16, device="cuda") for _ in hs]

        def body():
            for h, y in zip(hs, ys):
                sc.in_proj_decode(h, w_in, w, slots, pool, y=y)

        if graph:
            side = torch.cuda.Stream()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.stream(side):
                with torch.cuda.graph(g, stream=side):
                    body()
            g.replay()
        else:
            body()
        torch.cuda.synchronize()
        return [host(t) for t in ys + [pool]]

    eager, graphed = run(False), run(True)
    for a, b in zip(eager, graphed):
        assert_bits(b, a, "graph vs eager")
    # and the three steps against the oracle, token by token
    ref = c["pool"].copy()
    for t, got in zip(tokens, eager[:3]):
        st, y_ref = layer.in_proj_decode("bf16", t, c["w_in"], c["w"], c["slots"], ref)
        assert st == oracle.OK
        assert_close("bf16", got, y_ref, "y")
    assert_bits(eager[3], ref, "pool")
    assert sc.get_error() == 0


def test_more_sequences_than_staged_in_shared_memory():
    """600 sequences (more than the 512 cu_seqlens entries staged in shared
    memory): the epilogue looks rows up in global memory."""
    rng = np.random.default_rng(910)
    lengths = rng.integers(0, 4, size=600)
    c = make_case(rng, lengths, 64, 128, 3)
    y, pool = run_gpu(c)
    y_ref, pool_ref = run_oracle(c)
    assert sc.get_error() == 0
    assert_close("bf16", y, y_ref, "y")
    assert_bits(pool, pool_ref, "pool")


# ------------------------------------------------ in_proj fused with decode

def make_decode_case(rng, N, D, H, K, extra_slots=7, exact=True, with_bias=False):
    if exact:
        hidden = dyadic(rng, (N, D), 8, -3)
        w_in = dyadic(rng, (3 * H, D), 8, -6)
    else:
        hidden = oracle.round_bf16(rng.standard_normal((N, D)))
        w_in = oracle.round_bf16(rng.standard_normal((3 * H, D)) / np.sqrt(D))
    w = oracle.round_bf16(rng.standard_normal((H, K)) * np.sqrt(1 / 3))
    bias = oracle.round_bf16(rng.standard_normal(H) * 0.5) if with_bias else None
    n_slots = N + extra_slots
    slots = rng.permutation(n_slots)[:N].astype(np.int32)
    pool = np.full((n_slots, H, K), 0xDEAD, np.uint16)  # untouched slots keep this
    for s in slots:
        pool[s] = oracle.round_bf16(rng.standard_normal((H, K)))
    return dict(hidden=hidden, w_in=w_in, w=w, bias=bias, slots=slots, pool=pool,
                cu=np.arange(N + 1, dtype=np.int32), D=D, H=H, K=K)


def run_decode_gpu(c):
    pool = dev(c["pool"], "bf16")
    y = sc.in_proj_decode(dev(c["hidden"], "bf16"), dev(c["w_in"], "bf16"), dev(c["w"], "bf16"),
                          dev(c["slots"], "i32"), pool,
                          bias=None if c["bias"] is None else dev(c["bias"], "bf16"))
    torch.cuda.synchronize()
    return host(y), host(pool)


@pytest.mark.parametrize("N,D,H,K", [(1, 64, 64, 3), (5, 128, 64, 1), (37, 64, 192, 2),
                                     (129, 128, 64, 3), (300, 64, 128, 4),
                                     (256, 2048, 2048, 3)])
def test_in_proj_decode_exact_inputs(N, D, H, K):
    """Exact projections: y within the bf16 tolerance of the oracle, states bit
    for bit, untouched slots kept, and the same bits as shortconv_decode on
    the projection."""
    rng = np.random.default_rng(880 + N + K)
    c = make_decode_case(rng, N, D, H, K)
    y, pool = run_decode_gpu(c)
    assert sc.get_error() == 0
    ref = c["pool"].copy()
    st, y_ref = layer.in_proj_decode("bf16", c["hidden"], c["w_in"], c["w"], c["slots"], ref)
    assert st == oracle.OK
    assert_close("bf16", y, y_ref, "y")
    assert_bits(pool, ref, "pool")
    bcx = layer.in_proj("bf16", c["hidden"], c["w_in"])
    pool2 = dev(c["pool"], "bf16")
    y2 = sc.decode(dev(bcx, "bf16"), dev(c["w"], "bf16"), dev(c["slots"], "i32"), pool2)
    torch.cuda.synchronize()
    assert_bits(y, host(y2), "y against shortconv_decode")
    assert_bits(pool, host(pool2), "pool against shortconv_decode")


def test_in_proj_decode_with_bias():
    rng = np.random.default_rng(890)
    c = make_decode_case(rng, 77, 128, 128, 3, with_bias=True)
    y, pool = run_decode_gpu(c)
    assert sc.get_error() == 0
    ref = c["pool"].copy()
    st, y_ref = layer.in_proj_decode("bf16", c["hidden"], c["w_in"], c["w"], c["slots"], ref,
                                     bias=c["bias"])
    assert st == oracle.OK
    assert_close("bf16", y, y_ref, "y")
    assert_bits(pool, ref, "pool")


def test_in_proj_decode_normal_inputs_lfm2_shape():
    """Serving shape: 256 sequences, D = H = 2048, normal inputs; every output
    within its accumulation range (see _check_intervals), 64 sampled channels."""
    rng = np.random.default_rng(891)
    c = make_decode_case(rng, 256, 2048, 2048, 3, exact=False)
    y, pool = run_decode_gpu(c)
    assert sc.get_error() == 0
    ch = np.sort(np.concatenate([[0, 15, 16, 31, 32, 1023, 1024, 2047],
                                 rng.choice(np.arange(33, 2040), 56, replace=False)]))
    _check_intervals(c, y, pool, ch)


def test_in_proj_decode_continues_a_prefill_token_by_token():
    """A fused prefill of a sequence's first rows, then fused decode steps,
    equal the fused prefill of the whole sequence (exact projections)."""
    rng = np.random.default_rng(892)
    D, H, K, T = 128, 192, 3, 9
    hs = dyadic(rng, (T, D), 8, -3)
    w_in = dyadic(rng, (3 * H, D), 8, -6)
    w = oracle.round_bf16(rng.standard_normal((H, K)) * np.sqrt(1 / 3))
    pa = dev(np.zeros((2, H, K), np.uint16), "bf16")
    ya = sc.in_proj_prefill(dev(hs, "bf16"), dev(w_in, "bf16"), dev(w, "bf16"),
                            dev(np.array([0, T], np.int32), "i32"), dev(np.array([1], np.int32), "i32"),
                            pa)
    pb = dev(np.zeros((2, H, K), np.uint16), "bf16")
    yb = [sc.in_proj_prefill(dev(hs[:3], "bf16"), dev(w_in, "bf16"), dev(w, "bf16"),
                             dev(np.array([0, 3], np.int32), "i32"),
                             dev(np.array([1], np.int32), "i32"), pb)]
    for t in range(3, T):
        yb.append(sc.in_proj_decode(dev(hs[t:t + 1], "bf16"), dev(w_in, "bf16"), dev(w, "bf16"),
                                    dev(np.array([1], np.int32), "i32"), pb))
    torch.cuda.synchronize()
    assert_bits(np.concatenate([host(v) for v in yb]), host(ya), "y")
    assert_bits(host(pb), host(pa), "pool")
    assert sc.get_error() == 0


def test_in_proj_decode_bad_slot_skips_that_sequence():
    rng = np.random.default_rng(893)
    c = make_decode_case(rng, 40, 64, 64, 3)
    slots = c["slots"].copy()
    slots[7] = 10 ** 6
    pool = dev(c["pool"], "bf16")
    y = torch.full((40, 64), 3.0, dtype=torch.bfloat16, device="cuda")
    sc.in_proj_decode(dev(c["hidden"], "bf16"), dev(c["w_in"], "bf16"), dev(c["w"], "bf16"),
                      dev(slots, "i32"), pool, y=y)
    assert sc.get_error() == sc.DEV_BAD_SLOT
    ref = c["pool"].copy()
    keep = np.arange(40) != 7
    st, y_ref = layer.in_proj_decode("bf16", c["hidden"][keep], c["w_in"], c["w"],
                                     c["slots"][keep], ref)
    g = host(y)
    assert np.all(g[7] == np.uint16(0x4040)), "the skipped row was written"
    assert_close("bf16", g[keep], y_ref, "y")
    assert_bits(host(pool), ref, "pool")


@pytest.mark.parametrize("seed", range(8))
def test_in_proj_decode_seeded_shapes(seed):
    """Seeded shapes: N in 1..600 (ragged last tile), H a multiple of 64 up to
    320, D a multiple of 64 up to 384, K in 1..4, with or without a bias;
    exact projections, against the oracle."""
    rng = np.random.default_rng(7700 + seed)
    N = int(rng.integers(1, 601))
    D = 64 * int(rng.integers(1, 7))
    H = 64 * int(rng.integers(1, 6))
    K = int(rng.integers(1, 5))
    c = make_decode_case(rng, N, D, H, K, extra_slots=int(rng.integers(0, 9)),
                         with_bias=bool(rng.integers(0, 2)))
    y, pool = run_decode_gpu(c)
    assert sc.get_error() == 0
    ref = c["pool"].copy()
    st, y_ref = layer.in_proj_decode("bf16", c["hidden"], c["w_in"], c["w"], c["slots"], ref,
                                     bias=c["bias"])
    assert st == oracle.OK
    assert_close("bf16", y, y_ref, "y")
    assert_bits(pool, ref, "pool")
