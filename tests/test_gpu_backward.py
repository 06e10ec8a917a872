"""GPU backward (dB, dC, dx and the fp32 dW reduction) against the CPU oracle."""
import numpy as np
import pytest
import torch

import oracle
import lfm2_gated_short_gb300 as sc
from lfm2_gated_short_gb300 import workloads as wl
from fixtures import worked_example
from gpu_util import assert_bits, assert_close, assert_dw_close, dev, host

pytestmark = pytest.mark.gpu


def check_against_oracle(p, dbcx, dw, channels=None):
    """Compare GPU outputs with the oracle, optionally on a subset of channels.

    Channels are independent, so the oracle run on the columns of a channel
    subset is the same computation as the full run restricted to them.
    """
    H = p.H
    ch = np.arange(H) if channels is None else np.asarray(channels)
    cols = np.concatenate([ch, H + ch, 2 * H + ch])
    st, d_ref, dw_ref = oracle.backward(p.dtype, p.bcx[:, cols], p.w[ch], p.dy[:, ch])
    assert st == oracle.OK
    assert_close(p.dtype, dbcx[:, cols], d_ref, "dB|dC|dx")
    assert_dw_close(dw[ch], dw_ref)


def run(p):
    dbcx, dw = sc.backward(dev(p.bcx, p.dtype), dev(p.w, p.dtype), dev(p.dy, p.dtype))
    torch.cuda.synchronize()
    return host(dbcx), host(dw)


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_worked_example(dtype):
    ex = worked_example(dtype)
    dbcx, dw = sc.backward(dev(ex["bcx"], dtype), dev(ex["w"], dtype), dev(ex["dy"], dtype))
    d = host(dbcx)
    H = ex["H"]
    assert_bits(d[:, :H], ex["dB"], "dB")
    assert_bits(d[:, H:2 * H], ex["dC"], "dC")
    assert_bits(d[:, 2 * H:], ex["dx"], "dx")
    np.testing.assert_array_equal(host(dw), ex["dW"])


@pytest.mark.parametrize("K", [1, 2, 3, 4])
@pytest.mark.parametrize("T", [0, 1, 2, 5, 17, 301, 4099])
@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_backward_small(dtype, T, K):
    p = wl.training(T=T, H=256, K=K, seed=90 + K + T, dtype=dtype)
    dbcx, dw = run(p)
    check_against_oracle(p, dbcx, dw)
    if T == 0:
        assert np.all(dw == 0.0)


def test_backward_is_deterministic_and_overwrites_dw():
    p = wl.training(T=5000, H=512, K=3, seed=95)
    bcx, w, dy = dev(p.bcx, "bf16"), dev(p.w, "bf16"), dev(p.dy, "bf16")
    dw = torch.full((512, 3), 7.0, device="cuda")
    ws = torch.full((sc.backward_workspace_bytes(512, 3, 5000),), 0xFF, dtype=torch.uint8,
                    device="cuda")
    d1, w1 = sc.backward(bcx, w, dy, dw=dw, workspace=ws)
    w1 = host(w1)
    d2, w2 = sc.backward(bcx, w, dy, workspace=ws)
    assert_bits(host(d2), host(d1), "dbcx")
    assert_bits(host(w2), w1, "dW")


def test_backward_T65536_H2048_sampled_channels():
    """Long-sequence training shape: T=65536, H=2048, K=3; oracle on 64 channels."""
    p = wl.training()
    dbcx, dw = run(p)
    rng = np.random.default_rng(0)
    ch = np.sort(np.concatenate([[0, 7, 8, 255, 256, 2047],
                                 rng.choice(np.arange(9, 2040), 58, replace=False)]))
    check_against_oracle(p, dbcx, dw, ch)


@pytest.mark.parametrize("H", [2560, 4096])
def test_backward_channel_slices_wider_than_one_cta(H):
    p = wl.training(T=333, H=H, K=3, seed=96)
    dbcx, dw = run(p)
    check_against_oracle(p, dbcx, dw)


# ------------------------------------------- packed varlen, with states

def _varlen_case(lengths, H, K, seed, dtype="bf16", with_init=True, with_final=True):
    rng = np.random.default_rng(seed)
    lengths = np.asarray(lengths, np.int64)
    cu = np.r_[0, np.cumsum(lengths)].astype(np.int32)
    T, N = int(cu[-1]), len(lengths)
    bcx = wl.normal(rng, (T, 3 * H), 1.0, dtype)
    w = wl.normal(rng, (H, K), wl.WEIGHT_STD, dtype)
    dy = wl.normal(rng, (T, H), 1.0, dtype)
    init = wl.normal(rng, (N, H, K), 1.0, dtype) if with_init else None
    dfin = rng.standard_normal((N, H, K)).astype(np.float32) if with_final else None
    return dict(dtype=dtype, H=H, K=K, cu=cu, bcx=bcx, w=w, dy=dy, init=init, dfin=dfin)


def _run_varlen(c):
    dt = c["dtype"]
    out = sc.backward_varlen(dev(c["bcx"], dt), dev(c["w"], dt), dev(c["cu"], "i32"),
                             dev(c["dy"], dt),
                             init_states=None if c["init"] is None else dev(c["init"], dt),
                             d_final=None if c["dfin"] is None else dev(c["dfin"], "f32"))
    torch.cuda.synchronize()
    return host(out[0]), host(out[1]), host(out[2])


def _check_varlen(c, dbcx, dw, dinit, channels=None):
    H = c["H"]
    ch = np.arange(H) if channels is None else np.asarray(channels)
    cols = np.concatenate([ch, H + ch, 2 * H + ch])
    init = None if c["init"] is None else np.ascontiguousarray(c["init"][:, ch])
    dfin = None if c["dfin"] is None else np.ascontiguousarray(c["dfin"][:, ch].astype(np.float64))
    st, d_ref, dw_ref, di_ref = oracle.backward_varlen(
        c["dtype"], np.ascontiguousarray(c["bcx"][:, cols]), np.ascontiguousarray(c["w"][ch]),
        c["cu"], np.ascontiguousarray(c["dy"][:, ch]), init, dfin)
    assert st == oracle.OK
    assert_close(c["dtype"], dbcx[:, cols], d_ref, "dB|dC|dx")
    assert_dw_close(dw[ch], dw_ref)
    assert_dw_close(dinit[:, ch], di_ref, "d_init")


@pytest.mark.parametrize("K", [1, 2, 3, 4])
@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_backward_varlen_mixed_lengths(dtype, K):
    lengths = [5, 0, 1, 2, 3, 40, 0, 7, 64, 1, 130, 2]
    c = _varlen_case(lengths, 256, K, 200 + K, dtype)
    _check_varlen(c, *_run_varlen(c))


@pytest.mark.parametrize("with_init,with_final", [(False, False), (True, False), (False, True)])
def test_backward_varlen_optional_states(with_init, with_final):
    c = _varlen_case([17, 3, 0, 250, 9], 512, 3, 210, "bf16", with_init, with_final)
    _check_varlen(c, *_run_varlen(c))


def test_backward_varlen_many_sequences_across_row_ranges():
    rng = np.random.default_rng(211)
    lengths = rng.integers(0, 60, size=300)
    c = _varlen_case(lengths, 256, 4, 212)
    _check_varlen(c, *_run_varlen(c))


def test_dw_bits_do_not_depend_on_the_calls_in_between():
    """The launch picks its row split from the device and the shapes; calls
    with other widths in between (a different occupancy, the same slice
    count) must not change it, so dW and d_init keep their bits."""
    a = wl.training(T=3001, H=512, K=3, seed=740)
    b = wl.training(T=3001, H=64, K=3, seed=741)
    cu = np.array([0, 1000, 3001], np.int32)

    def run(t, varlen):
        args = (dev(t.bcx, "bf16"), dev(t.w, "bf16"))
        if varlen:
            out = sc.backward_varlen(args[0], args[1], dev(cu, "i32"), dev(t.dy, "bf16"))
            return host(out[1]), host(out[2])
        return host(sc.backward(args[0], args[1], dev(t.dy, "bf16"))[1]), None

    for varlen in (False, True):
        first = run(a, varlen)
        run(b, varlen)
        again = run(a, varlen)
        assert np.array_equal(first[0], again[0]), "dW bits"
        if varlen:
            assert np.array_equal(first[1], again[1]), "d_init bits"
    assert sc.get_error() == 0


def test_backward_varlen_more_sequences_than_staged_in_shared_memory():
    """900 sequences: past the 512 cu_seqlens entries staged in shared memory,
    so the kernel reads the offsets from global memory."""
    rng = np.random.default_rng(217)
    lengths = rng.integers(0, 12, size=900)
    c = _varlen_case(lengths, 128, 3, 218)
    _check_varlen(c, *_run_varlen(c))


def test_backward_varlen_one_fresh_sequence_matches_the_single_sequence_kernel():
    c = _varlen_case([3001], 512, 3, 213, with_init=False, with_final=False)
    dbcx, dw, _ = _run_varlen(c)
    d2, w2 = sc.backward(dev(c["bcx"], "bf16"), dev(c["w"], "bf16"), dev(c["dy"], "bf16"))
    assert_bits(dbcx, host(d2), "dbcx")
    np.testing.assert_array_equal(dw, host(w2))


@pytest.mark.parametrize("K", [2, 3, 4])
def test_split_T_backward_summed_on_the_host_equals_the_full_backward(K):
    """Sequence-parallel training emulated on one GPU: T rows split at T1.

    The first chunk's prefill leaves the state the second chunk starts from.
    The second chunk's backward starts from that state and returns d_init, the
    gradient of the state; the first chunk's backward takes it as d_final. The
    chunks' dB|dC|dx, and dW summed over them on the host, must equal the
    full-sequence backward: the oracle's within the tolerances, and the GPU's
    single-call backward within the dW tolerance."""
    T, T1, H = 3001, 1234, 256
    t = wl.training(T=T, H=H, K=K, seed=720 + K)
    w = dev(t.w, "bf16")
    pool = torch.zeros((1, H, K), dtype=torch.bfloat16, device="cuda")
    sc.prefill(dev(t.bcx[:T1], "bf16"), w, dev(np.array([0, T1]), "i32"),
               dev(np.array([0]), "i32"), pool)
    d_b, dw_b, dinit_b = sc.backward_varlen(
        dev(t.bcx[T1:], "bf16"), w, dev(np.array([0, T - T1]), "i32"), dev(t.dy[T1:], "bf16"),
        init_states=pool)
    d_a, dw_a, _ = sc.backward_varlen(
        dev(t.bcx[:T1], "bf16"), w, dev(np.array([0, T1]), "i32"), dev(t.dy[:T1], "bf16"),
        d_final=dinit_b)
    assert sc.get_error() == 0
    dbcx = np.concatenate([host(d_a), host(d_b)])
    dw = host(dw_a).astype(np.float64) + host(dw_b)
    st, d_ref, dw_ref = oracle.backward("bf16", t.bcx, t.w, t.dy)
    assert st == oracle.OK
    assert_close("bf16", dbcx, d_ref, "dB|dC|dx over both chunks")
    assert_dw_close(dw, dw_ref, "dW summed over the chunks")
    _, dw_full = sc.backward(dev(t.bcx, "bf16"), w, dev(t.dy, "bf16"))
    assert_dw_close(dw, host(dw_full), "dW against the single-call backward")


def test_backward_varlen_packed_lfm2_shapes_sampled_channels():
    """16 packed sequences, lengths U{64..2048}, H=2048, K=3, with states; 64 channels checked."""
    rng = np.random.default_rng(214)
    c = _varlen_case(rng.integers(64, 2048, size=16, endpoint=True), 2048, 3, 215)
    dbcx, dw, dinit = _run_varlen(c)
    ch = np.sort(np.concatenate([[0, 7, 8, 511, 512, 2047],
                                 rng.choice(np.arange(9, 2040), 58, replace=False)]))
    _check_varlen(c, dbcx, dw, dinit, ch)


def test_backward_varlen_bad_seqlens_zero_dw_and_set_the_error():
    c = _varlen_case([4, 5, 6], 64, 3, 216)
    bad = c["cu"].copy()
    bad[1], bad[2] = 9, 4                               # not non-decreasing
    dbcx0 = torch.full((15, 192), 3.0, dtype=torch.bfloat16, device="cuda")
    dbcx, dw, _ = sc.backward_varlen(dev(c["bcx"], "bf16"), dev(c["w"], "bf16"),
                                     dev(bad, "i32"), dev(c["dy"], "bf16"), dbcx=dbcx0)
    assert sc.get_error() == sc.DEV_BAD_SEQLENS
    assert np.all(host(dw) == 0.0)
    assert np.all(host(dbcx).view(np.uint16) == np.uint16(0x4040))  # 3.0 untouched
