"""Calls on several streams at once, each on its own buffers.

The library keeps no per-call state on the device besides the shared error
word, so work enqueued on different streams may overlap freely. Four streams
each run a different call (prefill, decode, verify + rollback, backward),
enqueued interleaved and repeated; every result must match the oracle.
"""
import numpy as np
import pytest
import torch

import oracle
import lfm2_gated_short_gb300 as sc
from lfm2_gated_short_gb300 import workloads as wl
from gpu_util import assert_bits, assert_close, assert_dw_close, dev, host

pytestmark = pytest.mark.gpu


def test_four_streams_interleaved():
    H, K, reps = 512, 3, 3
    streams = [torch.cuda.Stream() for _ in range(4)]
    p = wl.varlen_prefill(n_seqs=6, lo=20, hi=300, H=H, K=K, n_slots=10, seed=1100)
    d = wl.decode_serving(layers=1, steps=reps, batch=40, H=H, K=K, n_slots=64, seed=1101)
    v = wl.verify_serving(layers=1, batch=12, D=6, H=H, K=K, n_slots=20, seed=1102)
    t = wl.training(T=2000, H=H, K=K, seed=1103)
    # device inputs, made before any stream runs
    p_in = (dev(p.bcx, "bf16"), dev(p.w, "bf16"), dev(p.cu_seqlens, "i32"), dev(p.slot_ids, "i32"))
    p_pools = [dev(p.pool, "bf16") for _ in range(reps)]
    d_w, d_slots, d_pool = dev(d.w[0], "bf16"), dev(d.slot_ids, "i32"), dev(d.pools[0], "bf16")
    d_rows = [dev(d.bcx[0, s], "bf16") for s in range(reps)]
    v_in = (dev(v.bcx[0], "bf16"), dev(v.w[0], "bf16"), dev(v.slot_ids, "i32"))
    v_pools = [dev(v.pools[0], "bf16") for _ in range(reps)]
    v_acc = dev(v.accepted, "i32")
    t_in = (dev(t.bcx, "bf16"), dev(t.w, "bf16"), dev(t.dy, "bf16"))
    torch.cuda.synchronize()
    outs = {"p": [], "d": [], "v": [], "t": []}
    for r in range(reps):
        with torch.cuda.stream(streams[0]):
            outs["p"].append(sc.prefill(*p_in, p_pools[r]))
        with torch.cuda.stream(streams[1]):
            outs["d"].append(sc.decode(d_rows[r], d_w, d_slots, d_pool))
        with torch.cuda.stream(streams[2]):
            win, y = sc.verify(*v_in, v_pools[r], v.D)
            sc.rollback(win, v_acc, v_in[2], v_pools[r])
            outs["v"].append((win, y))
        with torch.cuda.stream(streams[3]):
            outs["t"].append(sc.backward(*t_in))
    torch.cuda.synchronize()
    assert sc.get_error() == 0
    # prefill: every repetition from the same initial pool
    ref = p.pool.copy()
    st, y_ref = oracle.prefill("bf16", p.bcx, p.w, p.cu_seqlens, p.slot_ids, ref)
    assert st == oracle.OK
    for r in range(reps):
        assert_close("bf16", host(outs["p"][r]), y_ref, f"prefill y, rep {r}")
        assert_bits(host(p_pools[r]), ref, f"prefill pool, rep {r}")
    # decode: consecutive steps on one pool, in stream order
    ref = d.pools[0].copy()
    for r in range(reps):
        st, y_ref = oracle.decode("bf16", d.bcx[0, r], d.w[0], d.slot_ids, ref)
        assert st == oracle.OK
        assert_close("bf16", host(outs["d"][r]), y_ref, f"decode y, step {r}")
    assert_bits(host(d_pool), ref, "decode pool")
    # verify + rollback: every repetition from the same initial pool
    st, win_ref, y_ref = oracle.verify("bf16", v.bcx[0], v.w[0], v.slot_ids, v.pools[0], v.D)
    assert st == oracle.OK
    ref = v.pools[0].copy()
    assert oracle.rollback("bf16", win_ref, v.accepted, v.slot_ids, ref) == oracle.OK
    for r in range(reps):
        assert_bits(host(outs["v"][r][0]), win_ref, f"verify windows, rep {r}")
        assert_close("bf16", host(outs["v"][r][1]), y_ref, f"verify y, rep {r}")
        assert_bits(host(v_pools[r]), ref, f"pool after rollback, rep {r}")
    # backward: deterministic, so every repetition has the same bits
    st, d_ref, dw_ref = oracle.backward("bf16", t.bcx, t.w, t.dy)
    assert st == oracle.OK
    for r in range(reps):
        assert_close("bf16", host(outs["t"][r][0]), d_ref, f"dB|dC|dx, rep {r}")
        assert_dw_close(host(outs["t"][r][1]), dw_ref)
        assert np.array_equal(host(outs["t"][r][1]), host(outs["t"][0][1])), "dW bits"


def test_host_threads_calling_at_once():
    """Four host threads, each with its own stream and buffers, call the
    library concurrently (the binding's C calls release the GIL). Results
    must match single-threaded calls bit for bit."""
    import threading
    H, K, n_iter = 256, 3, 15
    cases = []
    for j in range(4):
        p = wl.varlen_prefill(n_seqs=3 + j, lo=10, hi=200, H=H, K=K, n_slots=8, seed=1200 + j)
        cases.append(p)
    inputs = [(dev(p.bcx, "bf16"), dev(p.w, "bf16"), dev(p.cu_seqlens, "i32"),
               dev(p.slot_ids, "i32")) for p in cases]
    expect = []
    for j, p in enumerate(cases):  # single-threaded results first
        pool = dev(p.pool, "bf16")
        y = sc.prefill(*inputs[j], pool)
        dbcx, dw = sc.backward(inputs[j][0], inputs[j][1], y.repeat(1, 1))
        torch.cuda.synchronize()
        expect.append((host(y), host(pool), host(dbcx), host(dw)))
    results = [None] * 4
    errors = []

    def worker(j):
        try:
            s = torch.cuda.Stream()
            with torch.cuda.stream(s):
                for _ in range(n_iter):
                    pool = dev(cases[j].pool, "bf16")
                    y = sc.prefill(*inputs[j], pool)
                    dbcx, dw = sc.backward(inputs[j][0], inputs[j][1], y.repeat(1, 1))
            s.synchronize()
            results[j] = (host(y), host(pool), host(dbcx), host(dw))
        except Exception as e:  # reported below, on the main thread
            errors.append(e)

    threads = [threading.Thread(target=worker, args=(j,)) for j in range(4)]
    for th in threads:
        th.start()
    for th in threads:
        th.join()
    assert not errors, errors
    assert sc.get_error() == 0
    for j in range(4):
        for got, want, what in zip(results[j], expect[j], ("y", "pool", "dbcx", "dw")):
            assert np.array_equal(got, want), f"thread {j}: {what}"


def test_host_threads_calling_the_projections_at_once():
    """Four host threads, each with its own stream and buffers, call the
    tensor-core projections concurrently: a fused in_proj prefill (one
    sequence in threads 0 and 2, so that the fused kernel writes the state
    itself; three in threads 1 and 3, with the commit pass), out_proj on its
    output, and a fused decode step continuing the same slots. Results must
    match single-threaded calls bit for bit."""
    import threading
    D, H, K, n_iter = 64, 128, 3, 4
    rng = np.random.default_rng(1300)

    def dyadic(shape, lim, exp):
        return oracle.round_bf16(rng.integers(-lim, lim, size=shape, endpoint=True) * 2.0 ** exp)

    cases = []
    for j in range(4):
        lengths = [20000] if j % 2 == 0 else [700, 3, 5000]
        cu = np.r_[0, np.cumsum(lengths)].astype(np.int32)
        n = len(lengths)
        pool = np.zeros((n + 2, H, K), np.uint16)
        pool[:n] = oracle.round_bf16(rng.standard_normal((n, H, K)))
        cases.append(dict(hidden=dev(dyadic((int(cu[-1]), D), 8, -3), "bf16"),
                          w_in=dev(dyadic((3 * H, D), 8, -6), "bf16"),
                          w=dev(oracle.round_bf16(rng.standard_normal((H, K)) * 0.5), "bf16"),
                          cu=dev(cu, "i32"), slots=dev(np.arange(n, dtype=np.int32), "i32"),
                          w_out=dev(dyadic((256, H), 8, -6), "bf16"),
                          step=dev(dyadic((n, D), 8, -3), "bf16"), pool=pool))

    def run(c):
        pool = dev(c["pool"], "bf16")
        y = sc.in_proj_prefill(c["hidden"], c["w_in"], c["w"], c["cu"], c["slots"], pool)
        out = sc.out_proj(y, c["w_out"])
        y1 = sc.in_proj_decode(c["step"], c["w_in"], c["w"], c["slots"], pool)
        return y, pool, out, y1

    expect = []
    for c in cases:  # single-threaded results first
        r = run(c)
        torch.cuda.synchronize()
        expect.append(tuple(host(v) for v in r))
    results = [None] * 4
    errors = []

    def worker(j):
        try:
            s = torch.cuda.Stream()
            with torch.cuda.stream(s):
                for _ in range(n_iter):
                    r = run(cases[j])
            s.synchronize()
            results[j] = tuple(host(v) for v in r)
        except Exception as e:  # reported below, on the main thread
            errors.append(e)

    threads = [threading.Thread(target=worker, args=(j,)) for j in range(4)]
    for th in threads:
        th.start()
    for th in threads:
        th.join()
    assert not errors, errors
    assert sc.get_error() == 0
    for j in range(4):
        for got, want, what in zip(results[j], expect[j], ("y", "pool", "out", "decode y")):
            assert np.array_equal(got, want), f"thread {j}: {what}"
