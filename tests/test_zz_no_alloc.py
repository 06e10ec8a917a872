"""shortconv_backward_noalloc: the backward pass for callers that cannot
allocate device memory at call time (code inside a framework that owns all
device memory through its own pool, or latency-critical paths that cannot
afford an allocation's synchronization or an out-of-memory failure
mid-step). It keeps its scratch in a fixed array inside the library instead
of a caller workspace.

This file is collected last on purpose. It calls the entry point through the
C ABI and checks it, on two calls in a row, bit for bit against
shortconv_backward (which takes a caller workspace: the row split and the
fixed-order dW sum are the same, so the bits are too) and against the CPU
oracle. It must pass alone in a fresh process and after the other tests.
"""
import ctypes

import numpy as np
import pytest
import torch

import lfm2_gated_short_gb300 as sc
from lfm2_gated_short_gb300 import build as sc_build
from lfm2_gated_short_gb300 import workloads as wl
import oracle
from gpu_util import assert_bits, assert_close, assert_dw_close, dev, host

SCRATCH_LIMIT = 8 << 20  # bytes of fixed device scratch behind the call


def partial_bytes(H, K, T):
    """The fp32 dW partials the call keeps in its scratch, as the header states:
    one H*K block per row range, min(ceil(T / 16), 152) row ranges."""
    return min(max(-(-T // 16), 1), 152) * H * K * 4


def _noalloc():
    f = sc.lib().shortconv_backward_noalloc
    p, i32, i64 = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64
    f.argtypes = [i32, i32, i32, p, i64, p, p, p, p, p]
    f.restype = i32
    return f


def call_noalloc(bcx, w, dy):
    T = bcx.shape[0]
    H, K = w.shape
    dbcx = torch.empty_like(bcx)
    dw = torch.full((H, K), float("nan"), dtype=torch.float32, device=bcx.device)
    code = sc.SC_BF16 if bcx.dtype == torch.bfloat16 else sc.SC_F32
    st = _noalloc()(code, H, K, bcx.data_ptr(), T, w.data_ptr(), dy.data_ptr(),
                    dbcx.data_ptr(), dw.data_ptr(), torch.cuda.current_stream().cuda_stream)
    assert st == sc.SC_OK, sc.lib().shortconv_status_string(st)
    return dbcx, dw


def check_against_oracle(p, dbcx, dw, channels=None):
    """The oracle on a subset of channels (all of them when None): channels are
    independent, so its run on their columns is the full run restricted to them."""
    H = p.H
    ch = np.arange(H) if channels is None else np.asarray(channels)
    cols = np.concatenate([ch, H + ch, 2 * H + ch])
    st, d_ref, dw_ref = oracle.backward(p.dtype, p.bcx[:, cols], p.w[ch], p.dy[:, ch])
    assert st == oracle.OK
    assert_close(p.dtype, dbcx[:, cols], d_ref, "dB|dC|dx vs oracle")
    assert_dw_close(dw[ch], dw_ref, "dW vs oracle")


@pytest.mark.gpu
def test_two_calls_in_a_row_match_the_workspace_entry_point_and_the_oracle():
    rng = np.random.default_rng(0)
    sampled = np.sort(np.concatenate([[0, 7, 8, 255, 256, 2047],
                                      rng.choice(np.arange(9, 2040), 58, replace=False)]))
    cases = [(wl.training(T=5003, H=512, K=3, seed=301), None),
             (wl.training(T=65536, H=2048, K=3, seed=302), sampled)]
    for p, channels in cases:
        bcx, w, dy = dev(p.bcx, p.dtype), dev(p.w, p.dtype), dev(p.dy, p.dtype)
        assert partial_bytes(p.H, p.K, p.bcx.shape[0]) <= SCRATCH_LIMIT
        ref_dbcx, ref_dw = sc.backward(bcx, w, dy)
        ref_dbcx, ref_dw = host(ref_dbcx), host(ref_dw)
        for call in range(2):
            got_dbcx, got_dw = call_noalloc(bcx, w, dy)
            torch.cuda.synchronize()
            got_dbcx, got_dw = host(got_dbcx), host(got_dw)
            assert_bits(got_dbcx, ref_dbcx, f"dB|dC|dx, call {call}")
            assert_bits(got_dw, ref_dw, f"dW, call {call}")
            check_against_oracle(p, got_dbcx, got_dw, channels)
    assert sc.get_error() == 0


@pytest.mark.gpu
def test_fp32_call_matches_the_workspace_entry_point_and_the_oracle():
    p = wl.training(T=777, H=64, K=4, seed=303, dtype="f32")
    bcx, w, dy = dev(p.bcx, "f32"), dev(p.w, "f32"), dev(p.dy, "f32")
    ref_dbcx, ref_dw = sc.backward(bcx, w, dy)
    for call in range(2):
        got_dbcx, got_dw = call_noalloc(bcx, w, dy)
        torch.cuda.synchronize()
        assert_bits(host(got_dbcx), host(ref_dbcx), f"dB|dC|dx, call {call}")
        assert_bits(host(got_dw), host(ref_dw), f"dW, call {call}")
        check_against_oracle(p, host(got_dbcx), host(got_dw))


def test_sizes_beyond_the_scratch_are_rejected_before_any_work():
    # Fake aligned addresses: the size check answers before anything is touched,
    # and the call is only made once the size is known to exceed the scratch.
    sc_build.build()
    H, K, T = 8192, 4, 1025  # first row count whose partials exceed 8 MiB at H=8192, K=4
    assert partial_bytes(H, K, T) > SCRATCH_LIMIT
    assert partial_bytes(H, K, T - 1) <= SCRATCH_LIMIT
    assert partial_bytes(2048, 3, 2**31 - 1) <= SCRATCH_LIMIT
    # the caller-workspace size also holds the bias-gradient partials
    assert sc.backward_workspace_bytes(H, K, T) == partial_bytes(H, K, T) // K * (K + 1)
    base = 1 << 40
    st = _noalloc()(sc.SC_BF16, H, K, base, T, base + (1 << 34), base + (2 << 34),
                    base + (3 << 34), base + (4 << 34), None)
    assert st == sc.SC_EUNSUPPORTED
