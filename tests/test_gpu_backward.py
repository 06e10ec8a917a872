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
