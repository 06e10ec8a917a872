"""The oracle against the stored fixtures in tests/golden."""
import numpy as np
import pytest

import oracle
from lfm2_gated_short_gb300 import workloads as wl
from fixtures import store, tiny_fp32_golden, worked_example

DTYPES = ["f64", "f32", "bf16"]


@pytest.mark.parametrize("dtype", DTYPES)
def test_worked_example_forward(dtype):
    ex = worked_example(dtype)
    pool = ex["state"][None].copy()
    st, y = oracle.prefill(dtype, ex["bcx"], ex["w"], [0, ex["T"]], [0], pool)
    assert st == oracle.OK
    np.testing.assert_array_equal(y, ex["y"])
    np.testing.assert_array_equal(pool[0], ex["final_state"])


@pytest.mark.parametrize("dtype", DTYPES)
def test_worked_example_token_by_token_decode(dtype):
    ex = worked_example(dtype)
    pool = ex["state"][None].copy()
    for t in range(ex["T"]):
        st, y = oracle.decode(dtype, ex["bcx"][t:t + 1], ex["w"], [0], pool)
        assert st == oracle.OK
        np.testing.assert_array_equal(y[0], ex["y"][t])
        np.testing.assert_array_equal(pool[0], ex["windows"][t])


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("accepted", [0, 1, 2, 3, 4])
def test_worked_example_verify_and_rollback(dtype, accepted):
    ex = worked_example(dtype)
    pool = ex["state"][None].copy()
    st, win, y = oracle.verify(dtype, ex["bcx"], ex["w"], [0], pool, ex["T"])
    assert st == oracle.OK
    np.testing.assert_array_equal(y, ex["y"])
    np.testing.assert_array_equal(win[0], ex["windows"])
    np.testing.assert_array_equal(pool[0], ex["state"])          # verify only reads
    assert oracle.rollback(dtype, win, [accepted], [0], pool) == oracle.OK
    expect = ex["state"] if accepted == 0 else ex["windows"][accepted - 1]
    np.testing.assert_array_equal(pool[0], expect)


@pytest.mark.parametrize("dtype", DTYPES)
def test_worked_example_backward(dtype):
    ex = worked_example(dtype)
    st, dbcx, dw = oracle.backward(dtype, ex["bcx"], ex["w"], ex["dy"])
    assert st == oracle.OK
    H = ex["H"]
    np.testing.assert_array_equal(dbcx[:, :H], ex["dB"])
    np.testing.assert_array_equal(dbcx[:, H:2 * H], ex["dC"])
    np.testing.assert_array_equal(dbcx[:, 2 * H:], ex["dx"])
    np.testing.assert_array_equal(dw, ex["dW"])


def test_tiny_fp32_fixture_inputs_match_the_generator():
    g, p = tiny_fp32_golden(), wl.tiny_fp32()
    np.testing.assert_array_equal(g["bcx"], p.bcx)
    np.testing.assert_array_equal(g["w"], p.w)
    np.testing.assert_array_equal(g["decode_bcx"], p.decode_bcx)


def test_tiny_fp32_oracle_regression():
    g = tiny_fp32_golden()
    pool = np.zeros((1, g["H"], g["K"]), np.float32)
    st, y = oracle.prefill("f32", g["bcx"], g["w"], [0, g["T"]], [0], pool)
    assert st == oracle.OK
    np.testing.assert_array_equal(y, g["y_prefill"])
    np.testing.assert_array_equal(pool[0], g["state_after_prefill"])
    for s in range(g["steps"]):
        st, yd = oracle.decode("f32", g["decode_bcx"][s], g["w"], [0], pool)
        assert st == oracle.OK
        np.testing.assert_array_equal(yd[0], g["y_decode"][s])
    np.testing.assert_array_equal(pool[0], g["state_after_decode"])


def test_store_is_exact_for_the_worked_example_values():
    vals = np.array([800, 208, -120, 128, 112, 26, -14], np.float64)
    np.testing.assert_array_equal(oracle.bf16_to_f64(store(vals, "bf16")), vals)
