"""Plant a plausible mistake in a copy of the oracle and check the pins catch it.

Each mutant is one textual edit of ``oracle/shortconv_oracle.c`` (a dropped
term, a wrong operand or index, a transposed tap, a missing rounding, a
history leaking across sequences). It is compiled to a temporary library and
the pin and golden suites are run against it in a subprocess; the run must fail. The
unmodified copy must pass, so a failure is the mutant's doing.
"""
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "shortconv_oracle.c")

MUTANTS = {
    "taps_transposed": ("z += load(dt, w, (int64_t)h * K + k) * win[k];",
                        "z += load(dt, w, (int64_t)h * K + k) * win[K - 1 - k];"),
    "output_gate_dropped": ("store(dt, y, (y_row0 + r) * H + h, c * z);",
                            "store(dt, y, (y_row0 + r) * H + h, z);"),
    "input_gate_wrong_operand": ("double u = round_to(dt, b * x);",
                                 "double u = round_to(dt, c * x);"),
    "state_value_not_rounded": ("double u = round_to(dt, b * x);",
                                "double u = b * x;"),
    "window_not_reset_per_sequence": (
        "            for (int k = 0; k < K; ++k)\n                win[k] = load(dt, pool, base + k);\n"
        "            run_channel(dt, H, K, bcx, row0, len, w, bias, h, win, y, row0);",
        "            run_channel(dt, H, K, bcx, row0, len, w, bias, h, win, y, row0);"),
    "bf16_truncates": ("double r = nearbyint(d / spacing) * spacing;",
                       "double r = trunc(d / spacing) * spacing;"),
    "rollback_off_by_one": ("int64_t src = (((int64_t)i * D + (a - 1)) * H) * K;",
                            "int64_t src = (((int64_t)i * D + 0) * H) * K;"),
    "backward_du_index": ("int64_t q = s + K - 1 - k;", "int64_t q = s + k;"),
    "backward_dw_tap": ("int64_t p = t - K + 1 + k;\n                if (p >= 0)\n                    acc += dz[t] * u[p];",
                        "int64_t p = t - k;\n                if (p >= 0)\n                    acc += dz[t] * u[p];"),
    "varlen_init_ignored": ("ext[m] = init ? load(dt, init, sbase + m) : 0.0;",
                            "ext[m] = 0.0;"),
    "varlen_final_grad_dropped": ("dext[len + k] += d_final[sbase + k];",
                                  "dext[len + k] += 0.0 * d_final[sbase + k];"),
    "bias_ignored": ("        if (bias)\n            z += load(dt, bias, h);\n        store(dt, y,",
                     "        store(dt, y,"),
    "dbias_weighted": ("            for (int64_t t = 0; t < T; ++t)\n                acc += dz[t];\n            dbias[h] = acc;",
                       "            for (int64_t t = 0; t < T; ++t)\n                acc += dz[t] * u[t];\n            dbias[h] = acc;"),
    "backward_dx_uses_x": ("store(dt, dbcx, s * 3 * H + 2 * H + h, du * b);",
                           "store(dt, dbcx, s * 3 * H + 2 * H + h, du * x);"),
}


def _compile(src_text: str, out: str) -> None:
    c = out + ".c"
    with open(c, "w") as f:
        f.write(src_text)
    subprocess.run(["gcc", "-std=c11", "-O2", "-ffp-contract=off", "-fPIC", "-shared",
                    "-w", "-o", out, c, "-lm"], check=True)


def _run_pins(lib: str) -> subprocess.CompletedProcess:
    env = dict(os.environ, SHORTCONV_ORACLE_LIB=lib)
    return subprocess.run(
        [sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
         os.path.join(ROOT, "tests", "test_oracle_pins.py"),
         os.path.join(ROOT, "tests", "test_golden.py")],
        cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)


@pytest.fixture(scope="module")
def source():
    with open(SRC) as f:
        return f.read()


def test_unmodified_copy_passes_the_pins(source, tmp_path):
    lib = str(tmp_path / "liboracle_copy.so")
    _compile(source, lib)
    r = _run_pins(lib)
    assert r.returncode == 0, r.stdout[-2000:]


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(source, tmp_path, name):
    old, new = MUTANTS[name]
    assert source.count(old) >= 1, f"mutation site for {name} not found"
    lib = str(tmp_path / f"liboracle_{name}.so")
    _compile(source.replace(old, new, 1), lib)
    r = _run_pins(lib)
    assert r.returncode != 0, f"pins did not catch mutant {name}"
