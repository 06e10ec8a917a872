"""The bounds-checked build of the library, on the GPU.

Built with -DSC_BOUNDS_CHECK (_build/bounds/libshortconv.so), every global
load and store the kernels make through their memory helpers is checked
against the buffers the call was given; a refused access is skipped and
sets SC_DEV_OUT_OF_BOUNDS, nothing traps. This runs the whole guard-band
file (every call, the ragged shapes, against the oracle; each test also
asserts an empty error word, so any refused access fails it) in a child
process that loads that build, including the tests there that shorten a
record on purpose to show the checks refusing real accesses.
"""
import os
import subprocess
import sys

import pytest

from lfm2_gated_short_gb300 import build as sc_build

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)


def test_guard_band_cases_under_the_bounds_checked_build():
    lib = sc_build.build(bounds_check=True)
    env = dict(os.environ, SHORTCONV_LIBRARY=lib)
    r = subprocess.run(
        [sys.executable, "-m", "pytest", os.path.join(HERE, "test_gpu_guard_bands.py"), "-m",
         "gpu", "-q", "-rs", "-p", "no:cacheprovider"],
        cwd=ROOT, env=env, capture_output=True, text=True, timeout=1200)
    tail = (r.stdout + r.stderr)[-4000:]
    assert r.returncode == 0, tail
    assert " passed" in r.stdout and "skipped" not in r.stdout, tail
