"""Write tests/golden/tiny_fp32_oracle.json from the CPU oracle.

The tiny fp32 workload (one sequence, H=64, K=3, T=16 prefill from a zero
state, then 4 single-token decode steps; B, C, x ~ N(0, 1), w ~ N(0, 1/3))
is drawn with the seeded generator, run through the oracle only, and stored
with its inputs as float32 bit patterns. The file is a regression fixture: a
later change to the oracle's arithmetic that moves any bit shows up in
tests/test_golden.py.

Run from the repository root:  python tests/golden/make_golden.py
"""
import json
import os
import sys

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

import oracle  # noqa: E402
from lfm2_gated_short_gb300 import workloads as wl  # noqa: E402


def hexs(a: np.ndarray) -> str:
    return np.ascontiguousarray(a, dtype=np.float32).view(np.uint32).tobytes().hex()


def main() -> None:
    p = wl.tiny_fp32()
    pool = p.pool.copy()
    st, y = oracle.prefill("f32", p.bcx, p.w, p.cu_seqlens, p.slot_ids, pool)
    assert st == oracle.OK
    state_after_prefill = pool[0].copy()
    y_dec = []
    for step in range(p.decode_bcx.shape[0]):
        st, yd = oracle.decode("f32", p.decode_bcx[step], p.w, [0], pool)
        assert st == oracle.OK
        y_dec.append(yd[0])
    doc = {
        "what": "tiny fp32 ShortConv workload through the CPU oracle (regression fixture)",
        "written_by": "tests/golden/make_golden.py (calls only oracle/)",
        "encoding": "hex of little-endian float32 bit patterns, row-major",
        "H": p.H, "K": p.K, "T": p.T, "decode_steps": int(p.decode_bcx.shape[0]),
        "inputs": {"bcx": hexs(p.bcx), "w": hexs(p.w), "decode_bcx": hexs(p.decode_bcx)},
        "expected": {
            "y_prefill": hexs(y),
            "state_after_prefill": hexs(state_after_prefill),
            "y_decode": hexs(np.stack(y_dec)),
            "state_after_decode": hexs(pool[0]),
        },
    }
    with open(os.path.join(HERE, "tiny_fp32_oracle.json"), "w") as f:
        json.dump(doc, f, indent=1)
        f.write("\n")


if __name__ == "__main__":
    main()
