"""Load the stored fixtures under tests/golden as arrays of a given storage dtype."""
import json
import os

import numpy as np
import torch

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def store(values, dtype: str) -> np.ndarray:
    """Exact values (integers here) to storage: float32, bf16 bits or float64."""
    a = np.asarray(values, dtype=np.float64)
    if dtype == "f64":
        return a
    if dtype == "f32":
        return a.astype(np.float32)
    t = torch.from_numpy(a.astype(np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16).copy()


def worked_example(dtype: str) -> dict:
    """The hand-derived worked example expanded to H channels (channel h scales by h+1)."""
    with open(os.path.join(GOLDEN, "worked_example.json")) as f:
        doc = json.load(f)
    c0, H, K, T = doc["channel0"], doc["H"], doc["K"], doc["T"]
    s = np.arange(1, H + 1, dtype=np.float64)          # per-channel scale
    one = np.ones(H)
    col = lambda v, sc: np.outer(np.asarray(v, np.float64), sc)   # [T, H]
    B, C, X = col(c0["B"], s), col(c0["C"], one), col(c0["x"], one)
    out = {
        "H": H, "K": K, "T": T,
        "bcx": np.concatenate([B, C, X], 1),
        "w": np.tile(np.asarray(c0["w"], np.float64), (H, 1)),
        "state": np.outer(s, c0["state"]),
        "y": col(c0["y"], s),
        "final_state": np.outer(s, c0["final_state"]),
        "windows": np.einsum("h,jk->jhk", s, np.asarray(c0["windows"], np.float64)),
        "dy": col(c0["dy"], one),
        "dB": col(c0["dB"], one), "dC": col(c0["dC"], s), "dx": col(c0["dx"], s),
        "dW": np.outer(s, c0["dW"]),
    }
    for k in ("bcx", "w", "state", "y", "final_state", "windows", "dy", "dB", "dC", "dx"):
        out[k] = store(out[k], dtype)
    return out


def tiny_fp32_golden() -> dict:
    with open(os.path.join(GOLDEN, "tiny_fp32_oracle.json")) as f:
        doc = json.load(f)
    H, K, T, S = doc["H"], doc["K"], doc["T"], doc["decode_steps"]
    arr = lambda h, shape: np.frombuffer(bytes.fromhex(h), dtype=np.uint32).view(
        np.float32).reshape(shape).copy()
    i, e = doc["inputs"], doc["expected"]
    return {
        "H": H, "K": K, "T": T, "steps": S,
        "bcx": arr(i["bcx"], (T, 3 * H)), "w": arr(i["w"], (H, K)),
        "decode_bcx": arr(i["decode_bcx"], (S, 1, 3 * H)),
        "y_prefill": arr(e["y_prefill"], (T, H)),
        "state_after_prefill": arr(e["state_after_prefill"], (H, K)),
        "y_decode": arr(e["y_decode"], (S, H)),
        "state_after_decode": arr(e["state_after_decode"], (H, K)),
    }
