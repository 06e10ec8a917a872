"""Moving storage arrays between numpy (oracle side) and CUDA tensors, and the
parity tolerances.

Tolerances (the ShortConv target's stated bounds):
* fp32 outputs: max |gpu - oracle| <= 1e-5;
* bf16 outputs (y, dB, dC, dx): per element |gpu - oracle| <= 1e-2 + 2^-7 |oracle|;
* conv states and verify windows: bit-exact;
* dW (fp32 on the GPU, float64 in the oracle): |d_i| <= 1e-3 max(|ref_i|, rms(ref)).
"""
import numpy as np
import torch

import oracle

BF16_ATOL, BF16_RTOL, F32_ATOL, DW_RTOL = 1e-2, 2.0 ** -7, 1e-5, 1e-3


def dev(a: np.ndarray, dtype: str) -> torch.Tensor:
    a = np.ascontiguousarray(a)
    if dtype == "bf16":
        t = torch.from_numpy(a.view(np.int16).copy()).view(torch.bfloat16)
    elif dtype == "f32":
        t = torch.from_numpy(a.astype(np.float32, copy=True))
    elif dtype == "i32":
        t = torch.from_numpy(a.astype(np.int32, copy=True))
    else:
        raise ValueError(dtype)
    return t.cuda()


def host(t: torch.Tensor) -> np.ndarray:
    t = t.detach().cpu().contiguous()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16).copy()
    return t.numpy().copy()


def assert_close(dtype: str, got: np.ndarray, ref: np.ndarray, what: str = "") -> None:
    g, r = oracle.to_f64(dtype, got), oracle.to_f64(dtype, ref)
    assert g.shape == r.shape, (what, g.shape, r.shape)
    assert np.all(np.isfinite(g)), f"{what}: non-finite GPU output"
    if dtype == "f32":
        err = np.abs(g - r).max(initial=0.0)
        assert err <= F32_ATOL, f"{what}: max |err| {err:.3g} > {F32_ATOL}"
    else:
        bad = np.abs(g - r) > BF16_ATOL + BF16_RTOL * np.abs(r)
        assert not bad.any(), (
            f"{what}: {int(bad.sum())} of {bad.size} outside 1e-2 + 2^-7|ref|; first at "
            f"{np.argwhere(bad)[0]}: gpu {g[bad][0]} ref {r[bad][0]}")


def assert_dw_close(got: np.ndarray, ref: np.ndarray, what: str = "dW") -> None:
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    rms = np.sqrt(np.mean(ref ** 2)) if ref.size else 0.0
    bound = DW_RTOL * np.maximum(np.abs(ref), rms)
    bad = np.abs(got - ref) > bound
    assert not bad.any(), f"{what}: {int(bad.sum())} entries outside 1e-3 relative"


def assert_bits(got: np.ndarray, ref: np.ndarray, what: str = "") -> None:
    g = np.ascontiguousarray(got)
    r = np.ascontiguousarray(ref)
    assert g.shape == r.shape, (what, g.shape, r.shape)
    gv = g.view(np.uint16) if g.dtype == np.uint16 else g.view(np.uint32)
    rv = r.view(np.uint16) if r.dtype == np.uint16 else r.view(np.uint32)
    mism = gv != rv
    assert not mism.any(), f"{what}: {int(mism.sum())} of {mism.size} values differ in bits"
