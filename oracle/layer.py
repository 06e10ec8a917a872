"""The ShortConv layer's projections around the conv -- TEST INFRASTRUCTURE.

Only tests may import this module (with ``tests/``, ``__graft_entry__.smoke()``
and the CPU leg of ``bench.py``, like the rest of ``oracle/``).

The MAX LFM2 article ("MAX Pipelines 的 LFM2 架构支持", section
"短卷积实现（LFM2ShortConv）") gives the layer: ``in_proj`` projects the hidden
state to three parts b, c, xv; bx = b * xv feeds the causal conv; the output
c * conv_out goes through ``out_proj``. The article shows no bias on either
projection: both are plain linear maps here (the weight of a map from n to m
features is ``[m, n]``, so ``in_proj``'s is ``[3H, D]`` and ``out_proj``'s
``[D, H]``).

Each projection is its definition: the product in float64 (a library matmul),
then one rounding to the storage dtype (the projection's output is stored,
as the pages' layer stores b, c, xv before the conv). The conv part is the
pinned C oracle.
"""
from __future__ import annotations

import numpy as np

from . import DTYPES, decode, prefill, round_bf16, to_f64


def round_to(dtype: str, values: np.ndarray) -> np.ndarray:
    """One rounding of float64 values to the storage dtype (ties to even)."""
    if dtype == "bf16":
        return round_bf16(values)
    if dtype == "f32":
        return np.asarray(values, dtype=np.float64).astype(np.float32)
    if dtype == "f64":
        return np.asarray(values, dtype=np.float64)
    raise ValueError(f"dtype must be one of {sorted(DTYPES)}")


def linear(dtype: str, inp: np.ndarray, weight: np.ndarray) -> np.ndarray:
    """``round(inp @ weight^T)``: inp ``[T, n]``, weight ``[m, n]`` -> ``[T, m]``."""
    a, w = to_f64(dtype, inp), to_f64(dtype, weight)
    if a.ndim != 2 or w.ndim != 2 or a.shape[1] != w.shape[1]:
        raise ValueError(f"shapes {a.shape} and {w.shape} do not chain")
    return round_to(dtype, a @ w.T)


def in_proj(dtype: str, hidden: np.ndarray, w_in: np.ndarray) -> np.ndarray:
    """``bcx [T, 3H]`` with columns b | c | xv from ``hidden [T, D]`` and ``w_in [3H, D]``."""
    if w_in.shape[0] % 3:
        raise ValueError("w_in must have 3H rows")
    return linear(dtype, hidden, w_in)


def out_proj(dtype: str, y: np.ndarray, w_out: np.ndarray) -> np.ndarray:
    """``out [T, D]`` from the gated conv output ``y [T, H]`` and ``w_out [D, H]``."""
    return linear(dtype, y, w_out)


def in_proj_prefill(dtype, hidden, w_in, w, cu_seqlens, slot_ids, pool, bias=None):
    """``in_proj`` then the packed varlen prefill; ``pool`` in place; returns ``(status, y)``."""
    bcx = in_proj(dtype, hidden, w_in)
    return prefill(dtype, bcx, w, cu_seqlens, slot_ids, pool, bias=bias)


def in_proj_decode(dtype, hidden, w_in, w, slot_ids, pool, bias=None):
    """``in_proj`` then the decode of one token per sequence (row i of ``hidden``
    is sequence i's token); ``pool`` in place; returns ``(status, y)``."""
    bcx = in_proj(dtype, hidden, w_in)
    return decode(dtype, bcx, w, slot_ids, pool, bias=bias)
