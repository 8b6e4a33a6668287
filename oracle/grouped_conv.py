"""Oracle for the DFlash2 grouped dynamic depthwise convolution -- test infrastructure only.

Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py`` may
import this module. It shares no code with the product library.

The pages give the operation in closed form (prhub report on vLLM PR #52816 "DFlash2", the
motivation paragraph and change 1): inside a block, proposal position i sees earlier
positions of the same block through
    out[i, c] = sum_t (base[t, c] + delta[i, t, g(c)]) * x[i - t, c],
with every tap that reaches past the block boundary (i - t < 0) set to zero. base holds the
static per-channel taps, delta the dynamic per-position, per-group taps that the module's
"prepare" step projects from its input.

Readings (the pages leave these open): x is [B, T, C] (request b's block of T positions), base
is [taps, C], delta is [B, T, taps, G]; the G groups are contiguous channel ranges,
g(c) = c // (C / G); the block boundary is the start of each request's own block, so no tap
reads another request or the context.

The arithmetic is a sequential loop over positions and taps in float64 on the exactly
widened inputs (bf16 x is given as its uint16 bit patterns).

Pinning: ``tests/test_oracle_conv_pins.py`` checks a scalar brute force, the one-tap closed
form, a one-hot dynamic tap that shifts the block, causality, group isolation and linearity.
"""
from __future__ import annotations

import numpy as np


def widen(x, dtype: str) -> np.ndarray:
    a = np.asarray(x)
    if dtype == "bf16":
        return (a.astype(np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    if dtype == "f32":
        return a.astype(np.float32).astype(np.float64)
    raise ValueError(dtype)


def group_of_channel(C: int, G: int) -> np.ndarray:
    """g(c) for c in [0, C): contiguous groups of C / G channels."""
    assert C % G == 0
    return np.arange(C) // (C // G)


def grouped_conv(x, base, delta) -> np.ndarray:
    """out [B, T, C] float64 for x [B, T, C], base [taps, C], delta [B, T, taps, G] (float64)."""
    x = np.asarray(x, dtype=np.float64)
    base = np.asarray(base, dtype=np.float64)
    delta = np.asarray(delta, dtype=np.float64)
    B, T, C = x.shape
    taps = base.shape[0]
    G = delta.shape[3]
    g = group_of_channel(C, G)
    out = np.zeros((B, T, C))
    for i in range(T):
        for t in range(taps):
            if i - t < 0:
                continue  # the tap reaches past the block boundary
            coef = base[t][None, :] + delta[:, i, t, :][:, g]  # [B, C]
            out[:, i, :] += coef * x[:, i - t, :]
    return out
