"""Oracle for the draft pass's context K/V projection -- test infrastructure only.

Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py`` may
import this module. It shares no code with the product library.

The pages state that the drafter's cross-attention takes its context K/V from the target's
hidden states and its Q from the query embeddings (kenforever1 "dflash-gemma4-31b-notes",
the code lines under "why non-causal attention"). Reading: the projection is linear,
K[t] = h[t] W_k^T and V[t] = h[t] W_v^T, with W_k and W_v of shape [Hkv*D, hidden] (one
row per output feature). Token t sits at position pos0 + t of its request and is stored in
the paged cache at page page_table[(pos0 + t) // page_size], slot (pos0 + t) % page_size,
as Hkv heads of D features (feature n = head * D + d).

The arithmetic is numpy's matmul in float64 on the exactly widened bf16 inputs.

Pinning: ``tests/test_oracle_project_pins.py`` checks a plain triple loop on tiny sizes,
identity weights, linearity in h, and hand-computed page/slot coordinates.
"""
from __future__ import annotations

import numpy as np


def widen_bf16(bits) -> np.ndarray:
    """bf16 bit patterns (uint16 / int16 array) -> exact float64 values."""
    b = np.asarray(bits).astype(np.uint16).astype(np.uint32) << 16
    return b.view(np.float32).astype(np.float64)


def cache_coords(num_tokens: int, pos0: int, page_size: int, page_table) -> tuple:
    """(page id, slot) of every token of the request."""
    pt = np.asarray(page_table, dtype=np.int64)
    pos = pos0 + np.arange(num_tokens, dtype=np.int64)
    return pt[pos // page_size], pos % page_size


def project_kv(hidden, w_k, w_v, num_kv_heads: int, head_dim: int):
    """K, V [L, Hkv, D] float64 for hidden [L, H] and weights [Hkv*D, H] (float64 inputs)."""
    h = np.asarray(hidden, dtype=np.float64)
    k = h @ np.asarray(w_k, dtype=np.float64).T
    v = h @ np.asarray(w_v, dtype=np.float64).T
    L = h.shape[0]
    return k.reshape(L, num_kv_heads, head_dim), v.reshape(L, num_kv_heads, head_dim)
