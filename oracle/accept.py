"""Oracle for the verify step's longest-prefix acceptance -- test infrastructure only.

Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py`` may
import this module. It shares no code with the product library.

The pages describe the loop: the drafter guesses a block of 1 + num_speculative_tokens
queries, the target model verifies the whole block in parallel and the longest correct
prefix is accepted (kenforever1 "dflash-gemma4-31b-notes", the relation diagram, steps 3-4,
and the "DFlash speculative decode" box: guess a block, verify it, accept the correct
prefix, repeat).

Reading (greedy verification): a block is [x_0, d_1, ..., d_K] with K = T - 1 drafted
tokens after the bonus token x_0. The target's logits at block position j give its own
next token t_j = argmax_v logits[j, v] (smallest index among equal maxima). Draft d_i is
correct when d_i == t_{i-1}; the accepted length is the largest a in [0, K] with d_i ==
t_{i-1} for every i <= a; the token emitted after them is t_a (the target's own token at
the first mismatch, or after the whole block when all K are accepted).

The argmax is numpy's (first maximal index) on the logits widened exactly to float64
(bf16 is given as its uint16 bit patterns); the prefix rule is a plain loop.

Pinning: ``tests/test_oracle_accept_pins.py`` checks brute force over every draft pattern of tiny
blocks, the all-accepted and none-accepted closed forms, tie-breaking and the K = 0 case.
"""
from __future__ import annotations

import numpy as np


def _widen(logits, dtype: str) -> np.ndarray:
    a = np.asarray(logits)
    if dtype == "bf16":
        bits = a.astype(np.uint16).astype(np.uint32) << 16
        return bits.view(np.float32).astype(np.float64)
    if dtype == "f32":
        return a.astype(np.float32).astype(np.float64)
    raise ValueError(dtype)


def target_argmax(logits, dtype: str = "f32") -> np.ndarray:
    """t[b, j] = argmax over the last axis (first index among equal maxima). [B, T] int64."""
    return np.argmax(_widen(logits, dtype), axis=-1)


def accept_prefix(logits, draft, dtype: str = "f32"):
    """(accepted_len [B], next_token [B], target argmax [B, T]) for logits [B, T, V] and
    draft tokens [B, T - 1]."""
    t = target_argmax(logits, dtype)
    d = np.asarray(draft, dtype=np.int64)
    B, T = t.shape
    assert d.shape == (B, T - 1), (d.shape, B, T)
    acc = np.zeros(B, dtype=np.int64)
    nxt = np.zeros(B, dtype=np.int64)
    for b in range(B):
        a = 0
        while a < T - 1 and d[b, a] == t[b, a]:
            a += 1
        acc[b] = a
        nxt[b] = t[b, a]
    return acc, nxt, t
