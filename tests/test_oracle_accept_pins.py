"""Pins for the longest-prefix acceptance oracle (oracle/accept.py), CPU only.

They do not restate the oracle's formula. The argmax is checked against a pure-Python scan,
and the acceptance against a brute force over every draft pattern of tiny blocks. Closed
forms: all drafts accepted, the first one rejected, K = 0. Ties take the smallest index.
bf16 inputs are checked through their exact values.
"""
import itertools

import numpy as np
import pytest

from oracle import accept


def _scan_argmax(row):
    best, arg = None, None
    for v, x in enumerate(row):
        if best is None or x > best:
            best, arg = x, v
    return arg


def _brute_accept(targets, drafts):
    # count of leading drafts equal to the target's token at the previous position
    n = sum(1 for _ in itertools.takewhile(lambda p: p[0] == p[1], zip(drafts, targets)))
    return n, targets[n]


def test_argmax_matches_a_python_scan():
    rng = np.random.default_rng(0)
    x = rng.standard_normal((3, 5, 37)).astype(np.float32)
    t = accept.target_argmax(x, "f32")
    for b in range(3):
        for j in range(5):
            assert t[b, j] == _scan_argmax([float(v) for v in x[b, j]])


def test_every_draft_pattern_of_tiny_blocks():
    rng = np.random.default_rng(1)
    V, T = 4, 4  # K = 3 drafted tokens, V^K = 64 patterns per request
    logits = rng.standard_normal((2, T, V)).astype(np.float32)
    targets = [[_scan_argmax(list(logits[b, j])) for j in range(T)] for b in range(2)]
    patterns = list(itertools.product(range(V), repeat=T - 1))
    for pat in patterns:
        draft = np.array([pat, pat], dtype=np.int32)
        acc, nxt, _ = accept.accept_prefix(logits, draft, "f32")
        for b in range(2):
            ea, en = _brute_accept(targets[b], list(pat))
            assert (acc[b], nxt[b]) == (ea, en), (pat, b)


def test_all_accepted_and_first_rejected():
    rng = np.random.default_rng(2)
    logits = rng.standard_normal((3, 9, 50)).astype(np.float32)
    t = np.array([[_scan_argmax(list(logits[b, j])) for j in range(9)] for b in range(3)])
    acc, nxt, _ = accept.accept_prefix(logits, t[:, :8], "f32")
    assert list(acc) == [8, 8, 8] and list(nxt) == list(t[:, 8])
    wrong = t[:, :8].copy()
    wrong[:, 0] = (wrong[:, 0] + 1) % 50
    acc, nxt, _ = accept.accept_prefix(logits, wrong, "f32")
    assert list(acc) == [0, 0, 0] and list(nxt) == list(t[:, 0])


def test_ties_take_the_smallest_index():
    logits = np.zeros((1, 2, 10), dtype=np.float32)
    logits[0, 0, [7, 3]] = 5.0
    logits[0, 1, [9, 2, 4]] = 1.0
    acc, nxt, t = accept.accept_prefix(logits, np.array([[3]]), "f32")
    assert list(t[0]) == [3, 2] and acc[0] == 1 and nxt[0] == 2


def test_block_of_one_accepts_nothing():
    logits = np.arange(12, dtype=np.float32).reshape(2, 1, 6)
    acc, nxt, _ = accept.accept_prefix(logits, np.zeros((2, 0), dtype=np.int32), "f32")
    assert list(acc) == [0, 0] and list(nxt) == [5, 5]


def test_bf16_bits_are_widened_exactly():
    # 1.0078125 (0x3F81) and 1.0 (0x3F80) differ only in the last bf16 mantissa bit
    bits = np.array([[[0x3F80, 0x3F81, 0x3F80, 0xBF81]]], dtype=np.uint16)
    t = accept.target_argmax(bits, "bf16")
    assert t[0, 0] == 1
    with pytest.raises(ValueError):
        accept.target_argmax(bits, "f16")
