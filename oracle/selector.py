"""Oracle for the DFlash2 candidate-selector walk -- test infrastructure only.

Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py`` may
import this module. It shares no code with the product library.

The pages describe the selector (prhub report on vLLM PR #52816 "DFlash2", the motivation
paragraph and changes 1-2). It keeps the head's top-K candidates of every draft slot and scores
the transition between adjacent slots as
    edge(p -> c) = < A[p] * project(h), B[c] > + unary[c]
with a predecessor codebook A and a successor codebook B. It then walks from the verified anchor,
one slot after the other, carrying the previous choice in the loop. With temperature 0 it takes
the best edge. With T > 0 it steps by the inverse CDF and returns the K candidates' probabilities q
for lossless verification.

Readings (the pages leave these open): A and B are [V, E]; project(h) of slot s is given as a
vector proj[r, s] of length E (the projection itself is a linear layer outside the walk);
cand[r, s, k] are the K candidate tokens of slot s and unary[r, s, k] their unary scores; slot
0's predecessor is anchor[r]. Greedy takes the first maximal k. With T > 0,
q = softmax(edge / T) over the K candidates, and the walk takes the smallest k whose running
sum of q exceeds the given uniform u[r, s] (the last k if rounding leaves none).

The arithmetic is float64 on the exactly widened inputs, a plain sequential walk.

Pinning: ``tests/test_oracle_selector_pins.py`` checks a scalar brute force of the edge
formula, the unary-only case, the greedy path against exhaustive path enumeration when edges
do not depend on the predecessor, temperature limits and the inverse-CDF bins.
"""
from __future__ import annotations

import numpy as np


def widen_bf16(bits) -> np.ndarray:
    return (np.asarray(bits).astype(np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def edge_scores(A, B, proj_s, cand_s, unary_s, prev: int) -> np.ndarray:
    """edge(prev -> cand_s[k]) for the K candidates of one slot (float64 [K])."""
    a = np.asarray(A, dtype=np.float64)[prev] * np.asarray(proj_s, dtype=np.float64)
    Bc = np.asarray(B, dtype=np.float64)[np.asarray(cand_s)]
    return Bc @ a + np.asarray(unary_s, dtype=np.float64)


def walk(A, B, proj, cand, unary, anchor, temperature: float = 0.0, u=None):
    """(tokens [R, S], chosen k [R, S], path edge scores [R, S, K], q [R, S, K] or None)."""
    cand = np.asarray(cand)
    R, S, K = cand.shape
    tokens = np.zeros((R, S), dtype=np.int64)
    ks = np.zeros((R, S), dtype=np.int64)
    scores = np.zeros((R, S, K))
    q = np.zeros((R, S, K)) if temperature > 0 else None
    for r in range(R):
        prev = int(anchor[r])
        for s in range(S):
            e = edge_scores(A, B, proj[r, s], cand[r, s], unary[r, s], prev)
            scores[r, s] = e
            if temperature > 0:
                z = (e - e.max()) / temperature
                p = np.exp(z)
                p /= p.sum()
                q[r, s] = p
                cdf = np.cumsum(p)
                hit = np.nonzero(cdf > float(u[r, s]))[0]
                k = int(hit[0]) if hit.size else K - 1
            else:
                k = int(np.argmax(e))
            ks[r, s] = k
            tokens[r, s] = cand[r, s, k]
            prev = int(tokens[r, s])
    return tokens, ks, scores, q
