"""Pins for the candidate-selector walk oracle (oracle/selector.py), CPU only.

They do not restate the oracle's loop. A scalar brute force checks the edge formula. With A
constant and proj one, the edge no longer depends on the predecessor, so the greedy walk must
equal the per-slot argmax of <1, B[c]> + unary. When every edge is zero, the walk must take the
unary argmax. Exhaustive enumeration of all paths of a tiny instance checks that greedy is
the slot-by-slot best successor of the previous choice. The inverse-CDF bins are checked
against hand-computed probabilities, and a very small temperature against greedy.
"""
import itertools

import numpy as np

from oracle import selector as osel


def _inst(seed, R=2, S=4, K=3, V=11, E=5):
    rng = np.random.default_rng(seed)
    A = rng.standard_normal((V, E))
    B = rng.standard_normal((V, E))
    proj = rng.standard_normal((R, S, E))
    cand = rng.integers(0, V, size=(R, S, K))
    unary = rng.standard_normal((R, S, K))
    anchor = rng.integers(0, V, size=R)
    return A, B, proj, cand, unary, anchor


def test_edge_matches_scalar_brute_force():
    A, B, proj, cand, unary, anchor = _inst(0)
    tokens, ks, scores, _ = osel.walk(A, B, proj, cand, unary, anchor)
    R, S, K = cand.shape
    E = A.shape[1]
    for r in range(R):
        prev = anchor[r]
        for s in range(S):
            for k in range(K):
                c = cand[r, s, k]
                v = sum(A[prev, e] * proj[r, s, e] * B[c, e] for e in range(E)) + unary[r, s, k]
                assert abs(scores[r, s, k] - v) < 1e-12
            prev = tokens[r, s]


def test_predecessor_free_edges_give_per_slot_argmax():
    A, B, proj, cand, unary, anchor = _inst(1)
    A1 = np.ones_like(A)
    p1 = np.ones_like(proj)
    tokens, ks, _, _ = osel.walk(A1, B, p1, cand, unary, anchor)
    per_slot = B.sum(axis=1)[cand] + unary
    np.testing.assert_array_equal(ks, per_slot.argmax(axis=-1))


def test_zero_edges_take_the_unary_argmax_first_on_ties():
    A, B, proj, cand, unary, anchor = _inst(2)
    unary[0, 1] = [0.5, 0.5, 0.1]  # tie: the first index wins
    tokens, ks, _, _ = osel.walk(np.zeros_like(A), B, proj, cand, unary, anchor)
    np.testing.assert_array_equal(ks, unary.argmax(axis=-1))
    assert ks[0, 1] == 0


def test_greedy_is_the_best_successor_of_the_previous_choice():
    # enumerate every path; the greedy path is the one whose every step maximises the edge
    # from the path's own previous token
    A, B, proj, cand, unary, anchor = _inst(3, R=1, S=3, K=3, V=7, E=4)
    tokens, ks, _, _ = osel.walk(A, B, proj, cand, unary, anchor)
    K = cand.shape[2]
    found = []
    for path in itertools.product(range(K), repeat=3):
        prev, ok = anchor[0], True
        for s, k in enumerate(path):
            e = [float(np.sum(A[prev] * proj[0, s] * B[cand[0, s, j]]) + unary[0, s, j]) for j in range(K)]
            if e[k] != max(e):
                ok = False
                break
            prev = cand[0, s, k]
        if ok:
            found.append(path)
    assert found == [tuple(ks[0])]


def test_inverse_cdf_bins_and_limits():
    A, B, proj, cand, unary, anchor = _inst(4, R=1, S=1, K=3)
    A0 = np.zeros_like(A)  # edges are the unary scores alone
    unary[0, 0] = np.log([0.2, 0.5, 0.3])  # softmax at T = 1 gives q = (0.2, 0.5, 0.3)
    for u, k in ((0.0, 0), (0.19, 0), (0.21, 1), (0.69, 1), (0.71, 2), (0.999, 2)):
        _, ks, _, q = osel.walk(A0, B, proj, cand, unary, anchor, temperature=1.0, u=np.array([[u]]))
        assert ks[0, 0] == k, (u, k)
        np.testing.assert_allclose(q[0, 0], [0.2, 0.5, 0.3], atol=1e-12)
    # T = 2 flattens: q proportional to sqrt(p)
    _, _, _, q = osel.walk(A0, B, proj, cand, unary, anchor, temperature=2.0, u=np.array([[0.5]]))
    w = np.sqrt([0.2, 0.5, 0.3])
    np.testing.assert_allclose(q[0, 0], w / w.sum(), atol=1e-12)
    # a tiny temperature samples the greedy choice for any u in (0, 1)
    A, B, proj, cand, unary, anchor = _inst(5)
    g = osel.walk(A, B, proj, cand, unary, anchor)[1]
    for u in (0.01, 0.5, 0.99):
        t = osel.walk(A, B, proj, cand, unary, anchor, temperature=1e-9, u=np.full(cand.shape[:2], u))[1]
        np.testing.assert_array_equal(t, g)


def test_bf16_widening_is_exact():
    assert list(osel.widen_bf16(np.array([0x3F80, 0x4000, 0xC040], dtype=np.uint16))) == [1.0, 2.0, -3.0]
