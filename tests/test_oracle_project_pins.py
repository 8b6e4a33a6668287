"""Pins for the context K/V projection oracle (oracle/project.py), CPU only.

They do not restate the oracle's formula. A plain triple loop checks it on tiny sizes.
Identity weights select input columns, the projection is linear in h, and the cache
coordinates of a small example are written out by hand.
"""
import numpy as np

from oracle import project


def test_matches_a_triple_loop():
    rng = np.random.default_rng(0)
    L, H, Hkv, D = 3, 5, 2, 3
    h = rng.standard_normal((L, H))
    wk = rng.standard_normal((Hkv * D, H))
    wv = rng.standard_normal((Hkv * D, H))
    k, v = project.project_kv(h, wk, wv, Hkv, D)
    for t in range(L):
        for g in range(Hkv):
            for d in range(D):
                n = g * D + d
                sk = sum(h[t, i] * wk[n, i] for i in range(H))
                sv = sum(h[t, i] * wv[n, i] for i in range(H))
                assert abs(k[t, g, d] - sk) < 1e-12 and abs(v[t, g, d] - sv) < 1e-12


def test_identity_weights_select_columns_and_linearity():
    rng = np.random.default_rng(1)
    L, H, Hkv, D = 4, 12, 2, 4
    h = rng.standard_normal((L, H))
    eye = np.zeros((Hkv * D, H))
    eye[np.arange(Hkv * D), np.arange(Hkv * D)] = 1.0
    k, _ = project.project_kv(h, eye, eye, Hkv, D)
    np.testing.assert_array_equal(k.reshape(L, -1), h[:, : Hkv * D])
    h2 = rng.standard_normal((L, H))
    wk = rng.standard_normal((Hkv * D, H))
    a, _ = project.project_kv(h, wk, wk, Hkv, D)
    b, _ = project.project_kv(h2, wk, wk, Hkv, D)
    c, _ = project.project_kv(h + h2, wk, wk, Hkv, D)
    np.testing.assert_allclose(c, a + b, rtol=1e-12, atol=1e-12)


def test_cache_coordinates_by_hand():
    # page size 4, tokens at positions 13..18: pages 3, 3, 3, 4, 4, 4 of the table; slots 1, 2, 3, 0, 1, 2
    table = [7, 2, 9, 11, 5]
    pages, slots = project.cache_coords(6, 13, 4, table)
    assert list(pages) == [11, 11, 11, 5, 5, 5]
    assert list(slots) == [1, 2, 3, 0, 1, 2]


def test_bf16_widening_is_exact():
    bits = np.array([0x3F80, 0xC000, 0x3E20, 0x0000], dtype=np.uint16)
    assert list(project.widen_bf16(bits)) == [1.0, -2.0, 0.15625, 0.0]
