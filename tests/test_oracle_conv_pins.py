"""Pins for the grouped dynamic depthwise convolution oracle (oracle/grouped_conv.py), CPU only.

None restates the oracle's vectorised loop. A scalar brute force over every (b, i, c, t)
checks it on tiny sizes. The one-tap case reduces to a per-channel scale, and a one-hot
dynamic tap shifts the block with zeros at its start. Causality, group isolation and
linearity are invariants of the definition.
"""
import numpy as np

from oracle import grouped_conv as oc


def _rand(seed, B=2, T=5, C=6, taps=3, G=3):
    rng = np.random.default_rng(seed)
    return (rng.standard_normal((B, T, C)), rng.standard_normal((taps, C)),
            rng.standard_normal((B, T, taps, G)))


def test_matches_scalar_brute_force():
    x, base, delta = _rand(0)
    B, T, C = x.shape
    taps, G = base.shape[0], delta.shape[3]
    got = oc.grouped_conv(x, base, delta)
    for b in range(B):
        for i in range(T):
            for c in range(C):
                g = c // (C // G)
                s = 0.0
                for t in range(taps):
                    j = i - t
                    if j >= 0:
                        s += (base[t, c] + delta[b, i, t, g]) * x[b, j, c]
                assert abs(got[b, i, c] - s) < 1e-12


def test_one_tap_is_a_channel_scale():
    x, base, delta = _rand(1, taps=1)
    got = oc.grouped_conv(x, base, np.zeros_like(delta))
    np.testing.assert_allclose(got, x * base[0][None, None, :], rtol=0, atol=1e-15)


def test_one_hot_dynamic_tap_shifts_the_block():
    x, base, delta = _rand(2, T=7, taps=4)
    s = 2
    d = np.zeros_like(delta)
    d[:, :, s, :] = 1.0
    got = oc.grouped_conv(x, np.zeros_like(base), d)
    np.testing.assert_array_equal(got[:, :s, :], 0.0)  # taps before the block start are zero
    np.testing.assert_array_equal(got[:, s:, :], x[:, :-s, :])


def test_causal_inside_the_block():
    x, base, delta = _rand(3, T=6)
    ref = oc.grouped_conv(x, base, delta)
    x2 = x.copy()
    x2[:, 4:, :] += 10.0  # change positions 4 and 5
    got = oc.grouped_conv(x2, base, delta)
    np.testing.assert_array_equal(got[:, :4, :], ref[:, :4, :])
    assert np.abs(got[:, 4:, :] - ref[:, 4:, :]).max() > 1.0


def test_groups_are_contiguous_channel_ranges():
    x, base, delta = _rand(4, C=12, G=3)
    ref = oc.grouped_conv(x, base, delta)
    d2 = delta.copy()
    d2[:, :, :, 1] += 5.0  # group 1 = channels 4..7
    got = oc.grouped_conv(x, base, d2)
    changed = np.abs(got - ref).max(axis=(0, 1)) > 1e-9
    assert list(np.nonzero(changed)[0]) == [4, 5, 6, 7]


def test_linear_in_x_and_requests_independent():
    x, base, delta = _rand(5, B=3)
    rng = np.random.default_rng(6)
    x2 = rng.standard_normal(x.shape)
    a = oc.grouped_conv(x, base, delta)
    b = oc.grouped_conv(x2, base, delta)
    np.testing.assert_allclose(oc.grouped_conv(x + 2 * x2, base, delta), a + 2 * b, atol=1e-12)
    x3 = x.copy()
    x3[1] = x2[1]  # only request 1 changes
    c = oc.grouped_conv(x3, base, delta)
    np.testing.assert_array_equal(c[[0, 2]], a[[0, 2]])


def test_bf16_widening_is_exact():
    assert list(oc.widen(np.array([0x3F80, 0xBF00, 0x4049], dtype=np.uint16), "bf16")) == [1.0, -0.5, 3.140625]
