"""Pins for the fp64 oracle (CPU only).

The oracle is checked against things other than itself:
  * special cases that reduce to a library routine: torch's
    scaled_dot_product_attention in fp64 (global, GQA via repeat_interleave,
    a page table scattered by this test, and the lower-right causal mask
    torch.nn.attention.bias.causal_lower_right);
  * closed forms: Q = 0 gives the mean of the visible V and lse = log(count);
    a window of one key gives that key's V; V = 1 gives 1 (rows sum to one);
  * invariants the pages fix (non-causal: every block query sees every block
    key, so query/key permutations act as stated; causal: query i sees itself
    and its left only) and split-KV combine = unsplit result.
Each plausible slip (page vs slot index, GQA mapping, causal offset or
direction, window off-by-one, a dropped max term in lse, scale) fails one test.
"""
import json
import math
import os

import numpy as np
import pytest
import torch
import torch.nn.functional as F
from torch.nn.attention.bias import causal_lower_right

import oracle
import workloads

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "pages_facts.json")


# ----------------------------------------------------------------------------- helpers


def _scatter(logical_k, logical_v, page_size, pool_factor, gen):
    """Place per-request logical K/V ([L_b, Hkv, D] each) into a shuffled page pool.

    Written independently of the oracle: token t of request b goes to physical
    page table[b][t // page_size], slot t % page_size.
    """
    Hkv, D = logical_k[0].shape[1:]
    need = [(k.shape[0] + page_size - 1) // page_size for k in logical_k]
    pool = int(sum(need) * pool_factor) + 1
    perm = torch.randperm(pool, generator=gen)
    kc = torch.zeros(pool, page_size, Hkv, D, dtype=torch.float64)
    vc = torch.zeros(pool, page_size, Hkv, D, dtype=torch.float64)
    table = torch.zeros(len(logical_k), max(need), dtype=torch.int32)
    cur = 0
    for b, (k, v) in enumerate(zip(logical_k, logical_v)):
        for t in range(k.shape[0]):
            if t % page_size == 0:
                table[b, t // page_size] = int(perm[cur])
                cur += 1
            page = int(table[b, t // page_size])
            kc[page, t % page_size] = k[t]
            vc[page, t % page_size] = v[t]
    return kc, vc, table


def _logical_case(seed, B, T, Hq, Hkv, D, lens, page_size=4, pool_factor=2.0, fp32=True):
    gen = torch.Generator().manual_seed(seed)
    q = torch.randn(B * T, Hq, D, generator=gen, dtype=torch.float64)
    ks = [torch.randn(L, Hkv, D, generator=gen, dtype=torch.float64) for L in lens]
    vs = [torch.randn(L, Hkv, D, generator=gen, dtype=torch.float64) for L in lens]
    if fp32:  # values exactly representable in fp32 so both sides see the same numbers
        q = q.float().double()
        ks = [k.float().double() for k in ks]
        vs = [v.float().double() for v in vs]
    kc, vc, table = _scatter(ks, vs, page_size, pool_factor, gen)
    return q, ks, vs, kc, vc, table, torch.tensor(lens, dtype=torch.int32)


def _sdpa(q_b, k_b, v_b, scale, mask=None):
    """torch SDPA in fp64 for one request: q_b [T, Hq, D], k_b/v_b [L, Hkv, D]."""
    Hq, Hkv = q_b.shape[1], k_b.shape[1]
    kr = k_b.repeat_interleave(Hq // Hkv, dim=1)
    vr = v_b.repeat_interleave(Hq // Hkv, dim=1)
    out = F.scaled_dot_product_attention(
        q_b.transpose(0, 1)[None], kr.transpose(0, 1)[None], vr.transpose(0, 1)[None],
        attn_mask=mask, scale=scale)
    return out[0].transpose(0, 1)  # [T, Hq, D]


def _run(q, kc, vc, table, lens, T, **kw):
    return oracle.block_attn(q.float().numpy(), kc.float().numpy(), vc.float().numpy(),
                             table.numpy(), lens.numpy(), T, **kw)


# ----------------------------------------------------------------------------- library pins


@pytest.mark.parametrize("Hq,Hkv", [(4, 4), (6, 2), (8, 1)])
def test_global_noncausal_matches_sdpa_on_scattered_pages(Hq, Hkv):
    B, T, D = 3, 5, 16
    lens = [5, 23, 40]
    scale = 0.37
    q, ks, vs, kc, vc, table, sl = _logical_case(1, B, T, Hq, Hkv, D, lens)
    out, lse = _run(q, kc, vc, table, sl, T, causal=False, window=0, scale=scale)
    for b in range(B):
        ref = _sdpa(q[b * T:(b + 1) * T], ks[b], vs[b], scale)
        np.testing.assert_allclose(out[b * T:(b + 1) * T], ref.numpy(), rtol=1e-12, atol=1e-12)


def test_causal_matches_sdpa_lower_right():
    """Causal block attention = bottom-right aligned causal mask (query i at L - T + i)."""
    B, T, Hq, Hkv, D = 2, 7, 4, 2, 8
    lens = [7, 30]
    scale = 1.0 / math.sqrt(D)
    q, ks, vs, kc, vc, table, sl = _logical_case(2, B, T, Hq, Hkv, D, lens, page_size=4)
    out, _ = _run(q, kc, vc, table, sl, T, causal=True, window=0, scale=scale)
    for b in range(B):
        mask = causal_lower_right(T, lens[b]).to_dense()  # library-built bool mask [T, L]
        ref = _sdpa(q[b * T:(b + 1) * T], ks[b], vs[b], scale, mask=mask)
        np.testing.assert_allclose(out[b * T:(b + 1) * T], ref.numpy(), rtol=1e-12, atol=1e-12)


def test_causal_square_block_matches_sdpa_is_causal():
    """L == T: the whole sequence is the block; causal is the textbook lower triangle."""
    T, Hq, Hkv, D = 9, 2, 1, 8
    q, ks, vs, kc, vc, table, sl = _logical_case(3, 1, T, Hq, Hkv, D, [T], page_size=4)
    out, _ = _run(q, kc, vc, table, sl, T, causal=True, scale=0.5)
    kr, vr = ks[0].repeat_interleave(Hq, 1), vs[0].repeat_interleave(Hq, 1)
    ref = F.scaled_dot_product_attention(q.transpose(0, 1)[None], kr.transpose(0, 1)[None],
                                         vr.transpose(0, 1)[None], is_causal=True, scale=0.5)
    np.testing.assert_allclose(out, ref[0].transpose(0, 1).numpy(), rtol=1e-12, atol=1e-12)


def test_lse_matches_logsumexp_of_scores():
    B, T, Hq, Hkv, D = 2, 4, 4, 2, 8
    lens = [9, 17]
    q, ks, vs, kc, vc, table, sl = _logical_case(4, B, T, Hq, Hkv, D, lens)
    _, lse = _run(q, kc, vc, table, sl, T, scale=0.3)
    for b in range(B):
        for h in range(Hq):
            s = 0.3 * (q[b * T:(b + 1) * T, h] @ ks[b][:, h // (Hq // Hkv)].T)
            np.testing.assert_allclose(lse[b * T:(b + 1) * T, h], torch.logsumexp(s, 1).numpy(),
                                       rtol=1e-12, atol=1e-12)


# ----------------------------------------------------------------------------- closed forms


def _visible_count(L, T, i, causal, W):
    p = L - T + i
    hi = p if causal else L - 1
    lo = max(0, p - W + 1) if W > 0 else 0
    return hi - lo + 1


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("W", [0, 1, 3, 11, 100])
def test_zero_query_gives_mean_of_visible_values(causal, W):
    B, T, Hq, Hkv, D = 2, 5, 2, 1, 4
    lens = [12, 31]
    q, ks, vs, kc, vc, table, sl = _logical_case(5, B, T, Hq, Hkv, D, lens)
    q = torch.zeros_like(q)
    if W != 0 and W < T and not causal:
        pass  # narrower windows are still defined for the oracle
    out, lse = _run(q, kc, vc, table, sl, T, causal=causal, window=W, scale=1.0)
    for b, L in enumerate(lens):
        for i in range(T):
            n = _visible_count(L, T, i, causal, W)
            p = L - T + i
            hi = p if causal else L - 1
            lo = hi - n + 1
            mean = vs[b][lo:hi + 1].mean(0)  # [Hkv, D]
            for h in range(Hq):
                np.testing.assert_allclose(out[b * T + i, h], mean[h // (Hq // Hkv)].numpy(),
                                           rtol=1e-12, atol=1e-12)
                assert abs(lse[b * T + i, h] - math.log(n)) < 1e-12


@pytest.mark.parametrize("causal", [False, True])
def test_window_of_one_key(causal):
    """W = 1: query i sees only its own position p_i (causal) or [p_i, L) (non-causal)."""
    B, T, Hq, Hkv, D = 1, 6, 1, 1, 8
    L = 25
    q, ks, vs, kc, vc, table, sl = _logical_case(6, B, T, Hq, Hkv, D, [L])
    out, lse = _run(q, kc, vc, table, sl, T, causal=causal, window=1, scale=0.7)
    for i in range(T):
        p = L - T + i
        if causal or i == T - 1:
            np.testing.assert_allclose(out[i, 0], vs[0][p, 0].numpy(), rtol=0, atol=1e-13)
            s = 0.7 * float(q[i, 0] @ ks[0][p, 0])
            assert abs(lse[i, 0] - s) < 1e-12


def test_identical_keys_give_mean_and_shifted_lse():
    B, T, Hq, Hkv, D = 1, 3, 2, 2, 8
    L = 20
    q, ks, vs, kc, vc, table, sl = _logical_case(7, B, T, Hq, Hkv, D, [L])
    kc[:] = kc[int(table[0, 0]), 0]  # every slot of every page holds the same key rows
    ks = [kc[int(table[0, 0]), 0].expand(L, Hkv, D)]
    out, lse = _run(q, kc, vc, table, sl, T, scale=0.25)
    for i in range(T):
        for h in range(Hq):
            np.testing.assert_allclose(out[i, h], vs[0][:, h].mean(0).numpy(), rtol=1e-12, atol=1e-12)
            s = 0.25 * float(q[i, h] @ ks[0][0, h])
            assert abs(lse[i, h] - (s + math.log(L))) < 1e-12


def test_dominant_key_selects_its_value():
    B, T, Hq, Hkv, D = 1, 2, 1, 1, 4
    L = 10
    q, ks, vs, kc, vc, table, sl = _logical_case(8, B, T, Hq, Hkv, D, [L])
    q[:] = torch.tensor([1.0, 0, 0, 0], dtype=torch.float64)
    kc.zero_()
    page, slot = int(table[0, 3 // 4]), 3 % 4
    kc[page, slot, 0, 0] = 400.0  # key 3 dominates every other score by 400*scale
    out, _ = _run(q, kc, vc, table, sl, T, scale=1.0)
    for i in range(T):
        np.testing.assert_allclose(out[i, 0], vs[0][3, 0].numpy(), rtol=0, atol=1e-12)


@pytest.mark.parametrize("causal,W", [(False, 0), (True, 0), (False, 6), (True, 6)])
def test_unit_values_give_unit_output(causal, W):
    """Softmax rows sum to one: V = 1 gives out = 1 exactly (to rounding)."""
    B, T, Hq, Hkv, D = 2, 6, 4, 2, 8
    lens = [6, 33]
    q, ks, vs, kc, vc, table, sl = _logical_case(9, B, T, Hq, Hkv, D, lens)
    vc[:] = 1.0
    out, _ = _run(q, kc, vc, table, sl, T, causal=causal, window=W, scale=0.9)
    np.testing.assert_allclose(out, 1.0, rtol=0, atol=1e-13)


# ----------------------------------------------------------------------------- invariants


def test_noncausal_query_permutation_permutes_rows():
    B, T, Hq, Hkv, D = 2, 9, 4, 2, 8
    lens = [15, 40]
    q, ks, vs, kc, vc, table, sl = _logical_case(10, B, T, Hq, Hkv, D, lens)
    out, lse = _run(q, kc, vc, table, sl, T, scale=0.4)
    perm = torch.randperm(T, generator=torch.Generator().manual_seed(3))
    q2 = q.clone()
    for b in range(B):
        q2[b * T:(b + 1) * T] = q[b * T:(b + 1) * T][perm]
    out2, lse2 = _run(q2, kc, vc, table, sl, T, scale=0.4)
    for b in range(B):
        np.testing.assert_allclose(out2[b * T:(b + 1) * T], out[b * T:(b + 1) * T][perm.numpy()],
                                   rtol=1e-12, atol=1e-12)
        np.testing.assert_allclose(lse2[b * T:(b + 1) * T], lse[b * T:(b + 1) * T][perm.numpy()],
                                   rtol=1e-12, atol=1e-12)


def test_noncausal_key_permutation_leaves_output():
    """Non-causal, global: permuting the block's keys (with their values) changes nothing."""
    B, T, Hq, Hkv, D = 1, 8, 2, 1, 8
    L = 29
    q, ks, vs, kc, vc, table, sl = _logical_case(11, B, T, Hq, Hkv, D, [L])
    out, _ = _run(q, kc, vc, table, sl, T, scale=0.5)
    perm = torch.randperm(T, generator=torch.Generator().manual_seed(5)) + (L - T)
    k2, v2 = ks[0].clone(), vs[0].clone()
    k2[L - T:] = ks[0][perm]
    v2[L - T:] = vs[0][perm]
    kc2, vc2, table2 = _scatter([k2], [v2], 4, 2.0, torch.Generator().manual_seed(9))
    out2, _ = _run(q, kc2, vc2, table2, sl, T, scale=0.5)
    np.testing.assert_allclose(out2, out, rtol=1e-12, atol=1e-12)


def test_causal_row_ignores_keys_to_its_right():
    B, T, Hq, Hkv, D = 1, 8, 2, 2, 8
    L = 21
    q, ks, vs, kc, vc, table, sl = _logical_case(12, B, T, Hq, Hkv, D, [L])
    out, _ = _run(q, kc, vc, table, sl, T, causal=True, scale=0.5)
    i = 3
    p = L - T + i
    k2, v2 = ks[0].clone(), vs[0].clone()
    k2[p + 1:] = torch.randn(L - p - 1, Hkv, D, dtype=torch.float64).float().double()
    v2[p + 1:] = 5.0
    kc2, vc2, table2 = _scatter([k2], [v2], 4, 2.0, torch.Generator().manual_seed(1))
    out2, _ = _run(q, kc2, vc2, table2, sl, T, causal=True, scale=0.5)
    np.testing.assert_allclose(out2[: i + 1], out[: i + 1], rtol=1e-12, atol=1e-12)
    assert np.abs(out2[i + 1:] - out[i + 1:]).max() > 1e-3
    # non-causal rows do see them
    out3, _ = _run(q, kc2, vc2, table2, sl, T, causal=False, scale=0.5)
    out4, _ = _run(q, kc, vc, table, sl, T, causal=False, scale=0.5)
    assert np.abs(out3[0] - out4[0]).max() > 1e-3


def test_window_edge_key_is_seen_and_the_one_before_is_not():
    B, T, Hq, Hkv, D = 1, 4, 1, 1, 8
    L, W = 40, 7
    q, ks, vs, kc, vc, table, sl = _logical_case(13, B, T, Hq, Hkv, D, [L])
    base, _ = _run(q, kc, vc, table, sl, T, causal=True, window=W, scale=0.5)
    i = 2
    p = L - T + i
    for pos, must_change in ((p - W + 1, True), (p - W, False)):
        k2 = ks[0].clone()
        k2[pos] += 3.0
        kc2, vc2, t2 = _scatter([k2], [vs[0]], 4, 2.0, torch.Generator().manual_seed(2))
        out2, _ = _run(q, kc2, vc2, t2, sl, T, causal=True, window=W, scale=0.5)
        changed = np.abs(out2[i] - base[i]).max() > 1e-9
        assert changed == must_change, (pos, changed)


def test_window_covering_everything_equals_global():
    B, T, Hq, Hkv, D = 2, 5, 2, 1, 8
    lens = [9, 26]
    q, ks, vs, kc, vc, table, sl = _logical_case(14, B, T, Hq, Hkv, D, lens)
    for causal in (False, True):
        a, la = _run(q, kc, vc, table, sl, T, causal=causal, window=0, scale=0.5)
        b, lb = _run(q, kc, vc, table, sl, T, causal=causal, window=max(lens), scale=0.5)
        np.testing.assert_array_equal(a, b)
        np.testing.assert_array_equal(la, lb)


def test_block_of_one_is_causal_agnostic():
    q, ks, vs, kc, vc, table, sl = _logical_case(15, 3, 1, 4, 2, 8, [1, 7, 19])
    a, la = _run(q, kc, vc, table, sl, 1, causal=False, scale=0.5)
    b, lb = _run(q, kc, vc, table, sl, 1, causal=True, scale=0.5)
    np.testing.assert_array_equal(a, b)
    np.testing.assert_array_equal(la, lb)


def test_gqa_equals_mha_with_repeated_kv():
    B, T, Hq, Hkv, D = 2, 3, 6, 2, 8
    lens = [10, 14]
    q, ks, vs, kc, vc, table, sl = _logical_case(16, B, T, Hq, Hkv, D, lens)
    a, la = _run(q, kc, vc, table, sl, T, scale=0.5)
    kc2 = kc.repeat_interleave(Hq // Hkv, dim=2)
    vc2 = vc.repeat_interleave(Hq // Hkv, dim=2)
    b, lb = _run(q, kc2, vc2, table, sl, T, scale=0.5)
    np.testing.assert_allclose(a, b, rtol=1e-13, atol=1e-13)
    np.testing.assert_allclose(la, lb, rtol=1e-13, atol=1e-13)


def test_output_is_linear_in_v():
    B, T, Hq, Hkv, D = 1, 4, 2, 1, 8
    q, ks, vs, kc, vc, table, sl = _logical_case(17, B, T, Hq, Hkv, D, [18])
    vc_b = torch.randn(vc.shape, generator=torch.Generator().manual_seed(4), dtype=torch.float64)
    vc_b = vc_b.float().double()
    a, _ = _run(q, kc, vc, table, sl, T, scale=0.5)
    b, _ = _run(q, kc, vc_b, table, sl, T, scale=0.5)
    c, _ = _run(q, kc, (vc + 2 * vc_b).float().double(), table, sl, T, scale=0.5)
    np.testing.assert_allclose(c, a + 2 * b, rtol=1e-6, atol=1e-6)


@pytest.mark.parametrize("causal,W", [(False, 0), (True, 0), (False, 9), (True, 9)])
def test_split_combine_equals_unsplit(causal, W):
    B, T, Hq, Hkv, D = 2, 5, 4, 2, 8
    lens = [11, 47]
    q, ks, vs, kc, vc, table, sl = _logical_case(18, B, T, Hq, Hkv, D, lens)
    full, lfull = _run(q, kc, vc, table, sl, T, causal=causal, window=W, scale=0.6)
    bounds = [0, 3, 3, 16, 40, 41, 64]  # includes an empty chunk and chunks past every row
    parts, lses = [], []
    for kb, ke in zip(bounds[:-1], bounds[1:]):
        o, l = _run(q, kc, vc, table, sl, T, causal=causal, window=W, scale=0.6, key_range=(kb, ke))
        parts.append(o)
        lses.append(l)
    assert np.isneginf(np.stack(lses)).any()
    out, lse = oracle.split_combine(np.stack(parts), np.stack(lses))
    np.testing.assert_allclose(out, full, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(lse, lfull, rtol=1e-12, atol=1e-12)


def test_split_combine_single_chunk_and_all_empty():
    po = np.random.default_rng(0).standard_normal((1, 3, 4))
    pl = np.array([[0.5, -1.0, 2.0]])
    out, lse = oracle.split_combine(po, pl)
    np.testing.assert_allclose(out, po[0], rtol=1e-15)
    np.testing.assert_allclose(lse, pl[0], rtol=1e-15)
    out, lse = oracle.split_combine(np.zeros((2, 1, 4)), np.full((2, 1), -np.inf))
    assert np.isneginf(lse).all() and (out == 0).all()


def test_split_combine_two_chunk_closed_form():
    """Two chunks with lse a, b: weights e^a/(e^a+e^b), lse = log(e^a + e^b)."""
    o1, o2 = np.array([[1.0, 2.0]]), np.array([[3.0, -1.0]])
    a, b = 0.3, -1.2
    out, lse = oracle.split_combine(np.stack([o1, o2]), np.array([[a], [b]]))
    w1 = 1.0 / (1.0 + math.exp(b - a))
    np.testing.assert_allclose(out[0], w1 * o1[0] + (1 - w1) * o2[0], rtol=1e-14)
    assert abs(lse[0] - math.log(math.exp(a) + math.exp(b))) < 1e-14


# ----------------------------------------------------------------------------- host plumbing


def test_bf16_bits_are_widened_exactly():
    case = workloads.make_custom("t", 1, 3, 2, 1, 16, [20], dtype=torch.bfloat16, seed=3)
    a, la = oracle.block_attn(case.q, case.k_cache, case.v_cache, case.page_table, case.seq_lens, 3)
    b, lb = oracle.block_attn(case.q.float(), case.k_cache.float(), case.v_cache.float(),
                              case.page_table, case.seq_lens, 3)
    np.testing.assert_array_equal(a, b)
    np.testing.assert_array_equal(la, lb)


def test_row_sampler_matches_full():
    case = workloads.make_custom("t", 2, 4, 4, 2, 16, [9, 30], dtype=torch.bfloat16, seed=4)
    full, lfull = oracle.block_attn(case.q, case.k_cache, case.v_cache, case.page_table,
                                    case.seq_lens, 4, causal=True, window=5)
    rows = np.array([[0, 0, 0], [1, 3, 2], [1, 1, 3], [0, 2, 1]])
    o, l = oracle.block_attn_rows(case.q, case.k_cache, case.v_cache, case.page_table,
                                  case.seq_lens, 4, rows, causal=True, window=5)
    for r, (b, h, i) in enumerate(rows):
        np.testing.assert_array_equal(o[r], full[b * 4 + i, h])
        assert l[r] == lfull[b * 4 + i, h]


def test_out_of_range_page_is_an_error():
    case = workloads.make_custom("t", 1, 2, 1, 1, 8, [10], dtype=torch.float32, seed=5)
    bad = case.page_table.clone()
    bad[0, 0] = case.k_cache.shape[0]
    with pytest.raises(ValueError):
        oracle.block_attn(case.q, case.k_cache, case.v_cache, bad, case.seq_lens, 2)


def test_pages_facts_shape_the_named_workloads():
    facts = json.load(open(GOLDEN))
    T = facts["block_len_for_8_spec_tokens"]["value"]
    for bs, rows in facts["capture_sizes"]["value"].items():
        B = int(bs)
        lens = workloads._uniform_lens(B, 1024, 32768, seed=1234 + 2 + B)
        assert len(lens) == B and B * T == rows
        assert all(1024 <= L <= 32768 for L in lens)
    assert facts["max_head_size"]["value"] == 512
    assert facts["causal_default"]["value"] is False
    assert facts["dflash2_default_num_spec"]["value"] + 1 == 16
