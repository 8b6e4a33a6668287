"""GPU parity for dflash_selector_walk (through its C ABI) against oracle/selector.py.

The kernel scores edges in fp32 (lane-strided partial sums, then a shuffle tree); the oracle in
float64. Edge scores must agree within 1e-5 * (1 + sum_e |A[p,e] proj[e] B[c,e]| + |unary|),
several times the fp32 forward error of that summation. The walk's choices are integers taken
from those floats, so they are checked three ways:
  1. the kernel's path edges against the oracle's edges recomputed on the kernel's own path;
  2. each choice is valid under the oracle's edges within the tolerance: a maximal edge for
     temperature 0, the inverse-CDF bin of the uniform for T > 0, and q agrees to 1e-5;
  3. the whole path equals the oracle's own walk for every request whose decisions all have a
     margin (an edge gap above 1e-3 for temperature 0, a uniform farther than 1e-4 from its
     bin's edges for T > 0; the kernel's errors are near 1e-6). Most random requests qualify,
     and the test requires that most do.
"""
import numpy as np
import pytest
import torch

import speculative_decoding_block_dflash_gb300 as dfl
from oracle import selector as osel
from speculative_decoding_block_dflash_gb300 import build as build_mod

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    build_mod.build()
    dfl.load_library()


def _inputs(R, S, K, V, E, seed):
    g = torch.Generator(device="cuda").manual_seed(seed)
    A = torch.randn((V, E), generator=g, device="cuda").to(torch.bfloat16)
    B = torch.randn((V, E), generator=g, device="cuda").to(torch.bfloat16)
    proj = torch.randn((R, S, E), generator=g, device="cuda") / E ** 0.5
    cand = torch.randint(0, V, (R, S, K), generator=g, device="cuda", dtype=torch.int32)
    unary = torch.randn((R, S, K), generator=g, device="cuda")
    anchor = torch.randint(0, V, (R,), generator=g, device="cuda", dtype=torch.int32)
    u = torch.rand((R, S), generator=g, device="cuda")
    return A, B, proj, cand, unary, anchor, u


def _wide(t):
    return osel.widen_bf16(t.view(torch.int16).cpu().numpy())


def _check(A, B, proj, cand, unary, anchor, T, u, tokens, chosen, scores, q, min_exact=0.75):
    Ah, Bh = _wide(A), _wide(B)
    P = proj.cpu().numpy().astype(np.float64)
    C = cand.cpu().numpy()
    U = unary.cpu().numpy().astype(np.float64)
    an = anchor.cpu().numpy()
    uu = u.cpu().numpy().astype(np.float64)
    tk, ch, sc = tokens.cpu().numpy(), chosen.cpu().numpy(), scores.cpu().numpy().astype(np.float64)
    qq = q.cpu().numpy().astype(np.float64) if q is not None else None
    R, S, K = C.shape
    for r in range(R):
        prev = int(an[r])
        for s in range(S):
            e = osel.edge_scores(Ah, Bh, P[r, s], C[r, s], U[r, s], prev)
            mag = np.abs(Bh[C[r, s]] * (Ah[prev] * P[r, s])[None, :]).sum(axis=1) + np.abs(U[r, s])
            tol = 1e-5 * (1.0 + mag)
            assert np.all(np.abs(sc[r, s] - e) <= tol), (r, s, np.abs(sc[r, s] - e).max())
            k = int(ch[r, s])
            assert 0 <= k < K and tk[r, s] == C[r, s, k]
            if T == 0:
                assert e[k] >= e.max() - 2 * tol.max(), (r, s)
            else:
                p = np.exp((e - e.max()) / T)
                p /= p.sum()
                assert np.all(np.abs(qq[r, s] - p) <= 1e-5), (r, s)
                cdf = np.cumsum(p)
                assert k == 0 or cdf[k - 1] <= uu[r, s] + 1e-5, (r, s)
                assert k == K - 1 or cdf[k] > uu[r, s] - 1e-5, (r, s)
            prev = int(tk[r, s])
    # whole-path agreement where the oracle's own decisions are far from a tie
    ot, ok, osc, oq = osel.walk(Ah, Bh, P, C, U, an, temperature=T, u=uu)
    exact = 0
    for r in range(R):
        margin = np.inf
        for s in range(S):
            e = osc[r, s]
            if T == 0:
                top = np.sort(e)[::-1]
                margin = min(margin, top[0] - top[1] if K > 1 else np.inf)
            else:
                margin = min(margin, np.abs(np.cumsum(oq[r, s]) - uu[r, s]).min())
        if margin > (1e-3 if T == 0 else 1e-4):
            exact += 1
            np.testing.assert_array_equal(tk[r], ot[r])
            np.testing.assert_array_equal(ch[r], ok[r])
    assert exact >= min_exact * R, (exact, R)


@pytest.mark.parametrize("T", [0.0, 1.0, 0.5])
@pytest.mark.parametrize("R,S,K,V,E", [
    (1, 1, 1, 50, 8),         # one slot, one candidate
    (4, 15, 8, 5000, 256),    # 15 speculative slots, 8 candidates
    (3, 7, 33, 1000, 64),     # more candidates than a warp's lanes
    (2, 15, 64, 2000, 512),   # the most candidates, the largest staged rows
    (6, 3, 5, 300, 1024),
])
def test_matches_oracle(T, R, S, K, V, E):
    A, B, proj, cand, unary, anchor, u = _inputs(R, S, K, V, E, seed=R * 1000 + S * 10 + K + E)
    tokens, chosen, scores, q = dfl.selector_walk(A, B, proj, cand, unary, anchor, temperature=T,
                                                  uniforms=u if T > 0 else None)
    torch.cuda.synchronize()
    _check(A, B, proj, cand, unary, anchor, T, u, tokens, chosen, scores, q, min_exact=0.5 if R < 3 else 0.75)


def test_greedy_needs_no_q_and_reuses_the_workspace():
    A, B, proj, cand, unary, anchor, u = _inputs(8, 15, 8, 4000, 256, seed=3)
    ws = torch.zeros(dfl.selector_workspace_bytes(8, 15, 8), dtype=torch.uint8, device="cuda")
    first = dfl.selector_walk(A, B, proj, cand, unary, anchor, workspace=ws)
    second = dfl.selector_walk(A, B, proj, cand, unary, anchor, workspace=ws)  # counters were reset
    torch.cuda.synchronize()
    assert first[3] is None
    assert torch.equal(first[0], second[0]) and torch.equal(first[1], second[1])
    _check(A, B, proj, cand, unary, anchor, 0.0, u, *first)


def test_token_ids_outside_the_vocabulary_are_flagged():
    A, B, proj, cand, unary, anchor, u = _inputs(2, 4, 4, 100, 64, seed=4)
    cand[1, 2, 3] = 100  # one past the vocabulary
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    dfl.selector_walk(A, B, proj, cand, unary, anchor, device_error=err)
    torch.cuda.synchronize()
    assert int(err.item()) == dfl.DEVERR_TOKEN_ID


def test_cuda_graph_replay():
    A, B, proj, cand, unary, anchor, u = _inputs(4, 15, 8, 3000, 256, seed=5)
    ws = torch.zeros(dfl.selector_workspace_bytes(4, 15, 8), dtype=torch.uint8, device="cuda")
    tokens = torch.empty((4, 15), dtype=torch.int32, device="cuda")
    chosen = torch.empty_like(tokens)
    scores = torch.empty((4, 15, 8), device="cuda")
    q = torch.empty((4, 15, 8), device="cuda")
    s = torch.cuda.Stream()
    kw = dict(temperature=1.0, uniforms=u, workspace=ws, tokens=tokens, chosen=chosen, path_scores=scores, q=q,
              stream=s)
    with torch.cuda.stream(s):
        dfl.selector_walk(A, B, proj, cand, unary, anchor, **kw)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        dfl.selector_walk(A, B, proj, cand, unary, anchor, **kw)
    tokens.fill_(-1)
    graph.replay()
    torch.cuda.synchronize()
    _check(A, B, proj, cand, unary, anchor, 1.0, u, tokens, chosen, scores, q)


def test_full_size_batch32_sampling():
    # the bench's launch: 32 requests x 15 slots x 8 candidates over a 151936-token codebook of
    # width 256, temperature 1
    A, B, proj, cand, unary, anchor, u = _inputs(32, 15, 8, 151936, 256, seed=6)
    tokens, chosen, scores, q = dfl.selector_walk(A, B, proj, cand, unary, anchor, temperature=1.0, uniforms=u)
    torch.cuda.synchronize()
    _check(A, B, proj, cand, unary, anchor, 1.0, u, tokens, chosen, scores, q)


def test_one_workspace_serves_calls_of_different_sizes():
    # a larger call leaves edge tables where a smaller call's counters would sit if their
    # offset depended on the sizes; the fixed counter block keeps the smaller call correct
    big = _inputs(4, 15, 64, 2000, 512, seed=8)
    small = _inputs(8, 15, 8, 3000, 256, seed=9)
    need = max(dfl.selector_workspace_bytes(4, 15, 64), dfl.selector_workspace_bytes(8, 15, 8))
    ws = torch.zeros(need, dtype=torch.uint8, device="cuda")
    for A, B, proj, cand, unary, anchor, u in (big, small, big, small):
        out = dfl.selector_walk(A, B, proj, cand, unary, anchor, temperature=1.0, uniforms=u, workspace=ws)
        torch.cuda.synchronize()
        _check(A, B, proj, cand, unary, anchor, 1.0, u, *out, min_exact=0.5)
