"""GPU parity for dflash_project_kv (through its C ABI) against oracle/project.py.

The kernel rounds an fp32 tensor-core sum to bf16; the oracle sums the same bf16 inputs in
float64. The bar is the bf16 one: |kernel - oracle| <= 1e-2 + 1e-2 * |oracle| per element
(one bf16 rounding is at most 2^-9 relative; the fp32 accumulation error over a few
thousand terms of unit-scale products is far below that). Cache slots that no token maps to
must keep their sentinel bytes, which catches stray writes.
"""
import numpy as np
import pytest
import torch

import speculative_decoding_block_dflash_gb300 as dfl
from oracle import project as oracle_project
from speculative_decoding_block_dflash_gb300 import build as build_mod

pytestmark = pytest.mark.gpu

ATOL = 1e-2
RTOL = 1e-2
SENTINEL = -7.0  # exact in bf16


@pytest.fixture(scope="module", autouse=True)
def _built():
    build_mod.build()
    dfl.load_library()


def _host_f64(t):
    return oracle_project.widen_bf16(t.contiguous().view(torch.int16).cpu().numpy())


def _inputs(L, H, Hkv, D, page_size, num_pages, seed, stride=None):
    g = torch.Generator(device="cuda").manual_seed(seed)
    N = Hkv * D
    rows = torch.randn((L, stride or H), generator=g, device="cuda").to(torch.bfloat16)
    hidden = rows[:, :H]
    w_k = (torch.randn((N, H), generator=g, device="cuda") / H ** 0.5).to(torch.bfloat16)
    w_v = (torch.randn((N, H), generator=g, device="cuda") / H ** 0.5).to(torch.bfloat16)
    k_cache = torch.full((num_pages, page_size, Hkv, D), SENTINEL, device="cuda", dtype=torch.bfloat16)
    v_cache = torch.full_like(k_cache, SENTINEL)
    return hidden, w_k, w_v, k_cache, v_cache


def _slots(L, page_size, num_pages, seed, pos0=None):
    """Slot ids of a request whose tokens start at position pos0, pages from a shuffled table."""
    rng = np.random.default_rng(seed)
    if pos0 is None:
        pos0 = int(rng.integers(0, page_size * 3))
    need = (pos0 + L + page_size - 1) // page_size
    assert need <= num_pages
    table = rng.permutation(num_pages)[:need]
    pages, pos = oracle_project.cache_coords(L, pos0, page_size, table)
    return pages, pos, torch.from_numpy((pages * page_size + pos).astype(np.int32)).cuda()


def _check(hidden, w_k, w_v, k_cache, v_cache, pages, pos, rows=None):
    """Compare the cache slots of the given token rows (all by default) with the oracle."""
    Hkv, D = k_cache.shape[2], k_cache.shape[3]
    rows = np.arange(hidden.shape[0]) if rows is None else rows
    h = _host_f64(hidden[torch.from_numpy(rows).cuda()])
    e_k, e_v = oracle_project.project_kv(h, _host_f64(w_k), _host_f64(w_v), Hkv, D)
    pg = torch.from_numpy(pages[rows]).cuda()
    ps = torch.from_numpy(pos[rows]).cuda()
    for cache, e in ((k_cache, e_k), (v_cache, e_v)):
        got = cache[pg, ps].float().cpu().numpy().astype(np.float64)
        err = np.abs(got - e) - (ATOL + RTOL * np.abs(e))
        assert err.max() <= 0, f"max excess {err.max()} at {np.unravel_index(err.argmax(), err.shape)}"


def _untouched(cache, pages, pos):
    mask = torch.ones(cache.shape[:2], dtype=torch.bool, device="cuda")
    mask[torch.from_numpy(pages).cuda(), torch.from_numpy(pos).cuda()] = False
    rest = cache[mask]
    assert bool((rest == SENTINEL).all()), "a slot no token maps to was written"


@pytest.mark.parametrize("L,H,Hkv,D,page_size", [
    (1, 64, 1, 128, 16),       # one decode token, N below one feature tile
    (9, 320, 2, 128, 16),      # a verified block
    (200, 320, 2, 128, 16),    # two token tiles, ragged tail
    (130, 200, 3, 64, 32),     # hidden size not a multiple of 64; N = 192
    (257, 512, 5, 128, 16),    # N = 640: a partial last feature tile
    (300, 1024, 4, 512, 64),   # head_dim 512, 2 feature tiles per projection
])
def test_matches_oracle(L, H, Hkv, D, page_size):
    num_pages = (L + 3 * page_size) // page_size + 4
    hidden, w_k, w_v, k_cache, v_cache = _inputs(L, H, Hkv, D, page_size, num_pages, seed=L + H)
    pages, pos, slots = _slots(L, page_size, num_pages, seed=L)
    dfl.project_kv(hidden, w_k, w_v, slots, k_cache, v_cache)
    torch.cuda.synchronize()
    _check(hidden, w_k, w_v, k_cache, v_cache, pages, pos)
    _untouched(k_cache, pages, pos)
    _untouched(v_cache, pages, pos)


def test_strided_hidden_rows_and_many_tiles():
    # rows of a wider buffer; more tiles than CTA pairs (24 x 8 = 192 tiles of 256 x 256), so
    # that pairs loop over tiles
    L, H, Hkv, D, P = 6000, 256, 4, 256, 16
    num_pages = L // P + 8
    hidden, w_k, w_v, k_cache, v_cache = _inputs(L, H, Hkv, D, P, num_pages, seed=3, stride=H + 64)
    assert hidden.stride(0) == H + 64
    pages, pos, slots = _slots(L, P, num_pages, seed=4)
    dfl.project_kv(hidden, w_k, w_v, slots, k_cache, v_cache)
    torch.cuda.synchronize()
    _check(hidden, w_k, w_v, k_cache, v_cache, pages, pos)
    _untouched(k_cache, pages, pos)


def test_skipped_and_out_of_range_slots():
    L, H, Hkv, D, P = 40, 128, 2, 128, 16
    num_pages = 8
    hidden, w_k, w_v, k_cache, v_cache = _inputs(L, H, Hkv, D, P, num_pages, seed=7)
    pages, pos, slots = _slots(L, P, num_pages, seed=8, pos0=0)
    slots[5] = -1
    slots[6] = num_pages * P  # one past the pool: flagged and skipped
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    dfl.project_kv(hidden, w_k, w_v, slots, k_cache, v_cache, device_error=err)
    torch.cuda.synchronize()
    assert int(err.item()) == dfl.DEVERR_PAGE_ID
    keep = np.array([r for r in range(L) if r not in (5, 6)])
    _check(hidden, w_k, w_v, k_cache, v_cache, pages, pos, rows=keep)
    _untouched(k_cache, pages[keep], pos[keep])


def test_zero_tokens_is_a_no_op():
    hidden, w_k, w_v, k_cache, v_cache = _inputs(0, 64, 1, 128, 16, 2, seed=1)
    dfl.project_kv(hidden, w_k, w_v, torch.empty(0, dtype=torch.int32, device="cuda"), k_cache, v_cache)
    torch.cuda.synchronize()
    assert bool((k_cache == SENTINEL).all())


def test_cuda_graph_replay():
    L, H, Hkv, D, P = 64, 256, 2, 128, 16
    num_pages = 8
    hidden, w_k, w_v, k_cache, v_cache = _inputs(L, H, Hkv, D, P, num_pages, seed=11)
    pages, pos, slots = _slots(L, P, num_pages, seed=12)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        dfl.project_kv(hidden, w_k, w_v, slots, k_cache, v_cache)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        dfl.project_kv(hidden, w_k, w_v, slots, k_cache, v_cache)
    k_cache.fill_(SENTINEL)
    v_cache.fill_(SENTINEL)
    graph.replay()
    torch.cuda.synchronize()
    _check(hidden, w_k, w_v, k_cache, v_cache, pages, pos)


def test_full_size_prefill_sampled_rows():
    # an 8192-token context of 5376-wide hidden states into 4 KV heads of 512 (page 16),
    # the launch the benchmark times; 192 sampled token rows against the oracle
    L, H, Hkv, D, P = 8192, 5376, 4, 512, 16
    num_pages = L // P + 16
    hidden, w_k, w_v, k_cache, v_cache = _inputs(L, H, Hkv, D, P, num_pages, seed=21)
    pages, pos, slots = _slots(L, P, num_pages, seed=22)
    dfl.project_kv(hidden, w_k, w_v, slots, k_cache, v_cache)
    torch.cuda.synchronize()
    rng = np.random.default_rng(23)
    rows = np.unique(np.concatenate([rng.choice(L, 160, replace=False), np.arange(16), np.arange(L - 16, L)]))
    _check(hidden, w_k, w_v, k_cache, v_cache, pages, pos, rows=rows)
    _untouched(k_cache, pages, pos)
    _untouched(v_cache, pages, pos)


@pytest.mark.parametrize("split", [True, False])
def test_split_last_round_matches_oracle(split):
    # 5000 tokens into 4 x 512 features: 20 x 16 = 320 tiles of 256 x 256 on 76 CTA pairs leave
    # 16 for a fifth round, which the split runs as 32 halves along the hidden dimension
    L, H, Hkv, D, P = 5000, 512, 4, 512, 16
    num_pages = L // P + 8
    hidden, w_k, w_v, k_cache, v_cache = _inputs(L, H, Hkv, D, P, num_pages, seed=31)
    pages, pos, slots = _slots(L, P, num_pages, seed=32)
    ws = torch.zeros(dfl.load_library().dflash_project_kv_workspace_bytes(), dtype=torch.uint8, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    for _ in range(2):  # the second call reuses the workspace: its counters were reset
        k_cache.fill_(SENTINEL)
        v_cache.fill_(SENTINEL)
        dfl.project_kv(hidden, w_k, w_v, slots, k_cache, v_cache, device_error=err, workspace=ws if split else None,
                       split=split)
        torch.cuda.synchronize()
        assert int(err.item()) == 0
        _check(hidden, w_k, w_v, k_cache, v_cache, pages, pos)
        _untouched(k_cache, pages, pos)
    assert int(ws[:8192].view(torch.int32).abs().sum().item()) == 0  # the counter block is back at zero
