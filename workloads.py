"""Seeded synthetic inputs for DFlash block attention.

This module only draws random numbers and lays them out; it holds none of the
attention arithmetic. Both the CUDA path and the fp64 oracle receive the same
tensors from here (the oracle gets host copies).

Shapes follow Gemma-4-31B-like verify/draft workloads: a block of
T = 1 + num_speculative_tokens queries per request ("num_query_per_req =
1 + num_speculative_tokens", kenforever1 "dflash-gemma4-31b-notes"), global
layers with head_dim 512 and sliding-window layers, a paged KV cache of page
size 16 whose pages are scattered over a larger pool by a random permutation.

Named workloads (seed = 1234 + index):
  tiny            B=1, T=9, Hq=Hkv=1, D=64, L=128, identity page table, fp32
  global_verify   B=1, T=9, Hq=32, Hkv=4, D=512, L=8192, bf16, pool = 2x pages
  batch_sweep_bN  N in {1,2,4,8}: L_b ~ U[1024, 32768], otherwise as global_verify
  sliding         B=4, T=9, Hq=32, Hkv=16, D=256, W=1024, L=32768, bf16
  long_draft      B=8, T=16, Hq=32, Hkv=4, D=512, L=131072, 16 splits; K/V are a
                  projection of N(0,1) hidden states [L, 5376] through N(0, 0.02^2)
                  weights [5376, Hkv*D], stored bf16
"""
from __future__ import annotations

import dataclasses
import math
from typing import List, Optional, Sequence

import torch

PAGE_SIZE = 16


@dataclasses.dataclass
class Case:
    name: str
    q: torch.Tensor            # [B*T, Hq, D]
    k_cache: torch.Tensor      # [num_pages, page_size, Hkv, D]
    v_cache: torch.Tensor      # same
    page_table: torch.Tensor   # int32 [B, max_pages] (layer 0)
    seq_lens: torch.Tensor     # int32 [B]
    block_len: int
    causal: bool
    window: int
    scale: float
    num_splits: int = 0        # 0 = library chooses
    page_tables: Optional[List[torch.Tensor]] = None  # one per rotated layer (bench)

    @property
    def batch(self) -> int:
        return self.seq_lens.shape[0]

    @property
    def num_q_heads(self) -> int:
        return self.q.shape[1]

    @property
    def num_kv_heads(self) -> int:
        return self.k_cache.shape[2]

    @property
    def head_dim(self) -> int:
        return self.q.shape[2]

    @property
    def page_size(self) -> int:
        return self.k_cache.shape[1]

    def seq_lens_host(self) -> List[int]:
        return [int(x) for x in self.seq_lens.cpu().tolist()]


def _gen(device, seed):
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def _page_tables(seq_lens: Sequence[int], page_size: int, pool_pages: int, layers: int,
                 gen, device) -> List[torch.Tensor]:
    """Disjoint random page assignments, one per layer, from one shuffled pool."""
    need = [(L + page_size - 1) // page_size for L in seq_lens]
    max_pages = max(need)
    total = sum(need)
    if pool_pages < total * layers:
        raise ValueError("page pool too small")
    perm = torch.randperm(pool_pages, generator=gen, device=device).to(torch.int32)
    tables = []
    cursor = 0
    for _ in range(layers):
        pt = torch.zeros((len(seq_lens), max_pages), dtype=torch.int32, device=device)
        for b, n in enumerate(need):
            pt[b, :n] = perm[cursor:cursor + n]
            cursor += n
        tables.append(pt)
    return tables


def make_custom(name: str, batch: int, block_len: int, num_q_heads: int, num_kv_heads: int,
                head_dim: int, seq_lens: Sequence[int], dtype=torch.bfloat16,
                page_size: int = PAGE_SIZE, pool_factor: float = 2.0, layers: int = 1,
                causal: bool = False, window: int = 0, scale: Optional[float] = None,
                identity_pages: bool = False, seed: int = 0, device="cpu",
                num_splits: int = 0, value_std: float = 1.0) -> Case:
    """Generic seeded case: q, k, v ~ N(0, value_std^2), rounded once to `dtype`."""
    device = torch.device(device)
    gen = _gen(device, seed)
    seq_lens = [int(x) for x in seq_lens]
    assert len(seq_lens) == batch
    need = sum((L + page_size - 1) // page_size for L in seq_lens)
    if identity_pages:
        assert layers == 1
        pool = need
        tables = []
        pt = torch.zeros((batch, max((L + page_size - 1) // page_size for L in seq_lens)),
                         dtype=torch.int32, device=device)
        cursor = 0
        for b, L in enumerate(seq_lens):
            n = (L + page_size - 1) // page_size
            pt[b, :n] = torch.arange(cursor, cursor + n, dtype=torch.int32, device=device)
            cursor += n
        tables = [pt]
    else:
        pool = max(int(math.ceil(need * layers * pool_factor)), need * layers)
        tables = _page_tables(seq_lens, page_size, pool, layers, gen, device)
    q = (torch.randn((batch * block_len, num_q_heads, head_dim), generator=gen, device=device)
         * value_std).to(dtype)
    k = (torch.randn((pool, page_size, num_kv_heads, head_dim), generator=gen, device=device)
         * value_std).to(dtype)
    v = (torch.randn((pool, page_size, num_kv_heads, head_dim), generator=gen, device=device)
         * value_std).to(dtype)
    sl = torch.tensor(seq_lens, dtype=torch.int32, device=device)
    return Case(name=name, q=q, k_cache=k, v_cache=v, page_table=tables[0], seq_lens=sl,
                block_len=block_len, causal=causal, window=window,
                scale=(1.0 / math.sqrt(head_dim)) if scale is None else float(scale),
                num_splits=num_splits, page_tables=tables)


def _uniform_lens(batch: int, lo: int, hi: int, seed: int) -> List[int]:
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    return [int(x) for x in torch.randint(lo, hi + 1, (batch,), generator=g).tolist()]


def _projected_kv(case: Case, hidden: int, seed: int, chunk: int = 16384) -> None:
    """Fill the used pages of k/v with (N(0,1) hidden states) @ (N(0, 0.02^2) weights).

    Input preparation for the draft pass: context K/V come from target hidden
    states. Done chunk by chunk in bf16 on the case's device.
    """
    dev = case.q.device
    gen = _gen(dev, seed + 7)
    Hkv, D, P = case.num_kv_heads, case.head_dim, case.page_size
    w_k = (torch.randn((hidden, Hkv * D), generator=gen, device=dev) * 0.02).to(torch.bfloat16)
    w_v = (torch.randn((hidden, Hkv * D), generator=gen, device=dev) * 0.02).to(torch.bfloat16)
    for b, L in enumerate(case.seq_lens_host()):
        for t0 in range(0, L, chunk):
            t1 = min(L, t0 + chunk)
            h = torch.randn((t1 - t0, hidden), generator=gen, device=dev).to(torch.bfloat16)
            kk = (h @ w_k).view(t1 - t0, Hkv, D)
            vv = (h @ w_v).view(t1 - t0, Hkv, D)
            pos = torch.arange(t0, t1, device=dev)
            for pt in case.page_tables:
                pages = pt[b].long()[pos // P]
                case.k_cache[pages, pos % P] = kk
                case.v_cache[pages, pos % P] = vv


LONG_DRAFT = dict(B=8, T=16, Hq=32, Hkv=4, D=512, L=131072, splits=16)

CONFIG_NAMES = ["tiny", "global_verify", "batch_sweep_b1", "batch_sweep_b2", "batch_sweep_b4",
                "batch_sweep_b8", "sliding", "sliding_causal", "long_draft"]


def make_case(name: str, device="cuda", layers: int = 1, batch: Optional[int] = None) -> Case:
    """One of the named workloads above. `layers` > 1 adds disjoint page tables
    (distinct K/V per layer) so a benchmark can rotate through more bytes than L2.
    `batch` takes the first requests of long_draft only (its requests are alike, so a
    profiler can capture the same kernel on a fraction of the 17 GB cache)."""
    if name == "tiny":
        return make_custom(name, 1, 9, 1, 1, 64, [128], dtype=torch.float32, identity_pages=True,
                           scale=1.0 / 8.0, seed=1234 + 0, device=device)
    if name == "global_verify":
        return make_custom(name, 1, 9, 32, 4, 512, [8192], dtype=torch.bfloat16, pool_factor=2.0,
                           layers=layers, seed=1234 + 1, device=device)
    if name.startswith("batch_sweep_b"):
        B = int(name[len("batch_sweep_b"):])
        lens = _uniform_lens(B, 1024, 32768, seed=1234 + 2 + B)
        return make_custom(name, B, 9, 32, 4, 512, lens, dtype=torch.bfloat16, pool_factor=2.0,
                           layers=layers, seed=1234 + 2, device=device)
    if name in ("sliding", "sliding_causal"):
        return make_custom(name, 4, 9, 32, 16, 256, [32768] * 4, dtype=torch.bfloat16,
                           pool_factor=1.0, layers=layers, window=1024,
                           causal=(name == "sliding_causal"), seed=1234 + 3, device=device)
    if name == "long_draft":
        sh = LONG_DRAFT
        nb = sh["B"] if batch is None else batch
        case = make_custom(name, nb, sh["T"], sh["Hq"], sh["Hkv"], sh["D"], [sh["L"]] * nb,
                           dtype=torch.bfloat16, pool_factor=1.0, layers=layers, seed=1234 + 4, device=device,
                           num_splits=sh["splits"])
        _projected_kv(case, hidden=5376, seed=1234 + 4)
        return case
    raise KeyError(name)



def make_group_sample(name: str, keys: int, device="cpu", seed: int = 0) -> Case:
    """One (request, KV head) group of a named workload, restricted to its last `keys` keys.

    Same shapes per group (block_len, head_dim, the G query heads that share a KV head,
    page size) and the same value distributions as make_case(name), at batch 1 with a single
    KV head and seq_len = keys: what a CPU timing of the oracle on a bounded sample of that
    workload needs, without generating the whole K/V pool. For long_draft the K/V rows are a
    projection of N(0,1) hidden states of width 5376 through N(0, 0.02^2) weights of one head.
    Only the non-causal global workloads (global_verify, batch_sweep_b*, long_draft) are
    offered: their work is linear in the keys seen, so a sample scales to the full step.
    """
    shapes = {
        "global_verify": dict(T=9, Hq=32, Hkv=4, D=512),
        "long_draft": dict(T=16, Hq=32, Hkv=4, D=512),
    }
    if name.startswith("batch_sweep_b"):
        shapes[name] = dict(T=9, Hq=32, Hkv=4, D=512)
    sh = shapes[name]
    G = sh["Hq"] // sh["Hkv"]
    case = make_custom(name + "_group", 1, sh["T"], G, 1, sh["D"], [int(keys)], dtype=torch.bfloat16,
                       pool_factor=1.0, seed=seed, device=device)
    if name == "long_draft":
        dev = case.q.device
        gen = _gen(dev, seed + 7)
        hidden, D, P = 5376, sh["D"], case.page_size
        w_k = torch.randn((hidden, D), generator=gen, device=dev) * 0.02
        w_v = torch.randn((hidden, D), generator=gen, device=dev) * 0.02
        for t0 in range(0, int(keys), 4096):
            t1 = min(int(keys), t0 + 4096)
            h = torch.randn((t1 - t0, hidden), generator=gen, device=dev).to(torch.bfloat16).float()
            pos = torch.arange(t0, t1, device=dev)
            pages = case.page_table[0].long()[pos // P]
            case.k_cache[pages, pos % P, 0] = (h @ w_k).to(torch.bfloat16)
            case.v_cache[pages, pos % P, 0] = (h @ w_v).to(torch.bfloat16)
    return case
