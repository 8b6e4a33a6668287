#!/usr/bin/env python3
"""DFlash block attention benchmark: K/V HBM GB/s and block-queries/s.

A step is one dflash_block_attn call (argument check, split plan, paged K/V
staging, QK^T, masked online softmax, PV, split combine) over one layer's
paged KV cache for the workload below. Steps rotate over `layers` disjoint
page sets so the bytes touched between two visits of the same layer exceed
the 129 MB L2 (inputs larger than L2; no flush kernel in the timed region).
The timed loop replays one CUDA graph per layer (one captured call each):
the pages report FULL CUDA-graph capture as the way DFlash avoids being
launch-bound, and a Python/ctypes launch per 10 us kernel would be.

value = algorithmic K/V bytes per step (every visible (token, kv-head) row of
K and V once, bf16) / device time per step, summed over ranks.

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

WORKLOAD = "long_draft"
WORKLOAD_DESC = ("long-context split-KV draft cross-attention: batch 8, block_len 16 (num_spec 15), 32 q heads / "
                 "4 KV heads (GQA 8), head_dim 512, context 131072 tokens paged (page 16, shuffled page table), "
                 "16 split-KV chunks with LSE combine; K/V projected from N(0,1) hidden states of width 5376 "
                 "through N(0, 0.02^2) weights, bf16, causal=False")
# The other attention workloads, measured in the same run and reported under "workloads".
OTHER_WORKLOADS = ["global_verify", "batch_sweep_b1", "batch_sweep_b2", "batch_sweep_b4", "batch_sweep_b8",
                   "sliding", "sliding_causal"]
METRIC = "kv_hbm_gbs"
UNIT = "GB/s"
L2_BYTES = 129 * 1024 * 1024


def max_over_ranks(x: float) -> float:
    """The largest value of a per-rank float over the job (the slowest rank sets the job's
    time); the value itself when no process group is running."""
    import torch.distributed as tdist

    if not (tdist.is_available() and tdist.is_initialized()) or tdist.get_world_size() == 1:
        return float(x)
    dev = torch.device("cuda", torch.cuda.current_device()) if tdist.get_backend() == "nccl" else torch.device("cpu")
    t = torch.tensor([float(x)], dtype=torch.float64, device=dev)
    tdist.all_reduce(t, op=tdist.ReduceOp.MAX)
    return float(t.item())


def barrier():
    import torch.distributed as tdist

    if tdist.is_available() and tdist.is_initialized() and tdist.get_world_size() > 1:
        tdist.barrier()


def process_group_backend() -> str:
    """nccl with GPUs, gloo on a host without them (the CPU tests of the multi-rank path)."""
    return "nccl" if torch.cuda.is_available() else "gloo"


def env_int(name, default):
    try:
        return int(os.environ.get(name, default))
    except ValueError:
        return default


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20000)
    ap.add_argument("--warmup", type=int, default=200)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--config", default=WORKLOAD)
    ap.add_argument("--kernel", default="auto", choices=["auto", "simt", "tc", "tc_pair"])
    ap.add_argument("--splits", type=int, default=-1, help="-1: the workload's own (auto unless fixed)")
    ap.add_argument("--layers", type=int, default=0, help="page-set rotation count (0 = enough to exceed 4x L2)")
    ap.add_argument("--e2e-steps", type=int, default=500)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-other-workloads", action="store_true",
                    help="headline run only: skip the other attention workloads' extra key")
    ap.add_argument("--cpu-budget", type=float, default=20.0, help="seconds of oracle time for cpu_baseline")
    ap.add_argument("--ref-budget", type=float, default=120.0, help="seconds of oracle time for --impl reference")
    ap.add_argument("--capture", metavar="WORKLOAD", default=None,
                    help="profiler target: two block_attn calls on one layer of this attention workload, "
                         "nothing timed")
    ap.add_argument("--capture-batch", type=int, default=None,
                    help="with --capture long_draft: its first N requests (a capture-sized cache)")
    return ap.parse_args()


# ----------------------------------------------------------------------------- accounting


def visible_union_keys(case):
    """Keys any block query of each request can see (union of the rows' ranges)."""
    T, W = case.block_len, case.window
    n = 0
    for L in case.seq_lens_host():
        lo = max(0, L - T - W + 1) if W > 0 else 0
        n += L - lo
    return n


def kv_bytes_per_step(case):
    return visible_union_keys(case) * case.num_kv_heads * case.head_dim * case.k_cache.element_size() * 2


def io_bytes_per_step(case):
    q = case.q.numel() * case.q.element_size()
    return 2 * q + case.q.shape[0] * case.q.shape[1] * 4  # q in, out, lse


# ----------------------------------------------------------------------------- clocks


class ClockSampler:
    """nvidia-smi sampling of SM clock and throttle reasons while the timed loop runs."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int, period_ms: int = 50):
        self.gpu_index = gpu_index
        self.period_ms = period_ms
        self.proc = None
        self.lines = []
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.QUERY}", "--format=csv,noheader,nounits",
                 f"-lms", str(self.period_ms), "-i", str(self.gpu_index)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, FileNotFoundError):
            self.proc = None
            return
        self.thread = threading.Thread(target=self._reader, daemon=True)
        self.thread.start()
        time.sleep(0.3)  # let the first samples arrive before the timed region

    def _reader(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def stop(self):
        if self.proc is None:
            return
        time.sleep(0.1)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        if self.thread:
            self.thread.join(timeout=5)

    def summary(self, t0, t1):
        samples = []
        for ts, line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm, smax = float(parts[1]), float(parts[2])
            except ValueError:
                continue
            samples.append((ts, sm, smax, parts))
        inside = [s for s in samples if t0 <= s[0] <= t1]
        use = inside if inside else samples
        if not use:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no nvidia-smi samples"], "samples": 0}
        reasons = set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for _, _, _, parts in use:
            for name, val in zip(names, parts[5:9]):
                if val.lower() in ("active", "1", "yes"):
                    reasons.add(name)
        return {"sm_mhz": statistics.median(s[1] for s in use), "sm_max_mhz": max(s[2] for s in use),
                "reasons": sorted(reasons), "samples": len(inside),
                "samples_note": None if inside else "no sample fell inside the timed region; nearest samples used"}


# ----------------------------------------------------------------------------- oracle (CPU) legs


def host_copy_of_layer(case, layer=0):
    """Host copy of one layer's inputs with its pages compacted (index work only)."""
    pt = case.page_tables[layer]
    used = pt[:, : pt.shape[1]].reshape(-1).unique()
    remap = torch.full((case.k_cache.shape[0],), -1, dtype=torch.int32, device=pt.device)
    remap[used.long()] = torch.arange(used.numel(), dtype=torch.int32, device=pt.device)
    k = case.k_cache[used.long()].cpu()
    v = case.v_cache[used.long()].cpu()
    pt2 = remap[pt.long()].cpu()
    return dict(q=case.q.cpu(), k=k, v=v, pt=pt2, sl=case.seq_lens.cpu())


def time_oracle_full(case, budget_s, threads=None):
    """Oracle over whole steps (every row, every key) until the budget is used; seconds per step."""
    import oracle

    h = host_copy_of_layer(case)
    threads = threads or oracle.default_threads()
    times = []
    t_start = time.perf_counter()
    while True:
        t0 = time.perf_counter()
        oracle.block_attn(h["q"], h["k"], h["v"], h["pt"], h["sl"], case.block_len, causal=case.causal,
                          window=case.window, scale=case.scale, num_threads=threads)
        times.append(time.perf_counter() - t0)
        if time.perf_counter() - t_start > budget_s or len(times) >= 50:
            break
    return statistics.median(times), len(times), threads


def group_host_problem(case, b, g, kb):
    """Host copy of one (request b, KV head g) group of a case restricted to keys [kb, L_b): the
    G query heads' block rows and the pages that hold those keys, compacted (index work only).
    Returns the oracle's inputs and the key range in the compacted positions."""
    T, P = case.block_len, case.page_size
    G = case.num_q_heads // case.num_kv_heads
    L = case.seq_lens_host()[b]
    p0, p1 = kb // P, (L + P - 1) // P
    pages = case.page_table[b, p0:p1].long()
    k = case.k_cache[pages][:, :, g:g + 1, :].cpu()
    v = case.v_cache[pages][:, :, g:g + 1, :].cpu()
    q = case.q[b * T:(b + 1) * T, g * G:(g + 1) * G, :].cpu()
    pt = torch.arange(p1 - p0, dtype=torch.int32).view(1, -1)
    sl = torch.tensor([L - p0 * P], dtype=torch.int32)
    return dict(q=q, k=k, v=v, pt=pt, sl=sl, key_range=(kb - p0 * P, L - p0 * P))


def time_oracle_group_sample(case, budget_s, threads=None):
    """Oracle time per full step, estimated from whole (request, KV head) groups.

    Only for non-causal global workloads, whose oracle work is (rows x keys seen): groups are
    timed one after another (request-major) until about budget_s of oracle time is spent or
    every group is done, and a full step is the sampled time x (keys of all groups / keys of
    the sampled groups)."""
    import oracle

    assert not case.causal and case.window == 0
    threads = threads or oracle.default_threads()
    lens = case.seq_lens_host()
    t_sum, keys_done, groups = 0.0, 0, []
    for b in range(case.batch):
        for g in range(case.num_kv_heads):
            h = group_host_problem(case, b, g, 0)
            t0 = time.perf_counter()
            oracle.block_attn(h["q"], h["k"], h["v"], h["pt"], h["sl"], case.block_len, scale=case.scale,
                              key_range=h["key_range"], num_threads=threads)
            t_sum += time.perf_counter() - t0
            keys_done += lens[b]
            groups.append((b, g))
            if t_sum >= budget_s:
                break
        if t_sum >= budget_s:
            break
    total_keys = sum(lens) * case.num_kv_heads
    t_step = t_sum * total_keys / keys_done
    rows = case.block_len * (case.num_q_heads // case.num_kv_heads)
    sample = (f"{len(groups)} of {case.batch * case.num_kv_heads} (request, KV head) groups, each in full "
              f"({rows} rows x every key), {t_sum:.1f} s; scaled by keys to a full step")
    return t_step, sample, threads


def reference_arm(args, case):
    """--impl reference: the fp64 oracle on the host cores, each step a key chunk of every row."""
    import oracle

    h = host_copy_of_layer(case)
    threads = oracle.default_threads()
    L = max(case.seq_lens_host())
    # calibrate one full step, then size the per-step chunk to the budget
    t0 = time.perf_counter()
    oracle.block_attn(h["q"], h["k"], h["v"], h["pt"], h["sl"], case.block_len, causal=case.causal,
                      window=case.window, scale=case.scale, num_threads=threads)
    t_full = time.perf_counter() - t0
    n_steps = args.steps + args.warmup
    frac = min(1.0, args.ref_budget / max(1e-9, n_steps * t_full))
    chunk = max(case.page_size, int(L * frac) // case.page_size * case.page_size)
    chunk = min(chunk, L)
    kb = L - chunk  # the block's own keys and the context just before them
    for _ in range(args.warmup):
        oracle.block_attn(h["q"], h["k"], h["v"], h["pt"], h["sl"], case.block_len, causal=case.causal,
                          window=case.window, scale=case.scale, key_range=(kb, L), num_threads=threads)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle.block_attn(h["q"], h["k"], h["v"], h["pt"], h["sl"], case.block_len, causal=case.causal,
                          window=case.window, scale=case.scale, key_range=(kb, L), num_threads=threads)
    dt = (time.perf_counter() - t0) / max(1, args.steps)
    scale_up = L / chunk  # every row of this workload sees all L keys
    t_step = dt * scale_up
    value = kv_bytes_per_step(case) / t_step / 1e9
    sample = (f"each step: oracle over keys [{kb}, {L}) of all {case.q.shape[0] * case.q.shape[1]} rows "
              f"({chunk} of {L} keys); time scaled by {scale_up:.2f} to a full step")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": t_step * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": WORKLOAD_DESC},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": threads, "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "block_queries_per_s": case.batch / t_step,
    }
    print(json.dumps(line), flush=True)


def group_reference_arm(args):
    """--impl reference for long_draft: each step is the oracle over one (request, KV head) group
    of the workload restricted to its last keys (a group of the same shapes and distributions,
    generated on its own), scaled by the keys of every group to a full step."""
    import oracle
    import workloads

    sh = workloads.LONG_DRAFT
    threads = oracle.default_threads()
    n_steps = args.steps + args.warmup

    def make(keys):
        case = workloads.make_group_sample(WORKLOAD, keys, device="cpu", seed=1234 + 4)
        h = host_copy_of_layer(case)
        return case, h

    def run(case, h):
        t0 = time.perf_counter()
        oracle.block_attn(h["q"], h["k"], h["v"], h["pt"], h["sl"], case.block_len, scale=case.scale,
                          num_threads=threads)
        return time.perf_counter() - t0

    cal_keys = 512
    case, h = make(cal_keys)
    t_cal = run(case, h)
    keys = int(min(sh["L"], max(cal_keys, cal_keys * args.ref_budget / max(1e-6, n_steps * t_cal))))
    keys = max(case.page_size, keys // case.page_size * case.page_size)
    case, h = make(keys)
    for _ in range(args.warmup):
        run(case, h)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        run(case, h)
    dt = (time.perf_counter() - t0) / max(1, args.steps)
    total_keys = sh["B"] * sh["L"] * sh["Hkv"]
    t_step = dt * total_keys / keys
    kv = total_keys * sh["D"] * 2 * 2
    value = kv / t_step / 1e9
    sample = (f"each step: oracle over one (request, KV head) group (all {sh['T'] * sh['Hq'] // sh['Hkv']} rows) "
              f"and the last {keys} of its {sh['L']} keys, generated with the workload's shapes and "
              f"distributions; time scaled by {total_keys / keys:.0f} to a full step")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": t_step * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": WORKLOAD_DESC},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": threads, "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "block_queries_per_s": sh["B"] / t_step,
    }
    print(json.dumps(line), flush=True)


# ----------------------------------------------------------------------------- acceptance


def accept_reference_arm(args):
    """--impl reference --config accept_verify: the oracle on the host, full steps."""
    from oracle import accept as oracle_accept

    dev = "cuda" if torch.cuda.is_available() else "cpu"
    logits, draft = accept_inputs(dev, 1)
    host = logits[0].view(torch.int16).cpu().numpy().view(np.uint16)
    dh = draft.cpu().numpy()
    for _ in range(args.warmup):
        oracle_accept.accept_prefix(host, dh, "bf16")
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle_accept.accept_prefix(host, dh, "bf16")
    t_step = (time.perf_counter() - t0) / max(1, args.steps)
    per = host.size * 2
    value = per / t_step / 1e9
    line = {"impl": "reference", "metric": "logits_hbm_gbs", "value": value, "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": t_step * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": ACCEPT_DESC},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": 1, "kind": "oracle",
                             "sample": "full steps: numpy argmax over all rows, then the prefix loop"},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


ACCEPT_CONFIG = "accept_verify"
ACCEPT_DESC = ("verify-step acceptance: batch 8, block_len 9 (1 bonus + 8 drafts), bf16 target logits over a "
               "262144-entry vocabulary (synthetic; the pages do not state the vocabulary size), drafts that "
               "match the target on a random prefix")


def accept_inputs(dev, n_sets, B=8, T=9, V=262144, seed=1234 + 7):
    """n_sets disjoint logits buffers [B, T, V] bf16 ~ N(0, 1) and, per set, drafts equal to the
    target tokens up to a random per-request position (workloads-style seeded synthetic data)."""
    from oracle import accept as oracle_accept

    g = torch.Generator(device=dev).manual_seed(seed)
    logits = [torch.randn((B, T, V), generator=g, device=dev).to(torch.bfloat16) for _ in range(n_sets)]
    rng = np.random.default_rng(seed)
    drafts = []
    for x in logits[:1]:
        t = oracle_accept.target_argmax(x.view(torch.int16).cpu().numpy().view(np.uint16), "bf16")
        d = t[:, :T - 1].copy()
        for b in range(B):
            k = int(rng.integers(0, T))
            if k < T - 1:
                d[b, k] = (d[b, k] + 1) % V
        drafts.append(torch.from_numpy(d.astype(np.int32)).to(dev))
    return logits, drafts[0]


def accept_bench(args, dfl, dev, rank, world):
    per = 8 * 9 * 262144 * 2
    n_sets = args.layers or max(2, math.ceil(4 * L2_BYTES / per))
    logits, draft = accept_inputs(dev, n_sets)
    B, T, V = logits[0].shape
    ws = torch.zeros(dfl.accept_workspace_bytes(B, T), dtype=torch.uint8, device=dev)
    acc = torch.empty(B, dtype=torch.int32, device=dev)
    nxt = torch.empty(B, dtype=torch.int32, device=dev)
    side = torch.cuda.Stream(dev)
    with torch.cuda.stream(side):
        for x in logits:
            dfl.accept_prefix(x, draft, workspace=ws, accepted=acc, next_token=nxt, want_argmax=False, stream=side)
    torch.cuda.synchronize()
    graphs = []
    for x in logits:
        gr = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gr, stream=side):
            dfl.accept_prefix(x, draft, workspace=ws, accepted=acc, next_token=nxt, want_argmax=False, stream=side)
        graphs.append(gr)
    for k in range(max(3, args.warmup)):
        graphs[k % n_sets].replay()
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream(dev)
    sampler = ClockSampler(dev.index if dev.index is not None else 0)
    if rank == 0:
        sampler.start()
    ev0 = torch.cuda.Event(enable_timing=True)
    ev1 = torch.cuda.Event(enable_timing=True)
    barrier()
    torch.cuda.synchronize()
    t_wall0 = time.time()
    ev0.record(stream)
    for k in range(args.steps):
        graphs[k % n_sets].replay()
    ev1.record(stream)
    torch.cuda.synchronize()
    t_wall1 = time.time()
    if rank == 0:
        sampler.stop()
    ms = max_over_ranks(ev0.elapsed_time(ev1) / args.steps)
    value = world * per / (ms * 1e-3) / 1e9
    # end to end: drafts in from pinned memory, accepted length and next token back, every step
    d_h = draft.cpu().pin_memory()
    a_h = torch.empty(B, dtype=torch.int32).pin_memory()
    n_h = torch.empty(B, dtype=torch.int32).pin_memory()
    n_e2e = min(args.steps, args.e2e_steps)
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for k in range(n_e2e):
        draft.copy_(d_h, non_blocking=True)
        dfl.accept_prefix(logits[k % n_sets], draft, workspace=ws, accepted=acc, next_token=nxt, want_argmax=False)
        a_h.copy_(acc, non_blocking=True)
        n_h.copy_(nxt, non_blocking=True)
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(e0.elapsed_time(e1) / n_e2e)
    if rank != 0:
        return
    peak, peak_kind = measured_peaks()
    cpu = None
    if world == 1 and not args.no_cpu_baseline:
        from oracle import accept as oracle_accept

        host = logits[0].view(torch.int16).cpu().numpy().view(np.uint16)
        dh = draft.cpu().numpy()
        t0 = time.perf_counter()
        n_rep = 0
        while time.perf_counter() - t0 < min(args.cpu_budget, 10.0):
            oracle_accept.accept_prefix(host, dh, "bf16")
            n_rep += 1
        t_step = (time.perf_counter() - t0) / n_rep
        cpu = {"value": per / t_step / 1e9, "unit": UNIT, "cores": 1, "kind": "oracle",
               "sample": f"{n_rep} full steps (numpy argmax over all {B * T} rows, then the prefix loop)"}
    line = {
        "metric": "logits_hbm_gbs", "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": ACCEPT_DESC, "global_batch": B * world, "block_len": T, "vocab": V,
                   "l2": f"inputs larger than L2: {n_sets} rotated logits sets x {per / 1e6:.1f} MB",
                   "timed_path": "one CUDA-graph replay of one dflash_accept_prefix call per step",
                   "parallelism": f"replicas x{world}"},
        "blocks_per_s": world * B / (ms * 1e-3),
        "e2e": {"value": world * per / (e2e_ms * 1e-3) / 1e9, "unit": UNIT,
                "h2d_bytes_per_step": d_h.numel() * 4, "d2h_bytes_per_step": 2 * B * 4, "ms_per_step": e2e_ms,
                "note": "public Python API; drafts in, accepted length and next token out, every step; "
                        "the logits are device-resident"},
        "gpu_launches": args.steps,
        "roofline": {"bound": "hbm", "achieved": value / world, "peak": peak, "unit": "GB/s",
                     "frac": value / world / peak, "traffic": traffic_from_profiles("accept_kernel")[0],
                     "peak_kind": peak_kind, "kernel": "accept_kernel",
                     "achieved_basis": "logits bytes per launch / event-timed device time per step"},
        "clocks": sampler.summary(t_wall0, t_wall1),
    }
    if cpu:
        line["cpu_baseline"] = cpu
    print(json.dumps(line), flush=True)


# ----------------------------------------------------------------------------- context K/V projection


PROJECT_CONFIG = "project_prefill"
PROJECT_DESC = ("draft-pass context K/V projection of an 8192-token context: hidden 5376 -> 4 KV heads x 512 "
                "for K and for V (bf16 weights [2048, 5376] each), written into a paged cache of page size 16 "
                "through a shuffled page table (synthetic hidden states and random-init weights)")
PROJECT_SHAPE = dict(L=8192, H=5376, Hkv=4, D=512, P=16)


def project_inputs(dev, n_sets, seed=4321):
    """n_sets disjoint (hidden, w_k, w_v) sets, unit-variance outputs; one slot mapping over a
    shuffled page table; the two caches."""
    sh = PROJECT_SHAPE
    L, H, N, P = sh["L"], sh["H"], sh["Hkv"] * sh["D"], sh["P"]
    g = torch.Generator(device=dev).manual_seed(seed)
    sets = []
    for _ in range(n_sets):
        hidden = torch.randn((L, H), generator=g, device=dev).to(torch.bfloat16)
        w_k = (torch.randn((N, H), generator=g, device=dev) / H ** 0.5).to(torch.bfloat16)
        w_v = (torch.randn((N, H), generator=g, device=dev) / H ** 0.5).to(torch.bfloat16)
        sets.append((hidden, w_k, w_v))
    num_pages = 2 * L // P
    rng = np.random.default_rng(seed)
    table = rng.permutation(num_pages)[: L // P]
    pos = np.arange(L)
    slots = torch.from_numpy((table[pos // P] * P + pos % P).astype(np.int32)).to(dev)
    k_cache = torch.zeros((num_pages, P, sh["Hkv"], sh["D"]), dtype=torch.bfloat16, device=dev)
    v_cache = torch.zeros_like(k_cache)
    return sets, slots, k_cache, v_cache


def project_flops():
    sh = PROJECT_SHAPE
    return 2.0 * sh["L"] * sh["H"] * 2 * sh["Hkv"] * sh["D"]


def project_oracle_rate(budget_s, rows=256, seed=99):
    """The oracle (float64 numpy matmul) on a bounded sample of token rows: (TFLOP/s, sample text)."""
    from oracle import project as oracle_project

    sh = PROJECT_SHAPE
    H, N = sh["H"], sh["Hkv"] * sh["D"]
    rng = np.random.default_rng(seed)
    h = rng.standard_normal((rows, H))
    wk = rng.standard_normal((N, H)) / H ** 0.5
    wv = rng.standard_normal((N, H)) / H ** 0.5
    t0 = time.perf_counter()
    n = 0
    while n == 0 or time.perf_counter() - t0 < budget_s:
        oracle_project.project_kv(h, wk, wv, sh["Hkv"], sh["D"])
        n += 1
    dt = (time.perf_counter() - t0) / n
    rate = 2.0 * rows * H * 2 * N / dt / 1e12
    return rate, f"{n} oracle calls on {rows} of the {sh['L']} token rows (float64 numpy matmul, BLAS threads)"


def project_reference_arm(args):
    """--impl reference --config project_prefill: the oracle on the host cores."""
    budget = max(1.0, min(args.ref_budget, 120.0)) / max(1, args.steps + args.warmup)
    rate, sample = project_oracle_rate(budget)
    ms = project_flops() / (rate * 1e12) * 1e3
    line = {"impl": "reference", "metric": "projection_tflops", "value": rate, "unit": "TFLOP/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": PROJECT_DESC},
            "cpu_baseline": {"value": rate, "unit": "TFLOP/s", "cores": os.cpu_count(), "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": rate, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def project_bench(args, dfl, dev, rank, world):
    sh = PROJECT_SHAPE
    per_set = (sh["L"] * sh["H"] + 2 * sh["Hkv"] * sh["D"] * sh["H"]) * 2
    n_sets = args.layers or max(2, math.ceil(4 * L2_BYTES / per_set))
    sets, slots, k_cache, v_cache = project_inputs(dev, n_sets)
    side = torch.cuda.Stream(dev)
    with torch.cuda.stream(side):
        for hidden, w_k, w_v in sets:
            dfl.project_kv(hidden, w_k, w_v, slots, k_cache, v_cache, stream=side)
    torch.cuda.synchronize()
    graphs = []
    for hidden, w_k, w_v in sets:
        gr = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gr, stream=side):
            dfl.project_kv(hidden, w_k, w_v, slots, k_cache, v_cache, stream=side)
        graphs.append(gr)
    for k in range(max(3, args.warmup)):
        graphs[k % n_sets].replay()
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream(dev)
    sampler = ClockSampler(dev.index if dev.index is not None else 0)
    if rank == 0:
        sampler.start()
    ev0 = torch.cuda.Event(enable_timing=True)
    ev1 = torch.cuda.Event(enable_timing=True)
    barrier()
    torch.cuda.synchronize()
    t_wall0 = time.time()
    ev0.record(stream)
    for k in range(args.steps):
        graphs[k % n_sets].replay()
    ev1.record(stream)
    torch.cuda.synchronize()
    t_wall1 = time.time()
    if rank == 0:
        sampler.stop()
    ms = max_over_ranks(ev0.elapsed_time(ev1) / args.steps)
    flops = project_flops()
    value = world * flops / (ms * 1e-3) / 1e12
    # end to end: the hidden states and slot mapping in from pinned memory, the error word back,
    # every step. The inputs are double-buffered: a copy stream loads step k+1's hidden states
    # while the kernel of step k runs.
    h_h = sets[0][0].cpu().pin_memory()
    s_h = slots.cpu().pin_memory()
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    err_h = torch.empty(1, dtype=torch.int32).pin_memory()
    hbuf = [torch.empty_like(sets[0][0]) for _ in range(2)]
    sbuf = [torch.empty_like(slots) for _ in range(2)]
    copied = [torch.cuda.Event() for _ in range(2)]
    used = [torch.cuda.Event() for _ in range(2)]
    copier = torch.cuda.Stream(dev)
    n_e2e = max(2, min(args.steps, 20))
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    copier.wait_event(e0)
    for k in range(n_e2e):
        j = k % 2
        with torch.cuda.stream(copier):
            if k >= 2:
                copier.wait_event(used[j])
            hbuf[j].copy_(h_h, non_blocking=True)
            sbuf[j].copy_(s_h, non_blocking=True)
            copied[j].record(copier)
        stream.wait_event(copied[j])
        _, w_k, w_v = sets[k % n_sets]
        dfl.project_kv(hbuf[j], w_k, w_v, sbuf[j], k_cache, v_cache, device_error=err)
        used[j].record(stream)
        err_h.copy_(err, non_blocking=True)
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(e0.elapsed_time(e1) / n_e2e)
    if int(err_h.item()) != 0:
        raise RuntimeError(f"device error word {int(err_h.item())} after the projection")
    if rank != 0:
        return
    peak, peak_kind = measured_tflops()
    traffic, tnote = traffic_from_profiles("project_kv_kernel")
    cpu = None
    if world == 1 and not args.no_cpu_baseline:
        rate, sample = project_oracle_rate(min(args.cpu_budget, 10.0))
        cpu = {"value": rate, "unit": "TFLOP/s", "cores": os.cpu_count(), "kind": "oracle", "sample": sample}
    line = {
        "metric": "projection_tflops", "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": PROJECT_DESC, "tokens": sh["L"], "hidden": sh["H"], "num_kv_heads": sh["Hkv"],
                   "head_dim": sh["D"], "page_size": sh["P"],
                   "l2": f"inputs larger than L2: {n_sets} rotated (hidden, w_k, w_v) sets x {per_set / 1e6:.1f} MB",
                   "timed_path": "one CUDA-graph replay of one dflash_project_kv call per step",
                   "parallelism": f"replicas x{world}"},
        "e2e": {"value": world * flops / (e2e_ms * 1e-3) / 1e12, "unit": "TFLOP/s",
                "h2d_bytes_per_step": h_h.numel() * 2 + s_h.numel() * 4, "d2h_bytes_per_step": 4,
                "ms_per_step": e2e_ms,
                "note": "public Python API; hidden states and slot mapping in from pinned host memory (double-"
                        "buffered on a copy stream) and the error word back, every step; the weights and the "
                        "paged cache stay resident"},
        "gpu_launches": args.steps,
        "roofline": {"bound": "tensor", "achieved": value / world, "peak": peak, "unit": "TFLOP/s",
                     "frac": value / world / peak, "traffic": traffic, "peak_kind": peak_kind,
                     "kernel": "project_kv_kernel",
                     "achieved_basis": "2*L*H*(2*Hkv*D) flops per launch / event-timed device time per step",
                     "traffic_note": tnote},
        "clocks": sampler.summary(t_wall0, t_wall1),
    }
    if cpu:
        line["cpu_baseline"] = cpu
    print(json.dumps(line), flush=True)


# ----------------------------------------------------------------------------- DFlash2 grouped convolution


CONV_CONFIG = "conv_block"
CONV_DESC = ("DFlash2 grouped dynamic depthwise convolution over drafted blocks: 32 requests x 16 positions "
             "(1 + 15 speculative tokens, the DFlash2 default), 5120 channels in 8 contiguous groups, 4 taps, bf16 "
             "activations with fp32 static and dynamic taps (synthetic; the pages state neither the width, the "
             "group count nor the tap count)")
CONV_SHAPE = dict(B=32, T=16, C=5120, taps=4, G=8)


def conv_inputs(dev, n_sets, seed=2468):
    sh = CONV_SHAPE
    g = torch.Generator(device=dev).manual_seed(seed)
    sets = []
    for _ in range(n_sets):
        x = torch.randn((sh["B"], sh["T"], sh["C"]), generator=g, device=dev).to(torch.bfloat16)
        delta = torch.randn((sh["B"], sh["T"], sh["taps"], sh["G"]), generator=g, device=dev) * 0.25
        sets.append((x, delta, torch.empty_like(x)))
    base = torch.randn((sh["taps"], sh["C"]), generator=g, device=dev) * 0.5
    return sets, base


def conv_bytes():
    sh = CONV_SHAPE
    return (2 * sh["B"] * sh["T"] * sh["C"] * 2 + sh["B"] * sh["T"] * sh["taps"] * sh["G"] * 4
            + sh["taps"] * sh["C"] * 4)


def conv_oracle_rate(budget_s):
    from oracle import grouped_conv as oc

    sh = CONV_SHAPE
    rng = np.random.default_rng(7)
    x = rng.standard_normal((sh["B"], sh["T"], sh["C"]))
    base = rng.standard_normal((sh["taps"], sh["C"]))
    delta = rng.standard_normal((sh["B"], sh["T"], sh["taps"], sh["G"]))
    t0 = time.perf_counter()
    n = 0
    while n == 0 or time.perf_counter() - t0 < budget_s:
        oc.grouped_conv(x, base, delta)
        n += 1
    dt = (time.perf_counter() - t0) / n
    return conv_bytes() / dt / 1e9, f"{n} full oracle calls (float64 numpy loop over positions and taps)"


def conv_reference_arm(args):
    budget = max(1.0, min(args.ref_budget, 120.0)) / max(1, args.steps + args.warmup)
    rate, sample = conv_oracle_rate(budget)
    ms = conv_bytes() / (rate * 1e9) * 1e3
    line = {"impl": "reference", "metric": "conv_hbm_gbs", "value": rate, "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": CONV_DESC},
            "cpu_baseline": {"value": rate, "unit": UNIT, "cores": 1, "kind": "oracle", "sample": sample},
            "e2e": {"value": rate, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def conv_bench(args, dfl, dev, rank, world):
    per = conv_bytes()
    n_sets = args.layers or max(2, math.ceil(4 * L2_BYTES / per))
    sets, base = conv_inputs(dev, n_sets)
    side = torch.cuda.Stream(dev)
    with torch.cuda.stream(side):
        for x, delta, out in sets:
            dfl.grouped_conv(x, base, delta, out=out, stream=side)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=side):
        for x, delta, out in sets:
            dfl.grouped_conv(x, base, delta, out=out, stream=side)
    for _ in range(max(3, args.warmup)):
        graph.replay()
    torch.cuda.synchronize()
    reps = max(1, math.ceil(args.steps / n_sets))
    steps = reps * n_sets
    stream = torch.cuda.current_stream(dev)
    sampler = ClockSampler(dev.index if dev.index is not None else 0)
    if rank == 0:
        sampler.start()
    ev0 = torch.cuda.Event(enable_timing=True)
    ev1 = torch.cuda.Event(enable_timing=True)
    barrier()
    torch.cuda.synchronize()
    t_wall0 = time.time()
    ev0.record(stream)
    for _ in range(reps):
        graph.replay()
    ev1.record(stream)
    torch.cuda.synchronize()
    t_wall1 = time.time()
    if rank == 0:
        sampler.stop()
    ms = max_over_ranks(ev0.elapsed_time(ev1) / steps)
    value = world * per / (ms * 1e-3) / 1e9
    # end to end: x and delta in from pinned memory, out back, every step
    x0, d0, o0 = sets[0]
    x_h = x0.cpu().pin_memory()
    d_h = d0.cpu().pin_memory()
    o_h = torch.empty_like(o0, device="cpu").pin_memory()
    n_e2e = max(1, min(steps, 200))
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(n_e2e):
        x0.copy_(x_h, non_blocking=True)
        d0.copy_(d_h, non_blocking=True)
        dfl.grouped_conv(x0, base, d0, out=o0)
        o_h.copy_(o0, non_blocking=True)
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(e0.elapsed_time(e1) / n_e2e)
    if rank != 0:
        return
    peak, peak_kind = measured_peaks()
    cpu = None
    if world == 1 and not args.no_cpu_baseline:
        rate, sample = conv_oracle_rate(min(args.cpu_budget, 10.0))
        cpu = {"value": rate, "unit": UNIT, "cores": 1, "kind": "oracle", "sample": sample}
    sh = CONV_SHAPE
    line = {
        "metric": "conv_hbm_gbs", "value": value, "unit": UNIT, "n_gpus": world, "steps": steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": CONV_DESC, "global_batch": sh["B"] * world, "block_len": sh["T"],
                   "channels": sh["C"], "taps": sh["taps"], "groups": sh["G"],
                   "l2": f"inputs larger than L2: {n_sets} rotated (x, delta, out) sets x {per / 1e6:.2f} MB",
                   "timed_path": f"CUDA-graph replays of {n_sets} dflash_grouped_conv calls, one per step",
                   "parallelism": f"replicas x{world}"},
        "e2e": {"value": world * per / (e2e_ms * 1e-3) / 1e9, "unit": UNIT,
                "h2d_bytes_per_step": x_h.numel() * 2 + d_h.numel() * 4, "d2h_bytes_per_step": o_h.numel() * 2,
                "ms_per_step": e2e_ms,
                "note": "public Python API; x and delta in from pinned host memory, out back, every step"},
        "gpu_launches": steps,
        "roofline": {"bound": "hbm", "achieved": value / world, "peak": peak, "unit": "GB/s",
                     "frac": value / world / peak, "traffic": traffic_from_profiles("grouped_conv_kernel")[0],
                     "peak_kind": peak_kind, "kernel": "grouped_conv_kernel",
                     "achieved_basis": "x read + out written + delta + base bytes per launch / event-timed time"},
        "clocks": sampler.summary(t_wall0, t_wall1),
    }
    if cpu:
        line["cpu_baseline"] = cpu
    print(json.dumps(line), flush=True)


# ----------------------------------------------------------------------------- DFlash2 candidate selector


SEL_CONFIG = "selector_walk"
SEL_DESC = ("DFlash2 candidate-selector walk: 32 requests x 15 draft slots x 8 candidates per slot, predecessor "
            "and successor codebooks of 151936 x 256 bf16, temperature 1 (inverse-CDF sampling, q returned) "
            "(synthetic; the pages state neither the codebook width, the vocabulary nor K)")
SEL_SHAPE = dict(R=32, S=15, K=8, V=151936, E=256, T=1.0)


def sel_bytes():
    sh = SEL_SHAPE
    R, S, K, E = sh["R"], sh["S"], sh["K"], sh["E"]
    rows = R * ((1 + K) + (S - 1) * (2 * K))  # predecessor + candidate codebook rows gathered per call
    return rows * E * 2 + R * S * (E * 4 + K * 8 + 4) + R * S * (K * 8 + 8)


def sel_inputs(dev, n_sets, seed=1357):
    sh = SEL_SHAPE
    R, S, K, V, E = sh["R"], sh["S"], sh["K"], sh["V"], sh["E"]
    g = torch.Generator(device=dev).manual_seed(seed)
    A = torch.randn((V, E), generator=g, device=dev).to(torch.bfloat16)
    B = torch.randn((V, E), generator=g, device=dev).to(torch.bfloat16)
    sets = []
    for _ in range(n_sets):
        proj = torch.randn((R, S, E), generator=g, device=dev) / E ** 0.5
        cand = torch.randint(0, V, (R, S, K), generator=g, device=dev, dtype=torch.int32)
        unary = torch.randn((R, S, K), generator=g, device=dev)
        anchor = torch.randint(0, V, (R,), generator=g, device=dev, dtype=torch.int32)
        u = torch.rand((R, S), generator=g, device=dev)
        sets.append((proj, cand, unary, anchor, u))
    return A, B, sets


def sel_oracle_rate(budget_s):
    from oracle import selector as osel

    sh = SEL_SHAPE
    R, S, K, E = sh["R"], sh["S"], sh["K"], sh["E"]
    V = 4096  # the host sample gathers from a smaller codebook; the walk's arithmetic is the same
    rng = np.random.default_rng(11)
    A = rng.standard_normal((V, E))
    B = rng.standard_normal((V, E))
    proj = rng.standard_normal((R, S, E))
    cand = rng.integers(0, V, (R, S, K))
    unary = rng.standard_normal((R, S, K))
    anchor = rng.integers(0, V, R)
    u = rng.random((R, S))
    t0 = time.perf_counter()
    n = 0
    while n == 0 or time.perf_counter() - t0 < budget_s:
        osel.walk(A, B, proj, cand, unary, anchor, temperature=sh["T"], u=u)
        n += 1
    dt = (time.perf_counter() - t0) / n
    return sel_bytes() / dt / 1e9, f"{n} full oracle walks (float64, a {V}-row codebook)"


def sel_reference_arm(args):
    budget = max(1.0, min(args.ref_budget, 120.0)) / max(1, args.steps + args.warmup)
    rate, sample = sel_oracle_rate(budget)
    ms = sel_bytes() / (rate * 1e9) * 1e3
    line = {"impl": "reference", "metric": "selector_gather_gbs", "value": rate, "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": SEL_DESC},
            "cpu_baseline": {"value": rate, "unit": UNIT, "cores": 1, "kind": "oracle", "sample": sample},
            "e2e": {"value": rate, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def sel_bench(args, dfl, dev, rank, world):
    sh = SEL_SHAPE
    R, S, K, E = sh["R"], sh["S"], sh["K"], sh["E"]
    per = sel_bytes()
    n_sets = args.layers or max(2, math.ceil(4 * L2_BYTES / per))
    A, B, sets = sel_inputs(dev, n_sets)
    ws = torch.zeros(dfl.selector_workspace_bytes(R, S, K), dtype=torch.uint8, device=dev)
    tokens = torch.empty((R, S), dtype=torch.int32, device=dev)
    chosen = torch.empty_like(tokens)
    scores = torch.empty((R, S, K), device=dev)
    q = torch.empty((R, S, K), device=dev)
    side = torch.cuda.Stream(dev)

    def call(st, stream):
        proj, cand, unary, anchor, u = st
        dfl.selector_walk(A, B, proj, cand, unary, anchor, temperature=sh["T"], uniforms=u, workspace=ws,
                          tokens=tokens, chosen=chosen, path_scores=scores, q=q, stream=stream)

    with torch.cuda.stream(side):
        for st in sets:
            call(st, side)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=side):
        for st in sets:
            call(st, side)
    for _ in range(max(3, args.warmup)):
        graph.replay()
    torch.cuda.synchronize()
    reps = max(1, math.ceil(args.steps / n_sets))
    steps = reps * n_sets
    stream = torch.cuda.current_stream(dev)
    sampler = ClockSampler(dev.index if dev.index is not None else 0)
    if rank == 0:
        sampler.start()
    ev0 = torch.cuda.Event(enable_timing=True)
    ev1 = torch.cuda.Event(enable_timing=True)
    barrier()
    torch.cuda.synchronize()
    t_wall0 = time.time()
    ev0.record(stream)
    for _ in range(reps):
        graph.replay()
    ev1.record(stream)
    torch.cuda.synchronize()
    t_wall1 = time.time()
    if rank == 0:
        sampler.stop()
    ms = max_over_ranks(ev0.elapsed_time(ev1) / steps)
    value = world * per / (ms * 1e-3) / 1e9
    # end to end: the step's inputs in from pinned memory, tokens and q back, every step
    proj, cand, unary, anchor, u = sets[0]
    host_in = [t.cpu().pin_memory() for t in (proj, cand, unary, anchor, u)]
    tok_h = torch.empty_like(tokens, device="cpu").pin_memory()
    q_h = torch.empty_like(q, device="cpu").pin_memory()
    n_e2e = max(1, min(steps, 200))
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(n_e2e):
        for d, h in zip((proj, cand, unary, anchor, u), host_in):
            d.copy_(h, non_blocking=True)
        dfl.selector_walk(A, B, proj, cand, unary, anchor, temperature=sh["T"], uniforms=u, workspace=ws,
                          tokens=tokens, chosen=chosen, path_scores=scores, q=q)
        tok_h.copy_(tokens, non_blocking=True)
        q_h.copy_(q, non_blocking=True)
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(e0.elapsed_time(e1) / n_e2e)
    if rank != 0:
        return
    peak, peak_kind = measured_peaks()
    cpu = None
    if world == 1 and not args.no_cpu_baseline:
        rate, sample = sel_oracle_rate(min(args.cpu_budget, 10.0))
        cpu = {"value": rate, "unit": UNIT, "cores": 1, "kind": "oracle", "sample": sample}
    line = {
        "metric": "selector_gather_gbs", "value": value, "unit": UNIT, "n_gpus": world, "steps": steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": SEL_DESC, "global_batch": R * world, "slots": S, "candidates": K,
                   "vocab": sh["V"], "dim": E,
                   "l2": f"inputs larger than L2: 2 x {sh['V'] * E * 2 / 1e6:.0f} MB codebooks, {n_sets} rotated "
                         f"candidate sets of random rows",
                   "timed_path": f"CUDA-graph replays of {n_sets} dflash_selector_walk calls, one per step",
                   "parallelism": f"replicas x{world}"},
        "e2e": {"value": world * per / (e2e_ms * 1e-3) / 1e9, "unit": UNIT,
                "h2d_bytes_per_step": sum(h.numel() * h.element_size() for h in host_in),
                "d2h_bytes_per_step": tok_h.numel() * 4 + q_h.numel() * 4, "ms_per_step": e2e_ms,
                "note": "public Python API; projections, candidates, unary, anchors and uniforms in from pinned "
                        "host memory, tokens and q back, every step; the codebooks stay resident"},
        "gpu_launches": steps,
        "roofline": {"bound": "hbm", "achieved": value / world, "peak": peak, "unit": "GB/s",
                     "frac": value / world / peak, "traffic": traffic_from_profiles("selector_kernel")[0],
                     "peak_kind": peak_kind, "kernel": "selector_kernel",
                     "achieved_basis": "gathered codebook rows + proj + candidates + outputs per launch / "
                                       "event-timed time"},
        "clocks": sampler.summary(t_wall0, t_wall1),
    }
    if cpu:
        line["cpu_baseline"] = cpu
    print(json.dumps(line), flush=True)


# ----------------------------------------------------------------------------- GPU arm


def capture_case(args, dfl, dev):
    """Two calls of the workload's own plan on one layer (the second is the one a profiler
    captures with -s 1 -c 1); checks the device error word and prints the plan."""
    import workloads

    case = workloads.make_case(args.capture, device=dev, layers=1, batch=args.capture_batch)
    splits = case.num_splits if args.splits < 0 else args.splits
    for _ in range(2):
        dfl.block_attn(case.q, case.k_cache, case.v_cache, case.page_table, case.seq_lens, case.block_len,
                       causal=case.causal, window=case.window, scale=case.scale, num_splits=splits,
                       kernel=args.kernel)
    torch.cuda.synchronize()
    err = dfl.read_error()
    dims = dfl.make_dims(case.q, case.k_cache, case.page_table, case.block_len)
    plan = dfl.plan_info(dims, case.block_len, case.window, splits, args.kernel)
    print(json.dumps({"capture": args.capture, "batch": case.batch, "kv_bytes": kv_bytes_per_step(case),
                      "plan": plan, "error_word": err}), flush=True)
    assert err == 0, "device-side check failed"


def traffic_from_profiles(kernel_name, workload=None):
    """DRAM bytes per launch from the committed ncu summary of this kernel on this workload (records
    keyed "kernel@workload", or by the kernel alone for single-workload kernels), if the kernel
    source is unchanged since the capture."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None, None
    try:
        recs = json.load(open(path))
        rec = recs.get(f"{kernel_name}@{workload}") if workload else None
        if rec is None:
            rec = recs.get(kernel_name)
    except (ValueError, OSError):
        return None, None
    if not rec:
        return None, None
    if rec.get("source_sha256") != kernel_source_sha(rec.get("sources", [])):
        return None, "kernel changed since the ncu capture"
    return rec.get("dram_bytes_per_launch"), rec.get("note")


def kernel_source_sha(files):
    h = hashlib.sha256()
    for f in files:
        p = os.path.join(ROOT, f)
        if not os.path.exists(p):
            return None
        h.update(open(p, "rb").read())
    return h.hexdigest()


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        try:
            d = json.load(open(path))
            return float(d["hbm_gbs"]), "measured"
        except (ValueError, KeyError, OSError):
            pass
    return 6800.0, "fallback"


def measured_tflops():
    """Dense bf16 tensor peak: the measured burst figure (a kernel timed in short loops), else fallback."""
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        try:
            return float(json.load(open(path))["bf16_tflops"]), "measured (burst)"
        except (ValueError, KeyError, OSError):
            pass
    return 1900.0, "fallback"


def main():
    args = parse_args()
    rank = env_int("RANK", 0)
    world = env_int("WORLD_SIZE", 1)
    local = env_int("LOCAL_RANK", 0)
    dist = None
    if world > 1:
        import torch.distributed as dist_mod

        dist = dist_mod
        if process_group_backend() == "nccl":
            torch.cuda.set_device(local)
            dist.init_process_group("nccl", device_id=torch.device("cuda", local))
        else:
            dist.init_process_group("gloo")
    if args.impl == "reference":
        if rank != 0:
            if dist:
                dist.destroy_process_group()
            return
        if args.config == ACCEPT_CONFIG:
            accept_reference_arm(args)
            if dist:
                dist.destroy_process_group()
            return
        if args.config == PROJECT_CONFIG:
            project_reference_arm(args)
            if dist:
                dist.destroy_process_group()
            return
        if args.config == CONV_CONFIG:
            conv_reference_arm(args)
            if dist:
                dist.destroy_process_group()
            return
        if args.config == SEL_CONFIG:
            sel_reference_arm(args)
            if dist:
                dist.destroy_process_group()
            return
        if args.config == WORKLOAD:
            group_reference_arm(args)
            if dist:
                dist.destroy_process_group()
            return
        import workloads

        case = workloads.make_case(args.config, device="cuda" if torch.cuda.is_available() else "cpu")
        reference_arm(args, case)
        if dist:
            dist.destroy_process_group()
        return

    import workloads
    import speculative_decoding_block_dflash_gb300 as dfl
    from speculative_decoding_block_dflash_gb300 import build as build_mod

    if rank == 0:
        build_mod.build()
    if dist:
        dist.barrier()
    dfl.load_library()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)

    if args.capture:
        capture_case(args, dfl, dev)
        if dist:
            dist.destroy_process_group()
        return
    if args.config == ACCEPT_CONFIG:
        accept_bench(args, dfl, dev, rank, world)
        if dist:
            dist.destroy_process_group()
        return
    if args.config == PROJECT_CONFIG:
        project_bench(args, dfl, dev, rank, world)
        if dist:
            dist.destroy_process_group()
        return
    if args.config == CONV_CONFIG:
        conv_bench(args, dfl, dev, rank, world)
        if dist:
            dist.destroy_process_group()
        return
    if args.config == SEL_CONFIG:
        sel_bench(args, dfl, dev, rank, world)
        if dist:
            dist.destroy_process_group()
        return

    headline = args.config == WORKLOAD
    st = attn_setup(args.config, args, dfl, dev, workloads)
    case, splits, layers = st["case"], st["splits"], st["layers"]
    kv = kv_bytes_per_step(case)

    for k in range(max(3, args.warmup)):
        st["graphs"][k % layers].replay()
    torch.cuda.synchronize()

    stream = torch.cuda.current_stream(dev)
    sampler = ClockSampler(dev.index if dev.index is not None else 0, period_ms=20)
    if rank == 0:
        sampler.start()
    ev0 = torch.cuda.Event(enable_timing=True)
    ev1 = torch.cuda.Event(enable_timing=True)
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    t_wall0 = time.time()
    ev0.record(stream)
    for k in range(args.steps):
        st["graphs"][k % layers].replay()
    ev1.record(stream)
    torch.cuda.synchronize()
    t_wall1 = time.time()
    if dist:
        dist.barrier()
    ms_total = ev0.elapsed_time(ev1)
    ms_total_t = torch.tensor([ms_total], device=dev, dtype=torch.float64)
    if dist:
        dist.all_reduce(ms_total_t, op=dist.ReduceOp.MAX)
    ms_per_step = float(ms_total_t.item()) / args.steps
    value = world * kv / (ms_per_step * 1e-3) / 1e9
    bq = world * case.batch / (ms_per_step * 1e-3)

    # A clock record that covers what it times: at least one second of the same replays, with
    # the SM clock and throttle reasons sampled inside it (the timed region above can be
    # shorter than the sampling period).
    n_win = max(args.steps, int(math.ceil(1000.0 / max(1e-3, ms_per_step))))
    w0 = torch.cuda.Event(enable_timing=True)
    w1 = torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    tw0 = time.time()
    w0.record(stream)
    for k in range(n_win):
        st["graphs"][k % layers].replay()
    w1.record(stream)
    torch.cuda.synchronize()
    tw1 = time.time()
    win_ms = w0.elapsed_time(w1) / n_win
    if rank == 0:
        sampler.stop()

    # eager ctypes path, one call per step, for reference (not the headline)
    n_eager = min(args.steps, 2000)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    e0.record(stream)
    for k in range(n_eager):
        st["call"](k % layers)
    e1.record(stream)
    torch.cuda.synchronize()
    eager_ms = e0.elapsed_time(e1) / n_eager

    e2e = e2e_measure(st, args, dfl, dev, stream, dist)
    assert dfl.read_error(st["ws"]) == 0, "device-side check failed"

    info = st["plan"]
    kernel_name = info["kernel_name"]
    peak, peak_kind = measured_peaks()
    traffic, traffic_note = traffic_from_profiles(kernel_name, args.config)
    achieved = kv / (ms_per_step * 1e-3) / 1e9
    gpu_launches = args.steps * info["launches"]
    del st
    torch.cuda.empty_cache()

    # the other attention workloads, each on its own graphs (parity cases elsewhere; reported here)
    others = {}
    if headline and not args.no_other_workloads:
        for name in OTHER_WORKLOADS:
            others[name] = other_workload(name, args, dfl, dev, workloads, peak)
            torch.cuda.empty_cache()

    if rank != 0:
        if dist:
            dist.destroy_process_group()
        return

    clocks = sampler.summary(t_wall0, t_wall1)
    win_clocks = sampler.summary(tw0, tw1)
    clocks["window"] = {"replays": n_win, "seconds": tw1 - tw0, "ms_per_step": win_ms,
                        "sm_mhz": win_clocks["sm_mhz"], "sm_max_mhz": win_clocks["sm_max_mhz"],
                        "reasons": win_clocks["reasons"], "samples": win_clocks["samples"]}
    if not clocks["samples"]:
        # the timed region fell between two samples: the window's clocks stand for it
        clocks["sm_mhz"], clocks["sm_max_mhz"] = win_clocks["sm_mhz"], win_clocks["sm_max_mhz"]
        clocks["reasons"] = win_clocks["reasons"]
        clocks["samples_note"] = "no sample fell inside the timed region; the clocks are the 1 s window's"
    cpu = None
    if world == 1 and not args.no_cpu_baseline:
        case_cpu = workloads.make_case(args.config, device=dev, layers=1)
        if headline:
            t_step, sample, threads = time_oracle_group_sample(case_cpu, args.cpu_budget)
            cpu = {"value": kv / t_step / 1e9, "unit": UNIT, "cores": threads, "kind": "oracle", "sample": sample}
        else:
            t_step, n_rep, threads = time_oracle_full(case_cpu, args.cpu_budget)
            cpu = {"value": kv / t_step / 1e9, "unit": UNIT, "cores": threads, "kind": "oracle",
                   "sample": f"{n_rep} full steps of layer 0 (all {case_cpu.q.shape[0] * case_cpu.q.shape[1]} "
                             f"rows, every visible key), median {t_step * 1e3:.1f} ms per step"}
        del case_cpu
        if headline:
            # the global-layer verify workload on one host core, in full
            gv = workloads.make_case("global_verify", device=dev, layers=1)
            t1, n1, _ = time_oracle_full(gv, 0.0, threads=1)
            cpu["global_verify_1core"] = {"value": kv_bytes_per_step(gv) / t1 / 1e9, "unit": UNIT, "cores": 1,
                                          "ms_per_step": t1 * 1e3,
                                          "sample": "one full step (all 288 rows, every key) on one thread"}
            del gv
    line = {
        "metric": METRIC,
        "value": value,
        "unit": UNIT,
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": ms_per_step,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16" if case.q.dtype == torch.bfloat16 else "f32",
        "data": "synthetic",
        "config": {"workload": WORKLOAD_DESC if headline else args.config,
                   "global_batch": case.batch * world, "block_len": case.block_len,
                   "seq_len": max(case.seq_lens_host()), "splits": splits, "kernel": kernel_name,
                   "l2": f"inputs larger than L2: {layers} rotated page sets x {kv / 1e6:.1f} MB K/V",
                   "timed_path": "one CUDA-graph replay of one dflash_block_attn call per step",
                   "parallelism": f"replicas x{world}"},
        "block_queries_per_s": bq,
        "query_rows_per_s": bq * case.block_len * case.num_q_heads,
        "eager_ms_per_step": eager_ms,
        "e2e": e2e,
        "gpu_launches": gpu_launches,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "traffic": traffic, "peak_kind": peak_kind,
                     "kernel": kernel_name,
                     "achieved_basis": "algorithmic K/V bytes per launch / event-timed device time per step",
                     "traffic_note": traffic_note},
        "clocks": clocks,
    }
    if others:
        line["workloads"] = others
    if cpu:
        line["cpu_baseline"] = cpu
    print(json.dumps(line), flush=True)
    if dist:
        dist.destroy_process_group()


def attn_setup(name, args, dfl, dev, workloads, steps_hint=None):
    """Inputs of a named attention workload with enough rotated page sets ("layers") to exceed
    4x L2 between two visits, its workspace, and one captured CUDA graph per layer."""
    probe = workloads.make_case(name, device=dev, layers=1)
    per_layer = kv_bytes_per_step(probe)
    layers = args.layers or max(2, math.ceil(4 * L2_BYTES / max(1, per_layer)))
    del probe
    torch.cuda.empty_cache()
    case = workloads.make_case(name, device=dev, layers=layers)
    splits_req = case.num_splits if args.splits < 0 else args.splits
    dims = dfl.make_dims(case.q, case.k_cache, case.page_table, case.block_len)
    splits = dfl.plan_splits(dims, case.block_len, case.window, splits_req, args.kernel)
    ws = torch.zeros(dfl.workspace_bytes(dims, case.block_len, splits), dtype=torch.uint8, device=dev)
    out = torch.empty_like(case.q)
    lse = torch.empty(case.q.shape[:2], dtype=torch.float32, device=dev)

    def call(layer, stream=None):
        dfl.block_attn(case.q, case.k_cache, case.v_cache, case.page_tables[layer], case.seq_lens,
                       case.block_len, causal=case.causal, window=case.window, scale=case.scale, out=out,
                       lse=lse, num_splits=splits_req, kernel=args.kernel, workspace=ws, stream=stream)

    # one CUDA graph per layer (captured on a side stream after an eager warm-up)
    side = torch.cuda.Stream(device=dev)
    with torch.cuda.stream(side):
        for l in range(layers):
            call(l)
    torch.cuda.synchronize()
    graphs = []
    for l in range(layers):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=side):
            call(l)
        graphs.append(g)
    torch.cuda.synchronize()
    assert dfl.read_error(ws) == 0, "device-side check failed during warm-up"
    plan = dfl.plan_info(dims, case.block_len, case.window, splits_req, args.kernel)
    return dict(case=case, graphs=graphs, call=call, layers=layers, splits=splits, splits_req=splits_req,
                ws=ws, out=out, lse=lse, plan=plan)


def e2e_measure(st, args, dfl, dev, stream, dist):
    """End to end through the public API with host buffers: H2D of q / page_table / seq_lens from
    pinned memory, the call, D2H of out and lse -- every step. Inputs and results are double-
    buffered on two copy streams (one per direction), as a serving loop would run it: step k+1's
    inputs load and step k-1's results return while step k's kernels run."""
    case, layers, out, lse, ws = st["case"], st["layers"], st["out"], st["lse"], st["ws"]
    q_h = case.q.cpu().pin_memory()
    pts_h = [pt.cpu().pin_memory() for pt in case.page_tables]
    sl_h = case.seq_lens.cpu().pin_memory()
    out_h = [torch.empty(out.shape, dtype=out.dtype).pin_memory() for _ in range(2)]
    lse_h = [torch.empty(lse.shape, dtype=lse.dtype).pin_memory() for _ in range(2)]
    q_d = [torch.empty_like(case.q) for _ in range(2)]
    pt_d = [torch.empty_like(case.page_tables[0]) for _ in range(2)]
    sl_d = [torch.empty_like(case.seq_lens) for _ in range(2)]
    o_d = [torch.empty_like(out) for _ in range(2)]
    l_d = [torch.empty_like(lse) for _ in range(2)]
    copied = [torch.cuda.Event() for _ in range(2)]   # inputs j on the device
    computed = [torch.cuda.Event() for _ in range(2)]  # the call on inputs j / results j done
    drained = [torch.cuda.Event() for _ in range(2)]   # results j back on the host
    h2d = torch.cuda.Stream(dev)
    d2h = torch.cuda.Stream(dev)
    n_e2e = max(3, min(args.e2e_steps, args.steps))

    def run(n, e_start):
        h2d.wait_event(e_start)
        for k in range(n):
            j = k % 2
            with torch.cuda.stream(h2d):
                if k >= 2:
                    h2d.wait_event(computed[j])  # the call of step k-2 has read inputs j
                q_d[j].copy_(q_h, non_blocking=True)
                pt_d[j].copy_(pts_h[k % layers], non_blocking=True)
                sl_d[j].copy_(sl_h, non_blocking=True)
                copied[j].record(h2d)
            stream.wait_event(copied[j])
            if k >= 2:
                stream.wait_event(drained[j])  # results j of step k-2 are back on the host
            dfl.block_attn(q_d[j], case.k_cache, case.v_cache, pt_d[j], sl_d[j], case.block_len,
                           causal=case.causal, window=case.window, scale=case.scale, out=o_d[j], lse=l_d[j],
                           num_splits=st["splits_req"], kernel=args.kernel, workspace=ws)
            computed[j].record(stream)
            with torch.cuda.stream(d2h):
                d2h.wait_event(computed[j])
                out_h[j].copy_(o_d[j], non_blocking=True)
                lse_h[j].copy_(l_d[j], non_blocking=True)
                drained[j].record(d2h)
        for j in range(2):
            stream.wait_event(drained[j])

    e_w = torch.cuda.Event()
    e_w.record(stream)
    run(3, e_w)
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    run(n_e2e, e0)
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = e0.elapsed_time(e1) / n_e2e
    e2e_ms_t = torch.tensor([e2e_ms], device=dev, dtype=torch.float64)
    if dist:
        dist.all_reduce(e2e_ms_t, op=dist.ReduceOp.MAX)
    e2e_ms = float(e2e_ms_t.item())
    world = dist.get_world_size() if dist else 1
    h2d_bytes = q_h.numel() * q_h.element_size() + pts_h[0].numel() * 4 + sl_h.numel() * 4
    d2h_bytes = out_h[0].numel() * out_h[0].element_size() + lse_h[0].numel() * 4
    return {"value": world * kv_bytes_per_step(case) / (e2e_ms * 1e-3) / 1e9, "unit": UNIT,
            "h2d_bytes_per_step": h2d_bytes, "d2h_bytes_per_step": d2h_bytes, "ms_per_step": e2e_ms,
            "note": "public Python API, pinned host q/page_table/seq_lens in, out/lse back, every step, "
                    "double-buffered on one copy stream per direction (step k+1's inputs load and step k-1's "
                    "results return while step k runs); the KV cache is device-resident state"}


def other_workload(name, args, dfl, dev, workloads, peak):
    """Event-timed graph replays of another attention workload (its own split plan), for the
    "workloads" key of the line: microseconds per call, K/V GB/s and the fraction of peak."""
    sub = argparse.Namespace(**vars(args))
    sub.splits = -1
    st = attn_setup(name, sub, dfl, dev, workloads)
    case, layers = st["case"], st["layers"]
    kv = kv_bytes_per_step(case)
    for k in range(10):
        st["graphs"][k % layers].replay()
    torch.cuda.synchronize()
    n = max(200, min(5000, int(200e-3 / 40e-6)))
    stream = torch.cuda.current_stream(dev)
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for k in range(n):
        st["graphs"][k % layers].replay()
    b.record(stream)
    torch.cuda.synchronize()
    ms = a.elapsed_time(b) / n
    assert dfl.read_error(st["ws"]) == 0, f"device-side check failed on {name}"
    gbs = kv / (ms * 1e-3) / 1e9
    rec = {"us_per_call": ms * 1e3, "kv_bytes": kv, "gbs": gbs, "frac": gbs / peak, "splits": st["splits"],
           "kernel": st["plan"]["kernel_name"], "launches_per_call": st["plan"]["launches"], "replays": n,
           "l2": f"{layers} rotated page sets"}
    del st
    return rec


if __name__ == "__main__":
    main()
