"""GPU parity: libdflash_attn (through its C ABI) against the fp64 oracle.

Bars: bf16 outputs |gpu - oracle| <= 1e-2 + 1e-2*|oracle| element-wise (lse
too); fp32 outputs <= 1e-5 absolute; page-table indexing bit-exact (a shuffled
page table gives the same bits as the identity table over the same logical
K/V). Small cases span several key tiles with ragged tails; the named
workloads run at full size (every output where the oracle finishes in
seconds, sampled rows otherwise) with the library's own split plan.
"""
import math

import numpy as np
import pytest
import torch

import oracle
import workloads
import speculative_decoding_block_dflash_gb300 as dfl
from speculative_decoding_block_dflash_gb300 import build as build_mod

pytestmark = pytest.mark.gpu

BF16_TOL = 1e-2
FP32_TOL = 1e-5


@pytest.fixture(scope="module", autouse=True)
def _built():
    build_mod.build()
    oracle.build()
    dfl.load_library()


def _tc_available(case, kernel="tc"):
    dims = dfl.make_dims(case.q, case.k_cache, case.page_table, case.block_len)
    try:
        dfl.plan_splits(dims, case.block_len, case.window, 0, kernel)
        return True
    except dfl.DflashError:
        return False


GUARD = 4096  # elements of canary before and after each output buffer (16-byte multiples)


def _canary(dtype):
    # a finite bit pattern no kernel writes by chance (bf16 ~3.3e38, fp32 ~3.3e38)
    return (torch.int16, 0x7F7A) if dtype == torch.bfloat16 else (torch.int32, 0x7F7A5A5A)


def guarded(shape, dtype):
    """A contiguous view of `shape` in the middle of a larger buffer whose guard regions hold a
    canary pattern; check_guards() then proves the call wrote nothing outside the view."""
    n = int(np.prod(shape))
    buf = torch.empty(n + 2 * GUARD, dtype=dtype, device="cuda")
    itype, pat = _canary(dtype)
    buf.view(itype).fill_(pat)
    return buf, buf[GUARD:GUARD + n].view(shape)


def check_guards(buf, what):
    itype, pat = _canary(buf.dtype)
    bits = buf.view(itype)
    assert (bits[:GUARD] == pat).all().item() and (bits[-GUARD:] == pat).all().item(), \
        f"{what}: a write landed outside the output buffer"


def run(case, kernel="auto", num_splits=None, page_table=None, **kw):
    obuf, out = guarded(tuple(case.q.shape), case.q.dtype)
    lbuf, lse = guarded(tuple(case.q.shape[:2]), torch.float32)
    dfl.block_attn(case.q, case.k_cache, case.v_cache,
                   case.page_table if page_table is None else page_table,
                   case.seq_lens, case.block_len, causal=case.causal, window=case.window,
                   scale=case.scale, kernel=kernel, out=out, lse=lse,
                   num_splits=case.num_splits if num_splits is None else num_splits, **kw)
    torch.cuda.synchronize()
    check_guards(obuf, f"{case.name} out")
    check_guards(lbuf, f"{case.name} lse")
    return out, lse


def check_close(gpu, ref, tol_abs, tol_rel, what):
    g = gpu.detach().float().cpu().numpy().astype(np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert g.shape == ref.shape, (g.shape, ref.shape)
    assert np.isfinite(g).all(), f"{what}: non-finite GPU values"
    err = np.abs(g - ref)
    bound = tol_abs + tol_rel * np.abs(ref)
    bad = err > bound
    assert not bad.any(), (f"{what}: {bad.sum()} of {bad.size} elements out of tolerance; "
                           f"max err {err.max():.3e} at {np.unravel_index(err.argmax(), err.shape)}")


def tols(case):
    return (FP32_TOL, 0.0) if case.q.dtype == torch.float32 else (BF16_TOL, BF16_TOL)


def check_full(case, out, lse):
    ref_o, ref_l = oracle.block_attn(case.q, case.k_cache, case.v_cache, case.page_table, case.seq_lens,
                                     case.block_len, causal=case.causal, window=case.window, scale=case.scale)
    ta, tr = tols(case)
    check_close(out, ref_o, ta, tr, f"{case.name} out")
    check_close(lse, ref_l, ta, tr, f"{case.name} lse")


def sample_rows(case, per_request=6, seed=0):
    rng = np.random.default_rng(seed)
    rows = []
    for b in range(case.batch):
        picks = {(0, 0), (case.num_q_heads - 1, case.block_len - 1)}
        while len(picks) < per_request:
            picks.add((int(rng.integers(case.num_q_heads)), int(rng.integers(case.block_len))))
        rows += [(b, h, i) for h, i in sorted(picks)]
    return np.array(rows, dtype=np.int32)


def group_rows(case, seed=0):
    """Every output row of one (request, KV head) group per request: all G query heads x all T
    block positions, which at T = 16 and GQA 8 spans both halves of the tensor-core CTA pair
    (or both row groups of the single-CTA kernel)."""
    G = case.num_q_heads // case.num_kv_heads
    rng = np.random.default_rng(seed)
    rows = []
    for b in range(case.batch):
        g = int(rng.integers(case.num_kv_heads))
        rows += [(b, g * G + hh, i) for hh in range(G) for i in range(case.block_len)]
    return np.array(rows, dtype=np.int32)


def check_rows(case, out, lse, rows, what):
    ref_o, ref_l = oracle.block_attn_rows(case.q, case.k_cache, case.v_cache, case.page_table,
                                          case.seq_lens, case.block_len, rows, causal=case.causal,
                                          window=case.window, scale=case.scale)
    idx = torch.tensor(rows[:, 0] * case.block_len + rows[:, 2], device=out.device, dtype=torch.long)
    hh = torch.tensor(rows[:, 1], device=out.device, dtype=torch.long)
    ta, tr = tols(case)
    check_close(out[idx, hh], ref_o, ta, tr, f"{case.name} {what} out")
    check_close(lse[idx, hh], ref_l, ta, tr, f"{case.name} {what} lse")


def check_sampled(case, out, lse, per_request=6):
    rows = sample_rows(case, per_request)
    ref_o, ref_l = oracle.block_attn_rows(case.q, case.k_cache, case.v_cache, case.page_table,
                                          case.seq_lens, case.block_len, rows, causal=case.causal,
                                          window=case.window, scale=case.scale)
    idx = torch.tensor(rows[:, 0] * case.block_len + rows[:, 2], device=out.device, dtype=torch.long)
    hh = torch.tensor(rows[:, 1], device=out.device, dtype=torch.long)
    ta, tr = tols(case)
    check_close(out[idx, hh], ref_o, ta, tr, f"{case.name} sampled out")
    check_close(lse[idx, hh], ref_l, ta, tr, f"{case.name} sampled lse")


KERNELS = ["simt", "tc", "tc_pair"]


def maybe_skip(case, kernel):
    if kernel.startswith("tc") and (case.q.dtype != torch.bfloat16 or not _tc_available(case, kernel)):
        pytest.skip("tensor-core kernel does not cover this case")


# ----------------------------------------------------------------------------- small cases


def test_tiny_fp32_matches_oracle():
    case = workloads.make_case("tiny", device="cuda")
    out, lse = run(case)
    check_full(case, out, lse)


@pytest.mark.parametrize("kernel", KERNELS)
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("window", [0, 64])
@pytest.mark.parametrize("splits", [1, 3, 0])
def test_ragged_small_bf16(kernel, causal, window, splits):
    case = workloads.make_custom("ragged", 3, 9, 8, 2, 128, [9, 300, 777], causal=causal, window=window,
                                 seed=11, device="cuda")
    maybe_skip(case, kernel)
    out, lse = run(case, kernel=kernel, num_splits=splits)
    check_full(case, out, lse)


@pytest.mark.parametrize("kernel", KERNELS)
@pytest.mark.parametrize("D", [64, 256, 512])
@pytest.mark.parametrize("T", [9, 16])
def test_gqa8_head_dims(kernel, D, T):
    case = workloads.make_custom("gqa8", 2, T, 16, 2, D, [1000, 2500], seed=12 + D + T, device="cuda")
    maybe_skip(case, kernel)
    out, lse = run(case, kernel=kernel)
    check_full(case, out, lse)


@pytest.mark.parametrize("kernel", KERNELS)
@pytest.mark.parametrize("page_size", [8, 32, 64, 128])
def test_page_sizes(kernel, page_size):
    case = workloads.make_custom("pages", 2, 9, 16, 2, 256, [900, 2100], page_size=page_size, causal=True,
                                 window=300, seed=23 + page_size, device="cuda")
    maybe_skip(case, kernel)
    out, lse = run(case, kernel=kernel, num_splits=3)
    check_full(case, out, lse)


@pytest.mark.parametrize("T", [1, 2, 33, 64])
def test_block_len_extremes_simt(T):
    case = workloads.make_custom("blk", 2, T, 4, 1, 64, [T, T + 200], causal=True, seed=13 + T, device="cuda")
    out, lse = run(case, kernel="simt")
    check_full(case, out, lse)


def test_fp32_ragged_tight():
    case = workloads.make_custom("fp32", 2, 9, 4, 2, 64, [100, 333], dtype=torch.float32, causal=True,
                                 window=50, seed=14, device="cuda")
    out, lse = run(case, num_splits=4)
    check_full(case, out, lse)


# ----------------------------------------------------------------------------- named workloads, full size


@pytest.mark.parametrize("kernel", KERNELS)
def test_global_verify_full(kernel):
    case = workloads.make_case("global_verify", device="cuda")
    maybe_skip(case, kernel)
    out, lse = run(case, kernel=kernel)
    check_full(case, out, lse)


@pytest.mark.parametrize("kernel", KERNELS)
@pytest.mark.parametrize("name", ["sliding", "sliding_causal"])
def test_sliding_full(kernel, name):
    case = workloads.make_case(name, device="cuda")
    maybe_skip(case, kernel)
    out, lse = run(case, kernel=kernel)
    check_full(case, out, lse)


@pytest.mark.parametrize("kernel", KERNELS)
@pytest.mark.parametrize("B", [1, 2, 4, 8])
def test_batch_sweep_sampled(kernel, B):
    case = workloads.make_case(f"batch_sweep_b{B}", device="cuda")
    maybe_skip(case, kernel)
    out, lse = run(case, kernel=kernel)
    check_sampled(case, out, lse)
    if B == 8:
        check_rows(case, out, lse, group_rows(case, seed=B), "whole groups")


@pytest.mark.parametrize("kernel", KERNELS)
def test_long_draft_split16_groups(kernel):
    case = workloads.make_case("long_draft", device="cuda")
    maybe_skip(case, kernel)
    assert case.num_splits == 16
    out, lse = run(case, kernel=kernel)
    check_sampled(case, out, lse, per_request=4)
    # one whole (request, KV head) group per request: 128 rows x 131072 keys each
    check_rows(case, out, lse, group_rows(case, seed=5), "whole groups")
    del case
    torch.cuda.empty_cache()


def test_cta_pair_agrees_with_the_single_cta_kernel():
    # 8 heads x 16 positions at head_dim 512: one CTA pair per KV head (AUTO's choice), or two
    # single-CTA row groups that both read the K/V
    case = workloads.make_custom("pair_vs_tc", 2, 16, 32, 4, 512, [3000, 9000], seed=41, device="cuda")
    dims = dfl.make_dims(case.q, case.k_cache, case.page_table, case.block_len)
    assert dfl.plan_info(dims, case.block_len, 0, 0, "auto")["kernel_name"] == "tc_pair_attn_kernel"
    plan = dfl.plan_info(dims, case.block_len, 0, 0, "tc_pair")
    assert plan["kernel_name"] == "tc_pair_attn_kernel" and not plan["balanced"]
    # a persistent grid of CTA pairs: one per unit, or one per cluster slot when there are more
    units = case.batch * case.num_kv_heads * plan["num_splits"]
    assert plan["ctas"] % 2 == 0 and 2 <= plan["ctas"] <= 2 * units
    out, lse = run(case, kernel="tc_pair", num_splits=0)
    check_full(case, out, lse)
    a, la = run(case, kernel="tc", num_splits=plan["num_splits"])
    torch.testing.assert_close(out.float(), a.float(), atol=1e-2, rtol=1e-2)
    torch.testing.assert_close(lse, la, atol=1e-3, rtol=1e-3)


@pytest.mark.parametrize("T,Hq,Hkv,D", [(16, 16, 2, 512), (11, 16, 2, 256), (32, 16, 4, 256), (2, 8, 1, 512)])
@pytest.mark.parametrize("causal,window", [(False, 0), (True, 0), (False, 700), (True, 300)])
def test_cta_pair_shapes(T, Hq, Hkv, D, causal, window):
    # odd and even blocks, GQA 4 and 8, both head dims, ragged key tails, every mask
    if window and window < T:
        pytest.skip("window shorter than the block")
    case = workloads.make_custom("pair", 2, T, Hq, Hkv, D, [T + 5, 1337], causal=causal, window=window,
                                 seed=43 + T + D, device="cuda")
    maybe_skip(case, "tc_pair")
    for splits in (1, 3):
        out, lse = run(case, kernel="tc_pair", num_splits=splits)
        check_full(case, out, lse)


@pytest.mark.parametrize("D,Hkv,causal,window", [(512, 4, False, 0), (256, 4, True, 0), (512, 4, False, 700)])
def test_cta_pair_many_units_per_pair(D, Hkv, causal, window):
    # more (request, KV head, chunk) units than the device holds CTA pairs, so each pair runs
    # several units back to back with its ring, barriers and TMEM carried over; ragged lengths
    # leave some chunks with no keys at all (units without tiles)
    lens = [40, 3000, 17, 9000, 300, 5000, 64, 1200]
    case = workloads.make_custom("pairmany", 8, 16, 32, Hkv, D, lens, causal=causal, window=window,
                                 seed=45 + D, device="cuda")
    maybe_skip(case, "tc_pair")
    dims = dfl.make_dims(case.q, case.k_cache, case.page_table, case.block_len)
    splits = 12
    plan = dfl.plan_info(dims, case.block_len, window, splits, "tc_pair")
    units = case.batch * Hkv * splits
    assert plan["ctas"] < 2 * units, plan  # pairs take more than one unit each
    out, lse = run(case, kernel="tc_pair", num_splits=splits)
    check_full(case, out, lse)
    # the same call again on the same grid (the barriers' phases start over per launch)
    out2, lse2 = run(case, kernel="tc_pair", num_splits=splits)
    assert torch.equal(out, out2) and torch.equal(lse, lse2)


def test_cta_pair_garbage_beyond_seq_len_does_not_leak():
    """The pair reads V of the last, partial page in both CTAs: NaN/Inf there must not leak."""
    case = workloads.make_custom("pairnan", 2, 16, 16, 2, 512, [461, 790], seed=44, device="cuda")
    ref_o, ref_l = oracle.block_attn(case.q, case.k_cache, case.v_cache, case.page_table, case.seq_lens, 16,
                                     scale=case.scale)
    for b, L in enumerate(case.seq_lens_host()):
        last = int(case.page_table[b, (L - 1) // 16])
        case.k_cache[last, L % 16:] = float("nan")
        case.v_cache[last, L % 16:] = float("inf")
    for splits in (1, 2):
        out, lse = run(case, kernel="tc_pair", num_splits=splits)
        check_close(out, ref_o, BF16_TOL, BF16_TOL, "nan-poisoned pair out")
        check_close(lse, ref_l, BF16_TOL, BF16_TOL, "nan-poisoned pair lse")


# ----------------------------------------------------------------------------- exactness / invariants


@pytest.mark.parametrize("kernel", KERNELS)
def test_page_table_permutation_is_bit_exact(kernel):
    """Same logical K/V under the identity and a shuffled page table: identical bits."""
    case = workloads.make_custom("perm", 2, 9, 16, 2, 256, [700, 1500], identity_pages=True, seed=15,
                                 device="cuda")
    maybe_skip(case, kernel)
    a, la = run(case, kernel=kernel, num_splits=3)
    pool = case.k_cache.shape[0]
    perm = torch.randperm(pool, generator=torch.Generator().manual_seed(1)).cuda()
    k2 = torch.empty_like(case.k_cache)
    v2 = torch.empty_like(case.v_cache)
    k2[perm] = case.k_cache
    v2[perm] = case.v_cache
    pt2 = perm[case.page_table.long()].to(torch.int32)
    out2, lse2 = dfl.block_attn(case.q, k2, v2, pt2, case.seq_lens, case.block_len, scale=case.scale,
                                kernel=kernel, num_splits=3)
    torch.cuda.synchronize()
    assert torch.equal(a.view(torch.int16), out2.view(torch.int16))
    assert torch.equal(la, lse2)


@pytest.mark.parametrize("kernel", KERNELS)
def test_garbage_beyond_seq_len_does_not_leak(kernel):
    """Slots past L_b in the last page hold NaN/Inf: the output must not see them."""
    case = workloads.make_custom("nan", 2, 9, 8, 2, 128, [205, 390], seed=16, device="cuda")
    maybe_skip(case, kernel)
    ref_o, ref_l = oracle.block_attn(case.q, case.k_cache, case.v_cache, case.page_table, case.seq_lens, 9,
                                     scale=case.scale)
    for b, L in enumerate(case.seq_lens_host()):
        last = int(case.page_table[b, (L - 1) // 16])
        case.k_cache[last, L % 16:] = float("nan")
        case.v_cache[last, L % 16:] = float("inf")
    out, lse = run(case, kernel=kernel, num_splits=2)
    check_close(out, ref_o, BF16_TOL, BF16_TOL, "nan-poisoned out")
    check_close(lse, ref_l, BF16_TOL, BF16_TOL, "nan-poisoned lse")


@pytest.mark.parametrize("kernel", KERNELS)
def test_noncausal_query_permutation(kernel):
    case = workloads.make_custom("qperm", 1, 9, 8, 1, 128, [600], seed=17, device="cuda")
    maybe_skip(case, kernel)
    a, la = run(case, kernel=kernel)
    perm = torch.randperm(9, generator=torch.Generator().manual_seed(2)).cuda()
    case.q = case.q[perm].contiguous()
    b, lb = run(case, kernel=kernel)
    torch.testing.assert_close(b.float(), a[perm].float(), atol=2e-2, rtol=2e-2)
    torch.testing.assert_close(lb, la[perm], atol=1e-3, rtol=1e-3)


@pytest.mark.parametrize("kernel", KERNELS)
def test_split_counts_agree(kernel):
    case = workloads.make_custom("splits", 2, 16, 16, 2, 512, [3000, 5000], seed=18, device="cuda")
    maybe_skip(case, kernel)
    ref, lref = run(case, kernel=kernel, num_splits=1)
    for s in (2, 16, 0):
        out, lse = run(case, kernel=kernel, num_splits=s)
        torch.testing.assert_close(out.float(), ref.float(), atol=1e-2, rtol=1e-2)
        torch.testing.assert_close(lse, lref, atol=1e-3, rtol=1e-3)


@pytest.mark.parametrize("causal,window", [(False, 0), (True, 0), (False, 2048)])
def test_length_balanced_plan(causal, window):
    # Very different lengths under the auto plan: the tensor-core kernel deals one wave of
    # chunk slots to the requests by key span and combines in-kernel.
    case = workloads.make_custom("balanced", 4, 9, 32, 4, 512, [64, 9000, 1500, 300], causal=causal,
                                 window=window, seed=31, device="cuda")
    maybe_skip(case, "tc")
    dims = dfl.make_dims(case.q, case.k_cache, case.page_table, case.block_len)
    slots = dfl.plan_splits(dims, case.block_len, case.window, 0, "tc")
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    assert case.batch <= slots <= sms // case.num_kv_heads  # one wave of 4-CTA slots
    out, lse = run(case, kernel="tc", num_splits=0)
    check_full(case, out, lse)
    # the same call with the uniform plan of as many chunks agrees
    uni, luni = run(case, kernel="tc", num_splits=slots)
    torch.testing.assert_close(out.float(), uni.float(), atol=1e-2, rtol=1e-2)
    torch.testing.assert_close(lse, luni, atol=1e-3, rtol=1e-3)


def test_window_covering_everything_equals_global():
    case = workloads.make_custom("wg", 2, 9, 8, 2, 128, [300, 500], seed=19, device="cuda")
    a, la = run(case)
    case.window = 10000
    b, lb = run(case)
    torch.testing.assert_close(b.float(), a.float(), atol=1e-2, rtol=1e-2)
    torch.testing.assert_close(lb, la, atol=1e-3, rtol=1e-3)


def test_split_combine_matches_oracle():
    g = torch.Generator(device="cuda").manual_seed(20)
    S, rows, D = 7, 50, 512
    po = torch.randn(S, rows, D, device="cuda", generator=g)
    pl = torch.randn(S, rows, device="cuda", generator=g) * 3
    pl[2] = -float("inf")
    pl[:, 5] = -float("inf")  # an all-empty row
    out, lse = dfl.split_combine(po, pl, out_dtype=torch.float32)
    torch.cuda.synchronize()
    ref_o, ref_l = oracle.split_combine(po.cpu().numpy(), pl.cpu().numpy())
    ok = np.isfinite(ref_l)
    check_close(out[torch.tensor(ok, device="cuda")], ref_o[ok], FP32_TOL, FP32_TOL, "combine out")
    check_close(lse[torch.tensor(ok, device="cuda")], ref_l[ok], FP32_TOL, FP32_TOL, "combine lse")
    assert torch.isneginf(lse[5]).item() and (out[5] == 0).all().item()
    out_b, _ = dfl.split_combine(po, pl, out_dtype=torch.bfloat16)
    torch.cuda.synchronize()
    check_close(out_b[torch.tensor(ok, device="cuda")], ref_o[ok], BF16_TOL, BF16_TOL, "combine bf16 out")


# ----------------------------------------------------------------------------- device checks


def test_bad_page_id_is_reported_not_dereferenced():
    case = workloads.make_custom("badpage", 1, 9, 4, 1, 64, [200], seed=21, device="cuda")
    ws = torch.zeros(1 << 20, dtype=torch.uint8, device="cuda")
    pt = case.page_table.clone()
    pt[0, 3] = case.k_cache.shape[0] + 1000
    pt[0, 5] = -7
    dfl.block_attn(case.q, case.k_cache, case.v_cache, pt, case.seq_lens, 9, kernel="simt", workspace=ws)
    assert dfl.read_error(ws) & dfl.DEVERR_PAGE_ID
    assert dfl.read_error(ws) == 0  # cleared
    dfl.block_attn(case.q, case.k_cache, case.v_cache, case.page_table, case.seq_lens, 9, workspace=ws)
    assert dfl.read_error(ws) == 0


def test_bad_seq_len_is_reported():
    case = workloads.make_custom("badlen", 2, 9, 4, 1, 64, [200, 300], seed=22, device="cuda")
    ws = torch.zeros(1 << 20, dtype=torch.uint8, device="cuda")
    sl = case.seq_lens.clone()
    sl[1] = 5  # shorter than the block
    out, _ = dfl.block_attn(case.q, case.k_cache, case.v_cache, case.page_table, sl, 9, workspace=ws)
    assert dfl.read_error(ws) & dfl.DEVERR_SEQ_LEN
    assert (out[9:] == 0).all().item()
    sl[1] = 10 ** 6  # beyond max_pages * page_size
    dfl.block_attn(case.q, case.k_cache, case.v_cache, case.page_table, sl, 9, workspace=ws)
    assert dfl.read_error(ws) & dfl.DEVERR_SEQ_LEN


# ----------------------------------------------------------------------------- CUDA graphs


def test_cuda_graph_capture_and_replay():
    case = workloads.make_case("global_verify", device="cuda")
    ref, lref = run(case)
    dims = dfl.make_dims(case.q, case.k_cache, case.page_table, case.block_len)
    splits = dfl.plan_splits(dims, case.block_len, 0, 0)
    ws = torch.zeros(dfl.workspace_bytes(dims, case.block_len, splits), dtype=torch.uint8, device="cuda")
    out = torch.empty_like(case.q)
    lse = torch.empty(case.q.shape[:2], dtype=torch.float32, device="cuda")
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        dfl.block_attn(case.q, case.k_cache, case.v_cache, case.page_table, case.seq_lens, 9, out=out, lse=lse,
                       workspace=ws, num_splits=splits)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        dfl.block_attn(case.q, case.k_cache, case.v_cache, case.page_table, case.seq_lens, 9, out=out, lse=lse,
                       workspace=ws, num_splits=splits)
    out.zero_()
    g.replay()
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(out.view(torch.int16), ref.view(torch.int16))
    assert torch.equal(lse, lref)


def _plan_dims(B, T, Hq, Hkv, D, P, max_pages):
    d = dfl.Dims()
    d.batch, d.num_q_heads, d.num_kv_heads, d.head_dim = B, Hq, Hkv, D
    d.page_size, d.num_pages, d.max_pages, d.max_seq_len = P, B * max_pages, max_pages, 0
    d.dtype = dfl.BF16
    d.kv_stride_head, d.kv_stride_slot, d.kv_stride_page = D, Hkv * D, P * Hkv * D
    return d


def test_auto_plan_spreads_long_spans_over_waves():
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    # 8 requests of up to 131072 keys, blocks of 16 (two row groups per KV head): one wave of
    # balanced slots would stream ~55k keys each, so the plan is uniform chunks of ~7k keys
    long = _plan_dims(8, 16, 32, 4, 512, 16, 131072 // 16)
    assert dfl.plan_splits(long, 16, 0, 0, "tc") == -(-131072 // 7168)
    # up to 32768 keys over 8 requests keeps the one-wave length-balanced plan
    sweep = _plan_dims(8, 9, 32, 4, 512, 16, 32768 // 16)
    assert dfl.plan_splits(sweep, 9, 0, 0, "tc") == sms // 4
    # one request of 8192 keys: one wave (38 chunks on 152 SMs), each chunk rounded up to whole
    # 128-key tiles (256 keys), which leaves 32 chunks
    one = _plan_dims(1, 9, 32, 4, 512, 16, 8192 // 16)
    chunk = -(-(-(-8192 // (sms // 4))) // 128) * 128
    assert dfl.plan_splits(one, 9, 0, 0, "tc") == -(-8192 // chunk)
