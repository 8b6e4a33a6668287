"""dflash_block_attn_noalloc: the entry point for callers that cannot allocate.

Code that runs inside a custom allocator's own hooks, or in a runtime that
owns all device memory and forbids cudaMalloc, cannot hand dflash_block_attn
the workspace its split-KV partials need. The no-alloc entry point keeps that
scratch in a fixed array inside the library. These checks call
it through the C ABI and compare it with dflash_block_attn (same tolerance as
the parity tests: 1e-2 absolute + 1e-2 relative for bf16, 1e-5 for fp32) on two
calls in a row, so stale scratch contents from the first call cannot leak into
the second. This file is collected last on purpose.
"""
import ctypes

import pytest
import torch

import workloads
import speculative_decoding_block_dflash_gb300 as dfl
from speculative_decoding_block_dflash_gb300 import _binding as B
from speculative_decoding_block_dflash_gb300 import build as build_mod

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    build_mod.build()
    dfl.load_library()


def _reference(case, splits, kernel):
    ws = torch.zeros(64 << 20, dtype=torch.uint8, device="cuda")
    out, lse = dfl.block_attn(case.q, case.k_cache, case.v_cache, case.page_table, case.seq_lens, case.block_len,
                              causal=case.causal, window=case.window, scale=case.scale, num_splits=splits,
                              kernel=kernel, workspace=ws)
    torch.cuda.synchronize()
    return out, lse


def _noalloc(case, splits, kernel):
    out = torch.full_like(case.q, float("nan"))
    lse = torch.full(case.q.shape[:2], float("nan"), dtype=torch.float32, device="cuda")
    dfl.block_attn_noalloc(case.q, case.k_cache, case.v_cache, case.page_table, case.seq_lens, case.block_len,
                           causal=case.causal, window=case.window, scale=case.scale, out=out, lse=lse,
                           num_splits=splits, kernel=kernel)
    torch.cuda.synchronize()
    return out, lse


def _close(a, b, tol):
    torch.testing.assert_close(a.float(), b.float(), atol=tol, rtol=tol)


@pytest.mark.parametrize("kernel,dtype,tol", [("auto", torch.bfloat16, 1e-2), ("simt", torch.float32, 1e-5)])
def test_noalloc_matches_workspace_entry_point_twice(kernel, dtype, tol):
    # two different problems back to back through the same scratch
    first = workloads.make_custom("noalloc_a", 2, 9, 16, 2, 512 if dtype == torch.bfloat16 else 128,
                                  [3000, 5000], dtype=dtype, seed=71, device="cuda")
    second = workloads.make_custom("noalloc_b", 3, 9, 16, 2, 512 if dtype == torch.bfloat16 else 128,
                                   [700, 2500, 1300], dtype=dtype, causal=True, window=900, seed=72,
                                   device="cuda")
    for case, splits in ((first, 6), (second, 4)):
        ref_o, ref_l = _reference(case, splits, kernel)
        out, lse = _noalloc(case, splits, kernel)
        assert torch.isfinite(out.float()).all() and torch.isfinite(lse).all()
        _close(out, ref_o, tol)
        _close(lse, ref_l, tol)


def test_noalloc_unsplit_and_auto_plan():
    case = workloads.make_case("global_verify", device="cuda")
    for splits in (1, 0):
        ref_o, ref_l = _reference(case, splits, "auto")
        out, lse = _noalloc(case, splits, "auto")
        _close(out, ref_o, 1e-2)
        _close(lse, ref_l, 1e-2)


def test_noalloc_length_balanced_auto_plan():
    # B > 1 with the auto plan takes the length-balanced layout, which fits the scratch
    case = workloads.make_custom("noalloc_bal", 4, 9, 32, 4, 512, [64, 9000, 1500, 300], seed=74,
                                 device="cuda")
    ref_o, ref_l = _reference(case, 0, "auto")
    out, lse = _noalloc(case, 0, "auto")
    _close(out, ref_o, 1e-2)
    _close(lse, ref_l, 1e-2)


def test_noalloc_rejects_plans_beyond_its_scratch():
    lib = dfl.load_library()
    case = workloads.make_custom("noalloc_big", 8, 16, 32, 4, 512, [4096] * 8, seed=73, device="cuda")
    dims = B.make_dims(case.q, case.k_cache, case.page_table, case.block_len)
    need = dfl.workspace_bytes(dims, case.block_len, 32)
    assert need > 32 * 1024 * 1024
    out = torch.empty_like(case.q)
    st = lib.dflash_block_attn_noalloc(case.q.data_ptr(), case.k_cache.data_ptr(), case.v_cache.data_ptr(),
                                       case.page_table.data_ptr(), case.seq_lens.data_ptr(), ctypes.byref(dims),
                                       case.block_len, 0, 0, case.scale, out.data_ptr(), None, 32, 0, None)
    assert st == B.ERR_WORKSPACE
    assert "scratch" in lib.dflash_last_error_message().decode()


def test_noalloc_falls_back_when_the_auto_plan_does_not_fit():
    # 8 requests of 40000 keys in blocks of 16: the auto plan is 6 uniform chunks of ~7k keys,
    # whose fp32 partials (~50 MB) exceed the 32 MiB scratch; the no-alloc call falls back to a
    # plan that fits (for the CTA-pair kernel: the most uniform chunks that fit) and agrees
    case = workloads.make_custom("noalloc_long", 8, 16, 32, 4, 512, [40000] * 8, seed=75, device="cuda")
    dims = dfl.make_dims(case.q, case.k_cache, case.page_table, case.block_len)
    splits = dfl.plan_splits(dims, case.block_len, 0, 0, "auto")
    assert splits == -(-dims.max_pages * dims.page_size // 7168)
    assert dfl.workspace_bytes(dims, case.block_len, splits) > 32 * 1024 * 1024
    ref_o, ref_l = _reference(case, 0, "auto")
    out, lse = _noalloc(case, 0, "auto")
    _close(out, ref_o, 1e-2)
    _close(lse, ref_l, 1e-2)


def test_noalloc_bad_page_id_is_contained():
    # Device-side check bits land in the scratch's error word, which this entry point does not
    # report; what it guarantees is that the bad id is never dereferenced (its keys read as
    # zero, as in dflash_block_attn) and that the other requests are unaffected.
    case = workloads.make_custom("noalloc_badpage", 2, 9, 16, 2, 512, [900, 1400], seed=76, device="cuda")
    ref_o, ref_l = _reference(case, 3, "auto")
    pt = case.page_table.clone()
    pt[1, 10] = case.k_cache.shape[0] + 4096
    bad = workloads.Case(**{**case.__dict__, "page_table": pt})
    bad_ref_o, bad_ref_l = _reference(bad, 3, "auto")
    for _ in range(2):
        out, lse = _noalloc(bad, 3, "auto")
        assert torch.isfinite(out.float()).all() and torch.isfinite(lse).all()
        _close(out, bad_ref_o, 1e-2)  # the workspace entry point treats the page the same way
        _close(lse, bad_ref_l, 1e-2)
        _close(out[:9], ref_o[:9], 1e-2)  # request 0 does not see request 1's bad entry
        _close(lse[:9], ref_l[:9], 1e-2)
    # and a call with a good table right after is correct again
    out, lse = _noalloc(case, 3, "auto")
    _close(out, ref_o, 1e-2)
    _close(lse, ref_l, 1e-2)
