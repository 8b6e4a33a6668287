"""The tensor-core kernel's bounded waits: a wait that runs out reports
DFLASH_DEVERR_TIMEOUT, the call returns, and the workspace is fit for the next
call.

The in-kernel split combine (the flash-decoding style LSE merge of the split
chunks, prhub report on vLLM PR #52816 "DFlash2", review highlights: its
split-KV combine faulted in the FlashAttention backend) waits for every chunk
of its (request, row group) on a counter in the workspace. Here that counter
is preset on the host to a value that never reaches the split count, so every
CTA's arrival wait runs out; the wait limit is set to 1 ms through
dflash_opts.wait_limit_us so the call ends at once. No GPU fault, trap or hang
is involved: the kernel gives up on its own and returns.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads
import speculative_decoding_block_dflash_gb300 as dfl
from speculative_decoding_block_dflash_gb300 import _binding as B
from speculative_decoding_block_dflash_gb300 import build as build_mod

pytestmark = pytest.mark.gpu

COUNTER_OFF, COUNTER_BYTES = 256, 8192


@pytest.fixture(scope="module", autouse=True)
def _built():
    build_mod.build()
    oracle.build()
    dfl.load_library()


def _call(case, ws, wait_limit_us=0):
    out, lse = dfl.block_attn(case.q, case.k_cache, case.v_cache, case.page_table, case.seq_lens, case.block_len,
                              scale=case.scale, num_splits=0, kernel="tc", workspace=ws,
                              wait_limit_us=wait_limit_us)
    torch.cuda.synchronize()
    return out, lse


def test_combine_wait_runs_out_then_the_workspace_recovers():
    # global_verify's auto plan fills one wave of 152 CTAs, so the split chunks combine in
    # the kernel (cooperative launch): 4 (request, row group) counter pairs are used
    case = workloads.make_case("global_verify", device="cuda")
    dims = dfl.make_dims(case.q, case.k_cache, case.page_table, case.block_len)
    splits = dfl.plan_splits(dims, case.block_len, 0, 0, "tc")
    assert splits > 1
    ws = torch.zeros(dfl.workspace_bytes(dims, case.block_len, splits), dtype=torch.uint8, device="cuda")
    ctr = ws[COUNTER_OFF:COUNTER_OFF + COUNTER_BYTES].view(torch.int32)
    ctr[0::2] = -1_000_000  # arrivals that can never reach the split count
    groups = case.batch * case.num_kv_heads  # one row group per KV head at GQA 8 x T 9

    _call(case, ws, wait_limit_us=1000)
    c = ctr.cpu().numpy()
    # every CTA of a used group gave up, still counted itself, and the last one reset the pair
    assert (c[:2 * groups] == 0).all(), c[:2 * groups]
    assert (c[2 * groups::2] == -1_000_000).all()  # groups the call did not use are untouched
    err = dfl.read_error(ws)
    assert err & B.DEVERR_TIMEOUT, err
    # a reported timeout also clears the whole counter block
    assert (ctr.cpu().numpy() == 0).all()

    # the same workspace now gives the oracle's result, with the default limit and with 1 ms
    ref_o, ref_l = oracle.block_attn(case.q, case.k_cache, case.v_cache, case.page_table, case.seq_lens,
                                     case.block_len, scale=case.scale)
    for limit in (0, 1000):
        out, lse = _call(case, ws, wait_limit_us=limit)
        assert dfl.read_error(ws) == 0
        g = out.float().cpu().numpy()
        assert np.all(np.abs(g - ref_o) <= 1e-2 + 1e-2 * np.abs(ref_o))
        gl = lse.cpu().numpy()
        assert np.all(np.abs(gl - ref_l) <= 1e-2 + 1e-2 * np.abs(ref_l))
        assert (ctr.cpu().numpy() == 0).all()
