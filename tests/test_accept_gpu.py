"""GPU parity for dflash_accept_prefix (through its C ABI) against oracle/accept.py.

Every output is an integer, so the bar is bit-exact. The argmax over the vocabulary
decides in the logits' own precision on both sides: bf16 is widened exactly. Drafts are
built from the oracle's target tokens with one corrupted position per request, so that
the accepted lengths cover 0..K.
"""
import numpy as np
import pytest
import torch

import speculative_decoding_block_dflash_gb300 as dfl
from oracle import accept as oracle_accept
from speculative_decoding_block_dflash_gb300 import build as build_mod

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    build_mod.build()
    dfl.load_library()


def _host(logits):
    if logits.dtype == torch.bfloat16:
        return logits.view(torch.int16).cpu().numpy().view(np.uint16), "bf16"
    return logits.cpu().numpy(), "f32"


def _drafts(logits, seed):
    """Drafts equal to the target tokens except at one random position per request
    (position K, past the block, keeps them all)."""
    host, dt = _host(logits)
    t = oracle_accept.target_argmax(host, dt)
    B, T = t.shape
    rng = np.random.default_rng(seed)
    d = t[:, : T - 1].copy()
    V = logits.shape[-1]
    for b in range(B):
        k = rng.integers(0, T)  # 0..K
        if k < T - 1:
            d[b, k] = (d[b, k] + 1 + rng.integers(0, V - 1)) % V
    return torch.from_numpy(d.astype(np.int32)).to(logits.device)


def _check(logits, draft):
    acc, nxt, targ = dfl.accept_prefix(logits, draft)
    torch.cuda.synchronize()
    host, dt = _host(logits)
    e_acc, e_nxt, e_t = oracle_accept.accept_prefix(host, draft.cpu().numpy(), dt)
    np.testing.assert_array_equal(targ.cpu().numpy(), e_t)
    np.testing.assert_array_equal(acc.cpu().numpy(), e_acc)
    np.testing.assert_array_equal(nxt.cpu().numpy(), e_nxt)
    return e_acc


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("B,T", [(1, 1), (1, 2), (3, 9), (8, 16)])
@pytest.mark.parametrize("V", [1000, 4097, 32000])
def test_matches_oracle(dtype, B, T, V):
    g = torch.Generator(device="cuda").manual_seed(B * 1000 + T * 10 + V)
    logits = (torch.randn((B, T, V), generator=g, device="cuda") * 3).to(dtype)
    _check(logits, _drafts(logits, seed=V + T))


def test_full_vocab_batch8_block9_and_every_accept_length():
    # the verify shape of a batch of 8 blocks of 1 + 8 tokens over a 262144-entry vocabulary
    g = torch.Generator(device="cuda").manual_seed(5)
    logits = torch.randn((8, 9, 262144), generator=g, device="cuda").to(torch.bfloat16)
    host, dt = _host(logits)
    t = oracle_accept.target_argmax(host, dt)
    d = t[:, :8].copy()
    for b in range(8):  # request b accepts exactly b drafts
        d[b, b] = (d[b, b] + 17) % 262144
    draft = torch.from_numpy(d.astype(np.int32)).cuda()
    acc = _check(logits, draft)
    assert list(acc) == list(range(8))


def test_ties_across_slices_take_the_smallest_index():
    V = 200000
    logits = torch.full((2, 3, V), -1.0, device="cuda", dtype=torch.bfloat16)
    logits[0, 0, [150000, 7, 99999]] = 4.0   # the winner lies in the first slice
    logits[1, 2, [V - 1, 123456]] = 2.5
    logits[1, 0, 0] = 9.0
    draft = torch.tensor([[7, 0], [0, 0]], dtype=torch.int32, device="cuda")
    _check(logits, draft)


def test_negative_logits_padded_rows_and_reuse():
    V, stride = 5000, 5008
    g = torch.Generator(device="cuda").manual_seed(9)
    base = -torch.rand((4, 5, stride), generator=g, device="cuda") * 100 - 1  # all negative
    logits = base[:, :, :V]  # rows of stride 5008 elements
    assert logits.stride(1) == stride
    draft = _drafts(logits.contiguous(), seed=3)
    a1 = _check(logits, draft)
    a2 = _check(logits, draft)  # the same workspace, reset by the first call
    assert list(a1) == list(a2)


def test_cuda_graph_replay():
    g = torch.Generator(device="cuda").manual_seed(11)
    logits = torch.randn((4, 9, 50000), generator=g, device="cuda").to(torch.bfloat16)
    draft = _drafts(logits, seed=4)
    acc = torch.empty(4, dtype=torch.int32, device="cuda")
    nxt = torch.empty(4, dtype=torch.int32, device="cuda")
    ws = torch.zeros(dfl.accept_workspace_bytes(4, 9), dtype=torch.uint8, device="cuda")
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        dfl.accept_prefix(logits, draft, workspace=ws, accepted=acc, next_token=nxt, want_argmax=False)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        dfl.accept_prefix(logits, draft, workspace=ws, accepted=acc, next_token=nxt, want_argmax=False)
    acc.fill_(-1)
    nxt.fill_(-1)
    graph.replay()
    graph.replay()
    torch.cuda.synchronize()
    host, dt = _host(logits)
    e_acc, e_nxt, _ = oracle_accept.accept_prefix(host, draft.cpu().numpy(), dt)
    np.testing.assert_array_equal(acc.cpu().numpy(), e_acc)
    np.testing.assert_array_equal(nxt.cpu().numpy(), e_nxt)


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_rows_off_16_byte_boundaries(dtype):
    # rows starting 1 element past a boundary, of an odd stride: scalar head, vector body, tail
    V, stride = 7001, 7003
    g = torch.Generator(device="cuda").manual_seed(13)
    base = torch.randn((3, 4, stride), generator=g, device="cuda").to(dtype)
    logits = base[:, :, 1:V + 1]
    assert logits.data_ptr() % 16 != 0
    _check(logits, _drafts(logits.contiguous(), seed=6))
