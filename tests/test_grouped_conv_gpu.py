"""GPU parity for dflash_grouped_conv (through its C ABI) against oracle/grouped_conv.py.

The kernel sums at most 64 fp32 products per output. The oracle sums the same widened
inputs in float64. The bars are 1e-2 absolute + 1e-2 relative for bf16 outputs (one bf16
rounding is at most 2^-9 relative) and 1e-5 absolute + 1e-5 relative for fp32 outputs.
"""
import numpy as np
import pytest
import torch

import speculative_decoding_block_dflash_gb300 as dfl
from oracle import grouped_conv as oc
from speculative_decoding_block_dflash_gb300 import build as build_mod

pytestmark = pytest.mark.gpu

TOL = {torch.bfloat16: (1e-2, 1e-2), torch.float32: (1e-5, 1e-5)}


@pytest.fixture(scope="module", autouse=True)
def _built():
    build_mod.build()
    dfl.load_library()


def _inputs(B, T, C, taps, G, dtype, seed):
    g = torch.Generator(device="cuda").manual_seed(seed)
    x = torch.randn((B, T, C), generator=g, device="cuda").to(dtype)
    base = torch.randn((taps, C), generator=g, device="cuda") * 0.5
    delta = torch.randn((B, T, taps, G), generator=g, device="cuda") * 0.25
    return x, base, delta


def _host_x(x):
    if x.dtype == torch.bfloat16:
        return oc.widen(x.view(torch.int16).cpu().numpy(), "bf16")
    return oc.widen(x.cpu().numpy(), "f32")


def _check(x, base, delta, out):
    exp = oc.grouped_conv(_host_x(x), base.cpu().numpy().astype(np.float64), delta.cpu().numpy().astype(np.float64))
    got = out.float().cpu().numpy().astype(np.float64)
    atol, rtol = TOL[x.dtype]
    excess = np.abs(got - exp) - (atol + rtol * np.abs(exp))
    assert excess.max() <= 0, f"max excess {excess.max()} at {np.unravel_index(excess.argmax(), excess.shape)}"


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("B,T,C,taps,G", [
    (1, 1, 8, 1, 1),          # one position, one tap
    (2, 16, 512, 4, 8),       # a DFlash2 block of 16 positions
    (3, 9, 300, 3, 3),        # channels not a multiple of the CTA width
    (2, 9, 256, 20, 2),       # more taps than positions
    (4, 16, 5120, 16, 5120),  # one group per channel, taps spanning the block
    (2, 64, 1024, 64, 4),     # the longest block and tap count
    (2, 16, 301, 4, 7),       # an odd channel count (one-channel kernel)
    (2, 16, 4096, 4, 2048),   # delta too large to stage: read from global memory
    (5, 12, 1030, 8, 515),    # groups of two channels, a ragged last CTA
    (2, 16, 510, 4, 2),       # odd group size: a channel pair straddles two groups
])
def test_matches_oracle(dtype, B, T, C, taps, G):
    x, base, delta = _inputs(B, T, C, taps, G, dtype, seed=B * 100 + T + C + taps)
    out = dfl.grouped_conv(x, base, delta)
    torch.cuda.synchronize()
    _check(x, base, delta, out)


def test_one_hot_tap_shifts_the_block_exactly():
    # base = 0, delta one-hot on tap 3: out is x shifted by 3 positions, zeros at the block start
    B, T, C, taps, G = 3, 16, 640, 5, 4
    x, _, _ = _inputs(B, T, C, taps, G, torch.float32, seed=1)
    base = torch.zeros((taps, C), device="cuda")
    delta = torch.zeros((B, T, taps, G), device="cuda")
    delta[:, :, 3, :] = 1.0
    out = dfl.grouped_conv(x, base, delta)
    torch.cuda.synchronize()
    assert bool((out[:, :3] == 0).all())
    assert torch.equal(out[:, 3:], x[:, :-3])


def test_full_size_batch32():
    # the bench's launch: 32 blocks of 16 positions, 5120 channels, 4 taps, 8 groups
    x, base, delta = _inputs(32, 16, 5120, 4, 8, torch.bfloat16, seed=77)
    out = torch.full_like(x, 3.0)
    dfl.grouped_conv(x, base, delta, out=out)
    torch.cuda.synchronize()
    _check(x, base, delta, out)


def test_cuda_graph_replay():
    x, base, delta = _inputs(4, 16, 1024, 4, 8, torch.bfloat16, seed=5)
    out = torch.empty_like(x)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        dfl.grouped_conv(x, base, delta, out=out, stream=s)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        dfl.grouped_conv(x, base, delta, out=out, stream=s)
    out.zero_()
    graph.replay()
    torch.cuda.synchronize()
    _check(x, base, delta, out)
