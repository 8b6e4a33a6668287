"""The C-ABI library without a GPU: it loads, exports every declared entry
point, and rejects bad arguments on the host before any CUDA call."""
import ctypes
import os
import re

import pytest
import torch

import speculative_decoding_block_dflash_gb300 as dfl
from speculative_decoding_block_dflash_gb300 import _binding as B
from speculative_decoding_block_dflash_gb300 import build as build_mod

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "dflash_attn.h")

# Fake device addresses are only ever used in calls that must fail host-side
# validation; on a machine with a GPU these tests are skipped so that a
# validation slip can never hand such an address to a kernel.
cpu_only = pytest.mark.skipif(torch.cuda.is_available(), reason="fake-pointer validation runs on CPU-only hosts")


@pytest.fixture(scope="module")
def lib():
    build_mod.build()
    return dfl.load_library()


def declared_functions():
    text = open(HEADER).read()
    return re.findall(r"DFLASH_API\s+[\w\s\*]+?\b(dflash_\w+)\s*\(", text)


def test_header_declares_the_binding_surface():
    names = declared_functions()
    assert sorted(names) == sorted(B.EXPORTED)
    assert "dflash_block_attn" in names and "dflash_split_combine" in names


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name
    # nothing but the C ABI is exported
    out = os.popen(f"nm -D --defined-only {B.LIB_PATH}").read()
    exported = {ln.split()[-1] for ln in out.splitlines() if " T " in ln}
    assert exported == set(declared_functions())


def test_abi_version_matches_header(lib):
    m = re.search(r"#define DFLASH_ABI_VERSION (\d+)", open(HEADER).read())
    assert lib.dflash_abi_version() == int(m.group(1))


def test_status_strings(lib):
    for s in range(6):
        assert lib.dflash_status_string(s).decode()
    assert lib.dflash_status_string(99).decode() == "unknown status"


def good_dims(**kw):
    d = B.Dims()
    vals = dict(batch=2, num_q_heads=32, num_kv_heads=4, head_dim=512, page_size=16, num_pages=1024,
                max_pages=512, max_seq_len=0, dtype=B.BF16)
    vals.update(kw)
    for k, v in vals.items():
        setattr(d, k, v)
    d.kv_stride_head = kw.get("kv_stride_head", d.head_dim)
    d.kv_stride_slot = kw.get("kv_stride_slot", d.num_kv_heads * d.head_dim)
    d.kv_stride_page = kw.get("kv_stride_page", d.page_size * d.num_kv_heads * d.head_dim)
    return d


def test_workspace_layout(lib):
    d = good_dims()
    T = 9
    n1 = lib.dflash_workspace_bytes(ctypes.byref(d), T, 1)
    assert n1 == 256 + 8192  # error word + fixed counter block
    S = 16
    rows = 2 * T * 32
    n = lib.dflash_workspace_bytes(ctypes.byref(d), T, S)
    rnd = lambda x: (x + 255) // 256 * 256
    assert n == 256 + 8192 + rnd(4 * rows * S) + rnd(4 * rows * S * 512)
    assert lib.dflash_workspace_bytes(ctypes.byref(d), T, 0) == 0
    assert lib.dflash_workspace_bytes(ctypes.byref(good_dims(head_dim=520)), T, 1) == 0


def test_plan_splits_explicit_and_invalid(lib):
    d = good_dims()
    assert lib.dflash_plan_splits(ctypes.byref(d), 9, 0, 7, 0) == 7
    assert lib.dflash_plan_splits(ctypes.byref(d), 9, 0, 300, 0) == -B.ERR_INVALID_ARG
    assert lib.dflash_plan_splits(ctypes.byref(good_dims(num_kv_heads=5)), 9, 0, 0, 0) == -B.ERR_INVALID_ARG
    assert lib.dflash_plan_splits(ctypes.byref(good_dims(head_dim=72)), 9, 0, 0, 0) == -B.ERR_UNSUPPORTED
    auto = lib.dflash_plan_splits(ctypes.byref(d), 9, 0, 0, 0)
    assert 1 <= auto <= 256
    # a sliding window bounds the useful split count by its span (per request: the
    # length-balanced plan deals its slots over the batch's requests)
    assert lib.dflash_plan_splits(ctypes.byref(d), 9, 256, 0, 0) <= 2 * d.batch
    assert lib.dflash_plan_splits(ctypes.byref(good_dims(batch=1)), 9, 256, 0, 0) <= 2


def test_head_dim_512_accepted_and_above_rejected(lib):
    assert lib.dflash_plan_splits(ctypes.byref(good_dims(head_dim=512)), 9, 0, 1, 0) == 1
    assert lib.dflash_plan_splits(ctypes.byref(good_dims(head_dim=528)), 9, 0, 1, 0) == -B.ERR_INVALID_ARG


FAKE = 0x10000  # 64 KiB-aligned fake address, never dereferenced


def call(lib, dims=None, T=9, causal=0, window=0, scale=0.04, opts=None, **ptrs):
    p = dict(q=FAKE, k=FAKE, v=FAKE, pt=FAKE, sl=FAKE, out=FAKE, lse=FAKE)
    p.update(ptrs)
    d = dims if dims is not None else good_dims()
    return lib.dflash_block_attn(p["q"], p["k"], p["v"], p["pt"], p["sl"], ctypes.byref(d) if d else None, T,
                                 causal, window, scale, p["out"], p["lse"], ctypes.byref(opts) if opts else None)


@cpu_only
@pytest.mark.parametrize("kw,code", [
    (dict(dims=False), B.ERR_INVALID_ARG),
    (dict(q=0), B.ERR_INVALID_ARG),
    (dict(out=0), B.ERR_INVALID_ARG),
    (dict(q=FAKE + 2), B.ERR_INVALID_ARG),
    (dict(lse=FAKE + 2), B.ERR_INVALID_ARG),
    (dict(T=0), B.ERR_INVALID_ARG),
    (dict(T=65), B.ERR_INVALID_ARG),
    (dict(causal=2), B.ERR_INVALID_ARG),
    (dict(window=-1), B.ERR_INVALID_ARG),
    (dict(window=4), B.ERR_INVALID_ARG),          # window < block_len
    (dict(scale=0.0), B.ERR_INVALID_ARG),
    (dict(scale=float("nan")), B.ERR_INVALID_ARG),
    (dict(scale=float("inf")), B.ERR_INVALID_ARG),
])
def test_block_attn_rejects_bad_arguments(lib, kw, code):
    if kw.get("dims") is False:
        kw = dict(kw)
        kw["dims"] = None
        d = None
        st = lib.dflash_block_attn(FAKE, FAKE, FAKE, FAKE, FAKE, None, 9, 0, 0, 0.04, FAKE, FAKE, None)
        assert st == code
        return
    assert call(lib, **kw) == code
    assert lib.dflash_last_error_message().decode()


@cpu_only
@pytest.mark.parametrize("dkw,code", [
    (dict(num_kv_heads=3), B.ERR_INVALID_ARG),
    (dict(head_dim=40), B.ERR_UNSUPPORTED),
    (dict(head_dim=1024), B.ERR_INVALID_ARG),
    (dict(page_size=12), B.ERR_INVALID_ARG),
    (dict(page_size=512), B.ERR_INVALID_ARG),
    (dict(batch=0), B.ERR_INVALID_ARG),
    (dict(num_pages=0), B.ERR_INVALID_ARG),
    (dict(max_seq_len=512 * 16 + 1), B.ERR_INVALID_ARG),
    (dict(max_seq_len=4), B.ERR_INVALID_ARG),      # below block_len
    (dict(dtype=7), B.ERR_INVALID_ARG),
    (dict(kv_stride_slot=4 * 512 + 4), B.ERR_INVALID_ARG),   # 8-byte stride, not 16
    (dict(kv_stride_head=256), B.ERR_INVALID_ARG),
])
def test_block_attn_rejects_bad_dims(lib, dkw, code):
    assert call(lib, dims=good_dims(**dkw)) == code


@cpu_only
def test_split_needs_workspace(lib):
    o = B.Opts()
    o.num_splits = 4
    assert call(lib, opts=o) == B.ERR_WORKSPACE
    o.workspace = FAKE
    o.workspace_bytes = 1024
    assert call(lib, opts=o) == B.ERR_WORKSPACE
    o.workspace = FAKE + 16  # misaligned
    o.workspace_bytes = 1 << 40
    assert call(lib, opts=o) == B.ERR_WORKSPACE
    o.workspace = FAKE
    o.num_splits = 257
    assert call(lib, opts=o) == B.ERR_INVALID_ARG


@cpu_only
def test_forced_tc_kernel_rejects_fp32(lib):
    o = B.Opts()
    o.kernel = B.KERNELS["tc"]
    assert call(lib, dims=good_dims(dtype=B.FP32), opts=o) == B.ERR_UNSUPPORTED
    o.kernel = 9
    assert call(lib, opts=o) == B.ERR_INVALID_ARG


@cpu_only
@pytest.mark.parametrize("args,code", [
    ((0, FAKE, 2, 10, 64, B.FP32, FAKE, FAKE, None), B.ERR_INVALID_ARG),
    ((FAKE, FAKE, 0, 10, 64, B.FP32, FAKE, FAKE, None), B.ERR_INVALID_ARG),
    ((FAKE, FAKE, 257, 10, 64, B.FP32, FAKE, FAKE, None), B.ERR_INVALID_ARG),
    ((FAKE, FAKE, 2, 0, 64, B.FP32, FAKE, FAKE, None), B.ERR_INVALID_ARG),
    ((FAKE, FAKE, 2, 10, 66, B.FP32, FAKE, FAKE, None), B.ERR_INVALID_ARG),
    ((FAKE, FAKE, 2, 10, 1024, B.FP32, FAKE, FAKE, None), B.ERR_INVALID_ARG),
    ((FAKE, FAKE, 2, 10, 64, 3, FAKE, FAKE, None), B.ERR_INVALID_ARG),
    ((FAKE + 4, FAKE, 2, 10, 64, B.FP32, FAKE, FAKE, None), B.ERR_INVALID_ARG),
])
def test_split_combine_rejects_bad_arguments(lib, args, code):
    assert lib.dflash_split_combine(*args) == code


def test_read_error_rejects_null(lib):
    w = ctypes.c_uint32(0)
    assert lib.dflash_read_error(None, None, ctypes.byref(w), 0) == B.ERR_INVALID_ARG


def test_binding_refuses_to_run_without_the_library(tmp_path):
    with pytest.raises(RuntimeError):
        B.load_library(str(tmp_path / "missing.so"))


def test_accept_workspace_and_argument_checks(lib):
    # two regions, each 256-byte aligned: B*T 64-bit keys, then B int32 counters
    assert lib.dflash_accept_workspace_bytes(8, 9) == 768 + 256
    assert lib.dflash_accept_workspace_bytes(0, 9) == 0
    assert lib.dflash_accept_workspace_bytes(1000, 100) == 0  # B*T > 65535

    def acc(dtype=B.BF16, batch=2, T=9, V=1000, stride=1008, draft=FAKE, ws=FAKE, ws_bytes=1 << 20, logits=FAKE):
        return lib.dflash_accept_prefix(logits, dtype, batch, T, V, stride, draft, FAKE, FAKE, None, ws, ws_bytes,
                                        None)

    assert acc(dtype=7) == B.ERR_INVALID_ARG
    assert acc(V=0) == B.ERR_INVALID_ARG
    assert acc(stride=999) == B.ERR_INVALID_ARG          # shorter than a row
    assert acc(batch=70000) == B.ERR_INVALID_ARG
    assert acc(draft=None) == B.ERR_INVALID_ARG          # drafts needed when T > 1
    assert acc(logits=FAKE + 1) == B.ERR_INVALID_ARG     # logits aligned to their element size
    assert acc(dtype=B.FP32, logits=FAKE + 2) == B.ERR_INVALID_ARG
    assert acc(ws=None) == B.ERR_WORKSPACE
    assert acc(ws_bytes=64) == B.ERR_WORKSPACE
    assert acc(ws=FAKE + 16) == B.ERR_WORKSPACE
    assert b"workspace" in lib.dflash_last_error_message()


@cpu_only
def test_project_kv_argument_checks(lib):
    P = ctypes.c_void_p

    def proj(L=64, H=5376, stride=5376, hidden=FAKE, wk=FAKE, wv=FAKE, slots=FAKE, kc=FAKE, vc=FAKE, err=None,
             ws=None, **dkw):
        d = good_dims(**dkw)
        return lib.dflash_project_kv(P(hidden), L, H, stride, P(wk), P(wv), P(slots), P(kc), P(vc),
                                     ctypes.byref(d), P(err) if err else None, P(ws) if ws else None, 1 << 24, None)

    assert proj(L=0, hidden=None, slots=None) == B.OK  # no tokens: nothing is read or launched
    assert proj(dtype=B.FP32) == B.ERR_UNSUPPORTED
    assert proj(L=-1) == B.ERR_INVALID_ARG
    assert proj(L=(1 << 24) + 1) == B.ERR_INVALID_ARG
    assert proj(H=5370, stride=5370) == B.ERR_INVALID_ARG   # hidden size not a multiple of 8
    assert proj(stride=5368) == B.ERR_INVALID_ARG           # row stride shorter than a row
    assert proj(stride=5380) == B.ERR_INVALID_ARG           # row stride not a multiple of 8
    assert proj(head_dim=24) == B.ERR_INVALID_ARG           # head_dim not a multiple of 16
    assert proj(head_dim=1024) == B.ERR_INVALID_ARG
    assert proj(num_kv_heads=0) == B.ERR_INVALID_ARG
    assert proj(page_size=0) == B.ERR_INVALID_ARG
    assert proj(num_pages=0) == B.ERR_INVALID_ARG
    assert proj(kv_stride_head=516) == B.ERR_INVALID_ARG
    assert proj(hidden=None) == B.ERR_INVALID_ARG
    assert proj(slots=None) == B.ERR_INVALID_ARG
    assert proj(kc=FAKE + 8) == B.ERR_INVALID_ARG           # caches 16-byte aligned
    assert proj(wk=FAKE + 2) == B.ERR_INVALID_ARG
    assert proj(slots=FAKE + 2) == B.ERR_INVALID_ARG
    assert proj(err=FAKE + 1) == B.ERR_INVALID_ARG
    assert b"misaligned" in lib.dflash_last_error_message()
    assert proj(ws=FAKE + 16) == B.ERR_WORKSPACE       # the workspace is 256-byte aligned


@cpu_only
def test_grouped_conv_argument_checks(lib):
    P = ctypes.c_void_p

    def conv(x=FAKE, out=FAKE + 4096, dtype=B.BF16, B_=2, T=16, C=512, taps=4, G=8, base=FAKE, delta=FAKE):
        return lib.dflash_grouped_conv(P(x) if x else None, P(out) if out else None, dtype, B_, T, C, taps, G,
                                       P(base) if base else None, P(delta) if delta else None, None)

    assert conv(dtype=5) == B.ERR_INVALID_ARG
    assert conv(B_=0) == B.ERR_INVALID_ARG
    assert conv(B_=70000) == B.ERR_INVALID_ARG
    assert conv(T=0) == B.ERR_INVALID_ARG
    assert conv(T=65) == B.ERR_INVALID_ARG
    assert conv(taps=0) == B.ERR_INVALID_ARG
    assert conv(taps=65) == B.ERR_INVALID_ARG
    assert conv(G=7) == B.ERR_INVALID_ARG          # 512 channels do not split into 7 groups
    assert conv(G=0) == B.ERR_INVALID_ARG
    assert conv(x=None) == B.ERR_INVALID_ARG
    assert conv(delta=None) == B.ERR_INVALID_ARG
    assert conv(out=FAKE) == B.ERR_INVALID_ARG     # in place is rejected
    assert conv(x=FAKE + 1) == B.ERR_INVALID_ARG
    assert conv(dtype=B.FP32, out=FAKE + 4098) == B.ERR_INVALID_ARG
    assert conv(base=FAKE + 2) == B.ERR_INVALID_ARG
    assert b"misaligned" in lib.dflash_last_error_message()


@cpu_only
def test_selector_workspace_and_argument_checks(lib):
    P = ctypes.c_void_p
    # a fixed 256 KB counter block, then the R*S*K*K edge tables
    assert lib.dflash_selector_workspace_bytes(32, 15, 8) == 262144 + 32 * 15 * 64 * 4
    assert lib.dflash_selector_workspace_bytes(1, 1, 1) == 262144 + 256
    assert lib.dflash_selector_workspace_bytes(0, 15, 8) == 0
    assert lib.dflash_selector_workspace_bytes(2, 15, 65) == 0

    def walk(A=FAKE, V=1000, E=256, proj=FAKE, R=2, S=15, K=8, T=0.0, u=None, tokens=FAKE, ws=FAKE, ws_bytes=1 << 20,
             err=None):
        return lib.dflash_selector_walk(P(A) if A else None, P(FAKE), V, E, P(proj), P(FAKE), P(FAKE), P(FAKE), R, S, K,
                                        T, P(u) if u else None, P(tokens) if tokens else None, None, None, None,
                                        P(err) if err else None, P(ws) if ws else None, ws_bytes, None)

    assert walk(K=0) == B.ERR_INVALID_ARG
    assert walk(K=65) == B.ERR_INVALID_ARG
    assert walk(R=0) == B.ERR_INVALID_ARG
    assert walk(V=0) == B.ERR_INVALID_ARG
    assert walk(E=12) == B.ERR_INVALID_ARG            # dim not a multiple of 8
    assert walk(K=64, E=4096) == B.ERR_UNSUPPORTED    # the staged rows exceed shared memory
    assert walk(T=-1.0) == B.ERR_INVALID_ARG
    assert walk(T=float("nan")) == B.ERR_INVALID_ARG
    assert walk(T=0.7) == B.ERR_INVALID_ARG           # sampling needs uniforms
    assert walk(A=None) == B.ERR_INVALID_ARG
    assert walk(tokens=None) == B.ERR_INVALID_ARG
    assert walk(proj=FAKE + 4) == B.ERR_INVALID_ARG   # proj rows are read 16 bytes at a time
    assert walk(err=FAKE + 2) == B.ERR_INVALID_ARG
    assert walk(ws=None) == B.ERR_WORKSPACE
    assert walk(ws_bytes=1024) == B.ERR_WORKSPACE
    assert b"workspace" in lib.dflash_last_error_message()


def test_auto_plan_takes_uniform_waves_for_long_spans(lib):
    # the planner's host logic (no kernel runs): 8 requests of up to 131072 keys in blocks of 16
    # would give one balanced wave of ~55k-key chunks, so the auto plan takes uniform chunks of
    # about 7168 keys over several waves; up to 32768 keys keeps the one-wave balanced plan
    sms = torch.cuda.get_device_properties(0).multi_processor_count if torch.cuda.is_available() else 148
    long = good_dims(batch=8, max_pages=131072 // 16, num_pages=8 * (131072 // 16))
    assert lib.dflash_plan_splits(ctypes.byref(long), 16, 0, 0, 0) == -(-131072 // 7168)
    sweep = good_dims(batch=8, max_pages=32768 // 16, num_pages=8 * (32768 // 16))
    assert lib.dflash_plan_splits(ctypes.byref(sweep), 9, 0, 0, 0) == sms // 4
    # an explicit count is taken as given
    assert lib.dflash_plan_splits(ctypes.byref(long), 16, 0, 5, 0) == 5


def _cpu_inputs(B=2, T=9, Hq=4, Hkv=2, D=64, P=16, pages=8):
    q = torch.zeros((B * T, Hq, D), dtype=torch.bfloat16)
    k = torch.zeros((pages, P, Hkv, D), dtype=torch.bfloat16)
    v = torch.zeros_like(k)
    pt = torch.zeros((B, 4), dtype=torch.int32)
    sl = torch.full((B,), 20, dtype=torch.int32)
    return q, k, v, pt, sl


@pytest.mark.parametrize("entry", ["block_attn", "block_attn_noalloc"])
@pytest.mark.parametrize("bad", ["v_shape", "v_stride", "pt_int64", "sl_int64", "pt_slice", "q_rows", "out_dtype"])
def test_attention_entry_points_reject_mismatched_inputs_before_launch(lib, entry, bad):
    # v_cache is read with k_cache's geometry and the index tensors as int32, so both entry
    # points must refuse these before the library (or any kernel) sees a pointer
    q, k, v, pt, sl = _cpu_inputs()
    out = None
    if bad == "v_shape":
        v = torch.zeros((4,) + tuple(k.shape[1:]), dtype=k.dtype)
    elif bad == "v_stride":
        v = torch.zeros((k.shape[0], k.shape[1], k.shape[3], k.shape[2]), dtype=k.dtype).transpose(2, 3)
    elif bad == "pt_int64":
        pt = pt.to(torch.int64)
    elif bad == "sl_int64":
        sl = sl.to(torch.int64)
    elif bad == "pt_slice":
        pt = torch.zeros((2, 8), dtype=torch.int32)[:, :4]
    elif bad == "q_rows":
        q = q[:-1]
    elif bad == "out_dtype":
        out = torch.zeros(q.shape, dtype=torch.float32)
    fn = getattr(dfl, entry)
    with pytest.raises((ValueError, TypeError)):
        fn(q, k, v, pt, sl, 9, out=out)
