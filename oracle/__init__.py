"""fp64 CPU oracle for DFlash block attention -- test infrastructure only.

Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package. The product library never links, loads
or calls it, and this package imports nothing from the product package.

The arithmetic lives in ``dflash_oracle.c`` (plain loops, fp64), compiled here
with gcc into ``oracle/_build/liboracle.so``. This module only marshals numpy
arrays; see the C file for the definition each function follows.

Pinning: every function here is pinned by ``tests/test_oracle_pins.py`` against
closed forms, invariants and special cases that reduce to library routines
(torch scaled_dot_product_attention / scipy logsumexp in fp64). The sliding
window offset is pinned by the W = 1 closed form; the window reading itself
(left window of W keys ending at each query) is a reading of the pages.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "dflash_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the C oracle with gcc (portable flags: builds on x86_64 and aarch64)."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.check_call(
            ["gcc", "-O2", "-fPIC", "-shared", "-pthread", "-std=c11", "-o", tmp, _SRC, "-lm"]
        )
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            path = build()
            lib = ctypes.CDLL(path)
            f64p = ctypes.POINTER(ctypes.c_double)
            i32p = ctypes.POINTER(ctypes.c_int32)
            i32, i64, f64 = ctypes.c_int32, ctypes.c_int64, ctypes.c_double
            lib.oracle_block_attn.restype = ctypes.c_int
            vp = ctypes.c_void_p
            lib.oracle_block_attn.argtypes = [
                vp, vp, vp, i32, i32p, i32p,
                i32, i32, i32, i32, i32, i32, i32, i32,
                i64, i64, i64, i32, i32, f64, i32, i32, f64p, f64p, i32,
            ]
            lib.oracle_block_attn_rows.restype = ctypes.c_int
            lib.oracle_block_attn_rows.argtypes = [
                vp, vp, vp, i32, i32p, i32p,
                i32, i32, i32, i32, i32, i32, i32, i32,
                i64, i64, i64, i32, i32, f64, i32p, i64, f64p, f64p, i32,
            ]
            lib.oracle_split_combine.restype = ctypes.c_int
            lib.oracle_split_combine.argtypes = [f64p, f64p, i32, i64, i32, f64p, f64p]
            _lib = lib
    return _lib


def _ptr(a: np.ndarray, ctype):
    return a.ctypes.data_as(ctypes.POINTER(ctype))


def default_threads() -> int:
    return max(1, os.cpu_count() or 1)


def _as_host(x):
    """numpy view of an input: fp32 values, or uint16 bf16 bit patterns.

    A torch tensor is moved to the host; a bf16 tensor is reinterpreted as its
    16-bit patterns (no rounding), every other dtype is converted to fp32.
    """
    if hasattr(x, "detach") and hasattr(x, "dtype"):
        import torch  # only for tensors handed in by the tests

        t = x.detach().to("cpu").contiguous()
        if t.dtype == torch.bfloat16:
            return t.view(torch.int16).numpy().view(np.uint16)
        return t.to(torch.float32).numpy()
    a = np.asarray(x)
    if a.dtype == np.uint16:
        return np.ascontiguousarray(a)
    return np.ascontiguousarray(a, dtype=np.float32)


def _prep_inputs(q, k_cache, v_cache, page_table, seq_lens):
    q, k, v = _as_host(q), _as_host(k_cache), _as_host(v_cache)
    if not (q.dtype == k.dtype == v.dtype):
        raise ValueError("q, k_cache and v_cache must share one dtype")
    if k.shape != v.shape or k.ndim != 4:
        raise ValueError("k_cache/v_cache must both be [num_pages, page_size, Hkv, D]")
    in_dtype = 1 if q.dtype == np.uint16 else 0
    pt = np.ascontiguousarray(_as_int(page_table), dtype=np.int32)
    sl = np.ascontiguousarray(_as_int(seq_lens), dtype=np.int32)
    return q, k, v, pt, sl, in_dtype


def _as_int(x):
    if hasattr(x, "detach"):
        return x.detach().to("cpu").numpy()
    return np.asarray(x)


def block_attn(q, k_cache, v_cache, page_table, seq_lens, block_len, causal=False,
               window=0, scale=None, key_range=None, num_threads=None):
    """Plain fp64 block attention.

    q: [B*T, Hq, D]; k_cache, v_cache: [num_pages, page_size, Hkv, D];
    page_table: [B, max_pages] int32; seq_lens: [B] int32 (includes the block).
    key_range=(kb, ke) restricts the keys to positions in [kb, ke) (one split
    chunk); rows with no visible key then get lse=-inf and out=0.
    Returns (out [B*T, Hq, D] float64, lse [B*T, Hq] float64).
    """
    q, k, v, pt, sl, in_dtype = _prep_inputs(q, k_cache, v_cache, page_table, seq_lens)
    BT, Hq, D = q.shape
    T = int(block_len)
    B = BT // T
    num_pages, page_size, Hkv, Dk = k.shape
    if Dk != D or B * T != BT or pt.shape[0] != B or sl.shape[0] != B:
        raise ValueError("inconsistent shapes")
    if scale is None:
        scale = 1.0 / np.sqrt(D)
    kb, ke = (0, -1) if key_range is None else (int(key_range[0]), int(key_range[1]))
    out = np.zeros((BT, Hq, D), dtype=np.float64)
    lse = np.zeros((BT, Hq), dtype=np.float64)
    rc = _load().oracle_block_attn(
        q.ctypes.data, k.ctypes.data, v.ctypes.data, in_dtype,
        _ptr(pt, ctypes.c_int32), _ptr(sl, ctypes.c_int32),
        B, T, Hq, Hkv, D, page_size, num_pages, pt.shape[1],
        page_size * Hkv * D, Hkv * D, D,
        int(bool(causal)), int(window), float(scale), kb, ke,
        _ptr(out, ctypes.c_double), _ptr(lse, ctypes.c_double),
        int(num_threads or default_threads()),
    )
    if rc != 0:
        raise ValueError(f"oracle_block_attn failed with code {rc}")
    return out, lse


def block_attn_rows(q, k_cache, v_cache, page_table, seq_lens, block_len, rows,
                    causal=False, window=0, scale=None, num_threads=None):
    """The same definition for a sample of output rows.

    rows: int array [n, 3] of (b, h, i). Returns (out [n, D], lse [n]) float64.
    """
    q, k, v, pt, sl, in_dtype = _prep_inputs(q, k_cache, v_cache, page_table, seq_lens)
    BT, Hq, D = q.shape
    T = int(block_len)
    B = BT // T
    num_pages, page_size, Hkv, _ = k.shape
    rows = np.ascontiguousarray(rows, dtype=np.int32).reshape(-1, 3)
    n = rows.shape[0]
    if scale is None:
        scale = 1.0 / np.sqrt(D)
    out = np.zeros((n, D), dtype=np.float64)
    lse = np.zeros((n,), dtype=np.float64)
    rc = _load().oracle_block_attn_rows(
        q.ctypes.data, k.ctypes.data, v.ctypes.data, in_dtype,
        _ptr(pt, ctypes.c_int32), _ptr(sl, ctypes.c_int32),
        B, T, Hq, Hkv, D, page_size, num_pages, pt.shape[1],
        page_size * Hkv * D, Hkv * D, D,
        int(bool(causal)), int(window), float(scale),
        _ptr(rows, ctypes.c_int32), n,
        _ptr(out, ctypes.c_double), _ptr(lse, ctypes.c_double),
        int(num_threads or default_threads()),
    )
    if rc != 0:
        raise ValueError(f"oracle_block_attn_rows failed with code {rc}")
    return out, lse


def split_combine(partial_out, partial_lse):
    """LSE combine: partial_out [S, N..., D], partial_lse [S, N...] -> (out, lse) in fp64."""
    po = np.ascontiguousarray(partial_out, dtype=np.float64)
    pl = np.ascontiguousarray(partial_lse, dtype=np.float64)
    S = po.shape[0]
    D = po.shape[-1]
    inner = po.shape[1:-1]
    if pl.shape != (S,) + tuple(inner):
        raise ValueError("partial_lse shape mismatch")
    N = int(np.prod(inner)) if inner else 1
    out = np.zeros(tuple(inner) + (D,), dtype=np.float64)
    lse = np.zeros(tuple(inner), dtype=np.float64)
    _load().oracle_split_combine(
        _ptr(po, ctypes.c_double), _ptr(pl, ctypes.c_double), S, N, D,
        _ptr(out, ctypes.c_double), _ptr(lse, ctypes.c_double),
    )
    return out, lse
