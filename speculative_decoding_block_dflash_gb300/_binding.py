"""ctypes binding of libdflash_attn (argument marshalling only).

Every step of the attention runs in the library's CUDA kernels; this module
only turns torch tensors into the pointers, sizes and strides that
include/dflash_attn.h describes, picks the current CUDA stream, and keeps a
small per-device workspace cache. There is no CPU fallback: if the library is
missing, every call raises.
"""
from __future__ import annotations

import ctypes
import math
import os
import threading
from typing import Optional, Tuple

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "_lib", "libdflash_attn.so")

# dflash_status
OK, ERR_INVALID_ARG, ERR_UNSUPPORTED, ERR_CUDA, ERR_DEVICE_CHECK, ERR_WORKSPACE = range(6)
# dflash_dtype
BF16, FP32 = 0, 1
# dflash_kernel
KERNELS = {"auto": 0, "simt": 1, "tc": 2, "tc_pair": 3}
# device error bits
DEVERR_PAGE_ID, DEVERR_SEQ_LEN, DEVERR_TIMEOUT, DEVERR_TOKEN_ID = 1, 2, 4, 8

EXPORTED = (
    "dflash_block_attn",
    "dflash_block_attn_noalloc",
    "dflash_split_combine",
    "dflash_plan_splits",
    "dflash_plan_call",
    "dflash_workspace_bytes",
    "dflash_read_error",
    "dflash_status_string",
    "dflash_last_error_message",
    "dflash_abi_version",
    "dflash_accept_prefix",
    "dflash_accept_workspace_bytes",
    "dflash_project_kv",
    "dflash_project_kv_workspace_bytes",
    "dflash_grouped_conv",
    "dflash_selector_workspace_bytes",
    "dflash_selector_walk",
)


class Dims(ctypes.Structure):
    _fields_ = [
        ("batch", ctypes.c_int32),
        ("num_q_heads", ctypes.c_int32),
        ("num_kv_heads", ctypes.c_int32),
        ("head_dim", ctypes.c_int32),
        ("page_size", ctypes.c_int32),
        ("num_pages", ctypes.c_int32),
        ("max_pages", ctypes.c_int32),
        ("max_seq_len", ctypes.c_int32),
        ("dtype", ctypes.c_int32),
        ("kv_stride_page", ctypes.c_int64),
        ("kv_stride_slot", ctypes.c_int64),
        ("kv_stride_head", ctypes.c_int64),
    ]


class Opts(ctypes.Structure):
    _fields_ = [
        ("num_splits", ctypes.c_int32),
        ("kernel", ctypes.c_int32),
        ("workspace", ctypes.c_void_p),
        ("workspace_bytes", ctypes.c_size_t),
        ("stream", ctypes.c_void_p),
        ("wait_limit_us", ctypes.c_uint32),
    ]


class Plan(ctypes.Structure):
    _fields_ = [
        ("num_splits", ctypes.c_int32),
        ("kernel", ctypes.c_int32),
        ("balanced", ctypes.c_int32),
        ("launches", ctypes.c_int32),
        ("ctas", ctypes.c_int64),
    ]


KERNEL_NAMES = {1: "simt_attn_kernel", 2: "tc_attn_kernel", 3: "tc_pair_attn_kernel"}


class DflashError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"dflash status {status}: {message}")
        self.status = status


_lock = threading.Lock()
_lib = None


def load_library(path: Optional[str] = None):
    """Load libdflash_attn.so (built by build.py) and declare its signatures."""
    global _lib
    with _lock:
        if _lib is not None and path is None:
            return _lib
        p = path or LIB_PATH
        if not os.path.exists(p):
            raise RuntimeError(f"{p} is missing: build it with speculative_decoding_block_dflash_gb300.build.build()")
        lib = ctypes.CDLL(p)
        vp, i32, i64, f32 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_float
        dims_p, opts_p = ctypes.POINTER(Dims), ctypes.POINTER(Opts)
        lib.dflash_block_attn.restype = ctypes.c_int
        lib.dflash_block_attn.argtypes = [vp, vp, vp, vp, vp, dims_p, i32, i32, i32, f32, vp, vp, opts_p]
        lib.dflash_block_attn_noalloc.restype = ctypes.c_int
        lib.dflash_block_attn_noalloc.argtypes = [vp, vp, vp, vp, vp, dims_p, i32, i32, i32, f32, vp, vp, i32, i32, vp]
        lib.dflash_split_combine.restype = ctypes.c_int
        lib.dflash_split_combine.argtypes = [vp, vp, i32, i64, i32, i32, vp, vp, vp]
        lib.dflash_plan_splits.restype = i32
        lib.dflash_plan_splits.argtypes = [dims_p, i32, i32, i32, i32]
        lib.dflash_plan_call.restype = ctypes.c_int
        lib.dflash_plan_call.argtypes = [dims_p, i32, i32, i32, i32, ctypes.POINTER(Plan)]
        lib.dflash_workspace_bytes.restype = ctypes.c_size_t
        lib.dflash_workspace_bytes.argtypes = [dims_p, i32, i32]
        lib.dflash_read_error.restype = ctypes.c_int
        lib.dflash_read_error.argtypes = [vp, vp, ctypes.POINTER(ctypes.c_uint32), i32]
        lib.dflash_status_string.restype = ctypes.c_char_p
        lib.dflash_status_string.argtypes = [ctypes.c_int]
        lib.dflash_last_error_message.restype = ctypes.c_char_p
        lib.dflash_last_error_message.argtypes = []
        lib.dflash_abi_version.restype = i32
        lib.dflash_abi_version.argtypes = []
        lib.dflash_accept_workspace_bytes.restype = ctypes.c_size_t
        lib.dflash_accept_workspace_bytes.argtypes = [i32, i32]
        lib.dflash_accept_prefix.restype = ctypes.c_int
        lib.dflash_accept_prefix.argtypes = [vp, i32, i32, i32, i32, i64, vp, vp, vp, vp, vp, ctypes.c_size_t, vp]
        lib.dflash_project_kv.restype = ctypes.c_int
        lib.dflash_project_kv.argtypes = [vp, i32, i32, i64, vp, vp, vp, vp, vp, dims_p, vp, vp, ctypes.c_size_t, vp]
        lib.dflash_project_kv_workspace_bytes.restype = ctypes.c_size_t
        lib.dflash_project_kv_workspace_bytes.argtypes = []
        lib.dflash_grouped_conv.restype = ctypes.c_int
        lib.dflash_grouped_conv.argtypes = [vp, vp, i32, i32, i32, i32, i32, i32, vp, vp, vp]
        lib.dflash_selector_workspace_bytes.restype = ctypes.c_size_t
        lib.dflash_selector_workspace_bytes.argtypes = [i32, i32, i32]
        lib.dflash_selector_walk.restype = ctypes.c_int
        lib.dflash_selector_walk.argtypes = [vp, vp, i32, i32, vp, vp, vp, vp, i32, i32, i32, f32, vp, vp, vp, vp, vp,
                                             vp, vp, ctypes.c_size_t, vp]
        if path is None:
            _lib = lib
        return lib


def _check(status: int):
    if status != OK:
        lib = load_library()
        msg = lib.dflash_last_error_message().decode() or lib.dflash_status_string(status).decode()
        raise DflashError(status, msg)


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return BF16
    if t.dtype == torch.float32:
        return FP32
    raise TypeError(f"unsupported dtype {t.dtype} (bf16 or fp32)")


def make_dims(q: torch.Tensor, k_cache: torch.Tensor, page_table: torch.Tensor, block_len: int,
              max_seq_len: Optional[int] = None, batch: Optional[int] = None) -> Dims:
    """Dims for q [B*T, Hq, D] and a cache [num_pages, page_size, Hkv, D] (any strides, d contiguous)."""
    if q.dim() != 3 or k_cache.dim() != 4:
        raise ValueError("q must be [B*T, Hq, D] and k_cache [num_pages, page_size, Hkv, D]")
    B = batch if batch is not None else page_table.shape[0]
    d = Dims()
    d.batch = B
    d.num_q_heads = q.shape[1]
    d.num_kv_heads = k_cache.shape[2]
    d.head_dim = q.shape[2]
    d.page_size = k_cache.shape[1]
    d.num_pages = k_cache.shape[0]
    d.max_pages = page_table.shape[1]
    d.max_seq_len = int(max_seq_len) if max_seq_len else 0
    d.dtype = _dtype_code(q)
    d.kv_stride_page, d.kv_stride_slot, d.kv_stride_head = (int(s) for s in k_cache.stride()[:3])
    return d


def plan_splits(dims: Dims, block_len: int, window: int = 0, requested: int = 0, kernel: str = "auto") -> int:
    n = load_library().dflash_plan_splits(ctypes.byref(dims), int(block_len), int(window), int(requested),
                                          KERNELS[kernel])
    if n < 1:
        _check(-n)
    return n


def plan_info(dims: Dims, block_len: int, window: int = 0, requested: int = 0, kernel: str = "auto") -> dict:
    """What a call with these sizes runs (dflash_plan_call): split count, kernel, whether the
    splits are length-balanced, CTAs of the attention launch and kernel launches per call."""
    plan = Plan()
    _check(load_library().dflash_plan_call(ctypes.byref(dims), int(block_len), int(window), int(requested),
                                           KERNELS[kernel], ctypes.byref(plan)))
    return {"num_splits": plan.num_splits, "kernel": plan.kernel, "kernel_name": KERNEL_NAMES[plan.kernel],
            "balanced": bool(plan.balanced), "launches": plan.launches, "ctas": int(plan.ctas)}


def workspace_bytes(dims: Dims, block_len: int, num_splits: int) -> int:
    n = load_library().dflash_workspace_bytes(ctypes.byref(dims), int(block_len), int(num_splits))
    if n == 0:
        raise DflashError(ERR_INVALID_ARG, "invalid dims for workspace size")
    return n


def _check_attn_inputs(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor, page_table: torch.Tensor,
                       seq_lens: torch.Tensor, block_len: int, out: Optional[torch.Tensor],
                       lse: Optional[torch.Tensor]) -> None:
    """Checks the library cannot make from the pointers and dims alone: the dims carry
    k_cache's geometry only (the kernels and tensor maps read v_cache with it), and the
    index tensors are read as int32. Shared by both attention entry points."""
    if v_cache.shape != k_cache.shape or v_cache.stride() != k_cache.stride():
        raise ValueError("v_cache must match k_cache in shape and strides")
    if v_cache.dtype != k_cache.dtype or q.dtype != k_cache.dtype:
        raise TypeError("q, k_cache and v_cache must share one dtype")
    if not q.is_contiguous():
        raise ValueError("q must be contiguous")
    if page_table.dtype != torch.int32 or seq_lens.dtype != torch.int32:
        raise TypeError("page_table and seq_lens must be int32")
    if page_table.dim() != 2 or not page_table.is_contiguous():
        raise ValueError("page_table must be a contiguous [B, max_pages] tensor")
    if seq_lens.dim() != 1 or seq_lens.shape[0] != page_table.shape[0] or not seq_lens.is_contiguous():
        raise ValueError("seq_lens must be a contiguous [B] tensor matching page_table's rows")
    if q.dim() != 3 or q.shape[0] != page_table.shape[0] * int(block_len):
        raise ValueError("q must be [B*block_len, Hq, D] with B = page_table.shape[0]")
    if out is not None and (out.shape != q.shape or out.dtype != q.dtype or not out.is_contiguous()):
        raise ValueError("out must be a contiguous tensor of q's shape and dtype")
    if lse is not None and (tuple(lse.shape) != tuple(q.shape[:2]) or lse.dtype != torch.float32
                            or not lse.is_contiguous()):
        raise ValueError("lse must be a contiguous float32 [B*block_len, Hq] tensor")
    devs = {t.device for t in (q, k_cache, v_cache, page_table, seq_lens, out, lse) if t is not None}
    if len(devs) != 1 or next(iter(devs)).type != "cuda":
        raise ValueError("every tensor must be on one CUDA device")


_ws_cache = {}


def workspace_for(device: torch.device, nbytes: int) -> torch.Tensor:
    """A zero-initialised, 256-byte aligned device buffer of at least nbytes, cached per device."""
    key = (device.type, device.index)
    buf = _ws_cache.get(key)
    if buf is None or buf.numel() < nbytes:
        buf = torch.zeros(max(nbytes, 1 << 20), dtype=torch.uint8, device=device)
        _ws_cache[key] = buf
    return buf


def _stream_handle(stream) -> int:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def block_attn(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor, page_table: torch.Tensor,
               seq_lens: torch.Tensor, block_len: int, causal: bool = False, window: int = 0,
               scale: Optional[float] = None, out: Optional[torch.Tensor] = None,
               lse: Optional[torch.Tensor] = None, num_splits: int = 0, kernel: str = "auto",
               workspace: Optional[torch.Tensor] = None, max_seq_len: Optional[int] = None,
               stream=None, want_lse: bool = True,
               wait_limit_us: int = 0) -> Tuple[torch.Tensor, Optional[torch.Tensor]]:
    """DFlash block attention (include/dflash_attn.h, dflash_block_attn).

    q [B*T, Hq, D]; k_cache, v_cache [num_pages, page_size, Hkv, D] (head_dim
    contiguous); page_table int32 [B, max_pages]; seq_lens int32 [B] on the
    device. Returns (out [B*T, Hq, D] in q's dtype, lse fp32 [B*T, Hq] or None).
    wait_limit_us bounds every device-side wait of the tensor-core kernels (0 = 2 s).
    """
    lib = load_library()
    _check_attn_inputs(q, k_cache, v_cache, page_table, seq_lens, block_len, out, lse)
    dims = make_dims(q, k_cache, page_table, block_len, max_seq_len)
    if scale is None:
        scale = 1.0 / math.sqrt(q.shape[2])
    if out is None:
        out = torch.empty_like(q)
    if lse is None and want_lse:
        lse = torch.empty(q.shape[0], q.shape[1], dtype=torch.float32, device=q.device)
    splits = plan_splits(dims, block_len, window, num_splits, kernel)
    need = workspace_bytes(dims, block_len, splits)
    if workspace is None:
        workspace = workspace_for(q.device, need)
    opts = Opts()
    opts.num_splits = num_splits  # the caller's request: the library re-plans the same count (0 = auto)
    opts.kernel = KERNELS[kernel]
    opts.workspace = workspace.data_ptr()
    opts.workspace_bytes = workspace.numel() * workspace.element_size()
    opts.stream = _stream_handle(stream)
    opts.wait_limit_us = int(wait_limit_us)
    st = lib.dflash_block_attn(q.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(), page_table.data_ptr(),
                               seq_lens.data_ptr(), ctypes.byref(dims), int(block_len), int(bool(causal)),
                               int(window), float(scale), out.data_ptr(),
                               lse.data_ptr() if lse is not None else None, ctypes.byref(opts))
    _check(st)
    return out, lse


def block_attn_noalloc(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor, page_table: torch.Tensor,
                       seq_lens: torch.Tensor, block_len: int, causal: bool = False, window: int = 0,
                       scale: Optional[float] = None, out: Optional[torch.Tensor] = None,
                       lse: Optional[torch.Tensor] = None, num_splits: int = 0, kernel: str = "auto",
                       max_seq_len: Optional[int] = None, stream=None,
                       want_lse: bool = True) -> Tuple[torch.Tensor, Optional[torch.Tensor]]:
    """dflash_block_attn_noalloc: the same attention with the library's own fixed
    scratch instead of a workspace, for callers that cannot allocate device memory.
    The library call allocates nothing; for convenience this wrapper allocates out
    (and lse, when want_lse) with torch when they are not given, so a caller that
    must not allocate passes both."""
    lib = load_library()
    _check_attn_inputs(q, k_cache, v_cache, page_table, seq_lens, block_len, out, lse)
    dims = make_dims(q, k_cache, page_table, block_len, max_seq_len)
    if scale is None:
        scale = 1.0 / math.sqrt(q.shape[2])
    if out is None:
        out = torch.empty_like(q)
    if lse is None and want_lse:
        lse = torch.empty(q.shape[0], q.shape[1], dtype=torch.float32, device=q.device)
    st = lib.dflash_block_attn_noalloc(q.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(), page_table.data_ptr(),
                                       seq_lens.data_ptr(), ctypes.byref(dims), int(block_len), int(bool(causal)),
                                       int(window), float(scale), out.data_ptr(),
                                       lse.data_ptr() if lse is not None else None, int(num_splits),
                                       KERNELS[kernel], _stream_handle(stream))
    _check(st)
    return out, lse


def split_combine(partial_out: torch.Tensor, partial_lse: torch.Tensor, out_dtype=torch.float32,
                  out: Optional[torch.Tensor] = None, lse: Optional[torch.Tensor] = None,
                  stream=None) -> Tuple[torch.Tensor, torch.Tensor]:
    """Log-sum-exp combine (dflash_split_combine): partial_out fp32 [S, rows..., D],
    partial_lse fp32 [S, rows...] -> out [rows..., D] (out_dtype), lse [rows...]."""
    lib = load_library()
    if partial_out.dtype != torch.float32 or partial_lse.dtype != torch.float32:
        raise TypeError("partials must be fp32")
    if not (partial_out.is_contiguous() and partial_lse.is_contiguous()):
        raise ValueError("partials must be contiguous")
    S, D = partial_out.shape[0], partial_out.shape[-1]
    inner = tuple(partial_out.shape[1:-1])
    rows = int(math.prod(inner)) if inner else 1
    if out is None:
        out = torch.empty(inner + (D,), dtype=out_dtype, device=partial_out.device)
    if lse is None:
        lse = torch.empty(inner, dtype=torch.float32, device=partial_out.device)
    st = lib.dflash_split_combine(partial_out.data_ptr(), partial_lse.data_ptr(), S, rows, D,
                                  _dtype_code(out), out.data_ptr(), lse.data_ptr(), _stream_handle(stream))
    _check(st)
    return out, lse


_accept_ws = {}


def accept_workspace_bytes(batch: int, block_len: int) -> int:
    n = load_library().dflash_accept_workspace_bytes(int(batch), int(block_len))
    if n == 0:
        raise DflashError(1, "invalid batch/block_len for the acceptance workspace")
    return n


def accept_prefix(logits: torch.Tensor, draft: torch.Tensor, workspace: Optional[torch.Tensor] = None,
                  accepted: Optional[torch.Tensor] = None, next_token: Optional[torch.Tensor] = None,
                  target_argmax: Optional[torch.Tensor] = None, want_argmax: bool = True,
                  stream=None) -> Tuple[torch.Tensor, torch.Tensor, Optional[torch.Tensor]]:
    """Longest-prefix acceptance (dflash_accept_prefix): logits [B, T, V] bf16/fp32 (last
    dim contiguous), draft int32 [B, T-1] -> (accepted_len [B], next_token [B], target
    argmax [B, T] or None), int32 on the device. Without a workspace the call uses one cached
    per device: calls that may overlap (different streams) must each pass their own."""
    lib = load_library()
    if logits.dim() != 3 or logits.stride(2) != 1 or logits.stride(0) != logits.shape[1] * logits.stride(1):
        raise ValueError("logits must be [B, T, V] with contiguous rows of a common stride")
    B, T, V = logits.shape
    if draft.dtype != torch.int32 or tuple(draft.shape) != (B, T - 1) or not draft.is_contiguous():
        raise ValueError("draft must be a contiguous int32 [B, T-1] tensor")
    dev = logits.device
    if workspace is None:
        need = accept_workspace_bytes(B, T)
        key = (dev.type, dev.index)
        workspace = _accept_ws.get(key)
        if workspace is None or workspace.numel() < need:
            workspace = torch.zeros(max(need, 1 << 16), dtype=torch.uint8, device=dev)
            _accept_ws[key] = workspace
    if accepted is None:
        accepted = torch.empty(B, dtype=torch.int32, device=dev)
    if next_token is None:
        next_token = torch.empty(B, dtype=torch.int32, device=dev)
    if target_argmax is None and want_argmax:
        target_argmax = torch.empty(B, T, dtype=torch.int32, device=dev)
    st = lib.dflash_accept_prefix(logits.data_ptr(), _dtype_code(logits), B, T, V, logits.stride(1),
                                  draft.data_ptr() if draft.numel() else None, accepted.data_ptr(),
                                  next_token.data_ptr(),
                                  target_argmax.data_ptr() if target_argmax is not None else None,
                                  workspace.data_ptr(), workspace.numel() * workspace.element_size(),
                                  _stream_handle(stream))
    _check(st)
    return accepted, next_token, target_argmax


_proj_ws = {}


def project_kv(hidden: torch.Tensor, w_k: torch.Tensor, w_v: torch.Tensor, slot_mapping: torch.Tensor,
               k_cache: torch.Tensor, v_cache: torch.Tensor, device_error: Optional[torch.Tensor] = None,
               workspace: Optional[torch.Tensor] = None, split: bool = True, stream=None) -> None:
    """Context K/V projection into the paged cache (dflash_project_kv): hidden [L, H] bf16
    (rows of any stride, last dim contiguous), w_k / w_v [Hkv*D, H] bf16 contiguous,
    slot_mapping int32 [L] (page * page_size + position; < 0 skips the token), caches
    [num_pages, page_size, Hkv, D] bf16 (d contiguous, same strides). device_error: an
    optional int32/uint32 device word that receives DEVERR_* bits. With split (the default)
    the last round's tiles are split in two through a workspace (a zeroed one cached per
    device when none is given: calls that may overlap must each pass their own);
    split=False computes every tile whole."""
    lib = load_library()
    if split and workspace is None and hidden.numel():
        dev = hidden.device
        key = (dev.type, dev.index)
        workspace = _proj_ws.get(key)
        if workspace is None:
            workspace = torch.zeros(lib.dflash_project_kv_workspace_bytes(), dtype=torch.uint8, device=dev)
            _proj_ws[key] = workspace
    if not split:
        workspace = None
    if hidden.dim() != 2 or hidden.stride(1) != 1:
        raise ValueError("hidden must be [L, H] with a contiguous last dimension")
    if k_cache.dim() != 4 or k_cache.shape != v_cache.shape or k_cache.stride() != v_cache.stride():
        raise ValueError("k_cache and v_cache must be [num_pages, page_size, Hkv, D] of the same shape and strides")
    if k_cache.stride(3) != 1:
        raise ValueError("the caches' head_dim must be contiguous")
    L, H = hidden.shape
    N = k_cache.shape[2] * k_cache.shape[3]
    for name, w in (("w_k", w_k), ("w_v", w_v)):
        if tuple(w.shape) != (N, H) or not w.is_contiguous():
            raise ValueError(f"{name} must be a contiguous [{N}, {H}] tensor")
    if slot_mapping.dtype != torch.int32 or tuple(slot_mapping.shape) != (L,) or not slot_mapping.is_contiguous():
        raise ValueError("slot_mapping must be a contiguous int32 [L] tensor")
    for t in (hidden, w_k, w_v, k_cache, v_cache):
        if t.dtype != torch.bfloat16:
            raise TypeError("hidden, weights and caches must be bf16")
    d = Dims()
    d.batch = 1
    d.num_q_heads = k_cache.shape[2]
    d.num_kv_heads = k_cache.shape[2]
    d.head_dim = k_cache.shape[3]
    d.page_size = k_cache.shape[1]
    d.num_pages = k_cache.shape[0]
    d.max_pages = 1
    d.max_seq_len = 0
    d.dtype = BF16
    d.kv_stride_page, d.kv_stride_slot, d.kv_stride_head = (int(s) for s in k_cache.stride()[:3])
    st = lib.dflash_project_kv(hidden.data_ptr() if L else None, L, H, hidden.stride(0) if L else H,
                               w_k.data_ptr(), w_v.data_ptr(), slot_mapping.data_ptr() if L else None,
                               k_cache.data_ptr(), v_cache.data_ptr(), ctypes.byref(d),
                               device_error.data_ptr() if device_error is not None else None,
                               workspace.data_ptr() if workspace is not None else None,
                               workspace.numel() * workspace.element_size() if workspace is not None else 0,
                               _stream_handle(stream))
    _check(st)


def grouped_conv(x: torch.Tensor, base: torch.Tensor, delta: torch.Tensor, out: Optional[torch.Tensor] = None,
                 stream=None) -> torch.Tensor:
    """DFlash2 grouped dynamic depthwise convolution (dflash_grouped_conv): x [B, T, C] bf16/fp32,
    base float32 [taps, C], delta float32 [B, T, taps, G] -> out [B, T, C] of x's dtype."""
    lib = load_library()
    if x.dim() != 3 or not x.is_contiguous():
        raise ValueError("x must be a contiguous [B, T, C] tensor")
    B, T, C = x.shape
    if base.dim() != 2 or base.shape[1] != C or base.dtype != torch.float32 or not base.is_contiguous():
        raise ValueError("base must be a contiguous float32 [taps, C] tensor")
    taps = base.shape[0]
    if (delta.dim() != 4 or tuple(delta.shape[:3]) != (B, T, taps) or delta.dtype != torch.float32
            or not delta.is_contiguous()):
        raise ValueError("delta must be a contiguous float32 [B, T, taps, G] tensor")
    if out is None:
        out = torch.empty_like(x)
    elif out.shape != x.shape or out.dtype != x.dtype or not out.is_contiguous():
        raise ValueError("out must be a contiguous tensor of x's shape and dtype")
    st = lib.dflash_grouped_conv(x.data_ptr(), out.data_ptr(), _dtype_code(x), B, T, C, taps, delta.shape[3],
                                 base.data_ptr(), delta.data_ptr(), _stream_handle(stream))
    _check(st)
    return out


def selector_workspace_bytes(num_requests: int, num_slots: int, num_candidates: int) -> int:
    n = load_library().dflash_selector_workspace_bytes(int(num_requests), int(num_slots), int(num_candidates))
    if n == 0:
        raise DflashError(ERR_INVALID_ARG, "invalid sizes for the selector workspace")
    return n


_sel_ws = {}


def selector_walk(pred_codebook: torch.Tensor, succ_codebook: torch.Tensor, proj: torch.Tensor,
                  candidates: torch.Tensor, unary: torch.Tensor, anchor: torch.Tensor, temperature: float = 0.0,
                  uniforms: Optional[torch.Tensor] = None, workspace: Optional[torch.Tensor] = None,
                  tokens: Optional[torch.Tensor] = None, chosen: Optional[torch.Tensor] = None,
                  path_scores: Optional[torch.Tensor] = None, q: Optional[torch.Tensor] = None,
                  want_scores: bool = True, device_error: Optional[torch.Tensor] = None, stream=None):
    """DFlash2 candidate-selector walk (dflash_selector_walk). Codebooks bf16 [V, E]; proj float32
    [R, S, E]; candidates int32 [R, S, K]; unary float32 [R, S, K]; anchor int32 [R]; uniforms
    float32 [R, S] when temperature > 0. Returns (tokens [R, S], chosen [R, S], path_scores
    [R, S, K] or None, q [R, S, K] or None). Without a workspace the call uses one cached per
    device: calls that may overlap (different streams) must each pass their own."""
    lib = load_library()
    V, E = pred_codebook.shape
    R, S, K = candidates.shape
    for name, t, dt in (("pred_codebook", pred_codebook, torch.bfloat16), ("succ_codebook", succ_codebook, torch.bfloat16),
                        ("proj", proj, torch.float32), ("candidates", candidates, torch.int32),
                        ("unary", unary, torch.float32), ("anchor", anchor, torch.int32)):
        if t.dtype != dt or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous {dt} tensor")
    if tuple(succ_codebook.shape) != (V, E) or tuple(proj.shape) != (R, S, E) or tuple(unary.shape) != (R, S, K) \
            or tuple(anchor.shape) != (R,):
        raise ValueError("inconsistent selector shapes")
    dev = candidates.device
    if temperature > 0:
        if uniforms is None or uniforms.dtype != torch.float32 or tuple(uniforms.shape) != (R, S) \
                or not uniforms.is_contiguous():
            raise ValueError("temperature > 0 needs contiguous float32 uniforms [R, S]")
    if workspace is None:
        need = selector_workspace_bytes(R, S, K)
        key = (dev.type, dev.index)
        workspace = _sel_ws.get(key)
        if workspace is None or workspace.numel() < need:
            workspace = torch.zeros(max(need, 1 << 16), dtype=torch.uint8, device=dev)
            _sel_ws[key] = workspace
    if tokens is None:
        tokens = torch.empty((R, S), dtype=torch.int32, device=dev)
    if chosen is None:
        chosen = torch.empty((R, S), dtype=torch.int32, device=dev)
    if path_scores is None and want_scores:
        path_scores = torch.empty((R, S, K), dtype=torch.float32, device=dev)
    if q is None and temperature > 0:
        q = torch.empty((R, S, K), dtype=torch.float32, device=dev)
    st = lib.dflash_selector_walk(pred_codebook.data_ptr(), succ_codebook.data_ptr(), V, E, proj.data_ptr(),
                                  candidates.data_ptr(), unary.data_ptr(), anchor.data_ptr(), R, S, K,
                                  float(temperature), uniforms.data_ptr() if uniforms is not None else None,
                                  tokens.data_ptr(), chosen.data_ptr(),
                                  path_scores.data_ptr() if path_scores is not None else None,
                                  q.data_ptr() if q is not None else None,
                                  device_error.data_ptr() if device_error is not None else None,
                                  workspace.data_ptr(), workspace.numel() * workspace.element_size(),
                                  _stream_handle(stream))
    _check(st)
    return tokens, chosen, path_scores, q


def read_error(workspace: Optional[torch.Tensor] = None, clear: bool = True, stream=None) -> int:
    """The workspace's device error word (DEVERR_* bits); synchronises the stream."""
    lib = load_library()
    if workspace is None:
        if not torch.cuda.is_available():
            return 0
        workspace = _ws_cache.get(("cuda", torch.cuda.current_device()))
        if workspace is None:
            return 0
    word = ctypes.c_uint32(0)
    st = lib.dflash_read_error(workspace.data_ptr(), _stream_handle(stream), ctypes.byref(word), int(bool(clear)))
    if st not in (OK, ERR_DEVICE_CHECK):
        _check(st)
    return int(word.value)


def abi_version() -> int:
    return int(load_library().dflash_abi_version())
