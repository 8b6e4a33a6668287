"""DFlash block attention for one GB300 (sm_103a).

The compute lives in libdflash_attn.so (CUDA kernels behind the C ABI of
include/dflash_attn.h); this package is its thin Python binding.
"""
from ._binding import (  # noqa: F401
    BF16,
    DEVERR_PAGE_ID,
    DEVERR_SEQ_LEN,
    DEVERR_TIMEOUT,
    DEVERR_TOKEN_ID,
    EXPORTED,
    FP32,
    KERNELS,
    LIB_PATH,
    DflashError,
    Dims,
    Opts,
    abi_version,
    accept_prefix,
    accept_workspace_bytes,
    project_kv,
    grouped_conv,
    selector_walk,
    selector_workspace_bytes,
    block_attn,
    block_attn_noalloc,
    load_library,
    make_dims,
    plan_info,
    plan_splits,
    read_error,
    split_combine,
    workspace_bytes,
    workspace_for,
)
