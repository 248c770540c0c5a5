"""Masked flash-attention forward for GB300 (sm_103a).

The compute lives in ``libmfa_gb300.so`` (C ABI in ``include/fa.h``); this
package is its thin Python binding.  Build the library with
``masked_flash_attention_gb300.build.build()``.
"""
from ._lib import (  # noqa: F401
    EXPORTS,
    FA_DEBUG_NO_SKIP,
    FA_DEBUG_VALIDATE,
    FA_DEBUG_WITHHOLD,
    FA_OK,
    FaError,
    alloc_workspace,
    describe,
    fa_abi_version,
    fa_bwd,
    fa_bwd_plan,
    fa_check_device_error,
    fa_debug_dump_bytes_of,
    fa_fwd,
    fa_fwd_debug_dump,
    fa_fwd_kvcache,
    fa_fwd_kvcache_plan,
    fa_fwd_noalloc,
    fa_fwd_plan,
    fa_status_string,
    lib,
)
