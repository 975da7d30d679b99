"""GB300 (sm_103a) paged KV-cache attention.

The compute lives in libpkv.so (C ABI: include/pkv.h).  This package holds the
thin ctypes binding with the ABI's names, the host-side block manager, and the
build step.  Importing it does not load the library; the first call does, and
raises if the library was not built.
"""
from ._binding import (  # noqa: F401
    DEVERR,
    PKV_BF16,
    PKV_F32,
    PKV_FP8_E4M3,
    PkvError,
    decode_kernel_launches,
    decode_step,
    decode_step_kernel_launches,
    decode_step_shared_prefix,
    decode_step_shared_prefix_kernel_launches,
    decode_step_shared_prefix_workspace_bytes,
    decode_step_fp8,
    decode_step_fp8_kernel_launches,
    decode_workspace_bytes,
    get_device_error,
    header_functions,
    kv_append,
    kv_append_fp8,
    kv_block_copy,
    lib,
    library_path,
    paged_attention,
    paged_attention_kernel_launches,
    paged_attention_workspace_bytes,
    paged_decode_attention,
    paged_decode_attention_fp8,
    paged_decode_attention_noalloc,
    prefill_attention,
    selftest_bounded_wait,
)
from .blocks import BlockManager, OutOfBlocks, PrefixGroups  # noqa: F401


def build(force: bool = False) -> str:
    """Compile libpkv.so for sm_103a in-tree (nvcc) and return its path."""
    from . import _build
    return _build.build(force=force)
