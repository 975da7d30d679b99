"""ctypes binding of libpkv.so (the C ABI in include/pkv.h).

Argument marshalling only: each function checks that the torch tensors it is
given have the device, dtype, contiguity and shapes the C call expects, then
passes raw pointers, sizes and the current CUDA stream.  All computation runs in
the library's kernels; there is no fallback when the library is missing.
"""
from __future__ import annotations

import ctypes
import os
import re

import torch

from . import _build

PKV_OK, PKV_ERR_INVALID_ARG, PKV_ERR_UNSUPPORTED, PKV_ERR_WORKSPACE, PKV_ERR_CUDA = range(5)
PKV_F32, PKV_BF16, PKV_FP8_E4M3 = 0, 1, 2

DEVERR = {
    "slot": 1, "block": 2, "len": 4, "cu_seqlens": 8, "pair": 16, "timeout": 32, "layout": 64, "prefix": 128,
}

_DTYPES = {torch.float32: PKV_F32, torch.bfloat16: PKV_BF16, torch.uint8: PKV_FP8_E4M3}


class PkvError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"pkv status {status}: {message}")
        self.status = status


_lib = None


def library_path() -> str:
    return _build.LIB


def lib() -> ctypes.CDLL:
    """The loaded libpkv.so with argument types set.  Raises if it was never built."""
    global _lib
    if _lib is not None:
        return _lib
    path = library_path()
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is missing: build it first with "
                           "paged_kv_cache_165_gb300._build.build() (needs nvcc)")
    L = ctypes.CDLL(path)
    P, I, F, Z = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
    L.pkv_status_string.argtypes = [I]
    L.pkv_status_string.restype = ctypes.c_char_p
    L.pkv_last_error.argtypes = []
    L.pkv_last_error.restype = ctypes.c_char_p
    L.pkv_version.argtypes = []
    L.pkv_version.restype = I
    L.pkv_kv_append.argtypes = [P, P, P, P, I, P, I, I, I, I, I, P]
    L.pkv_kv_append.restype = I
    L.pkv_kv_block_copy.argtypes = [P, P, I, P, I, I, I, I, I, P]
    L.pkv_kv_block_copy.restype = I
    L.pkv_decode_workspace_bytes.argtypes = [I, I, I, I, I, I, I]
    L.pkv_decode_workspace_bytes.restype = Z
    L.pkv_paged_attention_workspace_bytes.argtypes = [I, I, I, I, I, I, I, I, I, I]
    L.pkv_paged_attention_workspace_bytes.restype = Z
    L.pkv_paged_attention.argtypes = [P, P, P, P, P, I, P, P, P, I, I, I, I, I, I, I, I, I, F, I, I, P,
                                      Z, P]
    L.pkv_paged_attention.restype = I
    L.pkv_paged_attention_kernel_launches.argtypes = [I, I, I, I, I, I, I, I, I, I, I, I]
    L.pkv_paged_attention_kernel_launches.restype = I
    L.pkv_kv_append_fp8.argtypes = [P, P, I, P, P, P, P, P, I, I, I, I, I, P]
    L.pkv_kv_append_fp8.restype = I
    L.pkv_paged_decode_attention_fp8.argtypes = [P, P, P, P, P, P, P, P, P, I, I, I, I, I, I, I, F, I, I,
                                                 P, Z, P]
    L.pkv_paged_decode_attention_fp8.restype = I
    L.pkv_decode_kernel_launches.argtypes = [I, I, I, I, I, I, I, I, I]
    L.pkv_decode_kernel_launches.restype = I
    L.pkv_paged_decode_attention.argtypes = [P, P, P, P, P, I, P, P, I, I, I, I, I, I, I, F, I, P,
                                             Z, P]
    L.pkv_paged_decode_attention.restype = I
    L.pkv_decode_step.argtypes = [P, P, P, P, P, P, P, P, I, P, P, I, I, I, I, I, I, I, F, I, P, Z, P]
    L.pkv_decode_step.restype = I
    L.pkv_decode_step_kernel_launches.argtypes = [I, I, I, I, I, I, I, I, I]
    L.pkv_decode_step_kernel_launches.restype = I
    L.pkv_decode_step_fp8.argtypes = [P, P, P, P, P, I, P, P, P, P, P, P, P, I, I, I, I, I, I, I, F, I, P, Z, P]
    L.pkv_decode_step_fp8.restype = I
    L.pkv_decode_step_fp8_kernel_launches.argtypes = [I, I, I, I, I, I, I, I, I]
    L.pkv_decode_step_fp8_kernel_launches.restype = I
    L.pkv_paged_decode_attention_noalloc.argtypes = [P, P, P, P, P, I, P, P, I, I, I, I, I, I, I,
                                                     F, I, P]
    L.pkv_paged_decode_attention_noalloc.restype = I
    L.pkv_decode_step_shared_prefix.argtypes = [P, P, P, P, P, P, P, P, I, P, P, P, P, P, I, I, I, I, I, I, I, I,
                                                I, I, I, F, I, P, Z, P]
    L.pkv_decode_step_shared_prefix.restype = I
    L.pkv_decode_step_shared_prefix_workspace_bytes.argtypes = [I] * 11
    L.pkv_decode_step_shared_prefix_workspace_bytes.restype = Z
    L.pkv_decode_step_shared_prefix_kernel_launches.argtypes = [I] * 13
    L.pkv_decode_step_shared_prefix_kernel_launches.restype = I
    L.pkv_selftest_bounded_wait.argtypes = [ctypes.c_ulonglong, I, I, P, P]
    L.pkv_selftest_bounded_wait.restype = I
    L.pkv_prefill_attention.argtypes = [P, P, P, P, P, I, P, I, I, I, I, I, I, F, P, P, P, I, I, P]
    L.pkv_prefill_attention.restype = I
    L.pkv_get_device_error.argtypes = [ctypes.POINTER(I), P]
    L.pkv_get_device_error.restype = I
    _lib = L
    return L


def header_functions() -> list:
    """Names of the functions include/pkv.h declares."""
    with open(os.path.join(_build.INCLUDE, "pkv.h")) as f:
        text = f.read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(pkv_[a-z_0-9]+)\s*\(", text)))


# ------------------------------------------------------------------ helpers

def _check(status: int) -> None:
    if status != PKV_OK:
        raise PkvError(status, lib().pkv_last_error().decode(errors="replace"))


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    if isinstance(stream, torch.cuda.Stream):
        return ctypes.c_void_p(stream.cuda_stream)
    return ctypes.c_void_p(int(stream))


def _ptr(t) -> ctypes.c_void_p:
    return ctypes.c_void_p(0 if t is None else t.data_ptr())


def _cuda(name, t, dtype=None):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.device.type != "cuda":
        raise ValueError(f"{name} must be on a CUDA device, got {t.device}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    return t


def _dtype(t) -> int:
    if t.dtype not in _DTYPES:
        raise TypeError(f"unsupported element type {t.dtype} (fp32, bf16 or uint8 E4M3 codes)")
    return _DTYPES[t.dtype]


# --------------------------------------------------------------------- ABI

def kv_append(k_new, v_new, k_cache, v_cache, slot_mapping, stream=None) -> None:
    """k_new/v_new [T][Hkv][d] -> cache slots slot_mapping[t] (int64, <0 skipped)."""
    _cuda("k_cache", k_cache)
    dt = _dtype(k_cache)
    _cuda("v_cache", v_cache, k_cache.dtype)
    _cuda("k_new", k_new, k_cache.dtype)
    _cuda("v_new", v_new, k_cache.dtype)
    _cuda("slot_mapping", slot_mapping, torch.int64)
    NB, Hkv, bs, d = k_cache.shape
    T = k_new.shape[0]
    if tuple(k_new.shape) != (T, Hkv, d) or tuple(v_new.shape) != (T, Hkv, d) or slot_mapping.numel() != T:
        raise ValueError("kv_append: shapes do not match [T][Hkv][d] / [T]")
    _check(lib().pkv_kv_append(_ptr(k_new), _ptr(v_new), _ptr(k_cache), _ptr(v_cache), dt,
                               _ptr(slot_mapping), T, Hkv, d, bs, NB, _stream(stream)))


def kv_append_fp8(k_new, v_new, k_codes, v_codes, k_scale, v_scale, slot_mapping, stream=None) -> None:
    """Quantise k_new/v_new [T][Hkv][d] (bf16 or fp32) into E4M3 codes [NB][Hkv][bs][d]
    (uint8) and fp32 row scales [NB][Hkv][bs] at slot_mapping[t] (int64, <0 skipped)."""
    _cuda("k_new", k_new)
    new_dt = _dtype(k_new)
    _cuda("v_new", v_new, k_new.dtype)
    for name, t in (("k_codes", k_codes), ("v_codes", v_codes)):
        _cuda(name, t, torch.uint8)
    for name, t in (("k_scale", k_scale), ("v_scale", v_scale)):
        _cuda(name, t, torch.float32)
    _cuda("slot_mapping", slot_mapping, torch.int64)
    NB, Hkv, bs, d = k_codes.shape
    T = k_new.shape[0]
    if tuple(k_new.shape) != (T, Hkv, d) or tuple(v_new.shape) != (T, Hkv, d) or \
            tuple(v_codes.shape) != (NB, Hkv, bs, d) or tuple(k_scale.shape) != (NB, Hkv, bs) or \
            tuple(v_scale.shape) != (NB, Hkv, bs) or slot_mapping.numel() != T:
        raise ValueError("kv_append_fp8: shapes do not match")
    _check(lib().pkv_kv_append_fp8(_ptr(k_new), _ptr(v_new), new_dt, _ptr(k_codes), _ptr(v_codes),
                                   _ptr(k_scale), _ptr(v_scale), _ptr(slot_mapping), T, Hkv, d, bs, NB,
                                   _stream(stream)))


def paged_decode_attention_fp8(out, q, k_codes, v_codes, k_scale, v_scale, block_table, context_lens,
                               scale, window=0, lse=None, num_splits=0, workspace=None, stream=None) -> None:
    """Decode attention (one query per sequence) over an E4M3 cache with row scales."""
    for name, t in (("k_codes", k_codes), ("v_codes", v_codes)):
        _cuda(name, t, torch.uint8)
    for name, t in (("k_scale", k_scale), ("v_scale", v_scale)):
        _cuda(name, t, torch.float32)
    _cuda("q", q, torch.float32)
    _cuda("out", out, torch.float32)
    _cuda("block_table", block_table, torch.int32)
    _cuda("context_lens", context_lens, torch.int32)
    if lse is not None:
        _cuda("lse", lse, torch.float32)
    NB, Hkv, bs, d = k_codes.shape
    B, Hq, dq = q.shape
    if dq != d or tuple(out.shape) != (B, Hq, d) or block_table.dim() != 2 or \
            block_table.shape[0] != B or context_lens.numel() != B or \
            (lse is not None and lse.numel() != B * Hq):
        raise ValueError("paged_decode_attention_fp8: shapes do not match")
    ws_bytes = 0
    if workspace is not None:
        _cuda("workspace", workspace)
        ws_bytes = workspace.numel() * workspace.element_size()
    _check(lib().pkv_paged_decode_attention_fp8(
        _ptr(out), _ptr(lse), _ptr(q), _ptr(k_codes), _ptr(v_codes), _ptr(k_scale), _ptr(v_scale),
        _ptr(block_table), _ptr(context_lens), B, Hq, Hkv, d, bs, block_table.shape[1], NB, float(scale),
        int(window), int(num_splits), _ptr(workspace), ws_bytes, _stream(stream)))


def kv_block_copy(k_cache, v_cache, pairs, stream=None) -> None:
    """Copy whole blocks: for each (src, dst) row of int32 pairs [n][2]."""
    _cuda("k_cache", k_cache)
    dt = _dtype(k_cache)
    _cuda("v_cache", v_cache, k_cache.dtype)
    _cuda("pairs", pairs, torch.int32)
    NB, Hkv, bs, d = k_cache.shape
    n = pairs.numel() // 2
    _check(lib().pkv_kv_block_copy(_ptr(k_cache), _ptr(v_cache), dt, _ptr(pairs), n, Hkv, d, bs,
                                   NB, _stream(stream)))


def decode_workspace_bytes(B, Hq, Hkv, d, bs, MBS, num_splits=0) -> int:
    return int(lib().pkv_decode_workspace_bytes(B, Hq, Hkv, d, bs, MBS, num_splits))


def decode_kernel_launches(B, Hq, Hkv, d, bs, MBS, NB, dtype, num_splits=0) -> int:
    """Kernels one paged_decode_attention call with these sizes enqueues (-1: rejected)."""
    dt = _DTYPES[dtype]
    return int(lib().pkv_decode_kernel_launches(B, Hq, Hkv, d, bs, MBS, NB, dt, num_splits))


def paged_decode_attention(out, q, k_cache, v_cache, block_table, context_lens, scale, lse=None,
                           num_splits=0, workspace=None, stream=None) -> None:
    """out [B][Hq][d] fp32 = attention of q [B][Hq][d] fp32 over the paged cache."""
    _cuda("k_cache", k_cache)
    dt = _dtype(k_cache)
    _cuda("v_cache", v_cache, k_cache.dtype)
    _cuda("q", q, torch.float32)
    _cuda("out", out, torch.float32)
    _cuda("block_table", block_table, torch.int32)
    _cuda("context_lens", context_lens, torch.int32)
    if lse is not None:
        _cuda("lse", lse, torch.float32)
    NB, Hkv, bs, d = k_cache.shape
    B, Hq, dq = q.shape
    if dq != d or tuple(out.shape) != (B, Hq, d) or block_table.dim() != 2 or \
            block_table.shape[0] != B or context_lens.numel() != B or \
            (lse is not None and lse.numel() != B * Hq):
        raise ValueError("paged_decode_attention: shapes do not match")
    MBS = block_table.shape[1]
    ws_bytes = 0
    if workspace is not None:
        _cuda("workspace", workspace)
        ws_bytes = workspace.numel() * workspace.element_size()
    _check(lib().pkv_paged_decode_attention(
        _ptr(out), _ptr(lse), _ptr(q), _ptr(k_cache), _ptr(v_cache), dt, _ptr(block_table),
        _ptr(context_lens), B, Hq, Hkv, d, bs, MBS, NB, float(scale), int(num_splits),
        _ptr(workspace), ws_bytes, _stream(stream)))


def decode_step(out, q, k_new, v_new, slot_mapping, k_cache, v_cache, block_table, context_lens, scale,
                lse=None, num_splits=0, workspace=None, stream=None) -> None:
    """One decode step: k_new/v_new [B][Hkv][d] (row b = sequence b's new token) go to
    slot_mapping[b] (int64, < 0: none), then out [B][Hq][d] fp32 = attention of q over the
    cache (context_lens count the new tokens).  One launch where the library fuses them."""
    _cuda("k_cache", k_cache)
    dt = _dtype(k_cache)
    _cuda("v_cache", v_cache, k_cache.dtype)
    _cuda("k_new", k_new, k_cache.dtype)
    _cuda("v_new", v_new, k_cache.dtype)
    _cuda("slot_mapping", slot_mapping, torch.int64)
    _cuda("q", q, torch.float32)
    _cuda("out", out, torch.float32)
    _cuda("block_table", block_table, torch.int32)
    _cuda("context_lens", context_lens, torch.int32)
    if lse is not None:
        _cuda("lse", lse, torch.float32)
    NB, Hkv, bs, d = k_cache.shape
    B, Hq, dq = q.shape
    if dq != d or tuple(out.shape) != (B, Hq, d) or tuple(k_new.shape) != (B, Hkv, d) or \
            tuple(v_new.shape) != (B, Hkv, d) or slot_mapping.numel() != B or block_table.dim() != 2 or \
            block_table.shape[0] != B or context_lens.numel() != B or \
            (lse is not None and lse.numel() != B * Hq):
        raise ValueError("decode_step: shapes do not match")
    ws_bytes = 0
    if workspace is not None:
        _cuda("workspace", workspace)
        ws_bytes = workspace.numel() * workspace.element_size()
    _check(lib().pkv_decode_step(
        _ptr(out), _ptr(lse), _ptr(q), _ptr(k_new), _ptr(v_new), _ptr(slot_mapping), _ptr(k_cache),
        _ptr(v_cache), dt, _ptr(block_table), _ptr(context_lens), B, Hq, Hkv, d, bs, block_table.shape[1],
        NB, float(scale), int(num_splits), _ptr(workspace), ws_bytes, _stream(stream)))


def decode_step_shared_prefix(out, q, k_new, v_new, slot_mapping, k_cache, v_cache, block_table, context_lens,
                              scale, groups, lse=None, num_splits=0, workspace=None, stream=None) -> None:
    """decode_step where the batch rows of each group in ``groups`` (a PrefixGroups on the
    device) share a prefix of physical blocks: the same results, with each group's prefix
    read once."""
    for name, t in (("k_cache", k_cache), ("v_cache", v_cache), ("k_new", k_new), ("v_new", v_new)):
        _cuda(name, t, k_cache.dtype)
    dt = _dtype(k_cache)
    _cuda("slot_mapping", slot_mapping, torch.int64)
    _cuda("q", q, torch.float32)
    _cuda("out", out, torch.float32)
    _cuda("block_table", block_table, torch.int32)
    _cuda("context_lens", context_lens, torch.int32)
    for name in ("prefix_tokens", "group_start", "group_seqs"):
        _cuda(name, getattr(groups, name), torch.int32)
    if lse is not None:
        _cuda("lse", lse, torch.float32)
    NB, Hkv, bs, d = k_cache.shape
    B, Hq, dq = q.shape
    if dq != d or tuple(out.shape) != (B, Hq, d) or tuple(k_new.shape) != (B, Hkv, d) or \
            tuple(v_new.shape) != (B, Hkv, d) or slot_mapping.numel() != B or block_table.dim() != 2 or \
            block_table.shape[0] != B or context_lens.numel() != B or groups.prefix_tokens.numel() != B or \
            (lse is not None and lse.numel() != B * Hq):
        raise ValueError("decode_step_shared_prefix: shapes do not match")
    ws_bytes = 0
    if workspace is not None:
        _cuda("workspace", workspace)
        ws_bytes = workspace.numel() * workspace.element_size()
    _check(lib().pkv_decode_step_shared_prefix(
        _ptr(out), _ptr(lse), _ptr(q), _ptr(k_new), _ptr(v_new), _ptr(slot_mapping), _ptr(k_cache),
        _ptr(v_cache), dt, _ptr(block_table), _ptr(context_lens), _ptr(groups.prefix_tokens),
        _ptr(groups.group_start), _ptr(groups.group_seqs), groups.n_groups, groups.n_members,
        groups.max_group_size, groups.max_prefix_tokens, B, Hq, Hkv, d, bs, block_table.shape[1], NB,
        float(scale), int(num_splits), _ptr(workspace), ws_bytes, _stream(stream)))


def decode_step_shared_prefix_workspace_bytes(B, Hq, Hkv, d, bs, MBS, groups, num_splits=0) -> int:
    return int(lib().pkv_decode_step_shared_prefix_workspace_bytes(
        B, Hq, Hkv, d, bs, MBS, int(num_splits), groups.n_groups, groups.n_members, groups.max_group_size,
        groups.max_prefix_tokens))


def decode_step_shared_prefix_kernel_launches(B, Hq, Hkv, d, bs, MBS, NB, dtype, groups, num_splits=0) -> int:
    return int(lib().pkv_decode_step_shared_prefix_kernel_launches(
        B, Hq, Hkv, d, bs, MBS, NB, _DTYPES[dtype], int(num_splits), groups.n_groups, groups.n_members,
        groups.max_group_size, groups.max_prefix_tokens))


def decode_step_kernel_launches(B, Hq, Hkv, d, bs, MBS, NB, dtype, num_splits=0) -> int:
    """Kernels one decode_step call with these sizes enqueues (-1: rejected)."""
    return int(lib().pkv_decode_step_kernel_launches(B, Hq, Hkv, d, bs, MBS, NB, _DTYPES[dtype],
                                                     int(num_splits)))


def paged_attention_workspace_bytes(B, Tq, max_q, Hq, Hkv, d, bs, MBS, window=0, num_splits=0) -> int:
    return int(lib().pkv_paged_attention_workspace_bytes(B, Tq, max_q, Hq, Hkv, d, bs, MBS, window,
                                                         num_splits))


def paged_attention_kernel_launches(B, Tq, max_q, Hq, Hkv, d, bs, MBS, NB, dtype, window=0,
                                    num_splits=0) -> int:
    """Kernels one paged_attention call with these sizes enqueues (-1: rejected)."""
    return int(lib().pkv_paged_attention_kernel_launches(B, Tq, max_q, Hq, Hkv, d, bs, MBS, NB,
                                                         _DTYPES[dtype], window, num_splits))


def paged_attention(out, q, k_cache, v_cache, block_table, context_lens, scale, cu_q=None, max_q=1,
                    window=0, lse=None, num_splits=0, workspace=None, stream=None) -> None:
    """Queries at the end of each cached sequence (causal, optional sliding window).

    q, out [Tq][Hq][d] fp32; cu_q int32 [B+1] (None: one query per sequence)."""
    _cuda("k_cache", k_cache)
    dt = _dtype(k_cache)
    _cuda("v_cache", v_cache, k_cache.dtype)
    _cuda("q", q, torch.float32)
    _cuda("out", out, torch.float32)
    _cuda("block_table", block_table, torch.int32)
    _cuda("context_lens", context_lens, torch.int32)
    if cu_q is not None:
        _cuda("cu_q", cu_q, torch.int32)
    if lse is not None:
        _cuda("lse", lse, torch.float32)
    NB, Hkv, bs, d = k_cache.shape
    Tq, Hq, dq = q.shape
    B = context_lens.numel()
    if dq != d or tuple(out.shape) != (Tq, Hq, d) or block_table.dim() != 2 or \
            block_table.shape[0] != B or (cu_q is not None and cu_q.numel() != B + 1) or \
            (cu_q is None and Tq != B) or (lse is not None and lse.numel() != Tq * Hq):
        raise ValueError("paged_attention: shapes do not match")
    ws_bytes = 0
    if workspace is not None:
        _cuda("workspace", workspace)
        ws_bytes = workspace.numel() * workspace.element_size()
    _check(lib().pkv_paged_attention(
        _ptr(out), _ptr(lse), _ptr(q), _ptr(k_cache), _ptr(v_cache), dt, _ptr(block_table),
        _ptr(context_lens), _ptr(cu_q), B, Tq, int(max_q), Hq, Hkv, d, bs, block_table.shape[1], NB,
        float(scale), int(window), int(num_splits), _ptr(workspace), ws_bytes, _stream(stream)))


def paged_decode_attention_noalloc(out, q, k_cache, v_cache, block_table, context_lens, scale,
                                   lse=None, num_splits=0, stream=None) -> None:
    """paged_decode_attention with the library's built-in split-K scratch (no workspace)."""
    _cuda("k_cache", k_cache)
    dt = _dtype(k_cache)
    _cuda("v_cache", v_cache, k_cache.dtype)
    _cuda("q", q, torch.float32)
    _cuda("out", out, torch.float32)
    _cuda("block_table", block_table, torch.int32)
    _cuda("context_lens", context_lens, torch.int32)
    if lse is not None:
        _cuda("lse", lse, torch.float32)
    NB, Hkv, bs, d = k_cache.shape
    B, Hq, dq = q.shape
    if dq != d or tuple(out.shape) != (B, Hq, d) or block_table.dim() != 2 or \
            block_table.shape[0] != B or context_lens.numel() != B or \
            (lse is not None and lse.numel() != B * Hq):
        raise ValueError("paged_decode_attention_noalloc: shapes do not match")
    _check(lib().pkv_paged_decode_attention_noalloc(
        _ptr(out), _ptr(lse), _ptr(q), _ptr(k_cache), _ptr(v_cache), dt, _ptr(block_table),
        _ptr(context_lens), B, Hq, Hkv, d, bs, block_table.shape[1], NB, float(scale),
        int(num_splits), _stream(stream)))


def prefill_attention(out, q, k, v, cu_seqlens, max_seqlen, scale, lse=None, k_cache=None,
                      v_cache=None, slot_mapping=None, stream=None) -> None:
    """Varlen causal attention of packed q [T][Hq][d], k/v [T][Hkv][d]; optional cache write."""
    _cuda("q", q)
    dt = _dtype(q)
    _cuda("k", k, q.dtype)
    _cuda("v", v, q.dtype)
    _cuda("out", out, torch.float32)
    _cuda("cu_seqlens", cu_seqlens, torch.int32)
    T, Hq, d = q.shape
    Hkv = k.shape[1]
    B = cu_seqlens.numel() - 1
    if tuple(k.shape) != (T, Hkv, d) or tuple(v.shape) != (T, Hkv, d) or tuple(out.shape) != (T, Hq, d):
        raise ValueError("prefill_attention: shapes do not match")
    if lse is not None:
        _cuda("lse", lse, torch.float32)
    bs = NB = 0
    if slot_mapping is not None:
        _cuda("slot_mapping", slot_mapping, torch.int64)
        _cuda("k_cache", k_cache, q.dtype)
        _cuda("v_cache", v_cache, q.dtype)
        NB, _, bs, _ = k_cache.shape
    _check(lib().pkv_prefill_attention(
        _ptr(out), _ptr(lse), _ptr(q), _ptr(k), _ptr(v), dt, _ptr(cu_seqlens), B, T,
        int(max_seqlen), Hq, Hkv, d, float(scale), _ptr(k_cache), _ptr(v_cache),
        _ptr(slot_mapping), bs, NB, _stream(stream)))


def selftest_bounded_wait(limit_ns, blocks, hold_tmem=True, gave_up=None, stream=None) -> None:
    """Run the kernels' bounded-wait failure path on purpose: `blocks` blocks wait on an
    mbarrier no copy completes, give up after limit_ns and tear down (PKV_DEVERR_TIMEOUT).
    gave_up: optional int32 device tensor of one element counting the threads that gave up."""
    if gave_up is not None:
        _cuda("gave_up", gave_up, torch.int32)
    _check(lib().pkv_selftest_bounded_wait(int(limit_ns), int(blocks), 1 if hold_tmem else 0, _ptr(gave_up),
                                           _stream(stream)))


def get_device_error(stream=None) -> int:
    """Synchronise the stream; return and clear the device error bits."""
    code = ctypes.c_int(0)
    _check(lib().pkv_get_device_error(ctypes.byref(code), _stream(stream)))
    return code.value


def decode_step_fp8(out, q, k_new, v_new, slot_mapping, k_codes, v_codes, k_scale, v_scale, block_table,
                    context_lens, scale, lse=None, num_splits=0, workspace=None, stream=None) -> None:
    """decode_step over an E4M3 cache: k_new/v_new [B][Hkv][d] (bf16 or fp32) are quantised
    into codes [NB][Hkv][bs][d] (uint8) and row scales [NB][Hkv][bs] (fp32) at
    slot_mapping[b], then out [B][Hq][d] fp32 = attention of q over the cache."""
    _cuda("k_new", k_new)
    new_dt = _dtype(k_new)
    _cuda("v_new", v_new, k_new.dtype)
    for name, t in (("k_codes", k_codes), ("v_codes", v_codes)):
        _cuda(name, t, torch.uint8)
    for name, t in (("k_scale", k_scale), ("v_scale", v_scale)):
        _cuda(name, t, torch.float32)
    _cuda("slot_mapping", slot_mapping, torch.int64)
    _cuda("q", q, torch.float32)
    _cuda("out", out, torch.float32)
    _cuda("block_table", block_table, torch.int32)
    _cuda("context_lens", context_lens, torch.int32)
    if lse is not None:
        _cuda("lse", lse, torch.float32)
    NB, Hkv, bs, d = k_codes.shape
    B, Hq, dq = q.shape
    if dq != d or tuple(out.shape) != (B, Hq, d) or tuple(k_new.shape) != (B, Hkv, d) or \
            tuple(v_new.shape) != (B, Hkv, d) or tuple(v_codes.shape) != (NB, Hkv, bs, d) or \
            tuple(k_scale.shape) != (NB, Hkv, bs) or tuple(v_scale.shape) != (NB, Hkv, bs) or \
            slot_mapping.numel() != B or block_table.dim() != 2 or block_table.shape[0] != B or \
            context_lens.numel() != B or (lse is not None and lse.numel() != B * Hq):
        raise ValueError("decode_step_fp8: shapes do not match")
    ws_bytes = 0
    if workspace is not None:
        _cuda("workspace", workspace)
        ws_bytes = workspace.numel() * workspace.element_size()
    _check(lib().pkv_decode_step_fp8(
        _ptr(out), _ptr(lse), _ptr(q), _ptr(k_new), _ptr(v_new), new_dt, _ptr(slot_mapping), _ptr(k_codes),
        _ptr(v_codes), _ptr(k_scale), _ptr(v_scale), _ptr(block_table), _ptr(context_lens), B, Hq, Hkv, d, bs,
        block_table.shape[1], NB, float(scale), int(num_splits), _ptr(workspace), ws_bytes, _stream(stream)))


def decode_step_fp8_kernel_launches(B, Hq, Hkv, d, bs, MBS, NB, new_dtype=torch.bfloat16, num_splits=0) -> int:
    """Kernels one decode_step_fp8 call with these sizes enqueues (-1: rejected)."""
    return int(lib().pkv_decode_step_fp8_kernel_launches(B, Hq, Hkv, d, bs, MBS, NB, _DTYPES[new_dtype],
                                                         int(num_splits)))
