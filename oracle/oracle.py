"""Plain CPU oracle for the paged KV-cache decode path (fp64).

TEST INFRASTRUCTURE.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
bench's CPU-baseline / reference arm import this module.  It shares no code with
the CUDA library and never imports it.

What each function follows:

* ``kv_append`` -- write each new token's K/V row to the cache slot named by
  ``slot_mapping`` (limoncc.com "大语言模型研究15——注意力机制优化之KV缓存" §2:
  compute only the new token's K/V and add it to the cache; zwjcode.cn "KV Cache
  的增量解码" §04 worked example).  A negative slot means padding: skip.
* ``kv_block_copy`` -- copy-on-write of a shared block: the whole block (all KV
  heads, all slots) of ``src`` is copied to ``dst`` (plumephp.com "KV Cache 优化与注
  意力机制加速" §4.3; 0539edu.com "从KV cache共享到批量调度…" §3.2).
* ``slot_of`` -- logical position ``pos`` of a sequence lives in physical block
  ``table[pos // bs]`` at offset ``pos % bs`` (plumephp.com §4.3, get_kv), i.e.
  slot ``table[pos // bs] * bs + pos % bs``.
* ``paged_decode`` / ``split_decode`` / ``prefill`` / ``attend_contiguous`` --
  the fp64 C routines in ``pkv_oracle.c`` (softmax(q K^T * scale) V with the
  GQA head mapping j = floor(i / m)); see that file's header.
* ``kv_cache_bytes`` -- 2 * L * N * H * T * d * b (zwjcode.cn §02; plumephp.com
  §3.2; limoncc.com §2 with H*d = d_model).

Arrays: caches are numpy arrays of raw element bits -- ``float32`` for an fp32
cache, ``uint16`` for bf16 -- shaped [NB][Hkv][bs][d].  Torch tensors are
accepted and converted (bf16 via a 16-bit integer view, no rounding).
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "pkv_oracle.c")
_LIB_DIR = os.path.join(_HERE, "_build")
_LIB = os.path.join(_LIB_DIR, "libpkv_oracle.so")

F32, BF16 = 0, 1


def build(force: bool = False) -> str:
    """Compile the C oracle with gcc (plain IEEE double: no fast-math, no FMA contraction)."""
    if not force and os.path.exists(_LIB) and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC):
        return _LIB
    os.makedirs(_LIB_DIR, exist_ok=True)
    tmp = _LIB + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread", "-ffp-contract=off",
           "-fno-fast-math", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB)
    return _LIB


_lib = None


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        P = ctypes.c_void_p
        lib.oracle_paged_decode.argtypes = [P, P, P, P, P, ctypes.c_int, P, P, ctypes.c_int,
                                            ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                            ctypes.c_int, ctypes.c_long, ctypes.c_double,
                                            ctypes.c_long, ctypes.c_int]
        lib.oracle_paged_decode.restype = ctypes.c_int
        lib.oracle_attend_contiguous.argtypes = [P, P, P, P, P, ctypes.c_long, ctypes.c_int,
                                                 ctypes.c_int, ctypes.c_int, ctypes.c_double]
        lib.oracle_attend_contiguous.restype = None
        lib.oracle_prefill.argtypes = [P, P, P, P, P, ctypes.c_int, P, ctypes.c_int, ctypes.c_int,
                                       ctypes.c_int, ctypes.c_int, ctypes.c_double, ctypes.c_int]
        lib.oracle_prefill.restype = ctypes.c_int
        lib.oracle_paged_attention.argtypes = [P, P, P, P, P, ctypes.c_int, P, P, P, ctypes.c_int,
                                               ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                               ctypes.c_int, ctypes.c_long, ctypes.c_double,
                                               ctypes.c_long, ctypes.c_int]
        lib.oracle_paged_attention.restype = ctypes.c_int
        _lib = lib
    return _lib


# ------------------------------------------------------------------ conversions

def to_numpy(x) -> np.ndarray:
    """numpy view of a host array or CPU torch tensor; bf16 becomes its uint16 bits."""
    if isinstance(x, np.ndarray):
        return x
    import torch  # only for the conversion of test inputs
    if isinstance(x, torch.Tensor):
        x = x.detach().cpu().contiguous()
        if x.dtype == torch.bfloat16:
            return x.view(torch.int16).numpy().view(np.uint16)
        return x.numpy()
    return np.asarray(x)


def _dtype_code(a: np.ndarray) -> int:
    if a.dtype == np.float32:
        return F32
    if a.dtype == np.uint16:
        return BF16
    raise TypeError(f"cache element type must be float32 or bf16 bits (uint16), got {a.dtype}")


def bf16_bits_to_f64(a: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns: they are the top 16 bits of an fp32."""
    return (a.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)


def to_f64(a) -> np.ndarray:
    a = to_numpy(a)
    return bf16_bits_to_f64(a) if a.dtype == np.uint16 else a.astype(np.float64)


def _c(a: np.ndarray, dtype=None) -> np.ndarray:
    return np.ascontiguousarray(a if dtype is None else a.astype(dtype, copy=False))


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


# --------------------------------------------------------------- cache writes

def slot_of(table_row, pos: int, bs: int) -> int:
    """Slot of logical position ``pos``: table[pos // bs] * bs + pos % bs."""
    return int(table_row[pos // bs]) * bs + pos % bs


def kv_append(k_cache, v_cache, k_new, v_new, slot_mapping) -> None:
    """In place: cache[slot // bs, :, slot % bs, :] = new[t] for each token t with slot >= 0.

    k_cache/v_cache [NB][Hkv][bs][d]; k_new/v_new [T][Hkv][d] of the same element type.
    """
    kc, vc = to_numpy(k_cache), to_numpy(v_cache)
    kn, vn = to_numpy(k_new), to_numpy(v_new)
    if kn.dtype != kc.dtype or vn.dtype != vc.dtype:
        raise TypeError("new K/V must have the cache's element type")
    bs = kc.shape[2]
    for t, s in enumerate(to_numpy(slot_mapping).tolist()):
        if s < 0:
            continue
        kc[s // bs, :, s % bs, :] = kn[t]
        vc[s // bs, :, s % bs, :] = vn[t]


def kv_block_copy(k_cache, v_cache, pairs) -> None:
    """In place, in pair order: cache[dst] = cache[src] for every (src, dst) pair."""
    kc, vc = to_numpy(k_cache), to_numpy(v_cache)
    for src, dst in to_numpy(pairs).reshape(-1, 2).tolist():
        kc[dst] = kc[src]
        vc[dst] = vc[src]


def kv_cache_bytes(layers: int, batch: int, heads: int, tokens: int, head_dim: int,
                   elem_bytes: int) -> int:
    """2 * L * N * H * T * d * b: K and V for every layer, sequence, head and token."""
    return 2 * layers * batch * heads * tokens * head_dim * elem_bytes


# ------------------------------------------------------------------- attention

def paged_decode(q, k_cache, v_cache, block_table, context_lens, scale: float,
                 chunk_tokens: int = 0, nthreads: int = 1):
    """softmax(scale * q K^T) V for one query per (sequence, head) over the paged cache.

    q [B][Hq][d] (fp32 values); caches [NB][Hkv][bs][d]; block_table int32
    [B][MBS]; context_lens int32 [B].  ``chunk_tokens`` > 0 computes the same
    result by split-K partials merged by log-sum-exp.  Returns (out [B][Hq][d],
    lse [B][Hq]) in float64.
    """
    qn = _c(to_numpy(q), np.float32)
    kc, vc = _c(to_numpy(k_cache)), _c(to_numpy(v_cache))
    dt = _dtype_code(kc)
    if _dtype_code(vc) != dt:
        raise TypeError("K and V caches differ in element type")
    table = _c(to_numpy(block_table), np.int32)
    lens = _c(to_numpy(context_lens), np.int32)
    B, Hq, d = qn.shape
    NB, Hkv, bs, d2 = kc.shape
    if d2 != d:
        raise ValueError("head_dim mismatch")
    MBS = table.shape[1] if table.ndim == 2 else 0
    out = np.zeros((B, Hq, d), np.float64)
    lse = np.zeros((B, Hq), np.float64)
    rc = _load().oracle_paged_decode(_ptr(out), _ptr(lse), _ptr(qn), _ptr(kc), _ptr(vc), dt,
                                     _ptr(table), _ptr(lens), B, Hq, Hkv, d, bs, MBS, NB,
                                     float(scale), int(chunk_tokens), int(nthreads))
    if rc != 0:
        raise ValueError("oracle: context length or block-table entry out of range")
    return out, lse


def paged_attention(q, k_cache, v_cache, block_table, context_lens, cu_q, scale: float,
                    window: int = 0, nthreads: int = 1):
    """Queries at the end of each cached sequence, causal, optional sliding window.

    Sequence b holds context_lens[b] tokens in the cache (its queries' own K/V
    among them) and owns query rows cu_q[b] .. cu_q[b+1]-1; its i-th of nq queries
    sits at position p = len - nq + i and sees keys lo .. p, lo = max(0, p - window
    + 1) for window > 0, else 0.  q [Tq][Hq][d] (fp32 values); caches
    [NB][Hkv][bs][d]; block_table int32 [B][MBS].  Returns (out [Tq][Hq][d],
    lse [Tq][Hq]) in float64.
    """
    qn = _c(to_numpy(q), np.float32)
    kc, vc = _c(to_numpy(k_cache)), _c(to_numpy(v_cache))
    dt = _dtype_code(kc)
    if _dtype_code(vc) != dt:
        raise TypeError("K and V caches differ in element type")
    table = _c(to_numpy(block_table), np.int32)
    lens = _c(to_numpy(context_lens), np.int32)
    cu = _c(to_numpy(cu_q), np.int32)
    Tq, Hq, d = qn.shape
    NB, Hkv, bs, d2 = kc.shape
    B = lens.shape[0]
    if d2 != d or cu.shape[0] != B + 1 or cu[-1] != Tq:
        raise ValueError("shape mismatch")
    MBS = table.shape[1] if table.ndim == 2 else 0
    out = np.zeros((Tq, Hq, d), np.float64)
    lse = np.zeros((Tq, Hq), np.float64)
    rc = _load().oracle_paged_attention(_ptr(out), _ptr(lse), _ptr(qn), _ptr(kc), _ptr(vc), dt,
                                        _ptr(table), _ptr(lens), _ptr(cu), B, Hq, Hkv, d, bs, MBS,
                                        NB, float(scale), int(window), int(nthreads))
    if rc != 0:
        raise ValueError("oracle: length, query count or block-table entry out of range")
    return out, lse


def attend_contiguous(q, K, V, scale: float):
    """Attention for one sequence without paging.

    q [Hq][d]; K, V [n][Hkv][d] (token-major, as appended); any element type.
    Returns (out [Hq][d], lse [Hq]) in float64.
    """
    qd = _c(to_f64(q))
    Kd = _c(np.transpose(to_f64(K), (1, 0, 2)))
    Vd = _c(np.transpose(to_f64(V), (1, 0, 2)))
    Hq, d = qd.shape
    Hkv, n, _ = Kd.shape
    out = np.zeros((Hq, d), np.float64)
    lse = np.zeros((Hq,), np.float64)
    _load().oracle_attend_contiguous(_ptr(out), _ptr(lse), _ptr(qd), _ptr(Kd), _ptr(Vd), n, Hq,
                                     Hkv, d, float(scale))
    return out, lse


def prefill(q, k, v, cu_seqlens, scale: float, nthreads: int = 1):
    """Varlen causal attention: token t of sequence b attends to keys 0..t of b.

    q [T][Hq][d], k/v [T][Hkv][d] (fp32 or bf16 bits, all the same type);
    cu_seqlens int32 [B+1].  Returns (out [T][Hq][d], lse [T][Hq]) in float64.
    """
    qn, kn, vn = _c(to_numpy(q)), _c(to_numpy(k)), _c(to_numpy(v))
    dt = _dtype_code(qn)
    if _dtype_code(kn) != dt or _dtype_code(vn) != dt:
        raise TypeError("q, k, v must share one element type")
    cu = _c(to_numpy(cu_seqlens), np.int32)
    T, Hq, d = qn.shape
    Hkv = kn.shape[1]
    B = cu.shape[0] - 1
    if B < 0 or (B >= 0 and (cu[0] != 0 or cu[-1] != T)):
        raise ValueError("cu_seqlens must start at 0 and end at the token count")
    out = np.zeros((T, Hq, d), np.float64)
    lse = np.zeros((T, Hq), np.float64)
    rc = _load().oracle_prefill(_ptr(out), _ptr(lse), _ptr(qn), _ptr(kn), _ptr(vn), dt,
                                _ptr(cu), B, Hq, Hkv, d, float(scale), int(nthreads))
    if rc != 0:
        raise ValueError("oracle: cu_seqlens must be non-decreasing")
    return out, lse
