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

F32, BF16, F64 = 0, 1, 2


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
    if a.dtype == np.float64:
        return F64
    raise TypeError(f"cache element type must be float32, bf16 bits (uint16) or float64, got {a.dtype}")


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


# ------------------------------------------------------------- FP8 (E4M3) cache
# The pages leave the low-bit format open: zwjcode.cn "KV Cache 的增量解码" §14 (low-bit
# K/V lowers memory and bandwidth; its error reaches every later query, so it must be
# validated) and plumephp.com "KV Cache 优化与注意力机制加速" §2.5 (FP8 attention on
# FP8 tensor cores).  The reading taken here: the OCP FP8 E4M3 format (1 sign, 4
# exponent bits with bias 7, 3 mantissa bits; no infinities, S.1111.111 is NaN; the
# largest finite value is 448) with one fp32 scale per cached row (token slot x KV
# head): scale = amax(row) / 448, code = E4M3(x / scale) rounded to nearest, ties to
# even, saturating at +-448; the cached value is code * scale.  A row of zeros stores
# scale 0 and codes 0.  Both divisions are fp32 operations.

E4M3_MAX = 448.0


def e4m3_decode(codes) -> np.ndarray:
    """float64 value of each E4M3 byte (NaN for S.1111.111)."""
    c = np.asarray(codes, np.uint8).astype(np.int64)
    sign = np.where(c & 0x80, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = c & 0x7
    val = np.where(e == 0, m * 2.0 ** -9, (1.0 + m / 8.0) * np.exp2(e - 7.0))
    val = np.where((e == 0xF) & (m == 0x7), np.nan, val)
    return sign * val


def e4m3_encode(x) -> np.ndarray:
    """E4M3 bytes of float32 values: nearest representable, ties to even, saturating."""
    x = np.asarray(x, np.float32).astype(np.float64)
    a = np.abs(x)
    # binade of a: 2^e <= a < 2^(e+1); normals from 2^-6, below them the spacing 2^-9
    _, ex = np.frexp(np.where(a > 0, a, 1.0))
    e = np.clip(ex - 1, -6, 8)
    quantum = np.exp2(e - 3.0)
    r = np.minimum(np.rint(a / quantum) * quantum, E4M3_MAX)   # rint: half to even
    # encode the rounded magnitude (it may have moved up one binade)
    _, er = np.frexp(np.where(r > 0, r, 1.0))
    er = er - 1
    normal = (r > 0) & (er >= -6)
    e_field = np.where(normal, er + 7, 0)
    m_field = np.where(normal, np.rint((r / np.exp2(er) - 1.0) * 8.0), np.rint(r / 2.0 ** -9))
    code = (e_field.astype(np.int64) << 3) | m_field.astype(np.int64)
    code = code | np.where(np.signbit(x), 0x80, 0)
    return code.astype(np.uint8)


def quantize_rows_e4m3(rows):
    """(codes, scales) of rows [..., d] (any float type, read as float32)."""
    x = to_f64(rows).astype(np.float32)
    amax = np.abs(x).max(axis=-1)
    scale = (amax / np.float32(E4M3_MAX)).astype(np.float32)
    safe = np.where(scale > 0, scale, np.float32(1.0)).astype(np.float32)
    y = (x / safe[..., None]).astype(np.float32)
    codes = np.where(scale[..., None] > 0, e4m3_encode(y), np.uint8(0)).astype(np.uint8)
    return codes, scale


def kv_append_fp8(k_codes, v_codes, k_scale, v_scale, k_new, v_new, slot_mapping) -> None:
    """In place: each new row (token t, KV head h) of K and V quantised into its slot.

    codes uint8 [NB][Hkv][bs][d], scales float32 [NB][Hkv][bs]; k_new/v_new [T][Hkv][d].
    """
    kc, vc, ks, vs = (to_numpy(a) for a in (k_codes, v_codes, k_scale, v_scale))
    kq, kscale = quantize_rows_e4m3(k_new)
    vq, vscale = quantize_rows_e4m3(v_new)
    bs = kc.shape[2]
    for t, s in enumerate(to_numpy(slot_mapping).tolist()):
        if s < 0:
            continue
        kc[s // bs, :, s % bs, :] = kq[t]
        vc[s // bs, :, s % bs, :] = vq[t]
        ks[s // bs, :, s % bs] = kscale[t]
        vs[s // bs, :, s % bs] = vscale[t]


def dequantize_fp8(codes, scales) -> np.ndarray:
    """float64 cache [NB][Hkv][bs][d]: code value * row scale, exact."""
    return e4m3_decode(to_numpy(codes)) * to_numpy(scales).astype(np.float64)[..., None]


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
