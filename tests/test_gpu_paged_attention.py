"""pkv_paged_attention on the GPU against the fp64 oracle: sliding-window decode on
every decode path, several queries per sequence (verification steps, prefill on top of
a cached prefix), ragged and empty query counts, blocks released outside the window,
and the device errors."""
import math
import os

import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_165_gb300 as pkv
from paged_kv_cache_165_gb300 import _build
from workloads import gen

from helpers import assert_attn_close, dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    _build.build()
    pkv.lib()
    pkv.get_device_error()


def make_case(seed, lens, nqs, hq, hkv, d, bs, dtype, spare=3):
    g = gen.generator(seed)
    per_seq = [gen.blocks_needed(n, bs) for n in lens]
    nb = sum(per_seq) + spare
    table = gen.block_table_from_order(gen.permutation(g, nb), per_seq)
    kc = gen.randn(g, (nb, hkv, bs, d), dtype)
    vc = gen.randn(g, (nb, hkv, bs, d), dtype)
    q = gen.randn(g, (sum(nqs), hq, d), torch.float32)
    cu = torch.tensor(np.concatenate([[0], np.cumsum(nqs)]), dtype=torch.int32)
    return q, kc, vc, table, torch.tensor(lens, dtype=torch.int32), cu


def release_outside_window(kc, vc, table, lens, nqs, window, bs):
    """Poison and unmap (-1) every block that lies wholly before each sequence's first
    visible position: the kernels must never read them."""
    kp, vp, tp = kc.clone(), vc.clone(), table.clone()
    for b, (L, nq) in enumerate(zip(lens, nqs)):
        lo = L - nq - window + 1
        for page in range(max(0, lo) // bs):
            blk = int(table[b, page])
            kp[blk] = float("nan")
            vp[blk] = float("nan")
            tp[b, page] = -1
    return kp, vp, tp


def run(q, kc, vc, table, lens, cu, scale, window, num_splits, one_per_seq):
    Tq, Hq, d = q.shape
    NB, Hkv, bs, _ = kc.shape
    B = lens.numel()
    max_q = int((cu[1:] - cu[:-1]).max()) if B else 0
    out = torch.full((Tq, Hq, d), float("nan"), device="cuda")
    lse = torch.full((Tq, Hq), float("nan"), device="cuda")
    ws = torch.zeros(max(16, pkv.paged_attention_workspace_bytes(B, Tq, max_q, Hq, Hkv, d, bs, table.shape[1],
                                                                   window, num_splits)),
                     dtype=torch.uint8, device="cuda")
    pkv.paged_attention(out, dev(q), dev(kc), dev(vc), dev(table), dev(lens), scale,
                        cu_q=None if one_per_seq else dev(cu), max_q=max_q, window=window, lse=lse,
                        num_splits=num_splits, workspace=ws)
    torch.cuda.synchronize()
    return out, lse


LENS = [1, 15, 16, 17, 100, 0, 257, 1000, 33]


@pytest.mark.parametrize("hq,hkv,d,dtype", [
    (8, 8, 128, torch.bfloat16),     # tensor-core decode, m = 1
    (16, 2, 128, torch.bfloat16),    # tensor-core decode, m = 8
    (64, 1, 128, torch.bfloat16),    # tcgen05 large-group decode
    (32, 2, 64, torch.bfloat16),     # tcgen05 large-group decode, d = 64
    (32, 2, 256, torch.bfloat16),    # large-group mma.sync kernel
    (8, 2, 96, torch.bfloat16),      # CUDA-core path
    (8, 2, 64, torch.float32),       # CUDA-core path, fp32 cache
])
@pytest.mark.parametrize("window", [1, 5, 16, 17, 100, 4096])
def test_sliding_window_decode_on_every_path(hq, hkv, d, dtype, window):
    lens = [max(n, 1) for n in LENS]
    nqs = [1] * len(lens)
    q, kc, vc, table, clens, cu = make_case(hq + d + window, lens, nqs, hq, hkv, d, 16, dtype)
    ref, ref_lse = oracle.paged_attention(q, kc, vc, table, clens, cu, 1 / math.sqrt(d), window)
    kp, vp, tp = release_outside_window(kc, vc, table, lens, nqs, window, 16)
    for s in (1, 3, 0):
        out, lse = run(q, kp, vp, tp, clens, cu, 1 / math.sqrt(d), window, s, one_per_seq=True)
        assert pkv.get_device_error() == 0
        assert_attn_close(out, ref, f"window {window} splits {s} out")
        assert_attn_close(lse, ref_lse, f"window {window} splits {s} lse")


def test_window_zero_equals_paged_decode():
    lens = [300, 17, 1000, 65]
    q, kc, vc, table, clens, cu = make_case(3, lens, [1] * 4, 64, 8, 128, 16, torch.bfloat16)
    out, lse = run(q, kc, vc, table, clens, cu, 0.088, 0, 0, one_per_seq=True)
    ref, ref_lse = oracle.paged_decode(q, kc, vc, table, clens, 0.088)
    assert_attn_close(out, ref, "out")
    assert_attn_close(lse, ref_lse, "lse")


@pytest.mark.parametrize("hq,hkv,d,dtype,bs", [
    (16, 2, 128, torch.bfloat16, 16), (8, 8, 64, torch.bfloat16, 32),
    (64, 1, 128, torch.bfloat16, 16), (8, 2, 40, torch.float32, 8),
])
@pytest.mark.parametrize("window", [0, 7, 64])
def test_several_queries_per_sequence(hq, hkv, d, dtype, bs, window):
    # ragged query counts, a sequence with none, one whose queries are all its tokens
    lens = [50, 300, 17, 9, 700, 64]
    nqs = [4, 1, 0, 9, 33, 5]
    q, kc, vc, table, clens, cu = make_case(hq * 3 + window, lens, nqs, hq, hkv, d, bs, dtype)
    scale = 1 / math.sqrt(d)
    ref, ref_lse = oracle.paged_attention(q, kc, vc, table, clens, cu, scale, window)
    if window:
        kc, vc, table = release_outside_window(kc, vc, table, lens, nqs, window, bs)
    for s in (1, 2, 0):
        out, lse = run(q, kc, vc, table, clens, cu, scale, window, s, one_per_seq=False)
        assert pkv.get_device_error() == 0
        assert_attn_close(out, ref, f"splits {s} out")
        assert_attn_close(lse, ref_lse, f"splits {s} lse")


def test_prefill_on_top_of_a_cached_prefix_equals_full_prefill():
    # the new tokens' rows of a prefill over prefix + new tokens (zwjcode.cn §07)
    P, N, hq, hkv, d, bs = 200, 56, 8, 2, 64, 16
    L = P + N
    g = gen.generator(31)
    qkv = [gen.randn(g, (L, h, d), torch.bfloat16) for h in (hq, hkv, hkv)]
    nb = gen.blocks_needed(L, bs) + 1
    table = gen.block_table_from_order(gen.permutation(g, nb), [gen.blocks_needed(L, bs)])
    kc = torch.zeros((nb, hkv, bs, d), dtype=torch.bfloat16, device="cuda")
    vc = torch.zeros_like(kc)
    slots = torch.tensor([oracle.slot_of(table[0], t, bs) for t in range(L)], device="cuda")
    pkv.kv_append(qkv[1].cuda(), qkv[2].cuda(), kc, vc, slots)
    full, full_lse = oracle.prefill(qkv[0], qkv[1], qkv[2], np.array([0, L], np.int32), 0.125)
    q_new = qkv[0][P:].float()
    out, lse = run(q_new, kc.cpu(), vc.cpu(), table, torch.tensor([L], dtype=torch.int32),
                   torch.tensor([0, N], dtype=torch.int32), 0.125, 0, 0, one_per_seq=False)
    assert_attn_close(out, full[P:], "new rows")
    assert_attn_close(lse, full_lse[P:], "new rows lse")


def poison_tails(kc, vc, table, lens, bs):
    """NaN / Inf in every slot past each sequence's length and in unused blocks."""
    kp, vp = kc.clone(), vc.clone()
    used = set()
    for b, n in enumerate(lens):
        for pos in range(n, gen.blocks_needed(n, bs) * bs):
            s = oracle.slot_of(table[b], pos, bs)
            kp[s // bs, :, s % bs] = float("nan")
            vp[s // bs, :, s % bs] = float("inf")
        used.update(int(x) for x in table[b, :gen.blocks_needed(n, bs)])
    for blk in range(kc.shape[0]):
        if blk not in used:
            kp[blk] = float("nan")
            vp[blk] = float("nan")
    return kp, vp


# many query rows per sequence (at least 64 in one sequence): the chunked-prefill kernel,
# 128 rows of one head per block over all of the sequence's keys
@pytest.mark.parametrize("hq,hkv,d,bs", [(16, 2, 128, 16), (8, 8, 64, 32), (64, 1, 128, 16), (32, 4, 64, 16),
                                         (8, 2, 128, 32)])
def test_chunked_prefill_kernel_ragged_rows(hq, hkv, d, bs):
    # a prefix plus 200 new rows (two row tiles), rows that are all of a sequence's tokens
    # (64, 129: no prefix), a single row, 300 rows over a 700-token prefix, 5 of 5
    lens = [300, 64, 1000, 129, 1000, 5]
    nqs = [200, 64, 1, 129, 300, 5]
    q, kc, vc, table, clens, cu = make_case(500 + hq + d + bs, lens, nqs, hq, hkv, d, bs, torch.bfloat16)
    kc, vc = poison_tails(kc, vc, table, lens, bs)
    B, Tq, max_q = len(lens), sum(nqs), max(nqs)
    assert pkv.paged_attention_kernel_launches(B, Tq, max_q, hq, hkv, d, bs, table.shape[1], kc.shape[0],
                                               torch.bfloat16, 0, 0) == 1
    assert pkv.paged_attention_workspace_bytes(B, Tq, max_q, hq, hkv, d, bs, table.shape[1], 0, 0) >= 0
    scale = 1 / math.sqrt(d)
    ref, ref_lse = oracle.paged_attention(q, kc, vc, table, clens, cu, scale)
    assert np.isfinite(ref).all()
    out, lse = run(q, kc, vc, table, clens, cu, scale, 0, 0, one_per_seq=False)
    assert pkv.get_device_error() == 0
    assert_attn_close(out, ref, "chunked prefill out")
    assert_attn_close(lse, ref_lse, "chunked prefill lse")


def test_chunked_prefill_kernel_equals_full_prefill_of_prefix_and_chunk():
    # the new rows of a prefill over prefix + chunk (zwjcode.cn §07), 200 rows over 300
    P, N, hq, hkv, d, bs = 300, 200, 8, 2, 128, 16
    L = P + N
    g = gen.generator(37)
    qkv = [gen.randn(g, (L, h, d), torch.bfloat16) for h in (hq, hkv, hkv)]
    nb = gen.blocks_needed(L, bs) + 1
    table = gen.block_table_from_order(gen.permutation(g, nb), [gen.blocks_needed(L, bs)])
    kc = torch.zeros((nb, hkv, bs, d), dtype=torch.bfloat16, device="cuda")
    vc = torch.zeros_like(kc)
    slots = torch.tensor([oracle.slot_of(table[0], t, bs) for t in range(L)], device="cuda")
    pkv.kv_append(qkv[1].cuda(), qkv[2].cuda(), kc, vc, slots)
    full, full_lse = oracle.prefill(qkv[0], qkv[1], qkv[2], np.array([0, L], np.int32), 1 / math.sqrt(d))
    out, lse = run(qkv[0][P:].float(), kc.cpu(), vc.cpu(), table, torch.tensor([L], dtype=torch.int32),
                   torch.tensor([0, N], dtype=torch.int32), 1 / math.sqrt(d), 0, 0, one_per_seq=False)
    assert pkv.get_device_error() == 0
    assert_attn_close(out, full[P:], "new rows")
    assert_attn_close(lse, full_lse[P:], "new rows lse")


def test_chunked_prefill_kernel_bad_block_id_reads_zeros():
    lens, nqs = [400, 200], [100, 70]
    q, kc, vc, table, clens, cu = make_case(41, lens, nqs, 16, 2, 128, 16, torch.bfloat16)
    bad = table.clone()
    bad[0, 3] = kc.shape[0] + 5                       # outside the cache: read as a zero page
    kz, vz = kc.clone(), vc.clone()
    zero = int(table[0, 3])
    kz[zero] = 0
    vz[zero] = 0
    out, lse = run(q, kc, vc, bad, clens, cu, 0.09, 0, 0, one_per_seq=False)
    assert pkv.get_device_error() & pkv.DEVERR["block"]
    ref, ref_lse = oracle.paged_attention(q, kz, vz, table, clens, cu, 0.09)
    assert_attn_close(out, ref, "bad block out")
    assert_attn_close(lse, ref_lse, "bad block lse")


def test_query_count_above_length_raises_cu_seqlens_error():
    lens = [5, 40]
    q, kc, vc, table, clens, cu = make_case(9, lens, [2, 3], 8, 2, 64, 16, torch.bfloat16)
    bad = torch.tensor([0, 2, 5], dtype=torch.int32)
    clens_bad = torch.tensor([1, 40], dtype=torch.int32)        # 2 queries, 1 token
    out, lse = run(q, kc, vc, table, clens_bad, bad, 0.1, 0, 1, one_per_seq=False)
    assert pkv.get_device_error() & pkv.DEVERR["cu_seqlens"]
    assert torch.all(out[:2] == 0) and torch.all(torch.isneginf(lse[:2]))
    ref, _ = oracle.paged_attention(q[2:], kc, vc, table[1:], clens_bad[1:], torch.tensor([0, 3], dtype=torch.int32), 0.1)
    assert_attn_close(out[2:], ref, "valid sequence")


def test_prefix_chunk_prefill_at_full_size():
    # the benched shape: 8 sequences with 4096 cached tokens each append a 512-token chunk
    # and attend it causally (bottom-right), 64 q / 8 kv heads, d 128, in the launch
    # configuration the bench uses
    P, N, B, hq, hkv, d, bs = 4096, 512, 8, 64, 8, 128, 16
    lens, nqs = [P + N] * B, [N] * B
    q, kc, vc, table, clens, cu = make_case(61, lens, nqs, hq, hkv, d, bs, torch.bfloat16, spare=1)
    scale = 1 / math.sqrt(d)
    out, lse = run(q, kc, vc, table, clens, cu, scale, 0, 0, one_per_seq=False)
    assert pkv.get_device_error() == 0
    # every row of every sequence (about 0.6 TFLOP of fp64 oracle work)
    ref, ref_lse = oracle.paged_attention(q, kc, vc, table, clens, cu, scale, nthreads=os.cpu_count() or 1)
    assert_attn_close(out, ref, "chunk out")
    assert_attn_close(lse, ref_lse, "chunk lse")
