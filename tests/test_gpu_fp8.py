"""FP8 (E4M3) KV cache on the GPU against the fp64 oracle: quantising appends bit-exact
(codes and row scales), block copies, and decode attention over the dequantised values on
the tensor-core and CUDA-core paths."""
import math

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


@pytest.mark.parametrize("dtype,d", [(torch.bfloat16, 128), (torch.float32, 64), (torch.bfloat16, 40)])
def test_kv_append_fp8_bit_exact(dtype, d):
    nb, hkv, bs, T = 9, 4, 16, 37
    g = gen.generator(d + 3)
    kn = gen.randn(g, (T, hkv, d), dtype) * 3.0
    vn = gen.randn(g, (T, hkv, d), dtype)
    kn[5, 2] = 0.0                                    # a row of zeros: scale 0, codes 0
    vn[7, 1, :3] = -0.0
    slots = torch.tensor(gen.permutation(g, nb * bs)[:T], dtype=torch.int64)
    slots[4] = -1                                     # padding token
    kc = torch.full((nb, hkv, bs, d), 0x5A, dtype=torch.uint8)
    vc = kc.clone()
    ks = torch.full((nb, hkv, bs), -7.0)
    vs = ks.clone()
    gkc, gvc, gks, gvs = dev(kc), dev(vc), dev(ks), dev(vs)
    pkv.kv_append_fp8(dev(kn), dev(vn), gkc, gvc, gks, gvs, dev(slots))
    assert pkv.get_device_error() == 0
    oracle.kv_append_fp8(kc, vc, ks, vs, kn, vn, slots)
    assert torch.equal(gkc.cpu(), kc) and torch.equal(gvc.cpu(), vc)
    assert torch.equal(gks.cpu(), ks) and torch.equal(gvs.cpu(), vs)


def test_kv_append_fp8_out_of_range_slot_is_skipped():
    kc = torch.zeros((2, 1, 16, 64), dtype=torch.uint8, device="cuda")
    vc = kc.clone()
    ks = torch.zeros((2, 1, 16), device="cuda")
    vs = ks.clone()
    new = torch.ones((2, 1, 64), dtype=torch.bfloat16, device="cuda")
    pkv.kv_append_fp8(new, new, kc, vc, ks, vs, torch.tensor([3, 32], device="cuda"))
    assert pkv.get_device_error() & pkv.DEVERR["slot"]
    assert kc[0, 0, 3].eq(0x7E).all() and ks[0, 0, 3].item() == float(np.float32(1.0) / np.float32(448.0))
    assert int(kc.ne(0).sum()) == 64


def test_fp8_block_copy_moves_codes_and_scales():
    nb, hkv, bs, d = 6, 2, 16, 128
    g = gen.generator(8)
    kc = torch.randint(0, 255, (nb, hkv, bs, d), generator=g, dtype=torch.uint8)
    vc = torch.randint(0, 255, (nb, hkv, bs, d), generator=g, dtype=torch.uint8)
    ks, vs = torch.rand((nb, hkv, bs), generator=g), torch.rand((nb, hkv, bs), generator=g)
    pairs = torch.tensor([[1, 4], [2, 0]], dtype=torch.int32)
    gk, gv, gks, gvs = dev(kc), dev(vc), dev(ks), dev(vs)
    pkv.kv_block_copy(gk, gv, dev(pairs))
    pkv.kv_block_copy(gks.view(nb, hkv, bs, 1), gvs.view(nb, hkv, bs, 1), dev(pairs))
    oracle.kv_block_copy(kc, vc, pairs)
    oracle.kv_block_copy(ks, vs, pairs)
    assert torch.equal(gk.cpu(), kc) and torch.equal(gv.cpu(), vc)
    assert torch.equal(gks.cpu(), ks) and torch.equal(gvs.cpu(), vs)


def fp8_case(seed, lens, hq, hkv, d, bs, spare=3, poison=True):
    g = gen.generator(seed)
    per_seq = [gen.blocks_needed(n, bs) for n in lens]
    nb = sum(per_seq) + spare
    table = gen.block_table_from_order(gen.permutation(g, nb), per_seq)
    k = gen.randn(g, (nb, hkv, bs, d), torch.bfloat16)
    v = gen.randn(g, (nb, hkv, bs, d), torch.bfloat16)
    kq, ks = oracle.quantize_rows_e4m3(k)
    vq, vs = oracle.quantize_rows_e4m3(v)
    kq, vq, ks, vs = (torch.from_numpy(np.ascontiguousarray(a)) for a in (kq, vq, ks, vs))
    if poison:   # unwritten slots: NaN codes and scales; never visible
        for b, n in enumerate(lens):
            for pos in range(n, per_seq[b] * bs):
                s = oracle.slot_of(table[b], pos, bs)
                kq[s // bs, :, s % bs] = 0x7F
                vq[s // bs, :, s % bs] = 0x7F
                ks[s // bs, :, s % bs] = float("nan")
                vs[s // bs, :, s % bs] = float("nan")
    q = gen.randn(g, (len(lens), hq, d), torch.float32)
    return q, kq, vq, ks, vs, table, torch.tensor(lens, dtype=torch.int32)


def run_fp8(q, kq, vq, ks, vs, table, lens, scale, window, num_splits):
    B, Hq, d = q.shape
    NB, Hkv, bs, _ = kq.shape
    out = torch.full((B, Hq, d), float("nan"), device="cuda")
    lse = torch.full((B, Hq), float("nan"), device="cuda")
    ws = torch.zeros(max(16, pkv.decode_workspace_bytes(B, Hq, Hkv, d, bs, table.shape[1], num_splits)),
                     dtype=torch.uint8, device="cuda")
    pkv.paged_decode_attention_fp8(out, dev(q), dev(kq), dev(vq), dev(ks), dev(vs), dev(table), dev(lens),
                                   scale, window=window, lse=lse, num_splits=num_splits, workspace=ws)
    torch.cuda.synchronize()
    return out, lse


@pytest.mark.parametrize("hq,hkv,d,bs", [
    (8, 8, 128, 16), (16, 4, 128, 16), (64, 8, 128, 16), (16, 2, 128, 32),   # tensor cores
    (32, 2, 128, 16), (8, 2, 64, 16), (8, 2, 128, 8),                       # CUDA cores
])
@pytest.mark.parametrize("window", [0, 50])
def test_fp8_decode_matches_the_dequantised_oracle(hq, hkv, d, bs, window):
    lens = [1, 15, 16, 17, 100, 0, 257, 1000, 33]
    q, kq, vq, ks, vs, table, clens = fp8_case(hq + d + bs + window, lens, hq, hkv, d, bs)
    kd, vd = oracle.dequantize_fp8(kq, ks), oracle.dequantize_fp8(vq, vs)
    scale = 1 / math.sqrt(d)
    # the empty sequence has no query position: out = 0, lse = -inf; the rest against
    # the oracle's attention over the dequantised cache
    live = [b for b, n in enumerate(lens) if n > 0]
    cu = torch.arange(len(live) + 1, dtype=torch.int32)
    ref, ref_lse = oracle.paged_attention(q[live], kd, vd, table[live], clens[live], cu, scale, window)
    for s in (1, 3, 0):
        out, lse = run_fp8(q, kq, vq, ks, vs, table, clens, scale, window, s)
        assert pkv.get_device_error() == 0
        assert_attn_close(out[live], ref, f"splits {s} out")
        assert_attn_close(lse[live], ref_lse, f"splits {s} lse")
        empty = lens.index(0)
        assert torch.all(out[empty] == 0) and torch.all(torch.isneginf(lse[empty]))


def test_fp8_decode_bad_block_reads_zeros_and_flags():
    lens = [200, 300]
    q, kq, vq, ks, vs, table, clens = fp8_case(5, lens, 16, 2, 128, 16, poison=False)
    bad = table.clone()
    bad[1, 2] = kq.shape[0] + 9
    out, _ = run_fp8(q, kq, vq, ks, vs, bad, clens, 0.1, 0, 0)
    assert pkv.get_device_error() & pkv.DEVERR["block"]
    assert torch.isfinite(out).all()
    kd, vd = oracle.dequantize_fp8(kq, ks), oracle.dequantize_fp8(vq, vs)
    ref, _ = oracle.paged_attention(q[:1], kd, vd, table[:1], clens[:1], torch.tensor([0, 1], dtype=torch.int32), 0.1)
    assert_attn_close(out[:1], ref, "good sequence")


def _fp8_step_case(seed, lens, hq, hkv, d, bs, new_dtype):
    """An FP8 cache, the new token of each sequence (rows of new_dtype) and its slot (the
    last position's); lens count the new token."""
    q, kq, vq, ks, vs, table, clens = fp8_case(seed, lens, hq, hkv, d, bs)
    g = gen.generator(seed + 1)
    k_new = gen.randn(g, (len(lens), hkv, d), new_dtype)
    v_new = gen.randn(g, (len(lens), hkv, d), new_dtype)
    slots = torch.tensor([oracle.slot_of(table[b], n - 1, bs) if n > 0 else -1 for b, n in enumerate(lens)],
                         dtype=torch.int64)
    return [q, kq, vq, ks, vs, table, clens, k_new, v_new, slots]


def _run_fp8_step(case, scale, num_splits, fused=True):
    q, kq, vq, ks, vs, table, clens, k_new, v_new, slots = case
    B, Hq, d = q.shape
    NB, Hkv, bs, _ = kq.shape
    out = torch.full((B, Hq, d), float("nan"), device="cuda")
    lse = torch.full((B, Hq), float("nan"), device="cuda")
    ws = torch.zeros(max(16, pkv.decode_workspace_bytes(B, Hq, Hkv, d, bs, table.shape[1], num_splits)),
                     dtype=torch.uint8, device="cuda")
    g = [dev(t) for t in (kq, vq, ks, vs)]
    if fused:
        pkv.decode_step_fp8(out, dev(q), dev(k_new), dev(v_new), dev(slots), *g, dev(table), dev(clens), scale,
                            lse=lse, num_splits=num_splits, workspace=ws)
    else:
        pkv.kv_append_fp8(dev(k_new), dev(v_new), *g, dev(slots))
        pkv.paged_decode_attention_fp8(out, dev(q), *g, dev(table), dev(clens), scale, lse=lse,
                                       num_splits=num_splits, workspace=ws)
    torch.cuda.synchronize()
    return out, lse, [t.cpu() for t in g]


def _same_bits(a, b):
    """Equal as stored bytes (the unwritten slots hold NaN scales)."""
    return torch.equal(a.view(torch.uint8), b.view(torch.uint8))


@pytest.mark.parametrize("hq,hkv,bs,new_dtype,fused", [
    (64, 8, 16, torch.bfloat16, True),     # tensor cores: the append runs inside the launch
    (8, 8, 16, torch.bfloat16, True),
    (16, 2, 32, torch.bfloat16, True),
    (64, 8, 16, torch.float32, False),     # fp32 new rows: kv_append_fp8 first
    (32, 2, 16, torch.bfloat16, False),    # 16 query heads per KV head: CUDA cores, append first
])
@pytest.mark.parametrize("num_splits", [0, 1, 3])
def test_fp8_decode_step_equals_append_then_decode(hq, hkv, bs, new_dtype, fused, num_splits):
    d = 128
    B = 8
    assert pkv.decode_step_fp8_kernel_launches(B, hq, hkv, d, bs, 200, 600, new_dtype, num_splits) == \
        pkv.decode_kernel_launches(B, hq, hkv, d, bs, 200, 600, torch.uint8, num_splits) + (0 if fused else 1)
    lens = [1, 16, 17, 700, 2049, 33, 5, 1000]
    case = _fp8_step_case(hq + bs + num_splits, lens, hq, hkv, d, bs, new_dtype)
    case[9][2] = -1                                   # sequence 2 has no new token this step
    scale = 1 / math.sqrt(d)
    out, lse, caches = _run_fp8_step(case, scale, num_splits)
    assert pkv.get_device_error() == 0
    ref_out, ref_lse, ref_caches = _run_fp8_step(case, scale, num_splits, fused=False)
    assert all(_same_bits(a, b) for a, b in zip(caches, ref_caches))
    assert torch.equal(out, ref_out) and torch.equal(lse, ref_lse)
    q, kq, vq, ks, vs, table, clens, k_new, v_new, slots = case
    want = [t.clone() for t in (kq, vq, ks, vs)]     # the oracle's codes and scales
    oracle.kv_append_fp8(*want, k_new, v_new, slots)
    assert all(_same_bits(a, b) for a, b in zip(caches, want))
    kd, vd = oracle.dequantize_fp8(want[0], want[2]), oracle.dequantize_fp8(want[1], want[3])
    ref, ref_l = oracle.paged_decode(q, kd, vd, table, clens, scale)
    assert_attn_close(out, ref, "decode_step_fp8 out")
    assert_attn_close(lse, ref_l, "decode_step_fp8 lse")


def test_fp8_decode_step_flags_a_slot_that_is_not_the_last_position():
    lens = [40, 0, 300]
    case = _fp8_step_case(78, lens, 16, 2, 128, 16, torch.bfloat16)
    table, k_new, v_new, slots = case[5], case[7], case[8], case[9]
    slots[0] = oracle.slot_of(table[0], 3, 16)        # an earlier position of sequence 0
    slots[1] = 5                                       # an empty sequence has no position
    out, lse, caches = _run_fp8_step(case, 0.1, 0)
    assert pkv.get_device_error() & pkv.DEVERR["slot"]
    want = [t.clone() for t in case[1:5]]              # only sequence 2's token is written
    oracle.kv_append_fp8(*want, k_new[2:], v_new[2:], slots[2:])
    assert all(_same_bits(a, b) for a, b in zip(caches, want))
