"""prefill_attention on the GPU: varlen causal attention vs the fp64 oracle, and the
cache it writes, bit-exact."""
import math

import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_165_gb300 as pkv
from paged_kv_cache_165_gb300 import _build
from workloads import gen

from helpers import assert_attn_close, assert_bits_equal, dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    _build.build()
    pkv.lib()
    pkv.get_device_error()


def run_prefill(p, scale, cache=None, max_seqlen=None):
    T, Hq, d = p.q.shape
    out = torch.full((T, Hq, d), float("nan"), device="cuda")
    lse = torch.full((T, Hq), float("nan"), device="cuda")
    kw = {}
    if cache is not None:
        kw = dict(k_cache=cache[0], v_cache=cache[1], slot_mapping=cache[2])
    pkv.prefill_attention(out, dev(p.q), dev(p.k), dev(p.v), dev(p.cu_seqlens),
                          max(p.lengths) if max_seqlen is None else max_seqlen, scale, lse=lse, **kw)
    torch.cuda.synchronize()
    return out, lse


LENS = [1, 7, 64, 65, 130, 0, 200, 63]


@pytest.mark.parametrize("hq,hkv", [(8, 8), (8, 2), (16, 2), (4, 1)])
@pytest.mark.parametrize("d", [64, 128])
def test_tensor_core_prefill_ragged(hq, hkv, d):
    p = gen.prefill_inputs(LENS, hq, hkv, d, torch.bfloat16, seed=hq * 10 + d)
    scale = 1 / math.sqrt(d)
    out, lse = run_prefill(p, scale)
    assert pkv.get_device_error() == 0
    ref, ref_lse = oracle.prefill(p.q, p.k, p.v, p.cu_seqlens, scale, nthreads=8)
    assert_attn_close(out, ref, f"prefill hq={hq} hkv={hkv} d={d}")
    assert_attn_close(lse, ref_lse, "prefill lse")


@pytest.mark.parametrize("nseq", [31, 40])
def test_tensor_core_prefill_one_long_prompt_among_short_ones(nseq):
    # one 3000-token prompt (24 query tiles) among 30 or 39 short ones: most (prompt,
    # query tile) blocks of the grid are past their prompt's end and return at once
    lens = ([3000] + [17 * (k % 5) + 1 for k in range(39)] + [0])[:nseq]
    p = gen.prefill_inputs(lens, 4, 1, 64, torch.bfloat16, seed=nseq)
    out, lse = run_prefill(p, 0.125)
    assert pkv.get_device_error() == 0
    ref, ref_lse = oracle.prefill(p.q, p.k, p.v, p.cu_seqlens, 0.125, nthreads=8)
    assert_attn_close(out, ref, f"prefill {nseq} prompts")
    assert_attn_close(lse, ref_lse, f"prefill {nseq} prompts lse")


@pytest.mark.parametrize("d", [64, 128])
def test_tensor_core_prefill_running_max_jumps(d):
    # scale 1 and keys growing along each prompt: the row maximum moves by far more than
    # 2^8 from one key tile to the next, so the lazy rescale of O runs on most tiles
    p = gen.prefill_inputs([300, 513, 1000, 129], 8, 2, d, torch.bfloat16, seed=d + 5)
    pos = torch.cat([torch.arange(n, dtype=torch.float32) for n in p.lengths])
    p.k.copy_((p.k.float() * (1 + pos / 96)[:, None, None]).to(torch.bfloat16))
    out, lse = run_prefill(p, 1.0)
    assert pkv.get_device_error() == 0
    ref, ref_lse = oracle.prefill(p.q, p.k, p.v, p.cu_seqlens, 1.0, nthreads=8)
    assert_attn_close(out, ref, f"prefill max jumps d={d}")
    assert_attn_close(lse, ref_lse, "prefill max jumps lse")


@pytest.mark.parametrize("dtype,d", [(torch.float32, 64), (torch.float32, 32), (torch.bfloat16, 96)])
def test_cuda_core_prefill(dtype, d):
    p = gen.prefill_inputs([3, 0, 17, 40], 8, 2, d, dtype, seed=d)
    out, lse = run_prefill(p, 0.2)
    ref, ref_lse = oracle.prefill(p.q, p.k, p.v, p.cu_seqlens, 0.2)
    assert_attn_close(out, ref, f"simt prefill {dtype} d={d}")
    assert_attn_close(lse, ref_lse, "simt prefill lse")


def test_prefill_writes_the_cache_and_decode_reads_it():
    """Prefill through cu_seqlens writing the paged cache, then one decode step per prompt."""
    lens = [5, 16, 47, 130]
    hq, hkv, d, bs = 16, 2, 128, 16
    p = gen.prefill_inputs(lens, hq, hkv, d, torch.bfloat16, seed=31)
    g = gen.generator(32)
    nb = sum(gen.blocks_needed(n + 1, bs) for n in lens) + 3
    bm = pkv.BlockManager(nb, bs, order=gen.permutation(g, nb))
    for s, n in enumerate(lens):
        bm.add_sequence(s, n)
    slots = torch.cat([bm.slot_mapping(s, range(n)) for s, n in enumerate(lens)])
    kc = gen.randn(g, (nb, hkv, bs, d), torch.bfloat16)
    vc = gen.randn(g, (nb, hkv, bs, d), torch.bfloat16)
    gk, gv = dev(kc), dev(vc)
    out, _ = run_prefill(p, 0.09, cache=(gk, gv, dev(slots)))
    assert pkv.get_device_error() == 0
    oracle.kv_append(kc, vc, p.k, p.v, slots)
    assert_bits_equal(gk, kc, "k_cache after prefill")
    assert_bits_equal(gv, vc, "v_cache after prefill")
    ref, _ = oracle.prefill(p.q, p.k, p.v, p.cu_seqlens, 0.09)
    assert_attn_close(out, ref, "prefill with cache write")
    # one decode step per prompt on top of the prefilled cache
    new_k = gen.randn(g, (len(lens), hkv, d), torch.bfloat16)
    new_v = gen.randn(g, (len(lens), hkv, d), torch.bfloat16)
    q = gen.randn(g, (len(lens), hq, d))
    step_slots, copies = bm.append_step(range(len(lens)))
    assert copies == []
    step_slots = torch.tensor(step_slots, dtype=torch.int64)
    pkv.kv_append(dev(new_k), dev(new_v), gk, gv, dev(step_slots))
    oracle.kv_append(kc, vc, new_k, new_v, step_slots)
    table, clens = bm.block_table(range(len(lens))), bm.context_lens(range(len(lens)))
    o = torch.empty((len(lens), hq, d), device="cuda")
    pkv.paged_decode_attention(o, dev(q), gk, gv, dev(table), dev(clens), 0.09, num_splits=1)
    ref_dec, _ = oracle.paged_decode(q, kc, vc, table, clens, 0.09)
    assert_attn_close(o, ref_dec, "decode after prefill")
    for s, n in enumerate(lens):   # decode step == the same row of a causal prefill of n+1 tokens
        K = torch.cat([p.k[p.cu_seqlens[s]:p.cu_seqlens[s + 1]], new_k[s:s + 1]])
        V = torch.cat([p.v[p.cu_seqlens[s]:p.cu_seqlens[s + 1]], new_v[s:s + 1]])
        r, _ = oracle.attend_contiguous(q[s], K, V, 0.09)
        assert_attn_close(o[s], r, "decode vs contiguous history")


def test_bad_cu_seqlens_sets_device_error():
    p = gen.prefill_inputs([4, 6], 4, 2, 64, torch.bfloat16, seed=3)
    bad = gen.PrefillInputs(p.lengths, torch.tensor([0, 7, 5], dtype=torch.int32), p.q, p.k, p.v)
    out, _ = run_prefill(bad, 0.1, max_seqlen=8)
    assert pkv.get_device_error() & pkv.DEVERR["cu_seqlens"]
    too_long = gen.PrefillInputs(p.lengths, p.cu_seqlens, p.q, p.k, p.v)
    out, _ = run_prefill(too_long, 0.1, max_seqlen=4)
    assert pkv.get_device_error() & pkv.DEVERR["cu_seqlens"]
    ref, _ = oracle.prefill(p.q, p.k, p.v, p.cu_seqlens, 0.1)
    assert_attn_close(out[:4], ref[:4], "rows within max_seqlen")
