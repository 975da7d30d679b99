"""The five workloads at full size, in the launch configuration bench.py times
(num_splits = 0: the library's own split-K plan; pkv_decode_step where the bench
calls it, kv_block_copy before it for the copy-on-write mix), against the fp64
oracle.

Caches are checked bit-exact in full, and attention outputs and lse of every
sequence and every head of every checked step (all 32 steps of the 70B cycle).
"""
import math
import os

import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_165_gb300 as pkv
from paged_kv_cache_165_gb300 import _build
from workloads import gen

from helpers import assert_attn_close, assert_bits_equal, dev

pytestmark = pytest.mark.gpu
THREADS = os.cpu_count() or 1


@pytest.fixture(scope="module", autouse=True)
def _lib():
    _build.build()
    pkv.lib()
    pkv.get_device_error()
    yield
    torch.cuda.empty_cache()


def decode(q, gk, gv, table, lens, scale):
    B, Hq, d = q.shape
    NB, Hkv, bs, _ = gk.shape
    ws = torch.zeros(max(pkv.decode_workspace_bytes(B, Hq, Hkv, d, bs, table.shape[1], 0), 16),
                     dtype=torch.uint8, device="cuda")
    out = torch.full((B, Hq, d), float("nan"), device="cuda")
    lse = torch.full((B, Hq), float("nan"), device="cuda")
    pkv.paged_decode_attention(out, q, gk, gv, table, lens, scale, lse=lse, workspace=ws)
    torch.cuda.synchronize()
    return out.cpu(), lse.cpu()


def check_sampled(out, lse, q, kc, vc, table, lens, scale, sample, what):
    idx = torch.tensor(sample)
    ref, ref_lse = oracle.paged_decode(q[idx], kc, vc, table[idx], lens[idx], scale, nthreads=THREADS)
    assert_attn_close(out[idx], ref, what + " out")
    assert_attn_close(lse[idx], ref_lse, what + " lse")


def check_all(out, lse, q, kc, vc, table, lens, scale, what):
    """Every sequence, every head."""
    check_sampled(out, lse, q, kc, vc, table, lens, scale, list(range(q.shape[0])), what)


def decode_step(q, k_new, v_new, slots, gk, gv, table, lens, scale):
    """pkv_decode_step as the bench times it: the appends inside the attention launch
    where the library fuses them."""
    B, Hq, d = q.shape
    NB, Hkv, bs, _ = gk.shape
    ws = torch.zeros(max(pkv.decode_workspace_bytes(B, Hq, Hkv, d, bs, table.shape[1], 0), 16),
                     dtype=torch.uint8, device="cuda")
    out = torch.full((B, Hq, d), float("nan"), device="cuda")
    lse = torch.full((B, Hq), float("nan"), device="cuda")
    pkv.decode_step(out, q, k_new, v_new, slots, gk, gv, table, lens, scale, lse=lse, workspace=ws)
    torch.cuda.synchronize()
    return out.cpu(), lse.cpu()


def run_decode_steps(inp, steps, check_steps, via_step=False):
    """Append + attend for `steps` consecutive steps (kv_append, then the decode; or one
    pkv_decode_step per step); the oracle checks every sequence of `check_steps`."""
    spec = inp.spec
    bs = spec.block_size
    kc, vc = inp.k_cache.clone(), inp.v_cache.clone()
    gk, gv = dev(kc), dev(vc)
    gtable = dev(inp.block_table)
    for c in range(steps):
        slots = torch.tensor([oracle.slot_of(inp.block_table[b], n + c, bs) for b, n in enumerate(inp.cached)])
        oracle.kv_append(kc, vc, inp.k_new[c], inp.v_new[c], slots)
        lens = torch.tensor([n + c + 1 for n in inp.cached], dtype=torch.int32)
        if via_step:
            out, lse = decode_step(dev(inp.q[c]), dev(inp.k_new[c]), dev(inp.v_new[c]), dev(slots), gk, gv,
                                   gtable, dev(lens), spec.scale)
        else:
            pkv.kv_append(dev(inp.k_new[c]), dev(inp.v_new[c]), gk, gv, dev(slots))
            if c in check_steps:
                out, lse = decode(dev(inp.q[c]), gk, gv, gtable, dev(lens), spec.scale)
        if c in check_steps:
            check_all(out, lse, inp.q[c], kc, vc, inp.block_table, lens, spec.scale, f"{spec.name} step {c}")
    assert pkv.get_device_error() == 0
    assert_bits_equal(gk, kc, f"{spec.name} k_cache")
    assert_bits_equal(gv, vc, f"{spec.name} v_cache")


@pytest.mark.parametrize("via_step", [False, True], ids=["append_then_decode", "decode_step"])
def test_llama2_7b_mha_decode(via_step):
    inp = gen.mha_7b_inputs()
    run_decode_steps(inp, 1, {0}, via_step)


@pytest.mark.parametrize("via_step", [False, True], ids=["append_then_decode", "decode_step"])
def test_llama2_70b_gqa_decode_32_steps(via_step):
    inp = gen.gqa_70b_inputs()
    run_decode_steps(inp, 32, set(range(32)), via_step)


@pytest.mark.parametrize("spec", [gen.LONG_GQA, gen.LONG_MQA], ids=["gqa", "mqa"])
def test_long_context_split_k_decode(spec):
    inp = gen.long_inputs(spec)
    run_decode_steps(inp, 1, {0}, via_step=True)


def test_long_context_varlen_prefill_writes_cache():
    lens = gen.long_prefill_lengths()
    hq, hkv, d, bs = 64, 8, 128, 16
    p = gen.prefill_inputs(lens, hq, hkv, d, torch.bfloat16, seed=4)
    g = gen.generator(44)
    nb = sum(gen.blocks_needed(n, bs) for n in lens) + 8
    bm = pkv.BlockManager(nb, bs, order=gen.permutation(g, nb))
    for s, n in enumerate(lens):
        bm.add_sequence(s, n)
    slots = torch.cat([bm.slot_mapping(s, range(n)) for s, n in enumerate(lens)])
    kc = torch.zeros((nb, hkv, bs, d), dtype=torch.bfloat16)
    vc = torch.zeros_like(kc)
    gk, gv = dev(kc), dev(vc)
    T = p.q.shape[0]
    out = torch.full((T, hq, d), float("nan"), device="cuda")
    lse = torch.full((T, hq), float("nan"), device="cuda")
    scale = 1 / math.sqrt(d)
    pkv.prefill_attention(out, dev(p.q), dev(p.k), dev(p.v), dev(p.cu_seqlens), max(lens), scale, lse=lse,
                          k_cache=gk, v_cache=gv, slot_mapping=dev(slots))
    torch.cuda.synchronize()
    assert pkv.get_device_error() == 0
    oracle.kv_append(kc, vc, p.k, p.v, slots)
    assert_bits_equal(gk, kc, "prefill k_cache")
    assert_bits_equal(gv, vc, "prefill v_cache")
    out, lse = out.cpu(), lse.cpu()
    # every row of every prompt, every query head (about 0.57 TFLOP of fp64 oracle work)
    ref, ref_lse = oracle.prefill(p.q, p.k, p.v, p.cu_seqlens, scale, nthreads=THREADS)
    assert_attn_close(out, ref, "prefill out")
    assert_attn_close(lse, ref_lse, "prefill lse")
    # one decode step on top of every prompt, reading the cache the prefill wrote
    new_k = gen.randn(g, (len(lens), hkv, d), torch.bfloat16)
    new_v = gen.randn(g, (len(lens), hkv, d), torch.bfloat16)
    q = gen.randn(g, (len(lens), hq, d))
    step_slots, copies = bm.append_step(range(len(lens)))
    step_slots = torch.tensor(step_slots)
    pkv.kv_append(dev(new_k), dev(new_v), gk, gv, dev(step_slots))
    oracle.kv_append(kc, vc, new_k, new_v, step_slots)
    table, clens = bm.block_table(range(len(lens))), bm.context_lens(range(len(lens)))
    dout, dlse = decode(dev(q), gk, gv, dev(table), dev(clens), scale)
    check_sampled(dout, dlse, q, kc, vc, table, clens, scale, list(range(len(lens))), "decode after prefill")


@pytest.mark.parametrize("route", ["append_then_decode", "decode_step", "shared_prefix"])
def test_continuous_batching_mix_with_prefix_sharing_and_cow(route):
    """256 sequences, lognormal lengths; 0..63 share a 4096-token prefix and form 32 fork
    pairs sharing their whole history, so each pair's first write into a shared partial
    block triggers copy-on-write (kv_block_copy) before the appends: kv_append then the
    decode, pkv_decode_step writing into the blocks just copied, or, as the bench's step,
    pkv_decode_step_shared_prefix reading the 64 sequences' shared prefix once."""
    spec = gen.MIX
    lay = gen.mix_layout()
    B, hq, hkv, d, bs = spec.batch, spec.q_heads, spec.kv_heads, spec.head_dim, spec.block_size
    unique_tokens = lay.prefix_tokens + sum(lay.lengths[s] - (lay.prefix_tokens if s < lay.prefix_seqs else 0)
                                            for s in range(B) if not (s < lay.prefix_seqs and s % 2 == 1))
    nb = gen.blocks_needed(unique_tokens, bs) + 2 * B + 64   # partial last blocks, new blocks, copies
    g = gen.generator(33)
    bm = pkv.BlockManager(nb, bs, order=gen.permutation(g, nb))
    kc = torch.zeros((nb, hkv, bs, d), dtype=torch.bfloat16)
    vc = torch.zeros_like(kc)
    root = B                                   # a sequence id outside the batch: the shared prefix
    bm.add_sequence(root, lay.prefix_tokens)
    oracle.kv_append(kc, vc, lay.tokens_k[0][:lay.prefix_tokens], lay.tokens_v[0][:lay.prefix_tokens],
                     bm.slot_mapping(root, range(lay.prefix_tokens)))
    for s in range(B):
        if s < lay.prefix_seqs and s % 2 == 1:
            bm.fork(s - 1, s)                  # the pair shares its whole history
            continue
        if s < lay.prefix_seqs:
            bm.fork(root, s)
            start = lay.prefix_tokens
        else:
            bm.add_sequence(s, 0)
            start = 0
        slots = []
        for _ in range(start, lay.lengths[s]):
            slot, copy = bm.append_slot(s)
            assert copy is None
            slots.append(slot)
        oracle.kv_append(kc, vc, lay.tokens_k[s][start:], lay.tokens_v[s][start:], torch.tensor(slots))
    bm.free_sequence(root)
    bm.audit()
    assert all(bm.refcount[blk] == lay.prefix_seqs for blk in bm.tables[0][:lay.prefix_tokens // bs])

    # one decode step for all 256 sequences: COW copies first, then the appends
    slots, copies = bm.append_step(range(B))
    bm.audit()
    partial_pairs = sum(1 for k in range(0, lay.prefix_seqs, 2) if lay.lengths[k] % bs != 0)
    assert len(copies) == partial_pairs > 0
    gk, gv = dev(kc), dev(vc)
    table, lens = bm.block_table(range(B)), bm.context_lens(range(B))
    pkv.kv_block_copy(gk, gv, dev(torch.tensor(copies, dtype=torch.int32)))
    if route == "shared_prefix":
        groups = bm.shared_prefix_groups(range(B))
        assert groups.n_groups == 1 and groups.n_members == lay.prefix_seqs
        assert groups.max_prefix_tokens == lay.prefix_tokens
        ws = torch.zeros(pkv.decode_step_shared_prefix_workspace_bytes(B, hq, hkv, d, bs, table.shape[1], groups),
                         dtype=torch.uint8, device="cuda")
        gout = torch.full((B, hq, d), float("nan"), device="cuda")
        glse = torch.full((B, hq), float("nan"), device="cuda")
        pkv.decode_step_shared_prefix(gout, dev(lay.q), dev(lay.k_new), dev(lay.v_new), dev(torch.tensor(slots)),
                                      gk, gv, dev(table), dev(lens), spec.scale, groups.to("cuda"), lse=glse,
                                      workspace=ws)
        torch.cuda.synchronize()
        out, lse = gout.cpu(), glse.cpu()
    elif route == "decode_step":
        out, lse = decode_step(dev(lay.q), dev(lay.k_new), dev(lay.v_new), dev(torch.tensor(slots)), gk, gv,
                               dev(table), dev(lens), spec.scale)
    else:
        pkv.kv_append(dev(lay.k_new), dev(lay.v_new), gk, gv, dev(torch.tensor(slots)))
        out, lse = decode(dev(lay.q), gk, gv, dev(table), dev(lens), spec.scale)
    oracle.kv_block_copy(kc, vc, torch.tensor(copies, dtype=torch.int32))
    oracle.kv_append(kc, vc, lay.k_new, lay.v_new, torch.tensor(slots))
    assert pkv.get_device_error() == 0
    assert_bits_equal(gk, kc, "mix k_cache")
    assert_bits_equal(gv, vc, "mix v_cache")
    check_all(out, lse, lay.q, kc, vc, table, lens, spec.scale, "mix")
    # isolation: each fork's output equals attention over its own logical history
    for s in (0, 1, 2, 3):
        K = torch.cat([lay.tokens_k[s], lay.k_new[s:s + 1]])
        V = torch.cat([lay.tokens_v[s], lay.v_new[s:s + 1]])
        ref, _ = oracle.attend_contiguous(lay.q[s], K, V, spec.scale)
        assert_attn_close(out[s], ref, f"mix sequence {s} vs its own history")
