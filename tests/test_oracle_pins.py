"""Pins for the fp64 oracle against what the pages and the mathematics fix.

No GPU.  Each test pins the oracle to something other than itself: a value the
pages print, a library routine (torch's fp64 scaled_dot_product_attention and
logsumexp), a closed form or invariant, or brute force on tiny inputs.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
from workloads import gen

from conftest import GOLDEN


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def _fp32_cache(nb, hkv, bs, d):
    return np.zeros((nb, hkv, bs, d), np.float32)


# ----------------------------------------------------------------- d = 1 example
# zwjcode.cn "KV Cache 的增量解码" §04: K = [1, 2, 0], V = [10, 20, 30], q = 1,
# scale 1 -> softmax ~ [0.245, 0.665, 0.090], o ~ 18.45.

def test_d1_example_contiguous_matches_printed_values():
    g = _golden("d1_worked_example.json")
    K = np.array(g["K_after_append"], np.float64).reshape(3, 1, 1)
    V = np.array(g["V_after_append"], np.float64).reshape(3, 1, 1)
    q = np.array([[g["q3"]]], np.float64)
    out, _ = oracle.attend_contiguous(q, K, V, g["scale"])
    assert round(out[0, 0], g["o3_printed_decimals"]) == g["o3_printed"]
    # softmax weights: with V = indicator of token t, the output is weight t
    weights = []
    for t in range(3):
        ind = np.zeros((3, 1, 1))
        ind[t] = 1.0
        w, _ = oracle.attend_contiguous(q, K, ind, g["scale"])
        weights.append(w[0, 0])
    assert [round(w, g["softmax_printed_decimals"]) for w in weights] == g["softmax_printed"]
    assert abs(sum(weights) - 1.0) < 1e-15


def test_d1_example_exact_value_and_lse():
    # closed form of the same three-token softmax (e = Euler's number), computed
    # with sympy at 40 digits: an evaluation that shares nothing with the oracle
    sympy = pytest.importorskip("sympy")
    e = sympy.E
    num = 10 * e**1 + 20 * e**2 + 30 * e**0
    den = e**1 + e**2 + e**0
    o_exact = float(sympy.N(num / den, 40))
    lse_exact = float(sympy.N(sympy.log(den), 40))
    g = _golden("d1_worked_example.json")
    K = np.array(g["K_after_append"], np.float64).reshape(3, 1, 1)
    V = np.array(g["V_after_append"], np.float64).reshape(3, 1, 1)
    out, lse = oracle.attend_contiguous(np.array([[1.0]]), K, V, 1.0)
    assert abs(out[0, 0] - o_exact) < 1e-12
    assert abs(lse[0] - lse_exact) < 1e-12


def test_d1_example_through_paged_cache_two_steps():
    """Prefill K^(2)=[1,2], V^(2)=[10,20] into a paged cache, append (k3=0, v3=30), decode q3=1."""
    g = _golden("d1_worked_example.json")
    bs = 16
    kc, vc = _fp32_cache(3, 1, bs, 1), _fp32_cache(3, 1, bs, 1)
    table = np.array([[2]], np.int32)            # logical block 0 -> physical block 2
    slots = [oracle.slot_of(table[0], p, bs) for p in range(2)]
    oracle.kv_append(kc, vc, np.array(g["K_before_append"], np.float32).reshape(2, 1, 1),
                     np.array(g["V_before_append"], np.float32).reshape(2, 1, 1), np.array(slots))
    snapshot_k = kc.copy()
    oracle.kv_append(kc, vc, np.array([[[g["k3"]]]], np.float32), np.array([[[g["v3"]]]], np.float32),
                     np.array([oracle.slot_of(table[0], 2, bs)]))
    # the cached entries are untouched by the append; only slot 2 of block 2 changed
    changed = np.argwhere(kc != snapshot_k)
    assert changed.tolist() == [] or changed.tolist() == [[2, 0, 2, 0]]
    assert kc[2, 0, :3, 0].tolist() == g["K_after_append"]
    assert vc[2, 0, :3, 0].tolist() == g["V_after_append"]
    out, _ = oracle.paged_decode(np.array([[[1.0]]], np.float32), kc, vc, table,
                                 np.array([3], np.int32), g["scale"])
    assert round(out[0, 0, 0], 2) == g["o3_printed"]


def test_d1_example_as_last_row_of_causal_prefill():
    g = _golden("d1_worked_example.json")
    q = np.array([0.3, -0.7, g["q3"]], np.float32).reshape(3, 1, 1)
    k = np.array(g["K_after_append"], np.float32).reshape(3, 1, 1)
    v = np.array(g["V_after_append"], np.float32).reshape(3, 1, 1)
    out, _ = oracle.prefill(q, k, v, np.array([0, 3], np.int32), g["scale"])
    assert round(out[2, 0, 0], 2) == g["o3_printed"]
    assert out[0, 0, 0] == 10.0                  # first token sees only itself


# ------------------------------------------------------------- library pins

def _random_paged(seed, lens, hq, hkv, d, bs, dtype, spare=3):
    g = gen.generator(seed)
    per_seq = [gen.blocks_needed(n, bs) for n in lens]
    nb = sum(per_seq) + spare
    table = gen.block_table_from_order(gen.permutation(g, nb), per_seq)
    kc = gen.randn(g, (nb, hkv, bs, d), dtype)
    vc = gen.randn(g, (nb, hkv, bs, d), dtype)
    q = gen.randn(g, (len(lens), hq, d), torch.float32)
    return q, kc, vc, table


def _logical_kv(cache, table_row, n, bs):
    """Walk the table a whole block at a time: [n][Hkv][d] of the sequence."""
    pages = [cache[int(p)] for p in table_row[: gen.blocks_needed(n, bs)]]   # [Hkv][bs][d] each
    if not pages:
        return cache.new_zeros((0, cache.shape[1], cache.shape[3]))
    return torch.cat([p.transpose(0, 1) for p in pages])[:n]


@pytest.mark.parametrize("hq,hkv", [(4, 4), (8, 2), (8, 1), (6, 3)])
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_decode_matches_torch_sdpa_fp64(hq, hkv, dtype):
    lens, d, bs, scale = [1, 15, 16, 17, 40], 32, 16, 0.37
    q, kc, vc, table = _random_paged(11, lens, hq, hkv, d, bs, dtype)
    out, lse = oracle.paged_decode(q, kc, vc, table, torch.tensor(lens, dtype=torch.int32), scale)
    for b, n in enumerate(lens):
        K = _logical_kv(kc, table[b], n, bs).double().transpose(0, 1)     # [Hkv][n][d]
        V = _logical_kv(vc, table[b], n, bs).double().transpose(0, 1)
        qb = q[b].double().unsqueeze(1)                                     # [Hq][1][d]
        ref = torch.nn.functional.scaled_dot_product_attention(
            qb.unsqueeze(0), K.unsqueeze(0), V.unsqueeze(0), scale=scale,
            enable_gqa=(hq != hkv))[0, :, 0]
        np.testing.assert_allclose(out[b], ref.numpy(), rtol=1e-12, atol=1e-12)
        Kx = K.repeat_interleave(hq // hkv, dim=0)                        # [Hq][n][d]
        scores = scale * torch.einsum("hd,hnd->hn", q[b].double(), Kx)
        np.testing.assert_allclose(lse[b], torch.logsumexp(scores, dim=-1).numpy(), rtol=1e-12, atol=1e-12)


def test_prefill_matches_torch_sdpa_causal_fp64():
    lens, hq, hkv, d, scale = [1, 7, 16, 33], 8, 2, 16, 0.25
    p = gen.prefill_inputs(lens, hq, hkv, d, torch.bfloat16, seed=5)
    out, lse = oracle.prefill(p.q, p.k, p.v, p.cu_seqlens, scale)
    cu = p.cu_seqlens.tolist()
    for b in range(len(lens)):
        sl = slice(cu[b], cu[b + 1])
        qb = p.q[sl].double().transpose(0, 1).unsqueeze(0)      # [1][Hq][n][d]
        kb = p.k[sl].double().transpose(0, 1).unsqueeze(0)
        vb = p.v[sl].double().transpose(0, 1).unsqueeze(0)
        ref = torch.nn.functional.scaled_dot_product_attention(qb, kb, vb, is_causal=True, scale=scale,
                                                               enable_gqa=True)[0].transpose(0, 1)
        np.testing.assert_allclose(out[sl], ref.numpy(), rtol=1e-12, atol=1e-12)


# ------------------------------------------------------- structure / invariants

def test_gqa_equals_mha_on_repeat_kv_expanded_cache():
    """limoncc.com §3.3 / §4.1: head i uses KV head floor(i/m); repeat_kv expands KV head j to j*m..j*m+m-1."""
    lens, hq, hkv, d, bs = [5, 23], 8, 2, 16, 16
    q, kc, vc, table = _random_paged(3, lens, hq, hkv, d, bs, torch.float32)
    lens_t = torch.tensor(lens, dtype=torch.int32)
    out_gqa, lse_gqa = oracle.paged_decode(q, kc, vc, table, lens_t, 0.25)
    m = hq // hkv
    kx = kc.repeat_interleave(m, dim=1)   # [NB][Hq][bs][d]: KV head j at positions j*m..j*m+m-1
    vx = vc.repeat_interleave(m, dim=1)
    out_mha, lse_mha = oracle.paged_decode(q, kx, vx, table, lens_t, 0.25)
    assert np.array_equal(out_gqa, out_mha) and np.array_equal(lse_gqa, lse_mha)
    # an interleaved mapping (head i -> KV head i % g) would read other data
    ki = kc[:, [i % hkv for i in range(hq)]]
    vi = vc[:, [i % hkv for i in range(hq)]]
    out_wrong, _ = oracle.paged_decode(q, ki, vi, table, lens_t, 0.25)
    assert not np.allclose(out_wrong, out_gqa)


def test_mqa_and_mha_are_the_special_cases():
    lens, d, bs = [9, 30], 8, 16
    q, kc, vc, table = _random_paged(4, lens, 4, 1, d, bs, torch.float32)
    lens_t = torch.tensor(lens, dtype=torch.int32)
    out, _ = oracle.paged_decode(q, kc, vc, table, lens_t, 0.5)
    for h in range(4):   # MQA: every head reads KV head 0 -> equals a single-head call per head
        o1, _ = oracle.paged_decode(q[:, h:h + 1], kc, vc, table, lens_t, 0.5)
        assert np.array_equal(out[:, h], o1[:, 0])


def test_paged_equals_contiguous_bit_exact():
    lens, hq, hkv, d, bs = [1, 16, 17, 50], 6, 2, 24, 16
    q, kc, vc, table = _random_paged(8, lens, hq, hkv, d, bs, torch.bfloat16)
    out, lse = oracle.paged_decode(q, kc, vc, table, torch.tensor(lens, dtype=torch.int32), 0.2)
    for b, n in enumerate(lens):
        K = _logical_kv(kc, table[b], n, bs)
        V = _logical_kv(vc, table[b], n, bs)
        o2, l2 = oracle.attend_contiguous(q[b], K, V, 0.2)
        assert np.array_equal(out[b], o2) and np.array_equal(lse[b], l2)


@pytest.mark.parametrize("chunk", [16, 32, 48, 4096])
def test_split_k_lse_merge_equals_one_pass(chunk):
    """plumephp.com §2.2 online_softmax_update applied to chunks == one-pass softmax."""
    lens, hq, hkv, d, bs = [0, 1, 16, 47, 130], 8, 4, 32, 16
    q, kc, vc, table = _random_paged(9, lens, hq, hkv, d, bs, torch.bfloat16)
    lens_t = torch.tensor(lens, dtype=torch.int32)
    o1, l1 = oracle.paged_decode(q, kc, vc, table, lens_t, 0.18)
    o2, l2 = oracle.paged_decode(q, kc, vc, table, lens_t, 0.18, chunk_tokens=chunk)
    np.testing.assert_allclose(o2, o1, rtol=0, atol=1e-12)
    np.testing.assert_allclose(l2[1:], l1[1:], rtol=1e-13, atol=0)
    assert np.all(np.isneginf(l1[0])) and np.all(np.isneginf(l2[0]))


def test_empty_sequence_gives_zero_output_and_minus_inf_lse():
    q, kc, vc, table = _random_paged(1, [0, 5], 2, 1, 8, 16, torch.float32)
    out, lse = oracle.paged_decode(q, kc, vc, table, torch.tensor([0, 5], dtype=torch.int32), 1.0)
    assert np.all(out[0] == 0.0) and np.all(np.isneginf(lse[0]))
    assert np.all(np.isfinite(out[1]))


def test_softmax_invariants():
    g = gen.generator(21)
    n, d = 12, 12
    K = gen.randn(g, (n, 1, d)).double()
    q = gen.randn(g, (2, d)).double()
    # constant V -> o equals that constant (weights sum to one)
    const = torch.full((n, 1, d), 3.25, dtype=torch.float64)
    o, _ = oracle.attend_contiguous(q, K, const, 0.3)
    np.testing.assert_allclose(o, 3.25, rtol=1e-15)
    # V = identity rows -> o[t] is softmax weight t; weights sum to 1 and match exp(s - lse)
    eye = torch.eye(n, dtype=torch.float64).reshape(n, 1, d)
    w, lse = oracle.attend_contiguous(q, K, eye, 0.3)
    np.testing.assert_allclose(w.sum(-1), 1.0, rtol=1e-15)
    s = 0.3 * (q @ K[:, 0].T).numpy()
    np.testing.assert_allclose(w, np.exp(s - lse[:, None]), rtol=1e-13)
    # a single token: o = v
    o1, l1 = oracle.attend_contiguous(q, K[:1], K[:1] * 2, 0.3)
    np.testing.assert_array_equal(o1, np.broadcast_to((K[0, 0] * 2).numpy(), o1.shape))
    # scale folds into q
    oa, _ = oracle.attend_contiguous(q, K, K, 0.3)
    ob, _ = oracle.attend_contiguous(q * 0.3, K, K, 1.0)
    np.testing.assert_allclose(oa, ob, rtol=1e-13, atol=1e-14)


def test_unwritten_slots_are_invisible():
    """zwjcode.cn §10: slots past the cached length must not affect the query."""
    lens, bs = [3, 17], 16
    q, kc, vc, table = _random_paged(2, lens, 4, 2, 8, bs, torch.float32, spare=0)
    lens_t = torch.tensor(lens, dtype=torch.int32)
    ref, lref = oracle.paged_decode(q, kc, vc, table, lens_t, 0.5)
    kp, vp = kc.clone(), vc.clone()
    for b, n in enumerate(lens):
        for pos in range(n, gen.blocks_needed(n, bs) * bs):
            s = oracle.slot_of(table[b], pos, bs)
            kp[s // bs, :, s % bs] = float("nan")
            vp[s // bs, :, s % bs] = float("inf")
    out, lse = oracle.paged_decode(q, kp, vp, table, lens_t, 0.5)
    assert np.array_equal(out, ref) and np.array_equal(lse, lref)


# ------------------------------------------------ incremental == full recompute

def test_incremental_decode_equals_full_causal_recompute():
    """zwjcode.cn §07: every position of a full causal forward equals the cached step."""
    n, hq, hkv, d, bs = 37, 4, 2, 16, 16
    p = gen.prefill_inputs([n], hq, hkv, d, torch.float32, seed=13)
    full, full_lse = oracle.prefill(p.q, p.k, p.v, p.cu_seqlens, 0.25)
    g = gen.generator(14)
    nb = gen.blocks_needed(n, bs) + 2
    table = gen.block_table_from_order(gen.permutation(g, nb), [gen.blocks_needed(n, bs)])
    kc, vc = _fp32_cache(nb, hkv, bs, d), _fp32_cache(nb, hkv, bs, d)
    for t in range(n):
        oracle.kv_append(kc, vc, p.k[t:t + 1], p.v[t:t + 1], np.array([oracle.slot_of(table[0], t, bs)]))
        step, step_lse = oracle.paged_decode(p.q[t:t + 1], kc, vc, table, np.array([t + 1], np.int32), 0.25)
        assert np.array_equal(step[0], full[t]) and np.array_equal(step_lse[0], full_lse[t])


def test_prefill_row_does_not_see_later_tokens():
    """zwjcode.cn §13: a query at position t sees keys 0..t only (causal alignment)."""
    lens = [9]
    p = gen.prefill_inputs(lens, 2, 1, 8, torch.float32, seed=17)
    out, _ = oracle.prefill(p.q, p.k, p.v, p.cu_seqlens, 0.5)
    k2, v2 = p.k.clone(), p.v.clone()
    k2[5:] = 1e3
    v2[5:] = -1e3
    out2, _ = oracle.prefill(p.q, k2, v2, p.cu_seqlens, 0.5)
    assert np.array_equal(out[:5], out2[:5])
    assert not np.allclose(out[5:], out2[5:])


def test_prefill_zero_length_sequences_are_tolerated():
    """0539edu.com §3.3: a length-0 request must not disturb the others."""
    hq, hkv, d = 4, 2, 8
    p = gen.prefill_inputs([3, 0, 5, 0], hq, hkv, d, torch.float32, seed=19)
    out, lse = oracle.prefill(p.q, p.k, p.v, p.cu_seqlens, 0.4)
    a = oracle.prefill(p.q[:3], p.k[:3], p.v[:3], torch.tensor([0, 3], dtype=torch.int32), 0.4)
    b = oracle.prefill(p.q[3:], p.k[3:], p.v[3:], torch.tensor([0, 5], dtype=torch.int32), 0.4)
    assert np.array_equal(out[:3], a[0]) and np.array_equal(out[3:], b[0])
    with pytest.raises(ValueError):
        oracle.prefill(p.q, p.k, p.v, torch.tensor([0, 5, 3, 8, 8], dtype=torch.int32), 0.4)


# ------------------------------------------------------------- cache writes

def test_kv_append_writes_named_slots_only():
    g = gen.generator(23)
    nb, hkv, bs, d = 4, 2, 8, 4
    kc = gen.randn(g, (nb, hkv, bs, d), torch.bfloat16)
    vc = gen.randn(g, (nb, hkv, bs, d), torch.bfloat16)
    k0, v0 = kc.clone(), vc.clone()
    kn = gen.randn(g, (3, hkv, d), torch.bfloat16)
    vn = gen.randn(g, (3, hkv, d), torch.bfloat16)
    slots = torch.tensor([13, -1, 0], dtype=torch.int64)          # -1: padding, skipped
    oracle.kv_append(kc, vc, kn, vn, slots)
    assert torch.equal(kc[1, :, 5], kn[0]) and torch.equal(vc[1, :, 5], vn[0])
    assert torch.equal(kc[0, :, 0], kn[2]) and torch.equal(vc[0, :, 0], vn[2])
    mask = torch.ones(nb, bs, dtype=torch.bool)
    mask[1, 5] = mask[0, 0] = False
    assert torch.equal(kc.transpose(1, 2)[mask], k0.transpose(1, 2)[mask])
    assert torch.equal(vc.transpose(1, 2)[mask], v0.transpose(1, 2)[mask])


def test_kv_block_copy_and_copy_on_write_isolation():
    """0539edu.com §4.3 isolation experiment, restated on a paged cache.

    Two sequences fork from one history whose last block is partial and shared.
    With copy-on-write each sequence's decode equals attention over its own
    logical tokens and the shared block is unchanged; writing into the shared
    block instead (no COW) corrupts the other sequence.
    """
    hq, hkv, d, bs, n = 4, 2, 8, 8, 11
    g = gen.generator(29)
    hist_k = gen.randn(g, (n, hkv, d))
    hist_v = gen.randn(g, (n, hkv, d))
    new_k = gen.randn(g, (2, hkv, d))
    new_v = gen.randn(g, (2, hkv, d))
    q = gen.randn(g, (2, hq, d))
    nb = 4
    kc, vc = _fp32_cache(nb, hkv, bs, d), _fp32_cache(nb, hkv, bs, d)
    shared = np.array([3, 1], np.int32)                  # the common history's blocks
    oracle.kv_append(kc, vc, hist_k, hist_v, np.array([oracle.slot_of(shared, p, bs) for p in range(n)]))
    before = kc[1].copy(), vc[1].copy()

    def expected(s):
        K = torch.cat([hist_k, new_k[s:s + 1]])
        V = torch.cat([hist_v, new_v[s:s + 1]])
        return oracle.attend_contiguous(q[s], K, V, 0.5)[0]

    # with copy-on-write: sequence 1 writes first, gets a private copy in block 0
    ck, cv = kc.copy(), vc.copy()
    oracle.kv_block_copy(ck, cv, np.array([[1, 0]], np.int32))
    tables = np.array([[3, 1], [3, 0]], np.int32)
    oracle.kv_append(ck, cv, new_k, new_v,
                     np.array([oracle.slot_of(tables[0], n, bs), oracle.slot_of(tables[1], n, bs)]))
    out, _ = oracle.paged_decode(q, ck, cv, tables, np.array([n + 1, n + 1], np.int32), 0.5)
    for s in range(2):
        np.testing.assert_allclose(out[s], expected(s), rtol=1e-13, atol=1e-13)
    assert np.array_equal(ck[1][:, : n - bs], before[0][:, : n - bs])   # shared history untouched
    # without copy-on-write both write into the shared block 1: one overwrites the other
    nk, nv = kc.copy(), vc.copy()
    tables = np.array([[3, 1], [3, 1]], np.int32)
    oracle.kv_append(nk, nv, new_k, new_v,
                     np.array([oracle.slot_of(tables[0], n, bs), oracle.slot_of(tables[1], n, bs)]))
    bad, _ = oracle.paged_decode(q, nk, nv, tables, np.array([n + 1, n + 1], np.int32), 0.5)
    assert not np.allclose(bad[0], expected(0))


# ----------------------------------------------------------- cache size formula

def test_cache_size_formula_matches_printed_values():
    g = _golden("kv_cache_sizes.json")
    for c in g["cases"]:
        nbytes = oracle.kv_cache_bytes(c["layers"], c["batch"], c["heads"], c["tokens"], c["head_dim"], c["bytes"])
        gib = nbytes / 2**30
        assert abs(gib - c["printed"]) <= c["printed_tolerance"] * c["printed"], c["source"]
    r = g["ratios"][0]
    full = oracle.kv_cache_bytes(80, 1, r["q_heads"], 4096, 128, 2)
    gqa = oracle.kv_cache_bytes(80, 1, r["kv_heads"], 4096, 128, 2)
    assert gqa / full == r["printed_ratio"]
    sizes = [oracle.kv_cache_bytes(80, 1, h, 4096, 128, 2) for h in g["ratios"][1]["kv_heads"]]
    assert [s // sizes[0] for s in sizes] == g["ratios"][1]["printed_ratio"]
    bad = g["garbled"][0]
    nbytes = oracle.kv_cache_bytes(bad["layers"], bad["batch"], bad["heads"], bad["tokens"], bad["head_dim"], bad["bytes"])
    assert nbytes == 160 * 2**30 and abs(nbytes / 1e9 - bad["printed"]) > 1.0


def test_paged_cache_bytes_equal_the_formula():
    """A paged cache holding exactly N sequences x T tokens has the formula's byte count."""
    hkv, d, bs, n_seq, tokens = 8, 128, 16, 3, 64
    nb = n_seq * tokens // bs
    k = torch.empty((nb, hkv, bs, d), dtype=torch.bfloat16)
    v = torch.empty_like(k)
    got = k.numel() * k.element_size() + v.numel() * v.element_size()
    assert got == oracle.kv_cache_bytes(1, n_seq, hkv, tokens, d, 2)


# ---------------------------------------------- queries at the end of the cache
# Queries sit at the last positions of their sequence and see keys up to their
# own position (zwjcode.cn "KV Cache 的增量解码" §13); a sliding window keeps the
# most recent W positions (zwjcode.cn §10, §15; plumephp.com §5.2).

def _multi_case(seed, lens, nq, hq, hkv, d, bs, dtype):
    q1, kc, vc, table = _random_paged(seed, lens, hq, hkv, d, bs, dtype)
    g = gen.generator(seed + 99)
    q = gen.randn(g, (nq * len(lens), hq, d), torch.float32)
    cu = np.arange(len(lens) + 1, dtype=np.int32) * nq
    return q, kc, vc, table, np.array(lens, np.int32), cu


def _sdpa_masked(q_rows, K, V, positions, window, scale):
    """torch fp64 SDPA with a boolean mask written from the definition."""
    L = K.shape[0]
    keys = torch.arange(L)[None, :]
    pos = torch.tensor(positions)[:, None]
    allowed = keys <= pos
    if window > 0:
        allowed &= keys > pos - window
    qh = q_rows.double().permute(1, 0, 2)[None]
    kh = K.double().permute(1, 0, 2)[None]
    vh = V.double().permute(1, 0, 2)[None]
    out = torch.nn.functional.scaled_dot_product_attention(qh, kh, vh, attn_mask=allowed[None, None],
                                                           scale=scale, enable_gqa=True)
    s = torch.einsum("hqd,hkd->hqk", qh[0], kh[0].repeat_interleave(qh.shape[1] // kh.shape[1], 0)) * scale
    lse = torch.logsumexp(s.masked_fill(~allowed[None], float("-inf")), -1)
    return out[0].permute(1, 0, 2), lse.permute(1, 0)


@pytest.mark.parametrize("nq,window", [(1, 0), (1, 7), (1, 1), (3, 0), (3, 5), (17, 0), (17, 16), (17, 100)])
def test_paged_attention_matches_torch_sdpa_with_explicit_mask(nq, window):
    lens, hq, hkv, d, bs = [40, 17, 33], 8, 2, 32, 16
    q, kc, vc, table, clens, cu = _multi_case(11 + nq + window, lens, nq, hq, hkv, d, bs, torch.bfloat16)
    scale = 0.177
    out, lse = oracle.paged_attention(q, kc, vc, table, clens, cu, scale, window)
    for b, L in enumerate(lens):
        K = _logical_kv(kc, table[b], L, bs)
        V = _logical_kv(vc, table[b], L, bs)
        rows = slice(cu[b], cu[b + 1])
        ref, ref_lse = _sdpa_masked(q[rows], K, V, list(range(L - nq, L)), window, scale)
        assert np.abs(out[rows] - ref.numpy()).max() < 1e-12
        assert np.abs(lse[rows] - ref_lse.numpy()).max() < 1e-12


def test_window_of_one_returns_the_own_value_row():
    lens, nq, hq, hkv, d, bs = [21, 48], 4, 4, 1, 16, 16
    q, kc, vc, table, clens, cu = _multi_case(5, lens, nq, hq, hkv, d, bs, torch.float32)
    out, lse = oracle.paged_attention(q, kc, vc, table, clens, cu, 0.3, window=1)
    for b, L in enumerate(lens):
        K = _logical_kv(kc, table[b], L, bs).double()
        V = _logical_kv(vc, table[b], L, bs).double()
        for i in range(nq):
            p, r = L - nq + i, cu[b] + i
            assert np.array_equal(out[r], V[p, 0][None].expand(hq, d).numpy())
            assert np.allclose(lse[r], (0.3 * q[r].double() @ K[p, 0]).numpy(), rtol=0, atol=1e-12)


def test_window_covering_everything_and_one_query_reduce_to_decode():
    lens, hq, hkv, d, bs = [300, 17, 1000, 65], 8, 2, 64, 16
    q, kc, vc, table, clens, cu = _multi_case(8, lens, 1, hq, hkv, d, bs, torch.bfloat16)
    full, full_lse = oracle.paged_attention(q, kc, vc, table, clens, cu, 0.125)
    wide, wide_lse = oracle.paged_attention(q, kc, vc, table, clens, cu, 0.125, window=1000)
    assert np.array_equal(full, wide) and np.array_equal(full_lse, wide_lse)
    dec, dec_lse = oracle.paged_decode(q, kc, vc, table, clens, 0.125)
    assert np.array_equal(full, dec) and np.array_equal(full_lse, dec_lse)


def test_queries_at_the_end_equal_the_last_rows_of_full_causal_prefill():
    # zwjcode.cn §07: the cached computation reproduces the full recomputation
    L, nq, hq, hkv, d, bs = 45, 9, 4, 2, 16, 16
    g = gen.generator(17)
    qkv = [gen.randn(g, (L, h, d), torch.float32) for h in (hq, hkv, hkv)]
    nb = gen.blocks_needed(L, bs) + 2
    kc, vc = _fp32_cache(nb, hkv, bs, d), _fp32_cache(nb, hkv, bs, d)
    table = gen.block_table_from_order(gen.permutation(g, nb), [gen.blocks_needed(L, bs)])
    oracle.kv_append(kc, vc, qkv[1].numpy(), qkv[2].numpy(),
                     np.array([oracle.slot_of(table[0], t, bs) for t in range(L)]))
    full, full_lse = oracle.prefill(qkv[0], qkv[1], qkv[2], np.array([0, L], np.int32), 0.25)
    out, lse = oracle.paged_attention(qkv[0][L - nq:], kc, vc, table, np.array([L], np.int32),
                                      np.array([0, nq], np.int32), 0.25)
    assert np.abs(out - full[L - nq:]).max() < 1e-12
    assert np.abs(lse - full_lse[L - nq:]).max() < 1e-12


def test_blocks_outside_the_window_are_never_read():
    lens, nq, hq, hkv, d, bs, W = [200, 130], 2, 4, 2, 32, 16, 40
    q, kc, vc, table, clens, cu = _multi_case(23, lens, nq, hq, hkv, d, bs, torch.float32)
    ref, ref_lse = oracle.paged_attention(q, kc, vc, table, clens, cu, 0.2, window=W)
    freed = table.clone()
    kp, vp = kc.clone(), vc.clone()
    for b, L in enumerate(lens):
        first_seen = L - nq - W + 1
        for page in range(first_seen // bs):          # whole blocks before the window
            kp[int(table[b, page])] = float("nan")
            vp[int(table[b, page])] = float("nan")
            freed[b, page] = -1
    out, lse = oracle.paged_attention(q, kp, vp, freed, clens, cu, 0.2, window=W)
    assert np.array_equal(out, ref) and np.array_equal(lse, ref_lse)


# ------------------------------------------------------------- FP8 (E4M3) cache
# zwjcode.cn §14 / plumephp.com §2.5 leave the low-bit format open; the oracle's reading
# is E4M3 with one fp32 scale per cached row.  The format pins against torch's
# float8_e4m3fn conversions; the quantisation against its own closed-form bounds.

def test_e4m3_decode_matches_torch_float8():
    codes = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).double().numpy()
    got = oracle.e4m3_decode(codes)
    assert np.array_equal(np.isnan(ref), np.isnan(got))
    assert np.array_equal(ref[~np.isnan(ref)], got[~np.isnan(got)])
    assert np.nanmax(got) == 448.0 and got[0x7E] == 448.0 and np.isnan(got[0x7F])


def test_e4m3_encode_rounds_to_nearest_even_like_torch():
    g = np.random.default_rng(0)
    x = (g.standard_normal(100000) * np.exp2(g.integers(-14, 9, 100000))).astype(np.float32)
    x = x[np.abs(x) <= 448]
    vals = np.unique(np.abs(oracle.e4m3_decode(np.arange(0x7F, dtype=np.uint8))))
    ties = ((vals[1:] + vals[:-1]) / 2).astype(np.float32)            # exactly halfway
    x = np.concatenate([x, ties, -ties, vals.astype(np.float32), np.float32([0.0, -0.0, 1e-30, -1e-30])])
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(oracle.e4m3_encode(x), ref)
    # saturation at the largest finite value
    assert oracle.e4m3_encode(np.float32([448.0001, -460.0])).tolist() == [0x7E, 0xFE]


def test_fp8_row_quantisation_bounds():
    g = gen.generator(41)
    rows = gen.randn(g, (6, 2, 64), torch.bfloat16)
    rows[3, 1] = 0.0                                   # an all-zero row
    codes, scale = oracle.quantize_rows_e4m3(rows)
    x = oracle.to_f64(rows)
    deq = oracle.e4m3_decode(codes) * scale.astype(np.float64)[..., None]
    assert scale[3, 1] == 0 and not codes[3, 1].any() and not deq[3, 1].any()
    for t in range(6):
        for h in range(2):
            if scale[t, h] == 0:
                continue
            i = np.abs(x[t, h]).argmax()
            assert abs(oracle.e4m3_decode(codes[t, h, i])) == 448.0   # the row's amax is +-448
            # each element within half an E4M3 spacing (relative 2^-4 for normals,
            # absolute 2^-10 * scale for subnormals)
            y = x[t, h] / np.float64(scale[t, h])
            spacing = np.where(np.abs(y) >= 2.0 ** -6, np.exp2(np.floor(np.log2(np.maximum(np.abs(y), 1e-300))) - 3),
                               2.0 ** -9)
            assert np.all(np.abs(deq[t, h] - x[t, h]) <= 0.5 * spacing * scale[t, h] * (1 + 1e-6))


def test_fp8_append_writes_named_slots_only():
    nb, hkv, bs, d = 5, 2, 16, 32
    kc = np.full((nb, hkv, bs, d), 0xAB, np.uint8)
    vc = kc.copy()
    ks = np.full((nb, hkv, bs), -1.0, np.float32)
    vs = ks.copy()
    g = gen.generator(2)
    kn, vn = gen.randn(g, (3, hkv, d), torch.bfloat16), gen.randn(g, (3, hkv, d), torch.bfloat16)
    oracle.kv_append_fp8(kc, vc, ks, vs, kn, vn, np.array([17, -1, 70]))
    kq, ksc = oracle.quantize_rows_e4m3(kn)
    assert np.array_equal(kc[1, :, 1], kq[0]) and np.array_equal(ks[1, :, 1], ksc[0])
    assert np.array_equal(kc[4, :, 6], kq[2])
    touched = np.zeros((nb, bs), bool)
    touched[1, 1] = touched[4, 6] = True
    assert np.all(kc.transpose(0, 2, 1, 3)[~touched] == 0xAB) and np.all(ks.transpose(0, 2, 1)[~touched] == -1)


def test_fp8_attention_is_attention_over_the_dequantised_cache():
    lens, hq, hkv, d, bs = [50, 17, 200], 8, 2, 32, 16
    q, kc, vc, table = _random_paged(61, lens, hq, hkv, d, bs, torch.float32)
    kq, ks = oracle.quantize_rows_e4m3(kc)
    vq, vs = oracle.quantize_rows_e4m3(vc)
    kd, vd = oracle.dequantize_fp8(kq, ks), oracle.dequantize_fp8(vq, vs)
    cu = np.arange(len(lens) + 1, dtype=np.int32)
    out, lse = oracle.paged_attention(q, kd, vd, table, np.array(lens, np.int32), cu, 0.2)
    for b, L in enumerate(lens):
        K = _logical_kv(torch.from_numpy(kd), table[b], L, bs)
        V = _logical_kv(torch.from_numpy(vd), table[b], L, bs)
        ref, ref_lse = _sdpa_masked(q[b:b + 1], K, V, [L - 1], 0, 0.2)
        assert np.abs(out[b] - ref[0].numpy()).max() < 1e-12
        assert np.abs(lse[b] - ref_lse[0].numpy()).max() < 1e-12
    # the quantisation error itself is what the pages warn about: visible, bounded
    exact, _ = oracle.paged_attention(q, kc, vc, table, np.array(lens, np.int32), cu, 0.2)
    assert 1e-4 < np.abs(out - exact).max() < 0.2
