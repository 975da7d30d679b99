"""Host block manager (allocation, fork, copy-on-write) checked against the oracle. No GPU."""
import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_165_gb300 import BlockManager, OutOfBlocks
from workloads import gen


def test_allocate_ceil_blocks_and_slots_match_the_oracle():
    """plumephp.com §4.3: allocate ceil(n/bs) blocks; get_kv(pos) = table[pos//bs][pos%bs]."""
    g = gen.generator(1)
    order = gen.permutation(g, 32)
    bm = BlockManager(32, 16, order=order)
    for s, n in enumerate([0, 1, 16, 17, 100]):
        bm.add_sequence(s, n)
        assert len(bm.tables[s]) == gen.blocks_needed(n, 16)
    bm.audit()
    table = bm.block_table(range(5))
    for s, n in enumerate([0, 1, 16, 17, 100]):
        mine = bm.slot_mapping(s, range(n)).tolist()
        ref = [oracle.slot_of(table[s].tolist(), p, 16) for p in range(n)]
        assert mine == ref
    used = set(x for row in table.tolist() for x in row if x >= 0)
    assert len(used) == sum(gen.blocks_needed(n, 16) for n in [0, 1, 16, 17, 100])


def test_fork_shares_blocks_and_counts_references():
    bm = BlockManager(8, 4)
    bm.add_sequence(0, 10)                 # 3 blocks
    bm.fork(0, 1)
    bm.fork(0, 2)
    assert bm.tables[1] == bm.tables[0] == bm.tables[2]
    assert [bm.refcount[b] for b in bm.tables[0]] == [3, 3, 3]
    bm.audit()
    bm.free_sequence(2)
    assert [bm.refcount[b] for b in bm.tables[0]] == [2, 2, 2]
    bm.audit()


def test_copy_on_write_only_for_a_shared_partial_last_block():
    bm = BlockManager(8, 4)
    bm.add_sequence(0, 6)                  # last block holds 2 of 4 tokens
    bm.fork(0, 1)
    last = bm.tables[0][-1]
    slot1, cp1 = bm.append_slot(1)         # first writer: shared block -> copy
    assert cp1 is not None and cp1[0] == last and bm.tables[1][-1] == cp1[1] != last
    assert slot1 == cp1[1] * 4 + 2
    slot0, cp0 = bm.append_slot(0)         # second writer: count now 1 -> in place
    assert cp0 is None and slot0 == last * 4 + 2
    bm.audit()
    # a full shared last block needs no copy: the next token opens a fresh block
    bm2 = BlockManager(8, 4)
    bm2.add_sequence(0, 8)
    bm2.fork(0, 1)
    s, cp = bm2.append_slot(1)
    assert cp is None and bm2.tables[1][:2] == bm2.tables[0] and len(bm2.tables[1]) == 3
    bm2.audit()


def test_out_of_blocks_and_bad_order():
    bm = BlockManager(2, 4)
    bm.add_sequence(0, 8)
    with pytest.raises(OutOfBlocks):
        bm.append_slot(0)
    with pytest.raises(ValueError):
        BlockManager(3, 4, order=[0, 0, 1])


def test_copy_on_write_keeps_every_sequence_isolated():
    """0539edu.com §4.3 isolation experiment on the block manager + oracle cache ops.

    A shared 37-token prompt, 4 forks, 3 decode steps each writing different
    tokens: every sequence's decode equals attention over its own logical history,
    whatever blocks the copies landed in.
    """
    hq, hkv, d, bs = 4, 2, 8, 16
    g = gen.generator(7)
    bm = BlockManager(24, bs, order=gen.permutation(g, 24))
    kc = gen.randn(g, (24, hkv, bs, d))
    vc = gen.randn(g, (24, hkv, bs, d))
    prompt_k = gen.randn(g, (37, hkv, d))
    prompt_v = gen.randn(g, (37, hkv, d))
    bm.add_sequence(0, 37)
    oracle.kv_append(kc, vc, prompt_k, prompt_v, bm.slot_mapping(0, range(37)))
    for child in (1, 2, 3):
        bm.fork(0, child)
    history = {s: ([prompt_k], [prompt_v]) for s in range(4)}
    for step in range(3):
        new_k = gen.randn(g, (4, hkv, d))
        new_v = gen.randn(g, (4, hkv, d))
        slots, copies = bm.append_step(range(4))
        if copies:
            oracle.kv_block_copy(kc, vc, torch.tensor(copies, dtype=torch.int32))
        oracle.kv_append(kc, vc, new_k, new_v, torch.tensor(slots))
        for s in range(4):
            history[s][0].append(new_k[s:s + 1])
            history[s][1].append(new_v[s:s + 1])
        bm.audit()
        q = gen.randn(g, (4, hq, d))
        out, _ = oracle.paged_decode(q, kc, vc, bm.block_table(range(4)), bm.context_lens(range(4)), 0.3)
        for s in range(4):
            ref, _ = oracle.attend_contiguous(q[s], torch.cat(history[s][0]), torch.cat(history[s][1]), 0.3)
            np.testing.assert_allclose(out[s], ref, rtol=1e-13, atol=1e-13)
    # the prompt's two full blocks are still shared by all four sequences
    assert all(bm.refcount[b] == 4 for b in bm.tables[0][:2])


def test_mix_layout_sharing_structure():
    """Prefix-sharing workload: pairs share everything, 0..63 share the prefix blocks."""
    lay = gen.mix_layout(batch=12, prefix_tokens=64, prefix_seqs=8, median=40)
    for k in range(0, 8, 2):
        assert lay.lengths[k] == lay.lengths[k + 1]
        assert torch.equal(lay.tokens_k[k], lay.tokens_k[k + 1])
    for s in range(8):
        assert torch.equal(lay.tokens_k[s][:64], lay.tokens_k[0][:64])
    assert all(16 <= n <= 32768 for n in lay.lengths)


def test_release_outside_window_frees_only_blocks_no_query_can_see():
    import numpy as np
    import oracle
    bs, W = 16, 40
    bm = BlockManager(40, bs, order=gen.permutation(gen.generator(4), 40))
    bm.add_sequence(0, 100)
    bm.add_sequence(1, 30)
    full_table = bm.block_table([0, 1], max_blocks=12)
    freed = bm.release_outside_window(0, W)          # first visible position 60: blocks 0..2
    assert len(freed) == 3 and bm.num_free == 40 - 7 - 2 + 3
    assert bm.release_outside_window(1, W) == []     # 30 tokens all inside the window
    bm.audit()
    table = bm.block_table([0, 1], max_blocks=12)
    assert table[0, :3].tolist() == [-1, -1, -1] and table[0, 3:7].tolist() == full_table[0, 3:7].tolist()
    with pytest.raises(KeyError):
        bm.slot(0, 47)
    # the windowed attention reads none of the released blocks
    g = gen.generator(5)
    kc = gen.randn(g, (40, 2, bs, 8), torch.float32)
    vc = gen.randn(g, (40, 2, bs, 8), torch.float32)
    q = gen.randn(g, (2, 4, 8), torch.float32)
    lens = np.array([100, 30], np.int32)
    cu = np.array([0, 1, 2], np.int32)
    ref, _ = oracle.paged_attention(q, kc, vc, full_table, lens, cu, 0.3, window=W)
    for blk in freed:
        kc[blk] = float("nan")
        vc[blk] = float("nan")
    out, _ = oracle.paged_attention(q, kc, vc, table, lens, cu, 0.3, window=W)
    assert np.array_equal(out, ref)
    # appending moves the window; a block is released once its last position leaves it
    for _ in range(12):
        bm.append_slot(0)
    assert bm.release_outside_window(0, W) == [int(full_table[0, 3])]   # 112 - 40 = 72 > 63
    bm.free_sequence(0)
    bm.free_sequence(1)
    bm.audit()
    assert bm.num_free == 40


def test_tiny_workload_draws_a_pool_of_8_blocks_with_3_free():
    """The tiny step: lengths {17, 40} plus one appended token each, over 8 physical blocks
    handed out in the order of a seeded permutation (2 + 3 used, 3 left in the pool)."""
    inp = gen.tiny_inputs()
    assert inp.num_blocks == 8 and tuple(inp.k_cache.shape) == (8, 2, 16, 64)
    order = gen.permutation(gen.generator(gen.TINY.seed), 8)
    table = inp.block_table.tolist()
    assert table[0][:2] == order[:2] and table[1] == order[2:5] and table[0][2] == -1
    used = {b for row in table for b in row if b >= 0}
    assert len(used) == 5 and used <= set(range(8))
    assert sorted(set(range(8)) - used) == sorted(order[5:])


def test_shared_prefix_groups_find_whole_common_blocks():
    """Rows forked from one prompt share its whole blocks; the group's prefix stops before
    the partial block each fork copied on write and before every member's last position."""
    bs = 16
    bm = BlockManager(64, bs, order=gen.permutation(gen.generator(3), 64))
    bm.add_sequence(100, 40)                  # a prompt of 40 tokens: 2 whole blocks + 8
    for s in (0, 1, 2):
        bm.fork(100, s)
    bm.add_sequence(3, 20)                     # a row in no group
    bm.fork(100, 4)
    bm.free_sequence(100)
    slots, copies = bm.append_step([0, 1, 2, 3, 4])
    assert len(copies) >= 3                    # the shared partial block is copied by its writers
    grp = bm.shared_prefix_groups([0, 1, 2, 3, 4])
    assert grp.n_groups == 1 and grp.n_members == 4
    assert grp.group_seqs.tolist() == [0, 1, 2, 4] and grp.group_start.tolist() == [0, 4]
    assert grp.prefix_tokens.tolist() == [32, 32, 32, 0, 32]
    assert grp.max_group_size == 4 and grp.max_prefix_tokens == 32
    for r in (0, 1, 2, 4):                     # the same physical blocks, ending before the new token
        assert bm.tables[r][:2] == bm.tables[0][:2] and bm.lengths[r] - 1 >= 32
    # a group needs two rows and one whole block
    assert bm.shared_prefix_groups([0, 3]).n_groups == 0
    assert bm.shared_prefix_groups([0, 1], min_blocks=3).n_groups == 0
