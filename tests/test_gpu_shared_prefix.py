"""pkv_decode_step_shared_prefix on the GPU: groups of sequences that share a prefix of
physical blocks (forks of a common prompt), the prefix read once per group and merged
with each sequence's own keys by log-sum-exp.  The results must be those of the plain
decode step: caches bit-exact against the oracle's append and copy-on-write, outputs and
lse within 2e-3 of the fp64 oracle over every sequence's whole context."""
import math

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


def build_case(seed, hq, hkv, d, bs, roots, loners, dtype=torch.bfloat16):
    """roots: [(prompt tokens, [own tokens of each fork])]; loners: lengths of rows in no
    group.  Histories are the cache's random content; copy-on-write copies are applied to
    the host caches as the block manager emits them.  Returns the state before one decode
    step of every row and the step's inputs."""
    g = gen.generator(seed)
    need = sum(gen.blocks_needed(p, bs) + sum(gen.blocks_needed(o + 1, bs) + 1 for o in owns) for p, owns in roots)
    need += sum(gen.blocks_needed(n + 1, bs) for n in loners) + 8
    bm = pkv.BlockManager(need, bs, order=gen.permutation(g, need))
    kc = gen.randn(g, (need, hkv, bs, d), dtype)
    vc = gen.randn(g, (need, hkv, bs, d), dtype)

    def copy(pair):
        if pair is not None:
            kc[pair[1]] = kc[pair[0]]
            vc[pair[1]] = vc[pair[0]]

    rows = []
    for r, (p, owns) in enumerate(roots):
        root = 10_000 + r
        bm.add_sequence(root, p)
        for own in owns:
            s = len(rows)
            bm.fork(root, s)
            for _ in range(own):
                copy(bm.append_slot(s)[1])
            rows.append(s)
        bm.free_sequence(root)
    for n in loners:
        s = len(rows)
        bm.add_sequence(s, n)
        rows.append(s)
    bm.audit()
    slots, copies = bm.append_step(rows)
    B = len(rows)
    q = gen.randn(g, (B, hq, d))
    k_new = gen.randn(g, (B, hkv, d), dtype)
    v_new = gen.randn(g, (B, hkv, d), dtype)
    return dict(bm=bm, rows=rows, kc=kc, vc=vc, q=q, k_new=k_new, v_new=v_new,
                slots=torch.tensor(slots, dtype=torch.int64),
                copies=torch.tensor(copies, dtype=torch.int32).reshape(-1, 2),
                table=bm.block_table(rows), lens=bm.context_lens(rows))


def run_step(c, groups, shared=True):
    B, hq, d = c["q"].shape
    NB, hkv, bs, _ = c["kc"].shape
    gk, gv = dev(c["kc"]), dev(c["vc"])
    if c["copies"].numel():
        pkv.kv_block_copy(gk, gv, dev(c["copies"]))
    out = torch.full((B, hq, d), float("nan"), device="cuda")
    lse = torch.full((B, hq), float("nan"), device="cuda")
    MBS = c["table"].shape[1]
    scale = 1 / math.sqrt(d)
    if shared:
        ws = torch.zeros(pkv.decode_step_shared_prefix_workspace_bytes(B, hq, hkv, d, bs, MBS, groups) + 16,
                         dtype=torch.uint8, device="cuda")
        pkv.decode_step_shared_prefix(out, dev(c["q"]), dev(c["k_new"]), dev(c["v_new"]), dev(c["slots"]), gk, gv,
                                      dev(c["table"]), dev(c["lens"]), scale, groups.to("cuda"), lse=lse,
                                      workspace=ws)
    else:
        ws = torch.zeros(pkv.decode_workspace_bytes(B, hq, hkv, d, bs, MBS) + 16, dtype=torch.uint8, device="cuda")
        pkv.decode_step(out, dev(c["q"]), dev(c["k_new"]), dev(c["v_new"]), dev(c["slots"]), gk, gv,
                        dev(c["table"]), dev(c["lens"]), scale, lse=lse, workspace=ws)
    torch.cuda.synchronize()
    return out, lse, gk, gv


def oracle_step(c):
    kc, vc = c["kc"].clone(), c["vc"].clone()
    if c["copies"].numel():
        oracle.kv_block_copy(kc, vc, c["copies"])
    oracle.kv_append(kc, vc, c["k_new"], c["v_new"], c["slots"])
    ref, ref_lse = oracle.paged_decode(c["q"], kc, vc, c["table"], c["lens"], 1 / math.sqrt(c["q"].shape[2]))
    return ref, ref_lse, kc, vc


# two groups (a 300-token prompt forked 5 ways, a 1000-token prompt forked 3 ways, forks
# whose own tokens run from 0 to 900), and rows in no group
ROOTS = [(300, [0, 1, 15, 16, 900]), (1000, [7, 200, 33])]
LONERS = [1, 17, 500, 2000]


@pytest.mark.parametrize("hq,hkv,d,bs", [(32, 8, 128, 16), (8, 8, 64, 32), (16, 2, 128, 16), (8, 1, 128, 16),
                                         (64, 4, 128, 16), (64, 1, 128, 16), (32, 2, 64, 32),   # tcgen05 decode
                                         (32, 2, 256, 16)])   # d 256: a plain step
def test_shared_prefix_step_equals_the_oracle_and_the_plain_step(hq, hkv, d, bs):
    c = build_case(hq + d + bs, hq, hkv, d, bs, ROOTS, LONERS)
    groups = c["bm"].shared_prefix_groups(c["rows"])
    assert groups.n_groups == 2 and groups.n_members == 8
    B, MBS = len(c["rows"]), c["table"].shape[1]
    plain = pkv.decode_step_kernel_launches(B, hq, hkv, d, bs, MBS, c["kc"].shape[0], torch.bfloat16)
    launches = pkv.decode_step_shared_prefix_kernel_launches(B, hq, hkv, d, bs, MBS, c["kc"].shape[0],
                                                             torch.bfloat16, groups)
    assert launches == (plain if d == 256 else plain + 2)
    out, lse, gk, gv = run_step(c, groups)
    assert pkv.get_device_error() == 0
    ref, ref_lse, kc, vc = oracle_step(c)
    assert_bits_equal(gk, kc, "k_cache")
    assert_bits_equal(gv, vc, "v_cache")
    assert_attn_close(out, ref, "shared-prefix out")
    assert_attn_close(lse, ref_lse, "shared-prefix lse")
    p_out, p_lse, _, _ = run_step(c, groups, shared=False)
    assert (out - p_out).abs().max().item() <= 1e-5 and (lse - p_lse).abs().max().item() <= 1e-5


def test_shared_prefix_step_without_groups_is_the_plain_step():
    c = build_case(5, 32, 8, 128, 16, ROOTS, LONERS)
    groups = c["bm"].shared_prefix_groups(c["rows"], min_members=99)
    assert groups.n_groups == 0
    out, lse, gk, gv = run_step(c, groups)
    p_out, p_lse, pk, pv = run_step(c, groups, shared=False)
    assert torch.equal(out, p_out) and torch.equal(lse, p_lse)
    assert torch.equal(gk, pk) and torch.equal(gv, pv)
    assert pkv.get_device_error() == 0


def test_shared_prefix_group_whose_members_differ_is_flagged():
    c = build_case(6, 32, 8, 128, 16, ROOTS, LONERS)
    groups = c["bm"].shared_prefix_groups(c["rows"])
    members = groups.group_seqs.tolist()
    bad = c["table"].clone()
    bad[members[1], 2] = bad[members[-1], -1]           # a member whose third block is another one
    c["table"] = bad
    run_step(c, groups)
    assert pkv.get_device_error() & pkv.DEVERR["prefix"]
    groups.prefix_tokens[members[0]] += c["kc"].shape[2]  # prefix lengths that disagree
    c["table"] = c["bm"].block_table(c["rows"])
    run_step(c, groups)
    assert pkv.get_device_error() & pkv.DEVERR["prefix"]


def test_shared_prefix_bad_group_descriptions_are_flagged_not_read():
    """Group offsets past the member list, a member that is no sequence of the batch and a
    group larger than the declared maximum raise PKV_DEVERR_PREFIX; the kernels' own range
    checks keep every access inside the arrays."""
    c = build_case(7, 32, 8, 128, 16, ROOTS, LONERS)
    good = c["bm"].shared_prefix_groups(c["rows"])
    B = len(c["rows"])
    bad_start = pkv.PrefixGroups(good.prefix_tokens, torch.tensor([0, 5, 9], dtype=torch.int32), good.group_seqs,
                                 good.max_group_size, good.max_prefix_tokens)      # 9 > the 8 members
    bad_seq = pkv.PrefixGroups(good.prefix_tokens, good.group_start,
                               torch.tensor(good.group_seqs.tolist()[:-1] + [B + 5], dtype=torch.int32),
                               good.max_group_size, good.max_prefix_tokens)        # sequence B + 5
    for groups in (bad_start, bad_seq):
        run_step(c, groups)
        assert pkv.get_device_error() & pkv.DEVERR["prefix"]
    run_step(c, good)
    assert pkv.get_device_error() == 0
    # 64 query heads a KV head: a group of 5 has 320 (member, head) rows, three 128-row tiles;
    # declared as a group of at most 1 (one tile), its rows would not all be computed
    c = build_case(8, 64, 1, 128, 16, ROOTS, LONERS)
    good = c["bm"].shared_prefix_groups(c["rows"])
    too_big = pkv.PrefixGroups(good.prefix_tokens, good.group_start, good.group_seqs, 1, good.max_prefix_tokens)
    run_step(c, too_big)
    assert pkv.get_device_error() & pkv.DEVERR["prefix"]
    run_step(c, good)
    assert pkv.get_device_error() == 0
