"""paged_decode_attention on the GPU against the fp64 oracle: small ragged cases,
every path (tensor-core bf16, CUDA-core fp32/bf16), one pass and split-K."""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_165_gb300 as pkv
from paged_kv_cache_165_gb300 import _build
from workloads import gen

from conftest import GOLDEN
from helpers import ATTN_ATOL, assert_attn_close, assert_bits_equal, dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    _build.build()
    pkv.lib()
    pkv.get_device_error()


def run_decode(q, kc, vc, table, lens, scale, num_splits=0, with_lse=True):
    B, Hq, d = q.shape
    NB, Hkv, bs, _ = kc.shape
    out = torch.full((B, Hq, d), float("nan"), device="cuda")
    lse = torch.full((B, Hq), float("nan"), device="cuda") if with_lse else None
    ws_bytes = pkv.decode_workspace_bytes(B, Hq, Hkv, d, bs, table.shape[1], num_splits)
    ws = torch.zeros(max(ws_bytes, 1), dtype=torch.uint8, device="cuda")
    pkv.paged_decode_attention(out, dev(q), dev(kc), dev(vc), dev(table), dev(lens), scale, lse=lse,
                               num_splits=num_splits, workspace=ws)
    torch.cuda.synchronize()
    return out, lse


def random_case(seed, lens, hq, hkv, d, bs, dtype, spare=4, poison=False):
    g = gen.generator(seed)
    per_seq = [gen.blocks_needed(n, bs) for n in lens]
    nb = sum(per_seq) + spare
    table = gen.block_table_from_order(gen.permutation(g, nb), per_seq)
    kc = gen.randn(g, (nb, hkv, bs, d), dtype)
    vc = gen.randn(g, (nb, hkv, bs, d), dtype)
    q = gen.randn(g, (len(lens), hq, d))
    if poison:   # unwritten slots past each length hold NaN / Inf: they must stay invisible
        for b, n in enumerate(lens):
            for pos in range(n, per_seq[b] * bs):
                s = oracle.slot_of(table[b], pos, bs)
                kc[s // bs, :, s % bs] = float("nan")
                vc[s // bs, :, s % bs] = float("inf")
        for blk in range(nb):
            if blk not in set(table.flatten().tolist()):
                kc[blk] = float("nan")
                vc[blk] = float("nan")
    return q, kc, vc, table, torch.tensor(lens, dtype=torch.int32)


def check(q, kc, vc, table, lens, scale, num_splits=0, what=""):
    out, lse = run_decode(q, kc, vc, table, lens, scale, num_splits)
    assert pkv.get_device_error() == 0
    ref, ref_lse = oracle.paged_decode(q, kc, vc, table, lens, scale)
    e1 = assert_attn_close(out, ref, what + " out")
    e2 = assert_attn_close(lse, ref_lse, what + " lse")
    return e1, e2


RAGGED = [1, 15, 16, 17, 31, 32, 33, 100, 0, 257]


@pytest.mark.parametrize("hq,hkv", [(8, 8), (8, 2), (16, 2), (12, 2), (32, 2), (16, 1)])
@pytest.mark.parametrize("d", [64, 128, 256])
@pytest.mark.parametrize("num_splits", [1, 3, 0])
def test_tensor_core_path_ragged(hq, hkv, d, num_splits):
    q, kc, vc, table, lens = random_case(hq * 1000 + d + num_splits, RAGGED, hq, hkv, d, 16, torch.bfloat16)
    check(q, kc, vc, table, lens, 1 / math.sqrt(d), num_splits, f"hq={hq} hkv={hkv} d={d} s={num_splits}")


@pytest.mark.parametrize("bs", [16, 32])
def test_block_sizes_and_poisoned_unwritten_slots(bs):
    q, kc, vc, table, lens = random_case(40 + bs, RAGGED, 16, 2, 128, bs, torch.bfloat16, poison=True)
    for s in (1, 2, 0):
        check(q, kc, vc, table, lens, 0.0884, s, f"bs={bs} s={s}")


@pytest.mark.parametrize("hq,hkv", [(9, 1), (16, 1), (48, 2), (64, 1), (128, 2)])
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("bs", [16, 32])
def test_large_group_path_ragged_and_poisoned(hq, hkv, d, bs):
    # 9..64 query heads per KV head: tcgen05 tiles of 64 keys gathered page by page, the
    # last tile of a chunk partly past the end, unwritten slots holding NaN / Inf
    lens = RAGGED + [2000, 64, 65, 127, 129]
    q, kc, vc, table, clens = random_case(hq * 7 + d + bs, lens, hq, hkv, d, bs, torch.bfloat16, poison=True)
    for s in (1, 3, 0):
        check(q, kc, vc, table, clens, 1 / math.sqrt(d), s, f"hq={hq} hkv={hkv} d={d} bs={bs} s={s}")


@pytest.mark.parametrize("hq,hkv,d", [(64, 1, 128), (32, 2, 64)])
def test_large_group_running_max_jumps(hq, hkv, d):
    # scale 1 and keys growing with their position: the row maximum moves by far more than
    # 2^8 between key tiles, so the lazy rescale of O runs on most tiles
    lens = [700, 2000, 129]
    q, kc, vc, table, clens = random_case(hq + d, lens, hq, hkv, d, 16, torch.bfloat16)
    for b, n in enumerate(lens):
        for pos in range(n):
            s = oracle.slot_of(table[b], pos, 16)
            kc[s // 16, :, s % 16] = (kc[s // 16, :, s % 16].float() * (1 + pos / 200)).to(torch.bfloat16)
    for s in (1, 0):
        check(q, kc, vc, table, clens, 1.0, s, f"max jumps hq={hq} d={d} s={s}")


@pytest.mark.parametrize("nseq", [200, 300])
def test_large_group_ragged_batch_in_both_launch_orders(nseq):
    # the tcgen05 kernel takes sequences longest first when there are at most 256 of them
    # (each block ranks the lengths) and in index order beyond; both against the oracle
    g = gen.generator(nseq)
    lens = [int(x) for x in torch.randint(1, 400, (nseq,), generator=g)]
    lens[7], lens[nseq - 3] = 1500, 0
    q, kc, vc, table, clens = random_case(nseq + 11, lens, 16, 1, 64, 16, torch.bfloat16)
    check(q, kc, vc, table, clens, 0.125, 0, f"{nseq} sequences")


def test_large_group_bad_block_id_reads_zeros():
    q, kc, vc, table, lens = random_case(81, [200, 700], 64, 1, 128, 16, torch.bfloat16)
    bad_table = table.clone()
    bad_table[1, 3] = kc.shape[0] + 5
    kz, vz = kc.clone(), vc.clone()
    for s in (1, 0):
        out, _ = run_decode(q, kc, vc, bad_table, lens, 0.1, s)
        assert pkv.get_device_error() & pkv.DEVERR["block"]
        assert torch.isfinite(out).all()
        assert_attn_close(out[:1], oracle.paged_decode(q[:1], kz, vz, table[:1], lens[:1], 0.1)[0], "good seq")


@pytest.mark.parametrize("dtype,d", [(torch.float32, 64), (torch.float32, 128), (torch.bfloat16, 96),
                                     (torch.float32, 40), (torch.bfloat16, 128)])
@pytest.mark.parametrize("bs", [8, 16])
def test_cuda_core_path(dtype, d, bs):
    # fp32 caches, head dims outside {64,128,256} and bs == 8 take the CUDA-core path
    q, kc, vc, table, lens = random_case(7 + d + bs, RAGGED, 8, 2, d, bs, dtype, poison=True)
    for s in (1, 0, 4):
        check(q, kc, vc, table, lens, 1 / math.sqrt(d), s, f"{dtype} d={d} bs={bs} s={s}")


def test_long_sequence_in_a_ragged_batch_splits_into_capped_chunks():
    # 160 sequences x 8 KV heads are units enough for one chunk per sequence, but one
    # sequence holds 10000 tokens: automatic chunks hold at most 8192 tokens, so it splits
    # into two chunks (313 and 312 of its 625 blocks), merged in place
    lens = [10000] + [50 + 7 * i for i in range(159)]
    B, hq, hkv, d, bs = len(lens), 8, 8, 128, 16
    q, kc, vc, table, lens_t = random_case(4242, lens, hq, hkv, d, bs, torch.bfloat16, spare=2)
    MBS = table.shape[1]
    assert MBS == 625
    counter_bytes = 256 << 10
    assert pkv.decode_workspace_bytes(B, hq, hkv, d, bs, MBS, 0) == counter_bytes + B * hq * 2 * (d + 1) * 4
    check(q, kc, vc, table, lens_t, 1 / math.sqrt(d), 0, "capped chunks")


@pytest.mark.parametrize("dtype,d", [(torch.bfloat16, 128), (torch.bfloat16, 64), (torch.bfloat16, 256),
                                     (torch.float32, 40), (torch.float32, 1), (torch.float32, 3)])
def test_separate_merge_of_many_chunks(dtype, d):
    # more chunks than the decode kernel merges in place: the LSE merge kernel folds them in
    # groups (one full pass of 4 x groups chunks, a ragged rest, groups with no chunk), and
    # for head dims that are not a multiple of 4 one thread per column
    lens = [5000, 1, 1700, 333, 4096]
    q, kc, vc, table, lens_t = random_case(900 + d, lens, 8, 2, d, 16, dtype, poison=True)
    for s in (9, 37, 300):
        check(q, kc, vc, table, lens_t, 1 / math.sqrt(d), s, f"{dtype} d={d} s={s}")


def test_tiny_config_append_then_decode():
    """Tiny workload: batch 2, 8 q / 2 kv heads, d 64, lengths {17, 40} + 1 appended, fp32,
    8 physical blocks in seeded-permutation order (5 used).  The 3 free blocks and the slots
    past each new length hold NaN / Inf, which must stay invisible; the step runs as
    kv_append + the attention (one pass and split-K) and as pkv_decode_step."""
    inp = gen.tiny_inputs()
    spec = inp.spec
    bs = spec.block_size
    assert inp.num_blocks == 8
    kc, vc = inp.k_cache.clone(), inp.v_cache.clone()
    used = set(inp.block_table.flatten().tolist()) - {-1}
    for blk in set(range(inp.num_blocks)) - used:
        kc[blk] = float("nan")
        vc[blk] = float("nan")
    for b, n in enumerate(inp.cached):
        for pos in range(n + 1, gen.blocks_needed(n + 1, bs) * bs):
            s = oracle.slot_of(inp.block_table[b], pos, bs)
            kc[s // bs, :, s % bs] = float("nan")
            vc[s // bs, :, s % bs] = float("inf")
    kc0, vc0 = kc.clone(), vc.clone()
    slots = torch.tensor([oracle.slot_of(inp.block_table[b], n, bs)
                          for b, n in enumerate(inp.cached)], dtype=torch.int64)
    gk, gv = dev(kc), dev(vc)
    pkv.kv_append(dev(inp.k_new[0]), dev(inp.v_new[0]), gk, gv, dev(slots))
    oracle.kv_append(kc, vc, inp.k_new[0], inp.v_new[0], slots)
    assert_bits_equal(gk, kc, "tiny k_cache")
    assert_bits_equal(gv, vc, "tiny v_cache")
    lens = torch.tensor([n + 1 for n in inp.cached], dtype=torch.int32)
    ref, ref_lse = oracle.paged_decode(inp.q[0], kc, vc, inp.block_table, lens, spec.scale)
    assert np.isfinite(ref).all()
    ws = torch.zeros(1 << 20, dtype=torch.uint8, device="cuda")
    for s in (1, 0, 2):
        out = torch.full((spec.batch, spec.q_heads, spec.head_dim), float("nan"), device="cuda")
        lse = torch.full((spec.batch, spec.q_heads), float("nan"), device="cuda")
        pkv.paged_decode_attention(out, dev(inp.q[0]), gk, gv, dev(inp.block_table), dev(lens),
                                   spec.scale, lse=lse, num_splits=s, workspace=ws)
        assert_attn_close(out, ref, f"tiny out, num_splits={s}")
        assert_attn_close(lse, ref_lse, f"tiny lse, num_splits={s}")
    # the same step through pkv_decode_step, on the cache as it was before the append
    gk2, gv2 = dev(kc0), dev(vc0)
    out = torch.full((spec.batch, spec.q_heads, spec.head_dim), float("nan"), device="cuda")
    lse = torch.full((spec.batch, spec.q_heads), float("nan"), device="cuda")
    pkv.decode_step(out, dev(inp.q[0]), dev(inp.k_new[0]), dev(inp.v_new[0]), dev(slots), gk2, gv2,
                    dev(inp.block_table), dev(lens), spec.scale, lse=lse, workspace=ws)
    assert_bits_equal(gk2, kc, "tiny k_cache via decode_step")
    assert_bits_equal(gv2, vc, "tiny v_cache via decode_step")
    assert_attn_close(out, ref, "tiny out via decode_step")
    assert_attn_close(lse, ref_lse, "tiny lse via decode_step")
    assert pkv.get_device_error() == 0


def _d1_golden():
    with open(os.path.join(GOLDEN, "d1_worked_example.json")) as f:
        return json.load(f)


@pytest.mark.parametrize("dtype,d", [(torch.float32, 1), (torch.bfloat16, 64)])
def test_d1_worked_example_on_gpu(dtype, d):
    """zwjcode.cn "KV Cache 的增量解码" §04: cache [1,2] / [10,20], append (0, 30), q = 1 -> 18.45.

    d = 1 runs on the CUDA-core path; the bf16 case embeds the one-dimensional head
    in the first lane of a 64-wide head (zeros elsewhere) to run the tensor-core path.
    """
    g = _d1_golden()
    bs = 16
    kc = torch.zeros((2, 1, bs, d), dtype=dtype)
    vc = torch.zeros_like(kc)
    table = torch.tensor([[1]], dtype=torch.int32)
    kc[1, 0, 0, 0], kc[1, 0, 1, 0] = g["K_before_append"]
    vc[1, 0, 0, 0], vc[1, 0, 1, 0] = g["V_before_append"]
    gk, gv = dev(kc), dev(vc)
    k3 = torch.zeros((1, 1, d), dtype=dtype)
    v3 = torch.zeros((1, 1, d), dtype=dtype)
    k3[0, 0, 0], v3[0, 0, 0] = g["k3"], g["v3"]
    pkv.kv_append(dev(k3), dev(v3), gk, gv, dev(torch.tensor([oracle.slot_of(table[0], 2, bs)])))
    q = torch.zeros((1, 1, d))
    q[0, 0, 0] = g["q3"]
    out, lse = run_decode(q, gk.cpu(), gv.cpu(), table, torch.tensor([3], dtype=torch.int32), g["scale"], 1)
    assert round(float(out[0, 0, 0]), g["o3_printed_decimals"]) == g["o3_printed"]
    oracle.kv_append(kc, vc, k3, v3, torch.tensor([oracle.slot_of(table[0], 2, bs)]))
    ref, ref_lse = oracle.paged_decode(q, kc, vc, table, torch.tensor([3], dtype=torch.int32), g["scale"])
    assert_attn_close(out, ref, "d1 out")
    assert_attn_close(lse, ref_lse, "d1 lse")


def test_lse_optional_and_empty_batch():
    q, kc, vc, table, lens = random_case(77, [5, 0, 40], 8, 2, 128, 16, torch.bfloat16)
    out, _ = run_decode(q, kc, vc, table, lens, 0.1, 0, with_lse=False)
    ref, _ = oracle.paged_decode(q, kc, vc, table, lens, 0.1)
    assert_attn_close(out, ref, "no-lse out")
    assert torch.all(out[1] == 0)
    empty = torch.empty((0, 8, 128), device="cuda")
    pkv.paged_decode_attention(empty, empty.clone(), dev(kc), dev(vc),
                               torch.empty((0, 4), dtype=torch.int32, device="cuda"),
                               torch.empty((0,), dtype=torch.int32, device="cuda"), 0.1)


def test_workspace_too_small_is_rejected():
    q, kc, vc, table, lens = random_case(78, [300, 300], 8, 2, 128, 16, torch.bfloat16)
    out = torch.empty((2, 8, 128), device="cuda")
    with pytest.raises(pkv.PkvError) as ei:
        pkv.paged_decode_attention(out, dev(q), dev(kc), dev(vc), dev(table), dev(lens), 0.1,
                                   num_splits=4, workspace=torch.empty(16, dtype=torch.uint8, device="cuda"))
    assert ei.value.status == 3


def test_bad_lengths_and_block_ids_raise_device_errors():
    q, kc, vc, table, lens = random_case(79, [20, 40], 8, 2, 128, 16, torch.bfloat16)
    bad_len = torch.tensor([20, 10_000], dtype=torch.int32)
    out, lse = run_decode(q, kc, vc, table, bad_len, 0.1, 1)
    assert pkv.get_device_error() & pkv.DEVERR["len"]
    assert torch.all(out[1] == 0) and torch.all(torch.isneginf(lse[1]))
    ref, _ = oracle.paged_decode(q[:1], kc, vc, table[:1], lens[:1], 0.1)
    assert_attn_close(out[:1], ref, "valid sequence next to a bad one")
    bad_table = table.clone()
    bad_table[1, 1] = kc.shape[0] + 3
    for s in (1, 0):
        out, _ = run_decode(q, kc, vc, bad_table, lens, 0.1, s)
        assert pkv.get_device_error() & pkv.DEVERR["block"]
        assert torch.isfinite(out).all()


def test_one_zeroed_workspace_serves_many_calls_and_shapes():
    """The arrival counters at the start of the workspace return to zero after every call,
    so a workspace zeroed once stays valid across calls with different shapes and splits."""
    ws = torch.zeros(16 << 20, dtype=torch.uint8, device="cuda")
    cases = [([300, 17, 1000, 0, 65], 16, 2, 128, 0), ([2000, 5], 64, 8, 128, 0),
             ([900] * 6, 8, 8, 64, 5), ([4000, 1, 33], 32, 4, 256, 0), ([300, 17, 1000, 0, 65], 16, 2, 128, 3)]
    for k, (lens, hq, hkv, d, s) in enumerate(cases):
        q, kc, vc, table, lens_t = random_case(500 + k, lens, hq, hkv, d, 16, torch.bfloat16)
        assert pkv.decode_workspace_bytes(len(lens), hq, hkv, d, 16, table.shape[1], s) <= ws.numel()
        out = torch.empty((len(lens), hq, d), device="cuda")
        lse = torch.empty((len(lens), hq), device="cuda")
        pkv.paged_decode_attention(out, dev(q), dev(kc), dev(vc), dev(table), dev(lens_t), 0.1, lse=lse,
                                   num_splits=s, workspace=ws)
        torch.cuda.synchronize()
        ref, ref_lse = oracle.paged_decode(q, kc, vc, table, lens_t, 0.1)
        assert_attn_close(out, ref, f"case {k}")
        assert_attn_close(lse, ref_lse, f"case {k} lse")
        assert int(ws[: 256 << 10].count_nonzero()) == 0     # counters back at zero
    assert pkv.get_device_error() == 0


@pytest.mark.parametrize("hq,hkv,lens,num_splits", [
    (64, 8, [3000, 5000, 700, 8000] * 4, 0),   # tensor-core split-K, merge fused in the kernel
    (64, 8, [300, 20], 1),                     # one pass
    (64, 1, [40000, 9000], 0),                 # large group kernel: separate merge kernel
    (32, 32, [2049] * 8, 0),
])
def test_decode_kernel_launches_counts_what_the_call_enqueues(hq, hkv, lens, num_splits):
    prof = pytest.importorskip("torch.profiler")
    q, kc, vc, table, clens = random_case(77, lens, hq, hkv, 128, 16, torch.bfloat16)
    args = [dev(t) for t in (q, kc, vc, table, clens)]
    B, NB, MBS = len(lens), kc.shape[0], table.shape[1]
    want = pkv.decode_kernel_launches(B, hq, hkv, 128, 16, MBS, NB, torch.bfloat16, num_splits)
    assert want in (1, 2)
    out = torch.empty((B, hq, 128), device="cuda")
    lse = torch.empty((B, hq), device="cuda")
    ws = torch.zeros(max(pkv.decode_workspace_bytes(B, hq, hkv, 128, 16, MBS, num_splits), 16),
                     dtype=torch.uint8, device="cuda")
    call = lambda: pkv.paged_decode_attention(out, args[0], args[1], args[2], args[3], args[4],
                                              1 / math.sqrt(128), lse=lse, num_splits=num_splits,
                                              workspace=ws)
    call()
    torch.cuda.synchronize()
    for _ in range(2):   # the first session of a process may start recording late
        with prof.profile(activities=[prof.ProfilerActivity.CUDA]) as p:
            call()
            torch.cuda.synchronize()
    names = [e.name for e in p.events() if e.device_type == torch.autograd.DeviceType.CUDA
             and "decode" in e.name]
    if not names:
        pytest.skip("the profiler recorded no kernels here")
    assert len(names) == want, names
    ref, ref_lse = oracle.paged_decode(q, kc, vc, table, clens, 1 / math.sqrt(128))
    assert_attn_close(out, ref, "out")
    assert_attn_close(lse, ref_lse, "lse")


# ------------------------------------------------------------------ decode_step (append + attend)

def _step_case(seed, lens, hq, hkv, d, bs, dtype):
    """A cache with lens[b] - 1 tokens written, the new token of each sequence, its slot
    (the last position's), and lens counting it."""
    q, kc, vc, table, clens = random_case(seed, lens, hq, hkv, d, bs, dtype)
    g = gen.generator(seed + 1)
    k_new = gen.randn(g, (len(lens), hkv, d), dtype)
    v_new = gen.randn(g, (len(lens), hkv, d), dtype)
    slots = torch.tensor([oracle.slot_of(table[b], n - 1, bs) if n > 0 else -1 for b, n in enumerate(lens)],
                         dtype=torch.int64)
    return q, kc, vc, table, clens, k_new, v_new, slots


def _run_step(q, kc, vc, table, clens, k_new, v_new, slots, scale, num_splits, fused=True):
    B, Hq, d = q.shape
    NB, Hkv, bs, _ = kc.shape
    out = torch.full((B, Hq, d), float("nan"), device="cuda")
    lse = torch.full((B, Hq), float("nan"), device="cuda")
    ws = torch.zeros(max(16, pkv.decode_workspace_bytes(B, Hq, Hkv, d, bs, table.shape[1], num_splits)),
                     dtype=torch.uint8, device="cuda")
    gk, gv = dev(kc), dev(vc)
    if fused:
        pkv.decode_step(out, dev(q), dev(k_new), dev(v_new), dev(slots), gk, gv, dev(table), dev(clens), scale,
                        lse=lse, num_splits=num_splits, workspace=ws)
    else:
        pkv.kv_append(dev(k_new), dev(v_new), gk, gv, dev(slots))
        pkv.paged_decode_attention(out, dev(q), gk, gv, dev(table), dev(clens), scale, lse=lse,
                                   num_splits=num_splits, workspace=ws)
    torch.cuda.synchronize()
    return out, lse, gk.cpu(), gv.cpu()


@pytest.mark.parametrize("hq,hkv,d,bs,dtype", [
    (64, 8, 128, 16, torch.bfloat16),    # the chunked kernel: the append runs inside it
    (8, 8, 64, 32, torch.bfloat16),
    (32, 8, 256, 16, torch.bfloat16),
    (16, 1, 128, 16, torch.bfloat16),    # the tcgen05 kernel: the append runs inside it too
    (32, 2, 64, 32, torch.bfloat16),
    (8, 2, 64, 16, torch.float32),       # CUDA-core path: kv_append first
])
@pytest.mark.parametrize("num_splits", [0, 1, 3])
def test_decode_step_equals_append_then_decode(hq, hkv, d, bs, dtype, num_splits):
    lens = [1, 16, 17, 700, 2049, 33, 5, 1000]
    case = _step_case(hq + d + bs + num_splits, lens, hq, hkv, d, bs, dtype)
    case[7][2] = -1                                   # sequence 2 has no new token this step
    out, lse, kc, vc = _run_step(*case, 1 / math.sqrt(d), num_splits)
    assert pkv.get_device_error() == 0
    ref_out, ref_lse, ref_kc, ref_vc = _run_step(*case, 1 / math.sqrt(d), num_splits, fused=False)
    assert torch.equal(kc, ref_kc) and torch.equal(vc, ref_vc)
    assert torch.equal(out, ref_out) and torch.equal(lse, ref_lse)
    q, kc0, vc0, table, clens, k_new, v_new, slots = case
    oracle.kv_append(kc0, vc0, k_new, v_new, slots)
    ref, ref_l = oracle.paged_decode(q, kc0, vc0, table, clens, 1 / math.sqrt(d))
    assert_attn_close(out, ref, "decode_step out")
    assert_attn_close(lse, ref_l, "decode_step lse")


@pytest.mark.parametrize("hq,hkv", [(16, 2), (16, 1)])   # chunked and tcgen05 kernels
def test_decode_step_flags_a_slot_that_is_not_the_last_position(hq, hkv):
    lens = [40, 0, 300]
    q, kc, vc, table, clens, k_new, v_new, slots = _step_case(77, lens, hq, hkv, 128, 16, torch.bfloat16)
    slots[0] = oracle.slot_of(table[0], 3, 16)        # an earlier position of sequence 0
    slots[1] = 5                                       # an empty sequence has no position
    out, lse, gk, gv = _run_step(q, kc, vc, table, clens, k_new, v_new, slots, 0.1, 0)
    assert pkv.get_device_error() & pkv.DEVERR["slot"]
    want_k, want_v = kc.clone(), vc.clone()          # only sequence 2's token is written
    oracle.kv_append(want_k, want_v, k_new[2:], v_new[2:], slots[2:])
    assert torch.equal(gk, want_k) and torch.equal(gv, want_v)


def test_decode_step_with_unaligned_new_rows_appends_first():
    lens = [100, 200]
    q, kc, vc, table, clens, k_new, v_new, slots = _step_case(9, lens, 16, 2, 128, 16, torch.bfloat16)
    B, Hq, d = q.shape
    NB, Hkv, bs, _ = kc.shape
    big_k = torch.zeros(B * Hkv * d + 1, dtype=torch.bfloat16, device="cuda")
    big_v = torch.zeros_like(big_k)
    kn = big_k[1:].view(B, Hkv, d)                    # 2-byte aligned, not 16
    vn = big_v[1:].view(B, Hkv, d)
    kn.copy_(dev(k_new))
    vn.copy_(dev(v_new))
    out = torch.empty((B, Hq, d), device="cuda")
    gk, gv = dev(kc), dev(vc)
    ws = torch.zeros(max(16, pkv.decode_workspace_bytes(B, Hq, Hkv, d, bs, table.shape[1], 0)),
                     dtype=torch.uint8, device="cuda")
    pkv.decode_step(out, dev(q), kn, vn, dev(slots), gk, gv, dev(table), dev(clens), 0.1, workspace=ws)
    torch.cuda.synchronize()
    assert pkv.get_device_error() == 0
    oracle.kv_append(kc, vc, k_new, v_new, slots)
    assert torch.equal(gk.cpu(), kc) and torch.equal(gv.cpu(), vc)
    assert_attn_close(out, oracle.paged_decode(q, kc, vc, table, clens, 0.1)[0], "unaligned rows")


@pytest.mark.parametrize("hq,hkv,d,dtype,fused", [(64, 8, 128, torch.bfloat16, True),
                                                   (16, 1, 128, torch.bfloat16, True),
                                                   (8, 2, 64, torch.float32, False)])
def test_decode_step_kernel_launches(hq, hkv, d, dtype, fused):
    B, bs, MBS, NB = 8, 16, 64, 600
    n = pkv.decode_kernel_launches(B, hq, hkv, d, bs, MBS, NB, dtype, 0)
    assert pkv.decode_step_kernel_launches(B, hq, hkv, d, bs, MBS, NB, dtype, 0) == n + (0 if fused else 1)
