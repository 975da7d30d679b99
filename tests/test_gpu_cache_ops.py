"""kv_append and kv_block_copy on the GPU: whole caches bit-exact against the oracle."""
import pytest
import torch

import oracle
import paged_kv_cache_165_gb300 as pkv
from paged_kv_cache_165_gb300 import _build
from workloads import gen

from helpers import assert_bits_equal, dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    _build.build()
    pkv.lib()
    pkv.get_device_error()


@pytest.mark.parametrize("dtype,d", [(torch.float32, 64), (torch.bfloat16, 128), (torch.bfloat16, 1),
                                     (torch.float32, 3), (torch.bfloat16, 256)])
def test_kv_append_bit_exact(dtype, d):
    g = gen.generator(100 + d)
    nb, hkv, bs, t = 11, 3, 16, 29
    kc = gen.randn(g, (nb, hkv, bs, d), dtype)
    vc = gen.randn(g, (nb, hkv, bs, d), dtype)
    kn = gen.randn(g, (t, hkv, d), dtype)
    vn = gen.randn(g, (t, hkv, d), dtype)
    slots = torch.randperm(nb * bs, generator=g)[:t].to(torch.int64)
    slots[3] = -1                                    # padding token
    slots[17] = -5
    gk, gv = dev(kc), dev(vc)
    pkv.kv_append(dev(kn), dev(vn), gk, gv, dev(slots))
    assert pkv.get_device_error() == 0
    oracle.kv_append(kc, vc, kn, vn, slots)
    assert_bits_equal(gk, kc, "k_cache")
    assert_bits_equal(gv, vc, "v_cache")


def test_kv_append_out_of_range_slot_sets_error_and_skips():
    g = gen.generator(3)
    nb, hkv, bs, d = 4, 2, 16, 64
    kc = gen.randn(g, (nb, hkv, bs, d), torch.bfloat16)
    vc = gen.randn(g, (nb, hkv, bs, d), torch.bfloat16)
    kn = gen.randn(g, (2, hkv, d), torch.bfloat16)
    vn = gen.randn(g, (2, hkv, d), torch.bfloat16)
    slots = torch.tensor([5, nb * bs + 7], dtype=torch.int64)
    gk, gv = dev(kc), dev(vc)
    pkv.kv_append(dev(kn), dev(vn), gk, gv, dev(slots))
    assert pkv.get_device_error() == pkv.DEVERR["slot"]
    assert pkv.get_device_error() == 0              # read-and-clear
    oracle.kv_append(kc, vc, kn[:1], vn[:1], slots[:1])
    assert_bits_equal(gk, kc, "k_cache")


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_kv_block_copy_bit_exact(dtype):
    g = gen.generator(5)
    nb, hkv, bs, d = 12, 8, 16, 128
    kc = gen.randn(g, (nb, hkv, bs, d), dtype)
    vc = gen.randn(g, (nb, hkv, bs, d), dtype)
    pairs = torch.tensor([[0, 5], [3, 7], [11, 2], [3, 9]], dtype=torch.int32)
    gk, gv = dev(kc), dev(vc)
    pkv.kv_block_copy(gk, gv, dev(pairs))
    assert pkv.get_device_error() == 0
    oracle.kv_block_copy(kc, vc, pairs)
    assert_bits_equal(gk, kc, "k_cache")
    assert_bits_equal(gv, vc, "v_cache")


def test_kv_block_copy_bad_pair_sets_error_and_skips():
    g = gen.generator(6)
    nb, hkv, bs, d = 4, 2, 16, 64
    kc = gen.randn(g, (nb, hkv, bs, d), torch.bfloat16)
    vc = gen.randn(g, (nb, hkv, bs, d), torch.bfloat16)
    pairs = torch.tensor([[0, 1], [2, nb], [-1, 3]], dtype=torch.int32)
    gk, gv = dev(kc), dev(vc)
    pkv.kv_block_copy(gk, gv, dev(pairs))
    assert pkv.get_device_error() == pkv.DEVERR["pair"]
    oracle.kv_block_copy(kc, vc, pairs[:1])
    assert_bits_equal(gk, kc, "k_cache")
    assert_bits_equal(gv, vc, "v_cache")


def test_kv_append_prefill_sized_scatter():
    """Long-context prefill size: 8 prompts, lengths uniform in [256, 4096], 8 KV heads, d 128."""
    lens = gen.long_prefill_lengths()
    total = sum(lens)
    g = gen.generator(7)
    hkv, d, bs = 8, 128, 16
    nb = sum(gen.blocks_needed(n) for n in lens) + 5
    bm = pkv.BlockManager(nb, bs, order=gen.permutation(g, nb))
    slots = []
    for s, n in enumerate(lens):
        bm.add_sequence(s, n)
        slots.append(bm.slot_mapping(s, range(n)))
    slots = torch.cat(slots)
    kc = torch.zeros((nb, hkv, bs, d), dtype=torch.bfloat16)
    vc = torch.zeros_like(kc)
    kn = gen.randn(g, (total, hkv, d), torch.bfloat16)
    vn = gen.randn(g, (total, hkv, d), torch.bfloat16)
    gk, gv = dev(kc), dev(vc)
    pkv.kv_append(dev(kn), dev(vn), gk, gv, dev(slots))
    assert pkv.get_device_error() == 0
    oracle.kv_append(kc, vc, kn, vn, slots)
    assert_bits_equal(gk, kc, "k_cache")
    assert_bits_equal(gv, vc, "v_cache")
