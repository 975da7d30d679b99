"""The no-allocation decode entry point, called through the C ABI, gives the same
results as the regular entry point that takes a caller workspace.

pkv_paged_decode_attention_noalloc serves callers that cannot call cudaMalloc --
plugins inside a host application that owns all device memory, and decode loops
that must not allocate or free mid-step because that synchronises the device.
Its split-K partials live in a scratch array built into the library, shared by
every call, so the test makes two calls in a row with different inputs: the
second must not see anything the first left behind.
"""
import ctypes
import math

import pytest
import torch

import paged_kv_cache_165_gb300 as pkv
from paged_kv_cache_165_gb300 import _binding, _build
from workloads import gen

from helpers import ATTN_ATOL

pytestmark = pytest.mark.gpu

SCRATCH_BYTES = 16 << 20   # PKV_NOALLOC_SCRATCH_BYTES in include/pkv.h


def _p(t):
    return ctypes.c_void_p(0 if t is None else t.data_ptr())


def _case(seed, lengths, hq=64, hkv=8, d=128, bs=16):
    g = gen.generator(seed)
    per_seq = [gen.blocks_needed(n, bs) for n in lengths]
    nb = sum(per_seq) + 3
    table = gen.block_table_from_order(gen.permutation(g, nb), per_seq)
    kc = gen.randn(g, (nb, hkv, bs, d), torch.bfloat16).cuda()
    vc = gen.randn(g, (nb, hkv, bs, d), torch.bfloat16).cuda()
    q = gen.randn(g, (len(lengths), hq, d)).cuda()
    return dict(q=q, kc=kc, vc=vc, table=table.cuda(),
                lens=torch.tensor(lengths, dtype=torch.int32).cuda(), hq=hq, hkv=hkv, d=d, bs=bs)


def _call(L, c, num_splits, noalloc, workspace=None):
    B = c["q"].shape[0]
    out = torch.full((B, c["hq"], c["d"]), float("nan"), device="cuda")
    lse = torch.full((B, c["hq"]), float("nan"), device="cuda")
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    common = (_p(out), _p(lse), _p(c["q"]), _p(c["kc"]), _p(c["vc"]), _binding.PKV_BF16,
              _p(c["table"]), _p(c["lens"]), B, c["hq"], c["hkv"], c["d"], c["bs"],
              c["table"].shape[1], c["kc"].shape[0], ctypes.c_float(1 / math.sqrt(c["d"])),
              num_splits)
    if noalloc:
        status = L.pkv_paged_decode_attention_noalloc(*common, stream)
    else:
        nbytes = 0 if workspace is None else workspace.numel()
        status = L.pkv_paged_decode_attention(*common, _p(workspace), nbytes, stream)
    return status, out, lse


@pytest.fixture(scope="module")
def L():
    _build.build()
    lib = pkv.lib()
    pkv.get_device_error()
    return lib


def test_noalloc_matches_workspace_entry_point_on_two_calls_in_a_row(L):
    first = _case(1, [700, 33, 4100, 1, 2048, 16, 3000, 257])
    second = _case(2, [5000, 9, 130, 4096, 64, 1500])          # other lengths, other data
    for c in (first, second):
        B = c["q"].shape[0]
        need = pkv.decode_workspace_bytes(B, c["hq"], c["hkv"], c["d"], c["bs"], c["table"].shape[1], 0)
        assert 0 < need <= SCRATCH_BYTES          # the split-K path, using the scratch array
    ref = []
    for c in (first, second):
        ws = torch.zeros(SCRATCH_BYTES, dtype=torch.uint8, device="cuda")
        status, out, lse = _call(L, c, 0, noalloc=False, workspace=ws)
        assert status == _binding.PKV_OK
        ref.append((out, lse))
    for c, (r_out, r_lse) in zip((first, second), ref):
        status, out, lse = _call(L, c, 0, noalloc=True)
        assert status == _binding.PKV_OK, L.pkv_last_error()
        torch.cuda.synchronize()
        assert torch.isfinite(out).all()
        assert (out - r_out).abs().max().item() <= ATTN_ATOL
        assert (lse - r_lse).abs().max().item() <= ATTN_ATOL
    assert pkv.get_device_error() == 0


def test_noalloc_rejects_sizes_beyond_its_scratch(L):
    # 256 sequences x 64 heads x 64 chunks of partials need far more than the scratch
    c = _case(3, [64] * 256)
    big_splits = 64
    B = c["q"].shape[0]
    assert pkv.decode_workspace_bytes(B, c["hq"], c["hkv"], c["d"], c["bs"], c["table"].shape[1],
                                      big_splits) > SCRATCH_BYTES
    c["table"] = torch.cat([c["table"], torch.full((B, 60), -1, dtype=torch.int32, device="cuda")], 1)
    status, out, _ = _call(L, c, big_splits, noalloc=True)
    assert status == _binding.PKV_ERR_WORKSPACE
    assert b"scratch" in L.pkv_last_error()
    torch.cuda.synchronize()
    assert torch.isnan(out).all()                  # nothing was enqueued
