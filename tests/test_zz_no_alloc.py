"""The no-allocation decode entry point, called through the C ABI, gives the same
results as the regular entry point that takes a caller workspace.

pkv_paged_decode_attention_noalloc serves callers that cannot call cudaMalloc --
plugins inside a host application that owns all device memory, and decode loops
that must not allocate or free mid-step because that synchronises the device.
Its split-K partials live in a scratch array built into the library, shared by
every call, so each case makes two calls in a row with different inputs: the
second must not see anything the first left behind.  Both entry points run the
same plan and the same kernels, so their outputs must be bit-identical; both are
also checked against the fp64 oracle.  The cases cover every kernel family: the
chunked kernel merging in place (arrival counters in the scratch), the chunked
kernel with the separate merge, the tcgen05 kernel (16 and 64 query heads per KV
head; one wave of blocks and several), the CUDA-core kernel over an fp32 cache,
and a one-pass call that needs no scratch.

This file is collected last, so a run that stops at the first failure has run
every other test before it.
"""
import ctypes
import math

import pytest
import torch

import oracle
import paged_kv_cache_165_gb300 as pkv
from paged_kv_cache_165_gb300 import _binding, _build
from workloads import gen

from helpers import ATTN_ATOL, assert_attn_close

pytestmark = pytest.mark.gpu

SCRATCH_BYTES = 16 << 20   # PKV_NOALLOC_SCRATCH_BYTES in include/pkv.h


def _p(t):
    return ctypes.c_void_p(0 if t is None else t.data_ptr())


def _case(seed, lengths, hq, hkv, d=128, bs=16, dtype=torch.bfloat16):
    g = gen.generator(seed)
    per_seq = [gen.blocks_needed(n, bs) for n in lengths]
    nb = sum(per_seq) + 3
    table = gen.block_table_from_order(gen.permutation(g, nb), per_seq)
    kc = gen.randn(g, (nb, hkv, bs, d), dtype)
    vc = gen.randn(g, (nb, hkv, bs, d), dtype)
    q = gen.randn(g, (len(lengths), hq, d))
    return dict(q=q, kc=kc, vc=vc, table=table, lens=torch.tensor(lengths, dtype=torch.int32),
                hq=hq, hkv=hkv, d=d, bs=bs, dt=_binding.PKV_BF16 if dtype == torch.bfloat16 else _binding.PKV_F32)


def _to_gpu(c):
    return {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in c.items()}


def _call(L, c, num_splits, noalloc, workspace=None):
    B = c["q"].shape[0]
    out = torch.full((B, c["hq"], c["d"]), float("nan"), device="cuda")
    lse = torch.full((B, c["hq"]), float("nan"), device="cuda")
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    common = (_p(out), _p(lse), _p(c["q"]), _p(c["kc"]), _p(c["vc"]), c["dt"],
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


def _lengths(seed, n, lo, hi):
    return gen.uniform_lengths(gen.generator(seed), n, lo, hi)


# (id, first call's lengths, second call's lengths, hq, hkv, cache dtype, num_splits,
#  kernels one call enqueues: 1 = one pass or merged in place, 2 = separate merge)
CASES = [
    ("chunked_merge_in_place", _lengths(10, 40, 1, 3000), _lengths(11, 40, 1, 2500) + [0], 64, 8,
     torch.bfloat16, 0, 1),
    ("chunked_separate_merge", [700, 33, 4100, 1, 2048, 16, 3000, 257], [5000, 9, 130, 4096, 64, 1500], 64, 8,
     torch.bfloat16, 0, 2),
    ("tcgen05_m16", [1200, 1, 4000, 333], [17, 2900, 0, 640, 128], 32, 2, torch.bfloat16, 0, 2),
    ("tcgen05_mqa_m64", [9000, 20, 4100], [130, 7000], 64, 1, torch.bfloat16, 0, 2),
    ("tcgen05_mqa_m64_5_splits", [9000, 20, 4100], [130, 7000], 64, 1, torch.bfloat16, 5, 2),
    ("tcgen05_m16_many_blocks", _lengths(12, 50, 1, 3000), _lengths(13, 50, 1, 2000), 32, 2,
     torch.bfloat16, 0, 2),
    ("cuda_core_f32", [300, 1, 1000, 47], [999, 12, 0, 530, 200], 8, 2, torch.float32, 3, 2),
    ("one_pass_no_scratch", [300, 1, 1000, 47], [999, 12, 0, 530], 64, 8, torch.bfloat16, 1, 1),
]


@pytest.mark.parametrize("name,lens1,lens2,hq,hkv,dtype,num_splits,launches", CASES, ids=[c[0] for c in CASES])
def test_noalloc_matches_workspace_entry_point_on_two_calls_in_a_row(L, name, lens1, lens2, hq, hkv, dtype,
                                                                    num_splits, launches):
    host = [_case(100 + i, lens, hq, hkv, dtype=dtype) for i, lens in enumerate((lens1, lens2))]
    cases = [_to_gpu(c) for c in host]
    for c in cases:
        B, MBS = c["q"].shape[0], c["table"].shape[1]
        need = pkv.decode_workspace_bytes(B, hq, hkv, c["d"], c["bs"], MBS, num_splits)
        assert need <= SCRATCH_BYTES
        assert (need > 0) == (num_splits != 1)   # the split-K cases use the scratch array
        assert pkv.decode_kernel_launches(B, hq, hkv, c["d"], c["bs"], MBS, c["kc"].shape[0], dtype,
                                          num_splits) == launches
    ref = []
    for c in cases:
        ws = torch.zeros(SCRATCH_BYTES, dtype=torch.uint8, device="cuda")
        status, out, lse = _call(L, c, num_splits, noalloc=False, workspace=ws)
        assert status == _binding.PKV_OK, L.pkv_last_error()
        ref.append((out, lse))
    for c, h, (r_out, r_lse) in zip(cases, host, ref):
        status, out, lse = _call(L, c, num_splits, noalloc=True)
        assert status == _binding.PKV_OK, L.pkv_last_error()
        torch.cuda.synchronize()
        assert torch.isfinite(out).all()
        assert torch.equal(out, r_out), f"{name}: out differs from the workspace entry point"
        assert torch.equal(lse, r_lse), f"{name}: lse differs from the workspace entry point"
        o_ref, l_ref = oracle.paged_decode(h["q"], h["kc"], h["vc"], h["table"], h["lens"], 1 / math.sqrt(h["d"]))
        assert_attn_close(out, o_ref, f"{name} out vs oracle", ATTN_ATOL)
        assert_attn_close(lse, l_ref, f"{name} lse vs oracle", ATTN_ATOL)
    assert pkv.get_device_error() == 0


def test_noalloc_rejects_sizes_beyond_its_scratch(L):
    # 256 sequences x 64 heads x 64 chunks of partials need far more than the scratch
    c = _to_gpu(_case(3, [64] * 256, 64, 8))
    big_splits = 64
    B = c["q"].shape[0]
    c["table"] = torch.cat([c["table"], torch.full((B, 60), -1, dtype=torch.int32, device="cuda")], 1)
    assert pkv.decode_workspace_bytes(B, c["hq"], c["hkv"], c["d"], c["bs"], c["table"].shape[1],
                                      big_splits) > SCRATCH_BYTES
    status, out, _ = _call(L, c, big_splits, noalloc=True)
    assert status == _binding.PKV_ERR_WORKSPACE
    assert b"scratch" in L.pkv_last_error()
    torch.cuda.synchronize()
    assert torch.isnan(out).all()                  # nothing was enqueued
