"""The kernels' failure path on the GPU, made to run without faulting anything.

Every wait of the library's kernels on an mbarrier is bounded; a wait that runs out
raises PKV_DEVERR_TIMEOUT, and its block lets go of its tensor memory and returns so
that the context stays usable.  pkv_selftest_bounded_wait runs exactly that path: its
blocks arm a barrier for bytes that no copy delivers (none is issued) and wait through
the kernels' own bounded wait with a 1 ms limit, holding all tensor-memory columns of
their SM.  Afterwards the tensor-core kernels, which allocate those columns, must still
run and match the oracle.
"""
import math
import time

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


def _decode_after(seed):
    """A tcgen05 decode (16 query heads per KV head) against the oracle."""
    lens = [300, 1, 129, 2000]
    hq, hkv, d, bs = 32, 2, 128, 16
    g = gen.generator(seed)
    per_seq = [gen.blocks_needed(n, bs) for n in lens]
    nb = sum(per_seq) + 2
    table = gen.block_table_from_order(gen.permutation(g, nb), per_seq)
    kc = gen.randn(g, (nb, hkv, bs, d), torch.bfloat16)
    vc = gen.randn(g, (nb, hkv, bs, d), torch.bfloat16)
    q = gen.randn(g, (len(lens), hq, d))
    clens = torch.tensor(lens, dtype=torch.int32)
    out = torch.full((len(lens), hq, d), float("nan"), device="cuda")
    lse = torch.full((len(lens), hq), float("nan"), device="cuda")
    ws = torch.zeros(max(pkv.decode_workspace_bytes(len(lens), hq, hkv, d, bs, table.shape[1], 3), 16),
                     dtype=torch.uint8, device="cuda")
    pkv.paged_decode_attention(out, dev(q), dev(kc), dev(vc), dev(table), dev(clens), 1 / math.sqrt(d),
                               lse=lse, num_splits=3, workspace=ws)
    ref, ref_lse = oracle.paged_decode(q, kc, vc, table, clens, 1 / math.sqrt(d))
    assert_attn_close(out, ref, "tcgen05 decode after a timeout")
    assert_attn_close(lse, ref_lse, "tcgen05 decode lse after a timeout")


def _prefill_after(seed):
    """A tcgen05 prefill against the oracle."""
    p = gen.prefill_inputs([200, 7, 129], 8, 2, 128, torch.bfloat16, seed=seed)
    T = p.q.shape[0]
    out = torch.full((T, 8, 128), float("nan"), device="cuda")
    pkv.prefill_attention(out, dev(p.q), dev(p.k), dev(p.v), dev(p.cu_seqlens), 200, 1 / math.sqrt(128))
    ref, _ = oracle.prefill(p.q, p.k, p.v, p.cu_seqlens, 1 / math.sqrt(128))
    assert_attn_close(out, ref, "tcgen05 prefill after a timeout")


@pytest.mark.parametrize("hold_tmem", [True, False], ids=["holding_tmem", "no_tmem"])
def test_a_wait_that_runs_out_reports_a_timeout_and_leaves_the_gpu_usable(hold_tmem):
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    blocks = 2 * sms
    gave_up = torch.zeros(1, dtype=torch.int32, device="cuda")
    assert pkv.get_device_error() == 0
    t0 = time.perf_counter()
    pkv.selftest_bounded_wait(1_000_000, blocks, hold_tmem=hold_tmem, gave_up=gave_up)
    code = pkv.get_device_error()        # synchronises: every block has returned
    elapsed = time.perf_counter() - t0
    assert code == pkv.DEVERR["timeout"]
    assert gave_up.item() == blocks * 128   # every thread's wait gave up
    assert elapsed < 10.0
    # the context is intact and the tensor memory was given back
    _decode_after(71)
    _prefill_after(72)
    assert pkv.get_device_error() == 0


def test_a_short_limit_on_a_stream_of_its_own_and_the_next_call_on_it():
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        pkv.selftest_bounded_wait(2_000_000, 4)
        assert pkv.get_device_error(stream=s) == pkv.DEVERR["timeout"]
        _decode_after(73)
    torch.cuda.synchronize()
    assert pkv.get_device_error() == 0
