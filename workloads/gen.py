"""Seeded random inputs and input structure for the five synthetic workloads.

Everything here is either a random draw (``torch.Generator`` seeded per
workload) or bookkeeping of *which* physical block a logical block is stored
in.  Values are drawn in fp32 ~ N(0, 1) and, where a workload stores bf16,
rounded once on the host by ``Tensor.to(torch.bfloat16)`` (round to nearest
even), so the oracle and the GPU read identical bits.

Workload shapes (one layer each; block size 16 throughout):

* ``TINY``   batch 2, 8 q heads / 2 kv heads, d 64, cached lengths {17, 40}
  then one appended token each, 8 physical blocks in seeded-permutation
  order, fp32 q/K/V, scale 1/sqrt(64).
* ``MHA_7B`` batch 32, 32 q heads = 32 kv heads, d 128, every sequence at
  2048 cached tokens, bf16 K/V, fp32 q, shuffled blocks, one append + attend.
* ``GQA_70B`` batch 64, 64 q / 8 kv heads, d 128, cached lengths uniform in
  [512, 8192], bf16 K/V, shuffled blocks, 32 consecutive decode steps.
* ``MIX``    batch 256, 32 q / 8 kv heads, d 128, lognormal lengths (median
  1024, sigma 1.0, clipped to [16, 32768]); sequences 0..63 share one
  4096-token prefix and form 32 fork pairs that also share their suffix.
* ``LONG``   batch 4, 64 q / 8 kv heads (and 1 kv head: MQA), d 128, 131072
  cached tokens, plus a varlen causal prefill of 8 prompts with lengths
  uniform in [256, 4096].
* ``SWA``    sliding-window decode shaped like Mistral-7B (the model the pages
  name for sliding windows): batch 64, 32 q / 8 kv heads, d 128, 16384 cached
  tokens per sequence, a window of the last 4096 tokens.
"""
from __future__ import annotations

import dataclasses
import math
from typing import List, Sequence

import torch

BLOCK_SIZE = 16


@dataclasses.dataclass(frozen=True)
class DecodeSpec:
    name: str
    seed: int
    batch: int
    q_heads: int
    kv_heads: int
    head_dim: int
    cache_dtype: torch.dtype
    block_size: int = BLOCK_SIZE
    steps: int = 1                 # consecutive decode steps (one token appended per sequence each)

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.head_dim)


TINY = DecodeSpec("tiny", 0, 2, 8, 2, 64, torch.float32)
MHA_7B = DecodeSpec("llama2_7b_mha", 1, 32, 32, 32, 128, torch.bfloat16)
GQA_70B = DecodeSpec("llama2_70b_gqa", 2, 64, 64, 8, 128, torch.bfloat16, steps=32)
MIX = DecodeSpec("mix_prefix_share", 3, 256, 32, 8, 128, torch.bfloat16)
LONG_GQA = DecodeSpec("long_gqa", 4, 4, 64, 8, 128, torch.bfloat16)
LONG_MQA = DecodeSpec("long_mqa", 4, 4, 64, 1, 128, torch.bfloat16)
SWA = DecodeSpec("mistral_7b_swa", 5, 64, 32, 8, 128, torch.bfloat16)
# chunked prefill on top of a cached prefix (prefix-cache hit): 8 sequences with 4096
# cached tokens each append and attend a chunk of 512 new tokens, causal within the chunk
PREFIX_CHUNK = DecodeSpec("prefix_chunk_prefill", 6, 8, 64, 8, 128, torch.bfloat16)

TINY_LENGTHS = (17, 40)
MHA_7B_LENGTH = 2048
GQA_70B_RANGE = (512, 8192)
MIX_MEDIAN, MIX_SIGMA, MIX_CLIP = 1024, 1.0, (16, 32768)
MIX_PREFIX_TOKENS, MIX_PREFIX_SEQS = 4096, 64
LONG_LENGTH = 131072
PREFILL_PROMPTS, PREFILL_RANGE = 8, (256, 4096)
SWA_LENGTH, SWA_WINDOW = 16384, 4096
PREFIX_LENGTH, PREFIX_CHUNK_LEN = 4096, 512


def generator(seed: int) -> torch.Generator:
    g = torch.Generator()
    g.manual_seed(seed)
    return g


def randn(gen: torch.Generator, shape: Sequence[int], dtype: torch.dtype = torch.float32) -> torch.Tensor:
    """N(0,1) draws in fp32, rounded once to ``dtype`` on the host."""
    x = torch.randn(tuple(shape), generator=gen, dtype=torch.float32)
    return x if dtype == torch.float32 else x.to(dtype)


def uniform_lengths(gen: torch.Generator, n: int, lo: int, hi: int) -> List[int]:
    """n integers uniform on [lo, hi] inclusive."""
    return torch.randint(lo, hi + 1, (n,), generator=gen).tolist()


def lognormal_lengths(gen: torch.Generator, n: int, median: float, sigma: float,
                      lo: int, hi: int) -> List[int]:
    """n lengths exp(ln(median) + sigma * N(0,1)), rounded and clipped to [lo, hi]."""
    z = torch.randn((n,), generator=gen, dtype=torch.float64)
    x = torch.exp(math.log(median) + sigma * z).round().clamp(lo, hi)
    return [int(v) for v in x.tolist()]


def permutation(gen: torch.Generator, n: int) -> List[int]:
    return torch.randperm(n, generator=gen).tolist()


def blocks_needed(tokens: int, block_size: int = BLOCK_SIZE) -> int:
    return -(-tokens // block_size)


def block_table_from_order(order: Sequence[int], blocks_per_seq: Sequence[int],
                           max_blocks: int | None = None, pad: int = -1) -> torch.Tensor:
    """Hand out physical block ids in ``order`` to sequence 0's logical blocks,
    then sequence 1's, and so on.  Unused table entries hold ``pad``.

    Returns int32 [batch][max_blocks].
    """
    mbs = max(blocks_per_seq) if max_blocks is None else max_blocks
    table = torch.full((len(blocks_per_seq), max(mbs, 1)), pad, dtype=torch.int32)
    k = 0
    for b, nb in enumerate(blocks_per_seq):
        if nb:
            table[b, :nb] = torch.tensor(order[k:k + nb], dtype=torch.int32)
        k += nb
    if k > len(order):
        raise ValueError("not enough physical blocks for the requested tables")
    return table


@dataclasses.dataclass
class DecodeInputs:
    """Host tensors for ``steps`` decode steps of one workload.

    ``k_cache``/``v_cache`` are [NB][Hkv][bs][d]; every slot (written or not)
    holds a random draw.  ``cached`` are the lengths before the first append.
    ``q[s]`` is [B][Hq][d] fp32; ``k_new[s]``/``v_new[s]`` are [B][Hkv][d].
    """
    spec: DecodeSpec
    cached: List[int]
    block_table: torch.Tensor
    num_blocks: int
    k_cache: torch.Tensor
    v_cache: torch.Tensor
    q: torch.Tensor            # [steps][B][Hq][d] fp32
    k_new: torch.Tensor        # [steps][B][Hkv][d]
    v_new: torch.Tensor


def decode_inputs(spec: DecodeSpec, cached: Sequence[int], spare_blocks: int = 0,
                  steps: int | None = None) -> DecodeInputs:
    """Draw a paged cache with room for ``steps`` appends per sequence.

    Physical blocks are a seeded permutation of ``0..NB-1`` handed out in
    order; ``spare_blocks`` extra blocks stay unreferenced (free pool).
    """
    steps = spec.steps if steps is None else steps
    gen = generator(spec.seed)
    bs = spec.block_size
    per_seq = [blocks_needed(n + steps, bs) for n in cached]
    nb = sum(per_seq) + spare_blocks
    order = permutation(gen, nb)
    table = block_table_from_order(order, per_seq)
    shape = (nb, spec.kv_heads, bs, spec.head_dim)
    k_cache = randn(gen, shape, spec.cache_dtype)
    v_cache = randn(gen, shape, spec.cache_dtype)
    b, hq, hkv, d = spec.batch, spec.q_heads, spec.kv_heads, spec.head_dim
    q = randn(gen, (steps, b, hq, d), torch.float32)
    k_new = randn(gen, (steps, b, hkv, d), spec.cache_dtype)
    v_new = randn(gen, (steps, b, hkv, d), spec.cache_dtype)
    return DecodeInputs(spec, list(cached), table, nb, k_cache, v_cache, q, k_new, v_new)


TINY_NUM_BLOCKS = 8


def tiny_inputs() -> DecodeInputs:
    """The tiny step over a pool of 8 physical blocks in seeded-permutation order: the two
    sequences take 2 + 3 of them (room for the appended token) and 3 stay free."""
    used = sum(blocks_needed(n + TINY.steps, TINY.block_size) for n in TINY_LENGTHS)
    return decode_inputs(TINY, TINY_LENGTHS, spare_blocks=TINY_NUM_BLOCKS - used)


def mha_7b_inputs() -> DecodeInputs:
    return decode_inputs(MHA_7B, [MHA_7B_LENGTH] * MHA_7B.batch)


def gqa_70b_lengths() -> List[int]:
    return uniform_lengths(generator(GQA_70B.seed + 1000), GQA_70B.batch, *GQA_70B_RANGE)


def gqa_70b_inputs(steps: int | None = None) -> DecodeInputs:
    return decode_inputs(GQA_70B, gqa_70b_lengths(), steps=steps)


def long_inputs(spec: DecodeSpec = LONG_GQA) -> DecodeInputs:
    return decode_inputs(spec, [LONG_LENGTH] * spec.batch)


# ---------------------------------------------------------------- prefix sharing

@dataclasses.dataclass
class MixLayout:
    """Logical structure of the continuous-batching mix.

    ``lengths[b]`` is sequence b's cached length.  Sequences ``0..63`` start
    with the same ``prefix_tokens`` tokens; pairs (2k, 2k+1) among them share
    their whole history (a fork at the current length, as for parallel
    sampling), so both members of a pair hold identical K/V for every cached
    position.  ``tokens_k[b]``/``tokens_v[b]`` hold each sequence's logical
    K/V rows [length][Hkv][d]; shared rows are the same tensor rows.
    """
    lengths: List[int]
    prefix_tokens: int
    prefix_seqs: int
    tokens_k: List[torch.Tensor]
    tokens_v: List[torch.Tensor]
    q: torch.Tensor             # [B][Hq][d] fp32
    k_new: torch.Tensor         # [B][Hkv][d]
    v_new: torch.Tensor


def mix_lengths(spec: DecodeSpec = MIX, prefix_tokens: int = MIX_PREFIX_TOKENS,
                prefix_seqs: int = MIX_PREFIX_SEQS) -> List[int]:
    """The lengths mix_layout draws (its generator's first draws), without the tokens."""
    lengths = lognormal_lengths(generator(spec.seed), spec.batch, MIX_MEDIAN, MIX_SIGMA, *MIX_CLIP)
    prefix_seqs = min(prefix_seqs, spec.batch - (spec.batch % 2))
    for k in range(0, prefix_seqs, 2):
        lengths[k] = lengths[k + 1] = min(prefix_tokens + lengths[k], MIX_CLIP[1])
    return lengths


def mix_layout(spec: DecodeSpec = MIX, batch: int | None = None,
               prefix_tokens: int = MIX_PREFIX_TOKENS, prefix_seqs: int = MIX_PREFIX_SEQS,
               median: float = MIX_MEDIAN, clip=MIX_CLIP) -> MixLayout:
    gen = generator(spec.seed)
    b = spec.batch if batch is None else batch
    hkv, d, dt = spec.kv_heads, spec.head_dim, spec.cache_dtype
    lengths = lognormal_lengths(gen, b, median, MIX_SIGMA, *clip)
    prefix_seqs = min(prefix_seqs, b - (b % 2))
    # sharing sequences: prefix + own suffix; a pair shares the suffix of its first member
    for k in range(0, prefix_seqs, 2):
        total = min(prefix_tokens + lengths[k], clip[1])
        lengths[k] = lengths[k + 1] = total
    prefix_k = randn(gen, (prefix_tokens, hkv, d), dt)
    prefix_v = randn(gen, (prefix_tokens, hkv, d), dt)
    tokens_k, tokens_v = [None] * b, [None] * b
    for s in range(b):
        if s < prefix_seqs and s % 2 == 1:
            tokens_k[s], tokens_v[s] = tokens_k[s - 1], tokens_v[s - 1]
            continue
        if s < prefix_seqs:
            n_own = lengths[s] - prefix_tokens
            own_k = randn(gen, (n_own, hkv, d), dt)
            own_v = randn(gen, (n_own, hkv, d), dt)
            tokens_k[s] = torch.cat([prefix_k, own_k])
            tokens_v[s] = torch.cat([prefix_v, own_v])
        else:
            tokens_k[s] = randn(gen, (lengths[s], hkv, d), dt)
            tokens_v[s] = randn(gen, (lengths[s], hkv, d), dt)
    q = randn(gen, (b, spec.q_heads, d), torch.float32)
    k_new = randn(gen, (b, hkv, d), dt)
    v_new = randn(gen, (b, hkv, d), dt)
    return MixLayout(lengths, prefix_tokens, prefix_seqs, tokens_k, tokens_v, q, k_new, v_new)


# ---------------------------------------------------------------- varlen prefill

@dataclasses.dataclass
class PrefillInputs:
    lengths: List[int]
    cu_seqlens: torch.Tensor    # int32 [B+1]
    q: torch.Tensor             # [T][Hq][d]
    k: torch.Tensor             # [T][Hkv][d]
    v: torch.Tensor


def prefill_inputs(lengths: Sequence[int], q_heads: int, kv_heads: int, head_dim: int,
                   dtype: torch.dtype, seed: int) -> PrefillInputs:
    gen = generator(seed)
    cu = [0]
    for n in lengths:
        cu.append(cu[-1] + int(n))
    t = cu[-1]
    q = randn(gen, (t, q_heads, head_dim), dtype)
    k = randn(gen, (t, kv_heads, head_dim), dtype)
    v = randn(gen, (t, kv_heads, head_dim), dtype)
    return PrefillInputs(list(lengths), torch.tensor(cu, dtype=torch.int32), q, k, v)


def long_prefill_lengths() -> List[int]:
    return uniform_lengths(generator(LONG_GQA.seed + 1000), PREFILL_PROMPTS, *PREFILL_RANGE)
