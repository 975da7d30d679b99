"""Host-side block manager: physical block pool, per-sequence block tables,
reference counts, fork and copy-on-write.

This is the bookkeeping that sits above the C ABI and produces its inputs
(block tables, slot mappings, copy pairs); nothing here runs on the GPU.

* Blocks of ``block_size`` tokens are handed out on demand from a free pool; a
  sequence's logical block j maps to a physical block through its table
  (plumephp.com "KV Cache 优化与注意力机制加速" §4.2-§4.3, BlockTable.allocate /
  get_kv).
* ``fork`` gives a new sequence the same table and increments every block's
  reference count (§4.3, BlockTable.fork).
* Before a sequence writes into a block whose count is above one, the block is
  copied to a fresh block which the writer takes over; the old block loses one
  reference (copy-on-write; 0539edu.com "从KV cache共享到批量调度…" §3.2, §5.2: the
  count is checked before the write).
* With a sliding window of W tokens (zwjcode.cn "KV Cache 的增量解码" §10;
  plumephp.com §5.2) ``release_outside_window`` gives back the blocks that hold
  only positions before the window: no later query of the sequence sees them.
  Their table entries become -1 and are never read.
* ``audit`` checks the invariant that every block's count equals the number of
  table entries that reference it (0539edu.com §5.2 suggests logging and checking
  every cache read/write per request).
* ``shared_prefix_groups`` finds the sequences of a batch whose leading blocks are
  the same physical blocks (a common prompt, forks) and describes them for
  pkv_decode_step_shared_prefix, which then reads each group's shared prefix once.
"""
from __future__ import annotations

import dataclasses
from collections import deque
from typing import Dict, Iterable, List, Optional, Sequence, Tuple

import torch


@dataclasses.dataclass
class PrefixGroups:
    """Groups of batch rows that share a prefix of whole physical blocks.

    ``prefix_tokens[b]`` is the number of leading tokens of batch row b in its group's
    shared prefix (0: no group); the members of group g are
    ``group_seqs[group_start[g]:group_start[g+1]]`` (batch rows).  Tensors are int32.
    """
    prefix_tokens: torch.Tensor
    group_start: torch.Tensor
    group_seqs: torch.Tensor
    max_group_size: int
    max_prefix_tokens: int

    @property
    def n_groups(self) -> int:
        return self.group_start.numel() - 1

    @property
    def n_members(self) -> int:
        return self.group_seqs.numel()

    def to(self, device) -> "PrefixGroups":
        return PrefixGroups(self.prefix_tokens.to(device), self.group_start.to(device), self.group_seqs.to(device),
                            self.max_group_size, self.max_prefix_tokens)


class OutOfBlocks(RuntimeError):
    pass


class BlockManager:
    def __init__(self, num_blocks: int, block_size: int = 16, order: Optional[Sequence[int]] = None):
        """``order``: the order in which free blocks are handed out (default 0..NB-1)."""
        if num_blocks < 1 or block_size < 1:
            raise ValueError("num_blocks and block_size must be positive")
        self.num_blocks = num_blocks
        self.block_size = block_size
        ids = list(range(num_blocks)) if order is None else [int(x) for x in order]
        if sorted(ids) != list(range(num_blocks)):
            raise ValueError("order must be a permutation of the block ids")
        self._free = deque(ids)
        self.refcount = [0] * num_blocks
        self.tables: Dict[int, List[int]] = {}
        self.lengths: Dict[int, int] = {}

    # ------------------------------------------------------------ pool
    @property
    def num_free(self) -> int:
        return len(self._free)

    def _alloc(self) -> int:
        if not self._free:
            raise OutOfBlocks("no free physical block")
        blk = self._free.popleft()
        self.refcount[blk] = 1
        return blk

    def _release(self, blk: int) -> None:
        self.refcount[blk] -= 1
        if self.refcount[blk] < 0:
            raise AssertionError(f"block {blk} released more often than referenced")
        if self.refcount[blk] == 0:
            self._free.append(blk)

    # ------------------------------------------------------- sequences
    def add_sequence(self, seq: int, num_tokens: int = 0) -> List[int]:
        """New sequence holding ``num_tokens`` tokens: ceil(n / bs) fresh blocks."""
        if seq in self.tables:
            raise KeyError(f"sequence {seq} exists")
        need = -(-num_tokens // self.block_size)
        if need > self.num_free:
            raise OutOfBlocks(f"sequence {seq} needs {need} blocks, {self.num_free} free")
        self.tables[seq] = [self._alloc() for _ in range(need)]
        self.lengths[seq] = num_tokens
        return list(self.tables[seq])

    def fork(self, parent: int, child: int) -> None:
        """``child`` shares all of ``parent``'s blocks (each count + 1)."""
        if child in self.tables:
            raise KeyError(f"sequence {child} exists")
        table = list(self.tables[parent])
        for blk in table:
            if blk >= 0:
                self.refcount[blk] += 1
        self.tables[child] = table
        self.lengths[child] = self.lengths[parent]

    def free_sequence(self, seq: int) -> None:
        for blk in self.tables.pop(seq):
            if blk >= 0:
                self._release(blk)
        del self.lengths[seq]

    def release_outside_window(self, seq: int, window: int) -> List[int]:
        """Give back the blocks of ``seq`` that hold only positions before its last
        ``window`` tokens; returns their ids.  The current query (position len - 1) sees
        positions len - window .. len - 1, and later queries see later ones."""
        if window <= 0:
            return []
        lo = self.lengths[seq] - window
        table = self.tables[seq]
        released = []
        for j in range(max(0, lo) // self.block_size):   # blocks ending at or before lo
            if table[j] >= 0:
                self._release(table[j])
                released.append(table[j])
                table[j] = -1
        return released

    def slot(self, seq: int, pos: int) -> int:
        """Cache slot of logical position ``pos``: table[pos // bs] * bs + pos % bs."""
        blk = self.tables[seq][pos // self.block_size]
        if blk < 0:
            raise KeyError(f"position {pos} of sequence {seq} lies in a released block")
        return blk * self.block_size + pos % self.block_size

    def append_slot(self, seq: int) -> Tuple[int, Optional[Tuple[int, int]]]:
        """Reserve the slot of the next token of ``seq``.

        Returns (slot, copy) where ``copy`` is a (src, dst) block pair that must be
        copied before the token is written (copy-on-write), or None.
        """
        pos = self.lengths[seq]
        table = self.tables[seq]
        copy = None
        if pos % self.block_size == 0:
            table.append(self._alloc())
        else:
            last = table[-1]
            if self.refcount[last] > 1:
                new = self._alloc()
                self._release(last)
                table[-1] = new
                copy = (last, new)
        self.lengths[seq] = pos + 1
        return self.slot(seq, pos), copy

    def append_step(self, seqs: Iterable[int]) -> Tuple[List[int], List[Tuple[int, int]]]:
        """One decode step: a slot for every sequence, plus the COW copies to run first."""
        slots, copies = [], []
        for s in seqs:
            slot, copy = self.append_slot(s)
            slots.append(slot)
            if copy is not None:
                copies.append(copy)
        return slots, copies

    # ---------------------------------------------------------- tensors
    def block_table(self, seqs: Sequence[int], max_blocks: Optional[int] = None,
                    pad: int = -1) -> torch.Tensor:
        mbs = max_blocks if max_blocks is not None else max(1, max(len(self.tables[s]) for s in seqs))
        out = torch.full((len(seqs), mbs), pad, dtype=torch.int32)
        for r, s in enumerate(seqs):
            t = self.tables[s]
            if len(t) > mbs:
                raise ValueError(f"sequence {s} has {len(t)} blocks > max_blocks {mbs}")
            if t:
                out[r, :len(t)] = torch.tensor(t, dtype=torch.int32)
        return out

    def context_lens(self, seqs: Sequence[int]) -> torch.Tensor:
        return torch.tensor([self.lengths[s] for s in seqs], dtype=torch.int32)

    def slot_mapping(self, seq: int, positions: Iterable[int]) -> torch.Tensor:
        return torch.tensor([self.slot(seq, p) for p in positions], dtype=torch.int64)

    # ----------------------------------------------------------- checks
    def shared_prefix_groups(self, seqs: Sequence[int], min_members: int = 2, min_blocks: int = 1) -> PrefixGroups:
        """Group the batch rows whose sequences start with the same physical blocks.

        Rows whose first block is the same shared block form a group; its prefix is the
        longest run of leading table entries common to every member, cut so that it ends
        before every member's last position (the step's new token is never in it).  Groups
        of fewer than ``min_members`` rows or ``min_blocks`` blocks are dropped.
        """
        seqs = list(seqs)
        by_first: Dict[int, List[int]] = {}
        for row, s in enumerate(seqs):
            t = self.tables[s]
            if t and self.refcount[t[0]] > 1:
                by_first.setdefault(t[0], []).append(row)
        bs = self.block_size
        prefix = [0] * len(seqs)
        starts, members = [0], []
        for rows in by_first.values():
            if len(rows) < min_members:
                continue
            tabs = [self.tables[seqs[r]] for r in rows]
            n = min(len(t) for t in tabs)
            pages = 0
            while pages < n and all(t[pages] == tabs[0][pages] for t in tabs):
                pages += 1
            pages = min(pages, min((self.lengths[seqs[r]] - 1) // bs for r in rows))
            if pages < min_blocks:
                continue
            for r in rows:
                prefix[r] = pages * bs
            members.extend(rows)
            starts.append(len(members))
        sizes = [b - a for a, b in zip(starts, starts[1:])]
        return PrefixGroups(torch.tensor(prefix, dtype=torch.int32), torch.tensor(starts, dtype=torch.int32),
                            torch.tensor(members, dtype=torch.int32), max(sizes, default=0), max(prefix, default=0))

    def audit(self) -> None:
        """Every block's count equals its table references; free blocks have count 0."""
        refs = [0] * self.num_blocks
        for table in self.tables.values():
            for blk in table:
                if blk >= 0:
                    refs[blk] += 1
        if refs != self.refcount:
            bad = [b for b in range(self.num_blocks) if refs[b] != self.refcount[b]][:8]
            raise AssertionError(f"refcount mismatch at blocks {bad}")
        free = set(self._free)
        if len(free) != len(self._free):
            raise AssertionError("a block is on the free list twice")
        for b in range(self.num_blocks):
            if (b in free) != (self.refcount[b] == 0):
                raise AssertionError(f"block {b}: free-list membership disagrees with its count")
