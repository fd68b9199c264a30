"""Host-side block manager: the logical -> physical map that the kernels consume.

This is the bookkeeping half of PagedAttention, kept on the host as in the
pages' system: the kernels only ever see, per sequence, a list of physical
block ids (the block table), per new token a physical slot (the slot mapping),
and per step a list of pending copy-on-write block copies.

Behaviour follows:

* CS349E Lecture 7 notes (KV Cache Management), §4.1 "块与块表": fixed-size
  blocks of B tokens, one block table per sequence, on-demand allocation (a new
  physical block only when the last one is full), so at most B-1 slots of a
  sequence are ever unused.
* same notes, §5.1 "并行采样：fork + 写时复制" and §5.3: fork shares every
  block and raises its reference count; appending into a shared (refcount > 1)
  last block first copies it (copy-on-write), so n samples forked from one
  prompt whose last block is partial cause n-1 copies, and none when the prompt
  length is a multiple of B (exercise 4 of the same notes); free lowers the
  counts and returns blocks that reach zero to the free list.
* CMU 15-779 Lecture 16 notes (LLM Serving 1), §3.3 "KV 块与块表": the block
  table walk-through with B = 4 (logical 0 -> physical 3, logical 1 -> physical
  2, a third block allocated only when the second is full).

A slot is ``physical_block * B + offset``; ``-1`` in a slot mapping means
"no write" (padding).
"""
from __future__ import annotations

from collections import deque
from dataclasses import dataclass, field


class OutOfBlocks(RuntimeError):
    """The free list is empty."""


@dataclass
class Sequence:
    seq_id: int
    num_tokens: int = 0
    block_ids: list = field(default_factory=list)


class BlockManager:
    """Reference-counted pool of ``num_blocks`` physical blocks of ``block_size`` tokens.

    ``free_order`` fixes the order in which free blocks are handed out (the
    synthetic workloads pass a seeded permutation so that a sequence's blocks
    land at scattered physical places).
    """

    def __init__(self, num_blocks: int, block_size: int, free_order=None):
        if num_blocks <= 0 or block_size <= 0:
            raise ValueError("num_blocks and block_size must be positive")
        self.num_blocks = num_blocks
        self.block_size = block_size
        order = list(range(num_blocks)) if free_order is None else [int(b) for b in free_order]
        if len(set(order)) != len(order) or any(b < 0 or b >= num_blocks for b in order):
            raise ValueError("free_order must list distinct block ids in [0, num_blocks)")
        self.free = deque(order)
        self.refcount = [0] * num_blocks
        for b in set(range(num_blocks)) - set(order):
            self.refcount[b] = 1  # held by someone outside this manager
        self.seqs: dict[int, Sequence] = {}
        self.copies_issued = 0

    # -- allocation -------------------------------------------------------
    def _take(self) -> int:
        if not self.free:
            raise OutOfBlocks("no free physical block")
        b = self.free.popleft()
        assert self.refcount[b] == 0
        self.refcount[b] = 1
        return b

    def _release(self, b: int) -> None:
        self.refcount[b] -= 1
        assert self.refcount[b] >= 0
        if self.refcount[b] == 0:
            self.free.append(b)

    def num_free(self) -> int:
        return len(self.free)

    # -- sequence operations (fork / append / free) ------------------------
    def add_sequence(self, seq_id: int, num_prompt_tokens: int) -> None:
        """Prefill: allocate ceil(n / B) blocks for an n-token prompt."""
        if seq_id in self.seqs:
            raise ValueError(f"sequence {seq_id} exists")
        B = self.block_size
        nblk = -(-num_prompt_tokens // B)
        if nblk > len(self.free):
            raise OutOfBlocks(f"prompt needs {nblk} blocks, {len(self.free)} free")
        self.seqs[seq_id] = Sequence(seq_id, num_prompt_tokens, [self._take() for _ in range(nblk)])

    def fork(self, parent_id: int, child_id: int) -> None:
        """The child shares every block of the parent (refcount + 1 each)."""
        if child_id in self.seqs:
            raise ValueError(f"sequence {child_id} exists")
        p = self.seqs[parent_id]
        for b in p.block_ids:
            self.refcount[b] += 1
        self.seqs[child_id] = Sequence(child_id, p.num_tokens, list(p.block_ids))

    def append_slot(self, seq_id: int):
        """Reserve the slot for the sequence's next token.

        Returns ``(slot, cow_pair)``; ``cow_pair`` is ``(src, dst)`` when the
        last block was shared and had to be copied before this write, else None.
        """
        seq = self.seqs[seq_id]
        B = self.block_size
        offset = seq.num_tokens % B
        pair = None
        if offset == 0:
            seq.block_ids.append(self._take())
        else:
            last = seq.block_ids[-1]
            if self.refcount[last] > 1:
                new = self._take()
                self.refcount[last] -= 1
                seq.block_ids[-1] = new
                pair = (last, new)
                self.copies_issued += 1
        seq.num_tokens += 1
        return seq.block_ids[-1] * B + offset, pair

    def free_sequence(self, seq_id: int) -> None:
        seq = self.seqs.pop(seq_id)
        for b in seq.block_ids:
            self._release(b)

    # -- views handed to the kernels ----------------------------------------
    def slot_of(self, seq_id: int, position: int) -> int:
        seq = self.seqs[seq_id]
        if not 0 <= position < seq.num_tokens:
            raise IndexError(position)
        B = self.block_size
        return seq.block_ids[position // B] * B + position % B

    def block_table(self, seq_id: int) -> list:
        return list(self.seqs[seq_id].block_ids)

    def context_len(self, seq_id: int) -> int:
        return self.seqs[seq_id].num_tokens


class NativeBlockManager:
    """The library's C++ block manager (``pa_bm_*`` in ``include/pa.h``), with prefix caching.

    Same operations as :class:`BlockManager` plus token-aware prefill that
    reuses cached block-aligned prefixes (chain hash of parent hash and block
    tokens) and LRU eviction of released cached blocks.
    """

    def __init__(self, num_blocks: int, block_size: int, prefix_caching: bool = True):
        import ctypes
        from . import library
        self._ct = ctypes
        self._lib = library()
        self._h = self._lib.pa_bm_create(int(num_blocks), int(block_size), 1 if prefix_caching else 0)
        if not self._h:
            raise ValueError("bad block manager sizes")
        self.num_blocks, self.block_size = num_blocks, block_size

    def __del__(self):
        h = getattr(self, "_h", None)
        if h:
            self._lib.pa_bm_destroy(h)
            self._h = None

    def _check(self, st, what):
        if st == 5:
            raise OutOfBlocks(what)
        if st != 0:
            raise ValueError(f"{what}: status {st}")

    def add_sequence(self, seq_id: int, tokens) -> int:
        """Prefill ``tokens``; returns how many leading tokens came from the prefix cache."""
        ct = self._ct
        toks = (ct.c_int32 * len(tokens))(*[int(t) for t in tokens])
        cached = ct.c_int32(0)
        self._check(self._lib.pa_bm_add_sequence(self._h, int(seq_id), toks, len(tokens), ct.byref(cached)),
                    "add_sequence")
        return int(cached.value)

    def fork(self, parent_id: int, child_id: int) -> None:
        self._check(self._lib.pa_bm_fork(self._h, int(parent_id), int(child_id)), "fork")

    def append_slot(self, seq_id: int, token: int = 0):
        ct = self._ct
        slot, src, dst = ct.c_int64(), ct.c_int64(), ct.c_int64()
        self._check(self._lib.pa_bm_append(self._h, int(seq_id), int(token), ct.byref(slot), ct.byref(src),
                                           ct.byref(dst)), "append")
        return int(slot.value), (None if src.value < 0 else (int(src.value), int(dst.value)))

    def free_sequence(self, seq_id: int) -> None:
        self._check(self._lib.pa_bm_free(self._h, int(seq_id)), "free")

    def block_table(self, seq_id: int) -> list:
        n = self._lib.pa_bm_block_table(self._h, int(seq_id), None, 0)
        if n < 0:
            raise KeyError(seq_id)
        buf = (self._ct.c_int32 * max(1, n))()
        self._lib.pa_bm_block_table(self._h, int(seq_id), buf, n)
        return list(buf[:n])

    def context_len(self, seq_id: int) -> int:
        return int(self._lib.pa_bm_context_len(self._h, int(seq_id)))

    def num_free(self) -> int:
        return int(self._lib.pa_bm_num_free(self._h))

    def stats(self) -> dict:
        out = (self._ct.c_int64 * 6)()
        self._lib.pa_bm_stats(self._h, out)
        return dict(zip(("queries", "hits", "evictions", "copies", "evictable", "cached"), list(out)))
