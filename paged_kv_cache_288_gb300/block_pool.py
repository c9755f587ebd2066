"""Host-side block pool: free list, reference counts, block tables, slots.

This is the bookkeeping that sits above the kernels (it is not timed):

* a pool of ``num_blocks`` fixed-size blocks with a free list; since all
  blocks have the same size any free block fits any request, so there is no
  external fragmentation (LLM의 Paged Attention, "Paged Attention의 핵심
  원리" item 1; serving-paged-attention, "블록으로 쪼개고 표로 잇는다");
* one block table per sequence, grown one block at a time as the sequence
  grows (same sections);
* sharing by copying a table and counting references, and copy-on-write when
  a sequence is about to write into a block someone else also holds
  (serving-paged-attention, "공유는 표를 베끼는 일이 된다": prefix sharing,
  parallel sampling, beam search);
* the slot of each new token, ``block * block_size + offset``, which is what
  ``pa_reshape_and_cache`` consumes (vLLM의 핵심 이해: PagedAttention,
  section 6, the token table).

``append`` returns the (src, dst) pairs that must be copied with
``pa_copy_blocks`` before the new tokens are written.
"""

import numpy as np


class OutOfBlocks(RuntimeError):
    """The pool has no free block left (the caller must preempt or wait)."""


class BlockPool:
    def __init__(self, num_blocks, block_size):
        if num_blocks <= 0 or block_size <= 0:
            raise ValueError("num_blocks and block_size must be positive")
        self.num_blocks = int(num_blocks)
        self.block_size = int(block_size)
        # lowest ids first, so that a fresh pool hands out 0, 1, 2, ...
        self._free = list(range(self.num_blocks - 1, -1, -1))
        self.refcount = np.zeros(self.num_blocks, dtype=np.int64)
        self.tables = {}
        self.lengths = {}

    # -- pool -------------------------------------------------------------

    @property
    def num_free(self):
        return len(self._free)

    def _take(self):
        if not self._free:
            raise OutOfBlocks(f"all {self.num_blocks} blocks are in use")
        b = self._free.pop()
        assert self.refcount[b] == 0
        self.refcount[b] = 1
        return b

    def _release(self, b):
        self.refcount[b] -= 1
        assert self.refcount[b] >= 0
        if self.refcount[b] == 0:
            self._free.append(b)

    # -- sequences --------------------------------------------------------

    def add_sequence(self, seq_id, num_tokens=0):
        """New sequence holding ``num_tokens`` tokens; returns their slots."""
        if seq_id in self.tables:
            raise KeyError(f"sequence {seq_id} exists")
        if -(-int(num_tokens) // self.block_size) > self.num_free:
            raise OutOfBlocks(f"{num_tokens} tokens need more than the {self.num_free} free blocks")
        self.tables[seq_id] = []
        self.lengths[seq_id] = 0
        slots, cow = self.append(seq_id, num_tokens)
        assert not cow
        return slots

    def fork(self, parent, child, num_tokens=None):
        """``child`` shares the first ``num_tokens`` tokens (default all) of ``parent``."""
        if child in self.tables:
            raise KeyError(f"sequence {child} exists")
        n = self.lengths[parent] if num_tokens is None else int(num_tokens)
        if not 0 <= n <= self.lengths[parent]:
            raise ValueError("cannot share more tokens than the parent holds")
        nb = -(-n // self.block_size)
        shared = self.tables[parent][:nb]
        for b in shared:
            self.refcount[b] += 1
        self.tables[child] = list(shared)
        self.lengths[child] = n

    def append(self, seq_id, num_tokens=1):
        """Grow a sequence; returns (slots of the new tokens, copy-on-write pairs)."""
        table = self.tables[seq_id]
        bs = self.block_size
        n = int(num_tokens)
        pos0 = self.lengths[seq_id]
        need = max(0, -(-(pos0 + n) // bs) - len(table))
        if n > 0 and pos0 // bs < len(table) and self.refcount[table[pos0 // bs]] > 1:
            need += 1  # the shared, partly filled block is copied first
        if need > self.num_free:
            raise OutOfBlocks(f"append of {n} tokens needs {need} blocks, {self.num_free} free")
        slots, cow = [], []
        for _ in range(int(num_tokens)):
            pos = self.lengths[seq_id]
            j, off = divmod(pos, bs)
            if j == len(table):
                table.append(self._take())
            elif self.refcount[table[j]] > 1:
                src = table[j]
                dst = self._take()
                self._release(src)
                table[j] = dst
                cow.append((src, dst))
            slots.append(table[j] * bs + off)
            self.lengths[seq_id] = pos + 1
        return slots, cow

    def free_sequence(self, seq_id):
        for b in self.tables.pop(seq_id):
            self._release(b)
        del self.lengths[seq_id]

    # -- views --------------------------------------------------------------

    def block_table_array(self, seq_ids, width=None, pad=0):
        """int32 [len(seq_ids), width] tables, unused entries set to ``pad``."""
        width = width or max([len(self.tables[s]) for s in seq_ids] + [1])
        out = np.full((len(seq_ids), width), pad, dtype=np.int32)
        for i, s in enumerate(seq_ids):
            t = self.tables[s]
            if len(t) > width:
                raise ValueError("table wider than width")
            out[i, :len(t)] = t
        return out

    def context_lens(self, seq_ids):
        return np.array([self.lengths[s] for s in seq_ids], dtype=np.int32)

    def tail_waste(self, seq_id):
        """Allocated but empty token slots of this sequence (its last block's tail)."""
        return len(self.tables[seq_id]) * self.block_size - self.lengths[seq_id]

    def used_blocks(self):
        return self.num_blocks - self.num_free
