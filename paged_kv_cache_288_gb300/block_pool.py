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

``PrefixCache`` adds automatic sharing of common prompt prefixes (prefix
caching, which caches the blocks of shared prompt beginnings so that they
are neither recomputed nor stored twice: LLM 추론 확장, 품질·비용 절충 필수,
the paragraph on prefix caching; serving-paged-attention, "공유는 표를
베끼는 일이 된다", the 100 requests with one system prompt). A full block
is found by a key that chains its token ids to the key of the block before
it, so equal keys mean equal prefixes up to and including that block.
"""

import hashlib
from collections import OrderedDict

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


def block_key(parent_key, token_ids):
    """Key of a full block: BLAKE2b-128 of the parent block's key and the
    block's token ids (int64, little endian). The first block's parent key is
    the empty byte string."""
    h = hashlib.blake2b(digest_size=16)
    h.update(parent_key)
    h.update(np.asarray(token_ids, dtype="<i8").tobytes())
    return h.digest()


class PrefixCache:
    """Full blocks of earlier prompts, found by their chained keys.

    The cache holds one reference of its own on every block it maps, so a
    cached block outlives the requests that filled it; such a block with no
    other holder is evictable, least recently used first, when the pool runs
    out of free blocks. Only full blocks are cached (a partly filled last
    block still changes).
    """

    def __init__(self, pool):
        self.pool = pool
        self.block_of = {}      # key -> physical block
        self.key_of = {}        # physical block -> key
        self._lru = OrderedDict()  # cached blocks nobody else holds, oldest first
        self.hits = 0
        self.misses = 0

    def _touch(self, b):
        if self.pool.refcount[b] == 1:
            self._lru[b] = True
            self._lru.move_to_end(b)
        else:
            self._lru.pop(b, None)

    def evict(self, n):
        """Return up to n evictable cached blocks to the free list."""
        done = 0
        while done < n and self._lru:
            b, _ = self._lru.popitem(last=False)
            del self.block_of[self.key_of.pop(b)]
            self.pool._release(b)
            done += 1
        return done

    def add_sequence(self, seq_id, token_ids):
        """New sequence for a prompt: its longest cached run of full blocks is
        shared; the rest is allocated. Returns (number of prompt tokens whose
        K/V are already cached, slots of the remaining prompt tokens, which
        the caller computes and writes with pa_reshape_and_cache)."""
        pool, bs = self.pool, self.pool.block_size
        tokens = np.asarray(token_ids, dtype=np.int64)
        n_full = len(tokens) // bs
        keys, key = [], b""
        for j in range(n_full):
            key = block_key(key, tokens[j * bs:(j + 1) * bs])
            keys.append(key)
        shared = []
        for k in keys:
            b = self.block_of.get(k)
            if b is None:
                break
            shared.append(b)
        self.hits += len(shared)
        self.misses += n_full - len(shared)
        need = -(-len(tokens) // bs) - len(shared)
        if need > pool.num_free:
            # evictable blocks other than the ones this request is about to share
            for b in shared:
                self._lru.pop(b, None)
            self.evict(need - pool.num_free)
        if need > pool.num_free:
            for b in shared:
                self._touch(b)
            raise OutOfBlocks(f"prompt of {len(tokens)} tokens needs {need} blocks, {pool.num_free} free")
        if seq_id in pool.tables:
            raise KeyError(f"sequence {seq_id} exists")
        for b in shared:
            pool.refcount[b] += 1
            self._lru.pop(b, None)
        pool.tables[seq_id] = list(shared)
        pool.lengths[seq_id] = len(shared) * bs
        slots, cow = pool.append(seq_id, len(tokens) - len(shared) * bs)
        assert not cow
        # the newly filled full blocks become cached (the caller writes them
        # in the same step, before any later request can read them)
        table = pool.tables[seq_id]
        for j in range(len(shared), n_full):
            b = table[j]
            if keys[j] not in self.block_of:
                self.block_of[keys[j]] = b
                self.key_of[b] = keys[j]
                pool.refcount[b] += 1
        return len(shared) * bs, slots

    def free_sequence(self, seq_id):
        """Release a sequence; its cached blocks stay cached (evictable once no
        other sequence holds them)."""
        blocks = list(self.pool.tables[seq_id])
        self.pool.free_sequence(seq_id)
        for b in blocks:
            if b in self.key_of:
                self._touch(b)


def shared_prefix_groups(block_tables, context_lens, block_size, min_shared_blocks=1):
    """Groups of consecutive sequences that share the leading blocks of their
    tables, in the form pa_decode_shared_prefix takes.

    Sharing a prompt prefix stores its blocks once and points every table at
    them (serving-paged-attention, "공유는 표를 베끼는 일이 된다"); this finds
    that sharing again from the tables themselves, so the decode can read the
    shared blocks once per group. Walking the batch in order, a sequence
    joins the current group while its first k table entries equal the group
    leader's for some k >= min_shared_blocks (k is the group's common run,
    shrunk as members join), and only blocks that lie wholly inside every
    member's context count. Returns (group_start int32 [G + 1], group_prefix
    int32 [G] in tokens); a sequence that shares nothing is a group of its
    own with prefix 0.
    """
    tables = np.asarray(block_tables)
    lens = np.asarray(context_lens, dtype=np.int64)
    B = len(lens)
    starts, prefixes = [0], []
    i = 0
    while i < B:
        full_i = int(lens[i]) // block_size  # whole blocks of the leader
        run = full_i
        j = i + 1
        while j < B:
            full_j = int(lens[j]) // block_size
            k = min(run, full_j)
            eq = tables[i, :k] == tables[j, :k]
            common = k if eq.all() else int(np.argmin(eq))
            if common < min_shared_blocks:
                break
            run = common
            j += 1
        shared = run if j - i > 1 else 0
        prefixes.append(shared * block_size)
        starts.append(j)
        i = j
    return np.asarray(starts, dtype=np.int32), np.asarray(prefixes, dtype=np.int32)
