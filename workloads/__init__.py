"""Seeded synthetic inputs for paged KV-cache decode.

Shared by the tests and by ``bench.py``: this module only draws inputs
(random token values, context lengths, physical block placement, slots of new
tokens, fp8 scales) and computes none of the operations under test. Neither
the oracle nor the CUDA library is imported here.

Inputs follow the shapes of the five workloads:

* ``tiny``: 4 sequences of 5/17/33/64 tokens, 4 query / 2 KV heads, head dim
  64, fp16, block size 16, a 64-block pool, then one appended token each.
* ``llama8b``: batch 64, 32/8 heads, head dim 128, bf16, block size 16,
  context lengths uniform in [128, 4096], pool 1.25x the need, table width 256.
* ``shared_prefix``: 100 sequences sharing a 1016-token prefix (64 blocks, the
  last one holding 8 tokens), each with a private suffix of 32..512 tokens
  that starts mid-block, fp16, 32/8/128.
* ``long_context``: batch 8, 32768 tokens each, bf16, 32/8/128, block size
  8/16/32/64.
* ``fp8_step``: batch 256, 32/8/128, block size 16, lognormal lengths (mean
  500, clipped to [16, 2048]), E4M3 KV with one float32 scale per (block, KV
  head), bf16 queries.
* ``prefill``: chunked prefill, 16 sequences with cached prefixes uniform in
  [0, 2048] tokens and a 512-token chunk of new queries each, 32/8/128, bf16,
  block size 16.

Random values are i.i.d. N(0, 1) drawn with ``torch.Generator('cpu')`` and
rounded to the storage type. Physical block ids are a seeded permutation of
the pool handed out in logical order. Unused table entries point at a
dedicated poison block whose every value is NaN, and the unused tail slots of
each sequence's last block are NaN too, so any read past a sequence's data
shows up as NaN in the output instead of an out-of-bounds access.
"""

from dataclasses import dataclass, field
import math

import numpy as np
import torch

F16 = "f16"
BF16 = "bf16"
FP8_E4M3 = "fp8_e4m3"

NAN_BITS = {F16: 0x7E00, BF16: 0x7FC0, FP8_E4M3: 0x7F}
_TORCH_16 = {F16: torch.float16, BF16: torch.bfloat16}


def elem_bytes(dtype):
    return 1 if dtype == FP8_E4M3 else 2


def _gen(seed):
    g = torch.Generator("cpu")
    g.manual_seed(int(seed))
    return g


def normal_bits(g, shape, dtype, chunk=1 << 24, sigma=1.0):
    """N(0, sigma^2) values rounded to f16/bf16, returned as raw uint16 bits
    (sigma = 1 leaves the N(0,1) draws unchanged)."""
    n = int(np.prod(shape)) if len(shape) else 1
    out = np.empty(n, dtype=np.uint16)
    for start in range(0, n, chunk):
        m = min(chunk, n - start)
        x = torch.randn(m, generator=g, dtype=torch.float32)
        if sigma != 1.0:
            x = x * float(sigma)
        x = x.to(_TORCH_16[dtype])
        out[start:start + m] = x.view(torch.int16).numpy().view(np.uint16)
    return out.reshape(shape)


def _bits_to_f32(bits, dtype):
    if dtype == F16:
        return bits.view(np.float16).astype(np.float32)
    return (bits.astype(np.uint32) << 16).view(np.float32)


@dataclass
class DecodeCase:
    """Everything one decode (optionally preceded by cache writes) needs."""

    name: str
    num_seqs: int
    num_heads: int
    num_kv_heads: int
    head_dim: int
    block_size: int
    num_blocks: int
    q_dtype: str
    kv_dtype: str
    scale: float
    q: np.ndarray                 # [B, Hq, d] raw bits
    k_cache: np.ndarray           # [Nb, Hkv, bs, d] raw bits
    v_cache: np.ndarray
    block_tables: np.ndarray      # int32 [B, max_blocks]
    context_lens: np.ndarray      # int32 [B]
    k_scale: np.ndarray = None    # float32 [Nb, Hkv] (fp8 only)
    v_scale: np.ndarray = None
    poison_block: int = -1
    # cache writes that precede the decode (new tokens)
    new_key: np.ndarray = None    # [T, Hkv, d] raw bits (source dtype)
    new_value: np.ndarray = None
    slot_mapping: np.ndarray = None  # int64 [T]
    src_dtype: str = None
    # copy-on-write pairs applied before the writes
    cow_pairs: np.ndarray = None  # int64 [P, 2]
    meta: dict = field(default_factory=dict)

    @property
    def max_blocks_per_seq(self):
        return int(self.block_tables.shape[1])

    @property
    def max_context_len(self):
        return int(self.context_lens.max()) if self.num_seqs else 0


def _assign_tables(g, nblocks_per_seq, num_blocks, width, poison_block):
    """Hand out a seeded permutation of the pool in logical order."""
    usable = [b for b in range(num_blocks) if b != poison_block]
    perm = torch.randperm(len(usable), generator=g).numpy()
    ids = np.asarray(usable, dtype=np.int64)[perm]
    tables = np.full((len(nblocks_per_seq), width), poison_block, dtype=np.int32)
    cursor = 0
    for i, nb in enumerate(nblocks_per_seq):
        tables[i, :nb] = ids[cursor:cursor + nb]
        cursor += nb
    return tables, ids[cursor:]


def _poison_tails(cache, tables, context_lens, block_size, dtype):
    nan = NAN_BITS[dtype]
    for i, ctx in enumerate(context_lens):
        ctx = int(ctx)
        if ctx <= 0:
            continue
        nb = -(-ctx // block_size)
        used_in_last = ctx - (nb - 1) * block_size
        if used_in_last < block_size:
            cache[tables[i, nb - 1], :, used_in_last:, :] = nan


def paged_case(seed, context_lens, num_heads, num_kv_heads, head_dim, block_size,
               dtype, *, pool_factor=1.25, table_width=None, name="custom",
               scale=None, append=False, q_dtype=None):
    """A 16-bit paged decode problem with random K/V already in the pool.

    With ``append=True`` the last token of every sequence is also returned as a
    new token (key, value, slot) so that a cache write can precede the decode;
    its slot holds unrelated random values before that write.
    """
    g = _gen(seed)
    ctx = np.asarray(context_lens, dtype=np.int64)
    nbs = [int(-(-c // block_size)) if c > 0 else 0 for c in ctx]
    need = sum(nbs)
    num_blocks = max(int(math.ceil(pool_factor * need)), need) + 1
    poison = int(torch.randint(num_blocks, (1,), generator=g).item())
    width = table_width or max(max(nbs) if nbs else 1, 1)
    tables, _ = _assign_tables(g, nbs, num_blocks, width, poison)
    shape = (num_blocks, num_kv_heads, block_size, head_dim)
    k_cache = normal_bits(g, shape, dtype)
    v_cache = normal_bits(g, shape, dtype)
    k_cache[poison] = NAN_BITS[dtype]
    v_cache[poison] = NAN_BITS[dtype]
    _poison_tails(k_cache, tables, ctx, block_size, dtype)
    _poison_tails(v_cache, tables, ctx, block_size, dtype)
    q_dtype = q_dtype or dtype
    q = normal_bits(g, (len(ctx), num_heads, head_dim), q_dtype)
    case = DecodeCase(
        name=name, num_seqs=len(ctx), num_heads=num_heads, num_kv_heads=num_kv_heads,
        head_dim=head_dim, block_size=block_size, num_blocks=num_blocks,
        q_dtype=q_dtype, kv_dtype=dtype,
        scale=float(scale if scale is not None else 1.0 / math.sqrt(head_dim)),
        q=q, k_cache=k_cache, v_cache=v_cache, block_tables=tables,
        context_lens=ctx.astype(np.int32), poison_block=poison)
    if append:
        T = len(ctx)
        case.new_key = normal_bits(g, (T, num_kv_heads, head_dim), dtype)
        case.new_value = normal_bits(g, (T, num_kv_heads, head_dim), dtype)
        slots = np.full(T, -1, dtype=np.int64)
        for i, c in enumerate(ctx):
            if c > 0:
                pos = int(c) - 1
                slots[i] = int(tables[i, pos // block_size]) * block_size + pos % block_size
        case.slot_mapping = slots
        case.src_dtype = dtype
    return case


def tiny(seed=1001):
    """Tiny case: lengths 5/17/33/64, 4/2 heads, d 64, fp16, 64-block pool.

    Returns (before, step): ``before`` is the decode problem at the initial
    lengths; ``step`` carries one new token per sequence (the 64-token
    sequence opens a fresh block) and the lengths after it.
    """
    g = _gen(seed)
    bs, Hq, Hkv, d, dtype = 16, 4, 2, 64, F16
    ctx0 = np.array([5, 17, 33, 64], dtype=np.int64)
    num_blocks = 64
    nbs_after = [int(-(-(c + 1) // bs)) for c in ctx0]
    perm = torch.randperm(num_blocks, generator=g).numpy().astype(np.int64)
    poison = int(perm[-1])
    width = max(nbs_after)
    tables = np.full((4, width), poison, dtype=np.int32)
    cursor = 0
    for i, nb in enumerate(nbs_after):
        tables[i, :nb] = perm[cursor:cursor + nb]
        cursor += nb
    shape = (num_blocks, Hkv, bs, d)
    k_cache = normal_bits(g, shape, dtype)
    v_cache = normal_bits(g, shape, dtype)
    k_cache[poison] = NAN_BITS[dtype]
    v_cache[poison] = NAN_BITS[dtype]
    _poison_tails(k_cache, tables, ctx0, bs, dtype)
    _poison_tails(v_cache, tables, ctx0, bs, dtype)
    # the block opened by the append is not referenced before it
    for i, c in enumerate(ctx0):
        if c % bs == 0:
            k_cache[tables[i, c // bs]] = NAN_BITS[dtype]
            v_cache[tables[i, c // bs]] = NAN_BITS[dtype]
    q0 = normal_bits(g, (4, Hq, d), dtype)
    before = DecodeCase(
        name="tiny", num_seqs=4, num_heads=Hq, num_kv_heads=Hkv, head_dim=d,
        block_size=bs, num_blocks=num_blocks, q_dtype=dtype, kv_dtype=dtype,
        scale=1.0 / math.sqrt(d), q=q0, k_cache=k_cache, v_cache=v_cache,
        block_tables=tables, context_lens=ctx0.astype(np.int32), poison_block=poison)
    new_key = normal_bits(g, (4, Hkv, d), dtype)
    new_value = normal_bits(g, (4, Hkv, d), dtype)
    slots = np.array([int(tables[i, c // bs]) * bs + int(c % bs) for i, c in enumerate(ctx0)],
                     dtype=np.int64)
    q1 = normal_bits(g, (4, Hq, d), dtype)
    step = DecodeCase(
        name="tiny_append", num_seqs=4, num_heads=Hq, num_kv_heads=Hkv, head_dim=d,
        block_size=bs, num_blocks=num_blocks, q_dtype=dtype, kv_dtype=dtype,
        scale=1.0 / math.sqrt(d), q=q1, k_cache=None, v_cache=None,
        block_tables=tables, context_lens=(ctx0 + 1).astype(np.int32), poison_block=poison,
        new_key=new_key, new_value=new_value, slot_mapping=slots, src_dtype=dtype)
    return before, step


def llama8b_lengths(seed=1002, num_seqs=64, lo=128, hi=4096):
    g = _gen(seed)
    return torch.randint(lo, hi + 1, (num_seqs,), generator=g).numpy().astype(np.int64)


def llama8b(seed=1002, num_seqs=64, append=True):
    """Batch-64 Llama-8B-shaped decode: 32/8 heads, d 128, bf16, bs 16."""
    ctx = llama8b_lengths(seed, num_seqs)
    return paged_case(seed + 100, ctx, 32, 8, 128, 16, BF16, pool_factor=1.25,
                      table_width=256, name="llama8b", append=append)


def long_context(block_size, seed=1004, num_seqs=8, context_len=32768):
    """Batch-8 x 32768-token decode for the split path, bf16, 32/8/128."""
    ctx = np.full(num_seqs, context_len, dtype=np.int64)
    return paged_case(seed + block_size, ctx, 32, 8, 128, block_size, BF16,
                      pool_factor=1.25, name=f"long_context_bs{block_size}", append=True)


def shared_prefix(seed=1003, num_seqs=100, prefix_len=1016, suffix_lo=32, suffix_hi=512,
                  num_heads=32, num_kv_heads=8, head_dim=128, block_size=16, dtype=F16):
    """Sequences sharing one prefix, each with a private suffix from mid-block.

    Prefix blocks are shared by every table. The prefix's last block is only
    partly filled, so each sequence first receives a private copy of it
    (``cow_pairs``: shared block -> private block, applied to K and V), then
    its suffix tokens are written (``new_key``/``new_value``/``slot_mapping``
    against the post-copy tables), then all sequences decode.
    """
    g = _gen(seed)
    bs = block_size
    suffix = torch.randint(suffix_lo, suffix_hi + 1, (num_seqs,), generator=g).numpy().astype(np.int64)
    ctx = prefix_len + suffix
    n_prefix = -(-prefix_len // bs)
    nbs = [int(-(-c // bs)) for c in ctx]
    private_need = sum(nb - n_prefix + 1 for nb in nbs)  # copy of the last shared block + suffix blocks
    need = n_prefix + private_need
    num_blocks = int(math.ceil(1.25 * need)) + 1
    perm = torch.randperm(num_blocks, generator=g).numpy().astype(np.int64)
    poison = int(perm[-1])
    shared = perm[:n_prefix]
    cursor = n_prefix
    width = max(nbs)
    tables = np.full((num_seqs, width), poison, dtype=np.int32)
    tables_before = np.full((num_seqs, width), poison, dtype=np.int32)
    cow = np.zeros((num_seqs, 2), dtype=np.int64)
    for i, nb in enumerate(nbs):
        tables_before[i, :n_prefix] = shared
        tables[i, :n_prefix - 1] = shared[:-1]
        own = perm[cursor:cursor + (nb - n_prefix + 1)]
        cursor += nb - n_prefix + 1
        tables[i, n_prefix - 1:nb] = own
        cow[i] = (shared[-1], own[0])
    shape = (num_blocks, num_kv_heads, bs, head_dim)
    k_cache = normal_bits(g, shape, dtype)
    v_cache = normal_bits(g, shape, dtype)
    # every block that is not prefix data starts out as NaN poison
    prefix_set = set(int(b) for b in shared)
    for b in range(num_blocks):
        if b not in prefix_set:
            k_cache[b] = NAN_BITS[dtype]
            v_cache[b] = NAN_BITS[dtype]
    last_used = prefix_len - (n_prefix - 1) * bs
    k_cache[shared[-1], :, last_used:, :] = NAN_BITS[dtype]
    v_cache[shared[-1], :, last_used:, :] = NAN_BITS[dtype]
    # suffix tokens and their slots in the post-copy tables
    T = int(suffix.sum())
    new_key = normal_bits(g, (T, num_kv_heads, head_dim), dtype)
    new_value = normal_bits(g, (T, num_kv_heads, head_dim), dtype)
    slots = np.empty(T, dtype=np.int64)
    t = 0
    for i in range(num_seqs):
        for pos in range(prefix_len, int(ctx[i])):
            slots[t] = int(tables[i, pos // bs]) * bs + pos % bs
            t += 1
    q = normal_bits(g, (num_seqs, num_heads, head_dim), dtype)
    return DecodeCase(
        name="shared_prefix", num_seqs=num_seqs, num_heads=num_heads,
        num_kv_heads=num_kv_heads, head_dim=head_dim, block_size=bs,
        num_blocks=num_blocks, q_dtype=dtype, kv_dtype=dtype,
        scale=1.0 / math.sqrt(head_dim), q=q, k_cache=k_cache, v_cache=v_cache,
        block_tables=tables, context_lens=ctx.astype(np.int32), poison_block=poison,
        new_key=new_key, new_value=new_value, slot_mapping=slots, src_dtype=dtype,
        cow_pairs=cow, meta={"tables_before_copy": tables_before, "shared_blocks": shared,
                             "prefix_len": prefix_len})


def fp8_lengths(seed=1005, num_seqs=256, mean=500.0, sigma=1.0, lo=16, hi=2048):
    g = _gen(seed)
    mu = math.log(mean) - sigma * sigma / 2.0
    z = torch.randn(num_seqs, generator=g, dtype=torch.float64).numpy()
    return np.clip(np.rint(np.exp(mu + sigma * z)), lo, hi).astype(np.int64)


def fp8_layer(seed, context_lens, num_heads=32, num_kv_heads=8, head_dim=128,
              block_size=16, src_dtype=BF16, pool_factor=1.25, name="fp8_layer",
              k_sigma=1.0, v_sigma=1.0):
    """One layer of an E4M3 KV cache, to be filled by cache writes.

    Every token of every sequence is a new token (bf16 N(0,1) key and value
    plus its slot, or N(0, k_sigma^2) / N(0, v_sigma^2) when given); the pool
    starts as NaN poison. Each (block, KV head) gets the scale amax/448 over
    the values that will be written into it (1.0 when that amax is 0), fixed
    before any write, as a caller would choose it.
    """
    g = _gen(seed)
    bs = block_size
    ctx = np.asarray(context_lens, dtype=np.int64)
    nbs = [int(-(-c // bs)) if c > 0 else 0 for c in ctx]
    need = sum(nbs)
    num_blocks = max(int(math.ceil(pool_factor * need)), need) + 1
    poison = int(torch.randint(num_blocks, (1,), generator=g).item())
    tables, _ = _assign_tables(g, nbs, num_blocks, max(max(nbs), 1), poison)
    T = int(ctx.sum())
    key = normal_bits(g, (T, num_kv_heads, head_dim), src_dtype, sigma=k_sigma)
    value = normal_bits(g, (T, num_kv_heads, head_dim), src_dtype, sigma=v_sigma)
    seq_of = np.repeat(np.arange(len(ctx)), ctx)
    pos = np.concatenate([np.arange(c) for c in ctx]) if T else np.zeros(0, np.int64)
    blk = tables[seq_of, pos // bs].astype(np.int64)
    slots = blk * bs + pos % bs
    k_amax = np.zeros((num_blocks, num_kv_heads), dtype=np.float32)
    v_amax = np.zeros((num_blocks, num_kv_heads), dtype=np.float32)
    ka = np.abs(_bits_to_f32(key, src_dtype)).max(axis=2)    # [T, Hkv]
    va = np.abs(_bits_to_f32(value, src_dtype)).max(axis=2)
    np.maximum.at(k_amax, blk, ka)
    np.maximum.at(v_amax, blk, va)
    k_scale = np.where(k_amax > 0, k_amax / np.float32(448.0), np.float32(1.0)).astype(np.float32)
    v_scale = np.where(v_amax > 0, v_amax / np.float32(448.0), np.float32(1.0)).astype(np.float32)
    shape = (num_blocks, num_kv_heads, bs, head_dim)
    k_cache = np.full(shape, NAN_BITS[FP8_E4M3], dtype=np.uint8)
    v_cache = np.full(shape, NAN_BITS[FP8_E4M3], dtype=np.uint8)
    q = normal_bits(g, (len(ctx), num_heads, head_dim), src_dtype)
    return DecodeCase(
        name=name, num_seqs=len(ctx), num_heads=num_heads, num_kv_heads=num_kv_heads,
        head_dim=head_dim, block_size=bs, num_blocks=num_blocks, q_dtype=src_dtype,
        kv_dtype=FP8_E4M3, scale=1.0 / math.sqrt(head_dim), q=q, k_cache=k_cache,
        v_cache=v_cache, block_tables=tables, context_lens=ctx.astype(np.int32),
        k_scale=k_scale, v_scale=v_scale, poison_block=poison, new_key=key,
        new_value=value, slot_mapping=slots.astype(np.int64), src_dtype=src_dtype)


def fp8_step_layer(layer, seed=1005, num_seqs=256):
    """Layer ``layer`` of the 32-layer fp8 decode step (lognormal lengths)."""
    ctx = fp8_lengths(seed, num_seqs)
    return fp8_layer(seed * 100 + layer, ctx, name=f"fp8_step_layer{layer}")


def random_small_case(seed, *, num_seqs, group, num_kv_heads, head_dim, block_size,
                      dtype, max_ctx, min_ctx=1, q_dtype=None, append=False):
    """Randomised small shapes for parity sweeps (lengths uniform in [min,max])."""
    g = _gen(seed)
    ctx = torch.randint(min_ctx, max_ctx + 1, (num_seqs,), generator=g).numpy().astype(np.int64)
    return paged_case(seed + 7, ctx, group * num_kv_heads, num_kv_heads, head_dim,
                      block_size, dtype, name=f"rand{seed}", append=append, q_dtype=q_dtype)


@dataclass
class PrefillCase:
    """A chunked-prefill problem: every sequence's last chunk of tokens are
    queries; the K/V of all its tokens (chunk included) are in the pool."""

    num_seqs: int
    num_heads: int
    num_kv_heads: int
    head_dim: int
    block_size: int
    num_blocks: int
    dtype: str
    scale: float
    q: np.ndarray                 # [T, Hq, d] raw bits, chunks packed in sequence order
    k_cache: np.ndarray           # [Nb, Hkv, bs, d] raw bits
    v_cache: np.ndarray
    block_tables: np.ndarray      # int32 [B, width]
    context_lens: np.ndarray      # int32 [B], chunk included
    query_start: np.ndarray       # int32 [B + 1]
    new_key: np.ndarray           # [T, Hkv, d]: the chunks' K/V, as stored in the pool
    new_value: np.ndarray
    slot_mapping: np.ndarray      # int64 [T]: the chunks' slots
    poison_block: int = -1

    @property
    def max_query_len(self):
        return int(np.diff(self.query_start).max()) if self.num_seqs else 0


def prefill_case(seed, prefix_lens, chunk_lens, num_heads, num_kv_heads, head_dim, block_size,
                 dtype, *, pool_factor=1.25, table_width=None):
    """Random K/V for every token of prefix + chunk, queries for the chunks."""
    g = _gen(seed)
    pre = np.asarray(prefix_lens, dtype=np.int64)
    chunk = np.asarray(chunk_lens, dtype=np.int64)
    ctx = pre + chunk
    bs = block_size
    nbs = [int(-(-c // bs)) for c in ctx]
    need = sum(nbs)
    num_blocks = max(int(math.ceil(pool_factor * need)), need) + 1
    poison = int(torch.randint(num_blocks, (1,), generator=g).item())
    width = table_width or max(max(nbs + [1]), 1)
    tables, _ = _assign_tables(g, nbs, num_blocks, width, poison)
    shape = (num_blocks, num_kv_heads, bs, head_dim)
    k_cache = normal_bits(g, shape, dtype)
    v_cache = normal_bits(g, shape, dtype)
    k_cache[poison] = NAN_BITS[dtype]
    v_cache[poison] = NAN_BITS[dtype]
    _poison_tails(k_cache, tables, ctx, bs, dtype)
    _poison_tails(v_cache, tables, ctx, bs, dtype)
    qs = np.zeros(len(ctx) + 1, dtype=np.int32)
    qs[1:] = np.cumsum(chunk)
    T = int(qs[-1])
    slots = np.empty(T, dtype=np.int64)
    t = 0
    for i in range(len(ctx)):
        for pos in range(int(pre[i]), int(ctx[i])):
            slots[t] = int(tables[i, pos // bs]) * bs + pos % bs
            t += 1
    blk, off = slots // bs, slots % bs
    new_key = k_cache[blk, :, off, :].copy() if T else np.zeros((0, num_kv_heads, head_dim), np.uint16)
    new_value = v_cache[blk, :, off, :].copy() if T else np.zeros((0, num_kv_heads, head_dim), np.uint16)
    q = normal_bits(g, (T, num_heads, head_dim), dtype)
    return PrefillCase(
        num_seqs=len(ctx), num_heads=num_heads, num_kv_heads=num_kv_heads, head_dim=head_dim,
        block_size=bs, num_blocks=num_blocks, dtype=dtype, scale=1.0 / math.sqrt(head_dim),
        q=q, k_cache=k_cache, v_cache=v_cache, block_tables=tables,
        context_lens=ctx.astype(np.int32), query_start=qs, new_key=new_key, new_value=new_value,
        slot_mapping=slots, poison_block=poison)


def prefill_llama8b(seed=1011, num_seqs=16, chunk=512, prefix_hi=2048):
    g = _gen(seed)
    pre = torch.randint(0, prefix_hi + 1, (num_seqs,), generator=g).numpy()
    return prefill_case(seed + 1, pre, [chunk] * num_seqs, 32, 8, 128, 16, BF16)

def grouped_prefix_case(seed, group_sizes, prefix_blocks, suffix_lo, suffix_hi, num_heads,
                        num_kv_heads, head_dim, block_size, dtype, pool_factor=1.25):
    """Sequences in groups whose tables share their leading blocks.

    Group g has group_sizes[g] consecutive sequences; all of them point their
    first prefix_blocks[g] table entries at the same physical blocks (random
    K/V, a seeded permutation of the pool), then own private blocks for a
    suffix of suffix_lo..suffix_hi tokens. Returns the DecodeCase plus the
    group description (group_start [G + 1], group_prefix [G] in tokens).
    """
    g = _gen(seed)
    bs = block_size
    B = int(sum(group_sizes))
    suffix = torch.randint(suffix_lo, suffix_hi + 1, (B,), generator=g).numpy().astype(np.int64)
    pre_tok = np.repeat(np.asarray(prefix_blocks, dtype=np.int64) * bs, group_sizes)
    ctx = pre_tok + suffix
    nbs = [int(-(-c // bs)) for c in ctx]
    need = int(sum(prefix_blocks)) + sum(nb - int(p // bs) for nb, p in zip(nbs, pre_tok))
    num_blocks = max(int(math.ceil(pool_factor * need)), need) + 1
    perm = torch.randperm(num_blocks, generator=g).numpy().astype(np.int64)
    poison = int(perm[-1])
    width = max(max(nbs), 1)
    tables = np.full((B, width), poison, dtype=np.int32)
    cursor = 0
    i = 0
    for gsize, pb in zip(group_sizes, prefix_blocks):
        shared = perm[cursor:cursor + pb]
        cursor += pb
        for _ in range(gsize):
            tables[i, :pb] = shared
            own = nbs[i] - pb
            tables[i, pb:pb + own] = perm[cursor:cursor + own]
            cursor += own
            i += 1
    shape = (num_blocks, num_kv_heads, bs, head_dim)
    k_cache = normal_bits(g, shape, dtype)
    v_cache = normal_bits(g, shape, dtype)
    k_cache[poison] = NAN_BITS[dtype]
    v_cache[poison] = NAN_BITS[dtype]
    _poison_tails(k_cache, tables, ctx, bs, dtype)
    _poison_tails(v_cache, tables, ctx, bs, dtype)
    q = normal_bits(g, (B, num_heads, head_dim), dtype)
    case = DecodeCase(
        name="grouped_prefix", num_seqs=B, num_heads=num_heads, num_kv_heads=num_kv_heads,
        head_dim=head_dim, block_size=bs, num_blocks=num_blocks, q_dtype=dtype, kv_dtype=dtype,
        scale=1.0 / math.sqrt(head_dim), q=q, k_cache=k_cache, v_cache=v_cache,
        block_tables=tables, context_lens=ctx.astype(np.int32), poison_block=poison)
    group_start = np.concatenate([[0], np.cumsum(group_sizes)]).astype(np.int32)
    group_prefix = (np.asarray(prefix_blocks, dtype=np.int64) * bs).astype(np.int32)
    return case, group_start, group_prefix
