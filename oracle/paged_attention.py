"""fp64 definitions of the paged KV-cache operations (oracle; test infrastructure).

Layout (a choice; the pages fix none beyond "blocks need not be contiguous"):
``k_cache`` and ``v_cache`` are ``[num_blocks, num_kv_heads, block_size,
head_dim]``; ``q`` and the decode output are ``[num_seqs, num_heads,
head_dim]``; ``block_tables`` is ``[num_seqs, max_blocks_per_seq]`` of
physical block ids; ``context_lens`` is ``[num_seqs]``; ``slot_mapping`` is
``[num_tokens]`` of ``block * block_size + offset`` or -1 (skip); fp8 scales
are ``[num_blocks, num_kv_heads]`` float32, one for K and one for V.

16-bit values are raw ``uint16`` bit patterns, 8-bit values raw ``uint8``
E4M3 codes. Arithmetic is float64 and follows the definitions literally:
gather the sequence through its table, then softmax(q K^T * scale) V.
"""

import numpy as np

from .ofp8 import e4m3_decode, e4m3_encode

F16 = "f16"
BF16 = "bf16"
FP8_E4M3 = "fp8_e4m3"


def bits_to_f64(bits, dtype):
    """Exact float64 value of raw 16-bit (f16 / bf16) or 8-bit (E4M3) codes."""
    bits = np.asarray(bits)
    if dtype == F16:
        return bits.astype(np.uint16).view(np.float16).astype(np.float64)
    if dtype == BF16:
        return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    if dtype == FP8_E4M3:
        return e4m3_decode(bits)
    raise ValueError(dtype)


def _bits_to_f32(bits, dtype):
    if dtype == F16:
        return bits.astype(np.uint16).view(np.float16).astype(np.float32)
    if dtype == BF16:
        return (bits.astype(np.uint32) << 16).view(np.float32)
    raise ValueError(dtype)


def reshape_and_cache(key, value, k_cache, v_cache, slot_mapping, block_size,
                      src_dtype, kv_dtype, k_scale=None, v_scale=None):
    """Write each new token's K and V into its slot, in place.

    vLLM의 핵심 이해: PagedAttention, section 6 (the token table records which
    page and which position inside it hold each token) and
    serving-paged-attention, section "블록으로 쪼개고 표로 잇는다" (a request
    borrows one free block at a time): slot = block * block_size + offset,
    so block = slot // block_size and offset = slot % block_size. A slot of -1
    marks a padding token that is not written. Slots of distinct tokens are
    distinct (two tokens in one slot is a caller error).

    16-bit caches receive the source bits unchanged. An 8-bit cache
    (serving-paged-attention, "실무에서 만지는 지점": KV stored in 8 bits)
    receives e4m3(float32(x) / scale[block, head]), the division in IEEE
    float32 and the encoding round-to-nearest-even with saturation; the scales
    belong to the caller and are only read.
    """
    slots = np.asarray(slot_mapping, dtype=np.int64)
    if kv_dtype != FP8_E4M3 and src_dtype != kv_dtype:
        raise ValueError("16-bit caches take sources of the same type")
    tokens = np.nonzero(slots >= 0)[0]
    # tokens are independent (slots are distinct), so they are taken in chunks
    for start in range(0, len(tokens), 4096):
        t = tokens[start:start + 4096]
        blk = slots[t] // block_size
        off = slots[t] % block_size
        if kv_dtype == FP8_E4M3:
            ks = np.asarray(k_scale, dtype=np.float32)[blk][:, :, None]
            vs = np.asarray(v_scale, dtype=np.float32)[blk][:, :, None]
            k_cache[blk, :, off, :] = e4m3_encode(_bits_to_f32(key[t], src_dtype) / ks)
            v_cache[blk, :, off, :] = e4m3_encode(_bits_to_f32(value[t], src_dtype) / vs)
        else:
            k_cache[blk, :, off, :] = key[t]
            v_cache[blk, :, off, :] = value[t]


def copy_blocks(k_caches, v_caches, block_mapping):
    """Copy whole physical blocks, K and V, in every layer, in place.

    serving-paged-attention, section "공유는 표를 베끼는 일이 된다": before a
    request writes into a block that other tables also point at, that block is
    copied to one of its own and its table entry is redirected (copy on
    write); LLM의 Paged Attention, "Paged Attention의 핵심 원리" item 3 says
    the same. ``block_mapping`` is a list of (src, dst) pairs.
    """
    for src, dst in block_mapping:
        for kc, vc in zip(k_caches, v_caches):
            kc[int(dst)] = kc[int(src)]
            vc[int(dst)] = vc[int(src)]


def swap_blocks(dst_k, dst_v, src_k, src_v, block_mapping):
    """Move whole blocks, K and V, in every layer, from the src pools to the
    dst pools (lists of per-layer arrays [num_blocks, ...]).

    serving-paged-attention, section "그래도 넘칠 때 — 선점": when the pool has
    no free block left, a request is preempted; the swap way moves its blocks
    to CPU memory and later back, so nothing is recomputed. Each (src, dst)
    pair of ``block_mapping`` copies block src of every src pool to block dst
    of the matching dst pool. Returns the pairs skipped because an index lies
    outside its pool (the library flags those and leaves them untouched).
    """
    skipped = []
    for src, dst in block_mapping:
        src, dst = int(src), int(dst)
        if not (0 <= src < src_k[0].shape[0] and 0 <= dst < dst_k[0].shape[0]):
            skipped.append((src, dst))
            continue
        for layer in range(len(src_k)):
            dst_k[layer][dst] = src_k[layer][src]
            dst_v[layer][dst] = src_v[layer][src]
    return skipped


def gather_sequence(cache, table_row, context_len, block_size, kv_head,
                    kv_dtype, scale=None):
    """One sequence's K (or V) rows for one KV head, in logical order, float64.

    serving-paged-attention, section "블록으로 쪼개고 표로 잇는다": the i-th
    logical block of a request lives in physical block table[i]; attention
    reads the scattered blocks through that table. Only the first
    ``context_len`` rows are data; the tail of the last block is not read
    (same page, table of wastes). 8-bit rows are decoded and multiplied by
    their block's scale.
    """
    if context_len <= 0:
        return np.zeros((0, cache.shape[-1]))
    nblocks = -(-context_len // block_size)
    ids = np.asarray(table_row[:nblocks], dtype=np.int64)
    rows = bits_to_f64(cache[ids, kv_head], kv_dtype)  # [nblocks, block_size, d]
    if kv_dtype == FP8_E4M3:
        rows = rows * np.asarray(scale, dtype=np.float32)[ids, kv_head].astype(np.float64)[:, None, None]
    return rows.reshape(nblocks * block_size, -1)[:context_len]


def paged_decode(q, k_cache, v_cache, block_tables, context_lens, scale,
                 block_size, q_dtype, kv_dtype, k_scale=None, v_scale=None):
    """Single-query attention of every sequence over its paged KV, float64.

    For sequence i and query head h, with G = num_heads / num_kv_heads and
    KV head g = h // G (contiguous grouping; LLM 추론 확장, 품질·비용 절충
    필수: under GQA several query heads share one KV head):

        K, V = the sequence's rows gathered through its block table
        s    = scale * (K @ q[i, h])
        out[i, h] = softmax(s) @ V

    The softmax subtracts max(s) before exponentiating; the online softmax of
    the same talk (three running variables) reaches this same value, so the
    oracle computes the plain definition. A sequence with context length 0
    gets an all-zero output.
    """
    qf = bits_to_f64(q, q_dtype)
    num_seqs, num_heads, head_dim = qf.shape
    num_kv_heads = k_cache.shape[1]
    group = num_heads // num_kv_heads
    out = np.zeros((num_seqs, num_heads, head_dim))
    for i in range(num_seqs):
        ctx = int(context_lens[i])
        if ctx <= 0:
            continue
        for g in range(num_kv_heads):
            K = gather_sequence(k_cache, block_tables[i], ctx, block_size, g, kv_dtype, k_scale)
            V = gather_sequence(v_cache, block_tables[i], ctx, block_size, g, kv_dtype, v_scale)
            for h in range(g * group, (g + 1) * group):
                s = scale * (K @ qf[i, h])
                p = np.exp(s - s.max())
                out[i, h] = (p @ V) / p.sum()
    return out


def paged_decode_partitioned(q, k_cache, v_cache, block_tables, context_lens,
                             scale, block_size, q_dtype, kv_dtype,
                             partition_size, k_scale=None, v_scale=None):
    """Split-context decode: per-partition softmax state, then a merge.

    Each partition p covers tokens [p*P, (p+1)*P) and yields its max m_p, its
    sum l_p = sum exp(s - m_p) and its normalised output o_p. The merge takes
    m = max_p m_p and returns sum_p exp(m_p - m) l_p o_p / sum_p exp(m_p - m)
    l_p. This is the state (running max, running sum, accumulator) of the
    online softmax in LLM 추론 확장, 품질·비용 절충 필수, carried across
    partitions instead of tiles. In exact arithmetic it equals
    ``paged_decode``.
    """
    qf = bits_to_f64(q, q_dtype)
    num_seqs, num_heads, head_dim = qf.shape
    num_kv_heads = k_cache.shape[1]
    group = num_heads // num_kv_heads
    out = np.zeros((num_seqs, num_heads, head_dim))
    for i in range(num_seqs):
        ctx = int(context_lens[i])
        if ctx <= 0:
            continue
        for g in range(num_kv_heads):
            K = gather_sequence(k_cache, block_tables[i], ctx, block_size, g, kv_dtype, k_scale)
            V = gather_sequence(v_cache, block_tables[i], ctx, block_size, g, kv_dtype, v_scale)
            for h in range(g * group, (g + 1) * group):
                ms, ls, os_ = [], [], []
                for start in range(0, ctx, partition_size):
                    s = scale * (K[start:start + partition_size] @ qf[i, h])
                    m_p = s.max()
                    e = np.exp(s - m_p)
                    ms.append(m_p)
                    ls.append(e.sum())
                    os_.append((e @ V[start:start + partition_size]) / e.sum())
                m = max(ms)
                w = np.array([np.exp(mp - m) * lp for mp, lp in zip(ms, ls)])
                out[i, h] = (w[:, None] * np.array(os_)).sum(axis=0) / w.sum()
    return out


def paged_prefill(q, k_cache, v_cache, block_tables, context_lens, query_start, scale,
                  block_size, q_dtype, kv_dtype):
    """Causal attention of each sequence's chunk of new query tokens over its
    paged KV, float64.

    The step before decode: a prompt (or a chunk of it, after earlier chunks
    are already cached) is attended with many queries at once (LLM 추론 확장,
    품질·비용 절충 필수, the prefill / decode split; serving-paged-attention,
    "블록으로 쪼개고 표로 잇는다": the same block tables serve both). Sequence i
    holds context_lens[i] tokens, the last n_i = query_start[i+1] -
    query_start[i] of which are its queries (their K/V already written).
    Query j of sequence i sits at position p = context_lens[i] - n_i + j and
    attends to the keys at positions 0..p:

        out[query_start[i] + j, h] = softmax(scale * K[0..p] q) V[0..p]

    with K, V the sequence's rows gathered through its table for KV head
    h // G. ``q`` and the result are [num_tokens, num_heads, head_dim].
    """
    qf = bits_to_f64(q, q_dtype)
    num_tokens, num_heads, head_dim = qf.shape
    num_kv_heads = k_cache.shape[1]
    group = num_heads // num_kv_heads
    out = np.zeros((num_tokens, num_heads, head_dim))
    for i in range(len(context_lens)):
        ctx = int(context_lens[i])
        q0, q1 = int(query_start[i]), int(query_start[i + 1])
        n = q1 - q0
        if n <= 0:
            continue
        for g in range(num_kv_heads):
            K = gather_sequence(k_cache, block_tables[i], ctx, block_size, g, kv_dtype)
            V = gather_sequence(v_cache, block_tables[i], ctx, block_size, g, kv_dtype)
            for j in range(n):
                p = ctx - n + j
                for h in range(g * group, (g + 1) * group):
                    s = scale * (K[:p + 1] @ qf[q0 + j, h])
                    w = np.exp(s - s.max())
                    out[q0 + j, h] = (w @ V[:p + 1]) / w.sum()
    return out