"""Closed-form memory accounting of a KV cache (oracle; test infrastructure).

These are the sizing rules the pages state in words. They pin the host-side
block pool and the bench's byte counts.
"""

import math


def kv_cache_bytes(num_layers, num_kv_heads, head_dim, num_tokens, bytes_per_value):
    """Bytes of K and V held for ``num_tokens`` tokens.

    serving-paged-attention, section "캐시가 얼마나 큰지부터" (how big the
    cache is): the size is the product of 2 (one copy for keys, one for
    values), the layer count, the KV-head count, the per-head dimension, the
    token count and the bytes of one value. The symbols of the printed formula
    were lost; the worked example of that section (32 layers, 8 KV heads,
    head dim 128, fp16 -> 128 KB per token) fixes this reading.
    """
    return 2 * num_layers * num_kv_heads * head_dim * num_tokens * bytes_per_value


def max_concurrent_requests(free_bytes, bytes_per_request):
    """How many whole requests fit in ``free_bytes``.

    serving-paged-attention, section "캐시가 얼마나 큰지부터": the memory left
    after the weights, divided into per-request shares, bounds the number of
    requests held at once (64 GB / 512 MB -> 128).
    """
    return free_bytes // bytes_per_request


def naive_waste_fraction(max_len, mean_len):
    """Fraction of a max-length reservation that holds no data.

    LLM의 Paged Attention, section "Paged Attention, 이것이 무엇일까요?": a
    request reserves memory for the maximum sequence length but fills only its
    actual length (2048 reserved, 500 used -> about 75 % wasted).
    """
    return 1.0 - mean_len / max_len


def paged_tail_waste_tokens(context_len, block_size):
    """Empty token slots of one sequence's last block.

    serving-paged-attention, section "블록으로 쪼개고 표로 잇는다", the table
    of wastes: only the tail of the last block is unused, at most
    ``block_size - 1`` tokens (15 for 16-token blocks).
    """
    if context_len <= 0:
        return 0
    nblocks = -(-context_len // block_size)
    return nblocks * block_size - context_len


def concurrent_capacity(num_blocks, block_size, mean_request_len):
    """Requests the pool holds at once: blocks x tokens per block / mean length.

    serving-paged-attention, section "실무에서 만지는 지점" (the knobs): the
    logged block count times the tokens per block is the total token capacity;
    divided by the mean request length it gives the concurrent requests.
    """
    return num_blocks * block_size / mean_request_len


def naive_vs_paged_bytes(lengths, max_len, block_size, bytes_per_token):
    """(naive bytes, paged bytes) for a population of requests.

    LLM의 Paged Attention, section "실제 구현과 성능 측정": the naive scheme
    reserves ``max_len`` tokens per request; the paged scheme allocates whole
    blocks on demand (serving-paged-attention, "블록으로 쪼개고 표로
    잇는다"), so each request holds ceil(len / block_size) blocks.
    """
    naive = len(lengths) * max_len * bytes_per_token
    paged = sum(math.ceil(n / block_size) * block_size for n in lengths) * bytes_per_token
    return naive, paged
