"""Host block pool: free list, on-demand growth, sharing, copy-on-write."""

import numpy as np
import pytest

import oracle
from paged_kv_cache_288_gb300 import BlockPool, OutOfBlocks, PrefixCache, block_key


def test_grows_one_block_at_a_time():
    pool = BlockPool(10, 16)
    slots = pool.add_sequence("a", 5)
    assert pool.used_blocks() == 1 and len(slots) == 5
    b0 = pool.tables["a"][0]
    assert slots == [b0 * 16 + i for i in range(5)]
    s, cow = pool.append("a", 11)
    assert pool.used_blocks() == 1 and not cow
    s, cow = pool.append("a", 1)  # token 17 opens a second block
    assert pool.used_blocks() == 2 and s == [pool.tables["a"][1] * 16]


def test_tail_waste_matches_closed_form():
    rng = np.random.default_rng(3)
    pool = BlockPool(100000, 16)
    for i, n in enumerate(rng.integers(1, 3000, 300)):
        pool.add_sequence(i, int(n))
        assert pool.tail_waste(i) == oracle.paged_tail_waste_tokens(int(n), 16) <= 15


def test_free_blocks_are_reused_by_anyone():
    pool = BlockPool(4, 8)
    pool.add_sequence("a", 16)
    pool.add_sequence("b", 16)
    with pytest.raises(OutOfBlocks):
        pool.add_sequence("c", 1)
    pool.free_sequence("a")
    assert pool.num_free == 2
    pool.add_sequence("c", 9)  # any two free blocks fit, wherever they are
    assert pool.num_free == 0


def test_capacity_rule_on_a_full_pool():
    pool = BlockPool(8192, 16)
    n = 0
    while True:
        try:
            pool.add_sequence(n, 512)
        except OutOfBlocks:
            break
        n += 1
    assert n == oracle.concurrent_capacity(8192, 16, 512) == 256


def test_fork_shares_then_copies_on_write():
    pool = BlockPool(20, 16)
    pool.add_sequence("p", 24)           # blocks: full, half full
    pool.fork("p", "c")
    a, b = pool.tables["p"]
    assert pool.tables["c"] == [a, b] and pool.refcount[a] == 2 and pool.refcount[b] == 2
    slots, cow = pool.append("c", 1)     # writes into the shared half-full block
    assert len(cow) == 1 and cow[0][0] == b
    new = cow[0][1]
    assert pool.tables["c"] == [a, new] and pool.refcount[b] == 1 and pool.refcount[new] == 1
    assert slots == [new * 16 + 8]
    slots, cow = pool.append("p", 1)     # the parent now owns b alone: no copy
    assert not cow and slots == [b * 16 + 8]


def test_prefix_sharing_pattern_of_one_hundred_requests():
    """100 requests over one 1016-token prompt: 64 shared blocks, 100 copies of the last."""
    pool = BlockPool(4000, 16)
    pool.add_sequence("prompt", 1016)
    total_cow = []
    for i in range(100):
        pool.fork("prompt", i)
        _, cow = pool.append(i, 40)
        total_cow += cow
    shared = pool.tables["prompt"]
    assert len(shared) == 64
    assert len(total_cow) == 100 and all(src == shared[-1] for src, _ in total_cow)
    for b in shared[:-1]:
        assert pool.refcount[b] == 101
    # the sharing saves what the closed form says
    per_token = oracle.kv_cache_bytes(32, 8, 128, 1, 2)
    private = 100 * (1016 + 40)
    used = pool.used_blocks() * 16
    assert used < private
    assert (private - used) * per_token > 0


def test_beam_pruning_frees_only_unshared_blocks():
    pool = BlockPool(20, 4)
    pool.add_sequence("root", 8)
    pool.fork("root", "beam1")
    pool.fork("root", "beam2")
    pool.append("beam1", 3)
    pool.append("beam2", 3)
    before = pool.num_free
    pool.free_sequence("beam2")
    assert pool.num_free == before + 1  # only beam2's own block returns
    assert all(pool.refcount[b] == 2 for b in pool.tables["root"])


def test_block_table_array_padding():
    pool = BlockPool(10, 4)
    pool.add_sequence(0, 9)
    pool.add_sequence(1, 2)
    t = pool.block_table_array([0, 1], width=4, pad=7)
    assert t.dtype == np.int32 and t.shape == (2, 4)
    assert list(t[1, 1:]) == [7, 7, 7]
    assert list(pool.context_lens([0, 1])) == [9, 2]


# ----------------------------------------------------------------------------
# prefix cache


def _prompt(seed, n):
    return np.random.default_rng(seed).integers(0, 32000, n)


def test_prefix_cache_shares_the_full_blocks_of_a_common_prefix():
    pool = BlockPool(64, 16)
    cache = PrefixCache(pool)
    common = _prompt(1, 40)
    a = np.concatenate([common, _prompt(2, 10)])
    b = np.concatenate([common, _prompt(3, 30)])
    cached, slots = cache.add_sequence("a", a)
    assert cached == 0 and len(slots) == 50
    cached, slots = cache.add_sequence("b", b)
    # 40 common tokens = 2 full blocks (32 tokens) + 8 in a block that differs
    assert cached == 32 and len(slots) == 70 - 32
    assert pool.tables["b"][:2] == pool.tables["a"][:2]
    assert pool.tables["b"][2] != pool.tables["a"][2]
    assert slots[0] == pool.tables["b"][2] * 16
    # refcounts: a, b and the cache hold the two shared blocks
    assert all(pool.refcount[x] == 3 for x in pool.tables["a"][:2])
    assert cache.hits == 2 and cache.misses == 3 + 2


def test_prefix_cache_keys_chain_the_whole_prefix():
    t = _prompt(4, 32)
    k1 = block_key(b"", t[:16])
    assert block_key(b"", t[:16]) == k1
    assert block_key(k1, t[16:]) != block_key(b"", t[16:])  # same tokens, other position
    u = t.copy()
    u[3] += 1  # an earlier change makes every later block different
    assert block_key(block_key(b"", u[:16]), u[16:]) != block_key(k1, t[16:])
    pool = BlockPool(16, 16)
    cache = PrefixCache(pool)
    cache.add_sequence("t", t)
    cached, _ = cache.add_sequence("u", u)
    assert cached == 0


def test_prefix_cache_keeps_blocks_after_the_request_and_evicts_oldest():
    pool = BlockPool(6, 4)
    cache = PrefixCache(pool)
    p, q = _prompt(5, 8), _prompt(6, 8)
    cache.add_sequence("p", p)
    cache.free_sequence("p")
    assert pool.num_free == 4  # the two full blocks stay cached
    cached, _ = cache.add_sequence("p2", p)
    assert cached == 8 and pool.num_free == 4
    cache.free_sequence("p2")
    cache.add_sequence("q", q)  # caches two more blocks: pool has 2 free
    cache.free_sequence("q")
    assert pool.num_free == 2
    # a 16-token prompt needs 4 blocks: the two oldest cached blocks (p's) go
    cached, _ = cache.add_sequence("r", _prompt(7, 16))
    assert cached == 0
    assert cache.add_sequence("q2", q)[0] == 8     # q is still cached
    with pytest.raises(OutOfBlocks):
        cache.add_sequence("p3", np.concatenate([p, p]))


def test_prefix_cache_one_hundred_requests_over_one_system_prompt():
    """The pages' example: 100 requests starting with the same system prompt
    keep one copy of its full blocks (1016 tokens: 63 full blocks + 8 tokens)."""
    pool = BlockPool(4000, 16)
    cache = PrefixCache(pool)
    system = _prompt(8, 1016)
    for i in range(100):
        suffix = _prompt(100 + i, 40)
        cached, slots = cache.add_sequence(i, np.concatenate([system, suffix]))
        assert cached == (0 if i == 0 else 63 * 16)
        assert len(slots) == 1056 - cached
    shared = pool.tables[0][:63]
    assert all(pool.tables[i][:63] == shared for i in range(100))
    assert all(pool.refcount[b] == 101 for b in shared)
    # blocks in use: 63 shared + per request ceil((1056 - 1008) / 16) = 3 own
    assert pool.used_blocks() == 63 + 100 * 3


def test_shared_prefix_groups_from_tables():
    """Groups found from the tables: consecutive sequences whose leading
    whole blocks agree, the common run shrinking as members join; a lone
    sequence has prefix 0; a partly filled last block is never shared."""
    from paged_kv_cache_288_gb300.block_pool import shared_prefix_groups
    t = np.array([
        [5, 6, 7, 9],     # 0: group A
        [5, 6, 7, 10],    # 1: group A (3 common blocks)
        [5, 6, 11, 12],   # 2: group A, common run shrinks to 2
        [20, 21, 0, 0],   # 3: alone
        [30, 31, 32, 0],  # 4: group B
        [30, 31, 33, 0],  # 5: group B (2 common blocks)
    ], dtype=np.int32)
    lens = np.array([64, 60, 50, 30, 40, 40])  # block size 16
    gs, gp = shared_prefix_groups(t, lens, 16)
    assert gs.tolist() == [0, 3, 4, 6]
    assert gp.tolist() == [32, 0, 32]
    # a shared block only partly inside a member's context does not count
    gs, gp = shared_prefix_groups(t[:2], np.array([64, 40]), 16)
    assert gs.tolist() == [0, 2] and gp.tolist() == [32]


def test_shared_prefix_groups_of_a_prefix_cache_batch():
    """100 requests with one 1016-token system prompt admitted through the
    prefix cache form one group sharing its 63 whole blocks."""
    from paged_kv_cache_288_gb300.block_pool import shared_prefix_groups
    rng = np.random.default_rng(3)
    pool = BlockPool(4000, 16)
    cache = PrefixCache(pool)
    system = rng.integers(0, 32000, 1016)
    for i in range(100):
        cache.add_sequence(i, np.concatenate([system, rng.integers(0, 32000, int(rng.integers(32, 513)))]))
    ids = list(range(100))
    gs, gp = shared_prefix_groups(pool.block_table_array(ids), pool.context_lens(ids), 16)
    assert gs.tolist() == [0, 100] and gp.tolist() == [1008]
