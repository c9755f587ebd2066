"""GPU parity of pa_decode against the fp64 oracle on small and edge cases."""

import numpy as np
import pytest
import torch

import oracle
import workloads
from workloads import F16, BF16, FP8_E4M3
from gpu_helpers import (DeviceCase, assert_close, dev, host_bits, oracle_decode, run_decode,
                         to_f64)
import paged_kv_cache_288_gb300 as pa

pytestmark = pytest.mark.gpu


def _check(case, partition_size=0, workspace=True):
    dc = DeviceCase(case)
    out = run_decode(pa, dc, partition_size=partition_size, workspace=workspace)
    ref = oracle_decode(case)
    torch.cuda.synchronize()
    assert dc.debug_err.item() == 0
    return assert_close(out, ref, case.q_dtype, case.kv_dtype, case.name), out, dc


def test_tiny_decode_append_decode():
    """Lengths 5/17/33/64, GQA 2, d 64, fp16; append one token each, decode again."""
    before, step = workloads.tiny()
    _check(before)
    dc = DeviceCase(before)
    # append through the library, then decode at the new lengths
    dstep = DeviceCase(step)
    pa.reshape_and_cache(dstep.new_key, dstep.new_value, dc.k_cache, dc.v_cache,
                         dstep.slot_mapping, debug_err=dc.debug_err)
    kc, vc = before.k_cache.copy(), before.v_cache.copy()
    oracle.reshape_and_cache(step.new_key, step.new_value, kc, vc, step.slot_mapping, 16, F16, F16)
    torch.cuda.synchronize()
    assert np.array_equal(host_bits(dc.k_cache), kc)
    assert np.array_equal(host_bits(dc.v_cache), vc)
    out = run_decode(pa, dstep, k_cache=dc.k_cache, v_cache=dc.v_cache)
    ref = oracle_decode(step, k_cache=kc, v_cache=vc)
    assert_close(out, ref, F16, F16, "tiny after append")
    assert dc.debug_err.item() == 0 and dstep.debug_err.item() == 0


SWEEP = [
    # (group, Hkv, d, bs, dtype)
    (1, 4, 128, 16, BF16), (2, 2, 64, 8, F16), (4, 2, 128, 32, BF16), (8, 1, 128, 64, F16),
    (4, 8, 128, 16, F16), (2, 3, 256, 16, BF16), (8, 2, 64, 16, BF16), (1, 1, 64, 64, F16),
    (4, 2, 256, 8, F16),
]


@pytest.mark.parametrize("group,Hkv,d,bs,dtype", SWEEP)
def test_random_shapes(group, Hkv, d, bs, dtype):
    seed = group * 10000 + Hkv * 1000 + d + bs
    case = workloads.random_small_case(seed, num_seqs=7, group=group, num_kv_heads=Hkv,
                                       head_dim=d, block_size=bs, dtype=dtype, max_ctx=700)
    _check(case)


# MQA and groups above 8 (LLM 추론 확장, 품질·비용 절충 필수: MHA, MQA and
# GQA): every query head of a group reads the same KV head
WIDE_GROUPS = [
    # (num_heads, num_kv_heads, d, bs, dtype)
    (32, 1, 128, 16, BF16), (16, 1, 128, 16, F16), (64, 1, 64, 32, BF16), (16, 2, 128, 8, BF16),
    (32, 4, 64, 16, F16), (24, 1, 128, 64, BF16),
]


@pytest.mark.parametrize("Hq,Hkv,d,bs,dtype", WIDE_GROUPS)
def test_mqa_and_wide_groups(Hq, Hkv, d, bs, dtype):
    lengths = [1, 17, 300, 1000, 2500, 64]
    case = workloads.paged_case(Hq * 100 + Hkv * 10 + bs, lengths, Hq, Hkv, d, bs, dtype,
                                name=f"mqa{Hq}/{Hkv}")
    _, out, dc = _check(case)
    ref = oracle_decode(case)
    # the split path and the schedule without a workspace take the same groups
    for part, ws in ((256 if 256 % bs == 0 else 512, True), (0, False)):
        other = run_decode(pa, dc, partition_size=part, workspace=ws)
        torch.cuda.synchronize()
        assert_close(other, ref, dtype, dtype, f"mqa part={part} ws={ws}")
    assert dc.debug_err.item() == 0


def test_mqa_fp8():
    """MQA over an 8-bit cache: 32 query heads, one KV head."""
    case = workloads.fp8_layer(880, [1, 40, 500, 1500], num_heads=32, num_kv_heads=1,
                               head_dim=128, block_size=16, src_dtype=BF16, name="mqa_fp8")
    dc = DeviceCase(case)
    pa.reshape_and_cache(dc.new_key, dc.new_value, dc.k_cache, dc.v_cache, dc.slot_mapping,
                         k_scale=dc.k_scale, v_scale=dc.v_scale, debug_err=dc.debug_err)
    kc, vc = case.k_cache.copy(), case.v_cache.copy()
    oracle.reshape_and_cache(case.new_key, case.new_value, kc, vc, case.slot_mapping, 16, BF16,
                             FP8_E4M3, case.k_scale, case.v_scale)
    ref = oracle_decode(case, k_cache=kc, v_cache=vc)
    for part in (0, 512):
        out = run_decode(pa, dc, partition_size=part)
        torch.cuda.synchronize()
        max_abs, _ = assert_close(out, ref, BF16, FP8_E4M3, f"mqa fp8 part={part}")
        assert max_abs <= 3e-2
    assert dc.debug_err.item() == 0


@pytest.mark.parametrize("bs", [8, 16, 32, 64])
def test_lengths_around_block_boundaries(bs):
    lengths = [1, 2, bs - 1, bs, bs + 1, 2 * bs - 1, 2 * bs, 2 * bs + 1, 5 * bs + 3]
    case = workloads.paged_case(500 + bs, lengths, 8, 2, 128, bs, BF16, name=f"edges{bs}")
    _check(case)


SPLIT_CASES = [(ps, bs) for ps in (16, 64, 512) for bs in (8, 16, 32) if ps % bs == 0]


@pytest.mark.parametrize("partition_size,bs", SPLIT_CASES)
def test_split_path_matches_oracle_and_other_schedules(partition_size, bs):
    lengths = [1, 15, 16, 17, 511, 512, 513, 1300, 2048]
    case = workloads.paged_case(600 + bs, lengths, 16, 4, 128, bs, BF16, name="split")
    (_, _), out_split, dc = _check(case, partition_size=partition_size)
    ref = oracle_decode(case)
    # the library's own schedule and the no-workspace schedule meet the same bound
    for ws in (True, False):
        other = run_decode(pa, dc, partition_size=0, workspace=ws)
        assert_close(other, ref, BF16, BF16, f"schedule workspace={ws}")
    # different schedules round P and the merges differently, never by more
    # than the parity tolerance between them
    a, b = to_f64(out_split, BF16), to_f64(run_decode(pa, dc), BF16)
    assert np.all(np.abs(a - b) <= 2e-3 + 1e-2 * np.abs(b))


@pytest.mark.parametrize("partition_size", [16, 32])
def test_split_path_partitions_shorter_than_the_ring(partition_size):
    """Partitions of one or two 16-token tiles and many more partitions than
    warps: in the claimed quarter a warp's loads run up to three tiles ahead,
    so it claims several partitions before it computes the first of them;
    they must be taken in the order they were claimed."""
    lengths = [12000, 9000, 7001, 5003, 3]
    case = workloads.paged_case(960 + partition_size, lengths, 16, 4, 128, 16, BF16, name=f"ring{partition_size}")
    _check(case, partition_size=partition_size)


def test_fp8_split_path_single_tile_partitions():
    """The E4M3 kernel (32-token tiles, two ring slots per warp) with 32-token
    partitions: every claimed partition is a single tile."""
    lengths = [9000, 7000, 5001, 33]
    case = workloads.fp8_layer(970, lengths, num_heads=16, num_kv_heads=4, head_dim=128,
                               block_size=16, src_dtype=BF16, name="fp8_ring")
    dc = DeviceCase(case)
    pa.reshape_and_cache(dc.new_key, dc.new_value, dc.k_cache, dc.v_cache, dc.slot_mapping,
                         k_scale=dc.k_scale, v_scale=dc.v_scale, debug_err=dc.debug_err)
    kc, vc = case.k_cache.copy(), case.v_cache.copy()
    oracle.reshape_and_cache(case.new_key, case.new_value, kc, vc, case.slot_mapping, 16, BF16,
                             FP8_E4M3, case.k_scale, case.v_scale)
    ref = oracle_decode(case, k_cache=kc, v_cache=vc)
    for part in (32, 0):
        out = run_decode(pa, dc, partition_size=part)
        torch.cuda.synchronize()
        max_abs, _ = assert_close(out, ref, BF16, FP8_E4M3, f"fp8 part={part}")
        assert max_abs <= 3e-2, max_abs
    assert dc.debug_err.item() == 0


def test_empty_and_single_token_sequences():
    lengths = [0, 1, 0, 3, 1]
    case = workloads.paged_case(700, lengths, 4, 2, 64, 16, F16, name="empty")
    (_, _), out, dc = _check(case)
    got = to_f64(out, F16)
    assert np.all(got[0] == 0) and np.all(got[2] == 0)
    # a single token: the output is that token's value row, rounded to fp16
    for i in (1, 4):
        blk = case.block_tables[i, 0]
        for h in range(4):
            want = oracle.bits_to_f64(case.v_cache[blk, h // 2, 0], F16)
            assert np.array_equal(got[i, h], want)


def test_no_workspace_still_correct():
    case = workloads.paged_case(701, [3000, 100, 4096], 32, 8, 128, 16, BF16, name="nows")
    _check(case, workspace=False)


def test_split_without_workspace_is_rejected():
    case = workloads.paged_case(702, [100], 4, 2, 64, 16, F16)
    dc = DeviceCase(case)
    with pytest.raises(pa.PaError):
        run_decode(pa, dc, partition_size=64, workspace=False)


def test_physical_permutation_gives_bit_identical_output():
    case = workloads.paged_case(703, [900, 37, 2000, 16], 32, 8, 128, 16, BF16, name="perm")
    dc = DeviceCase(case)
    out1 = run_decode(pa, dc)
    rng = np.random.default_rng(0)
    Nb2 = case.num_blocks + 33
    new_id = rng.permutation(Nb2)[:case.num_blocks]
    kc = np.full((Nb2,) + case.k_cache.shape[1:], workloads.NAN_BITS[BF16], np.uint16)
    vc = kc.copy()
    kc[new_id] = case.k_cache
    vc[new_id] = case.v_cache
    tables = torch.from_numpy(new_id[case.block_tables].astype(np.int32)).cuda()
    out2 = run_decode(pa, dc, k_cache=dev(kc, BF16), v_cache=dev(vc, BF16), block_tables=tables)
    torch.cuda.synchronize()
    assert torch.equal(out1.view(torch.int16), out2.view(torch.int16))


def test_shared_prefix_equals_private_copies_bit_identical():
    case = workloads.shared_prefix(seed=7, num_seqs=6, prefix_len=300, suffix_lo=5, suffix_hi=90)
    dc = DeviceCase(case)
    pa.copy_blocks(pa.pointer_array([dc.k_cache], "cuda"), pa.pointer_array([dc.v_cache], "cuda"),
                   dc.cow_pairs, case.num_blocks, 8 * 16 * 128 * 2)
    pa.reshape_and_cache(dc.new_key, dc.new_value, dc.k_cache, dc.v_cache, dc.slot_mapping)
    out_shared = run_decode(pa, dc)
    # private copies of every shared prefix block, one set per sequence
    kc, vc = host_bits(dc.k_cache), host_bits(dc.v_cache)
    shared = case.meta["shared_blocks"][:-1]
    extra_k, extra_v, tables = [], [], case.block_tables.copy()
    for i in range(case.num_seqs):
        for j, b in enumerate(shared):
            tables[i, j] = kc.shape[0] + len(extra_k)
            extra_k.append(kc[b])
            extra_v.append(vc[b])
    kc2 = np.concatenate([kc, np.stack(extra_k)])
    vc2 = np.concatenate([vc, np.stack(extra_v)])
    out_private = run_decode(pa, dc, k_cache=dev(kc2, F16), v_cache=dev(vc2, F16),
                             block_tables=torch.from_numpy(tables).cuda())
    torch.cuda.synchronize()
    assert torch.equal(out_shared.view(torch.int16), out_private.view(torch.int16))
    ref = oracle.paged_decode(case.q, kc, vc, case.block_tables, case.context_lens, case.scale,
                              16, F16, F16)
    assert_close(out_shared, ref, F16, F16, "shared prefix")


def test_bad_table_entries_are_flagged_and_skipped():
    case = workloads.paged_case(704, [40, 40], 4, 2, 64, 16, F16, name="badtable")
    tables = case.block_tables.copy()
    tables[0, 1] = case.num_blocks + 5   # out of range
    tables[1, 0] = -3
    dc = DeviceCase(case)
    out = run_decode(pa, dc, block_tables=torch.from_numpy(tables).cuda())
    torch.cuda.synchronize()
    assert dc.debug_err.item() & pa.DEVERR_BLOCK_RANGE
    assert torch.isfinite(out.float()).all()
    # the result equals attention over the remaining blocks only
    keep = case.context_lens.copy()
    ref = np.zeros((2, 4, 64))
    for i, drop in ((0, 1), (1, 0)):
        for h in range(4):
            rows_k, rows_v = [], []
            for j in range(3):
                if j == drop:
                    continue
                n = min(16, int(keep[i]) - 16 * j)
                b = case.block_tables[i, j]
                rows_k.append(oracle.bits_to_f64(case.k_cache[b, h // 2, :n], F16))
                rows_v.append(oracle.bits_to_f64(case.v_cache[b, h // 2, :n], F16))
            K, V = np.concatenate(rows_k), np.concatenate(rows_v)
            s = case.scale * K @ oracle.bits_to_f64(case.q[i, h], F16)
            w = np.exp(s - s.max())
            ref[i, h] = w @ V / w.sum()
    assert_close(out, ref, F16, F16, "skipped blocks")


def test_context_above_bound_is_flagged_and_clamped():
    case = workloads.paged_case(705, [64, 20], 4, 2, 64, 16, F16, name="clamp")
    dc = DeviceCase(case)
    ws = torch.empty(1, dtype=torch.uint8, device="cuda")
    out = torch.empty_like(dc.q)
    pa.decode(out, dc.q, dc.k_cache, dc.v_cache, dc.block_tables, dc.context_lens, case.scale,
              32, debug_err=dc.debug_err)
    torch.cuda.synchronize()
    assert dc.debug_err.item() & pa.DEVERR_CONTEXT_RANGE
    ref = oracle_decode(case, context_lens=np.array([32, 20], np.int32))
    assert_close(out, ref, F16, F16, "clamped")
    del ws


@pytest.mark.parametrize("q_dtype", [BF16, F16])
@pytest.mark.parametrize("bs", [8, 16, 64])
def test_fp8_kv_decode(q_dtype, bs):
    lengths = [1, 7, 16, 33, 250, 777]
    case = workloads.fp8_layer(800 + bs, lengths, num_heads=16, num_kv_heads=4, head_dim=128,
                               block_size=bs, src_dtype=q_dtype, name=f"fp8_bs{bs}")
    dc = DeviceCase(case)
    pa.reshape_and_cache(dc.new_key, dc.new_value, dc.k_cache, dc.v_cache, dc.slot_mapping,
                         k_scale=dc.k_scale, v_scale=dc.v_scale, debug_err=dc.debug_err)
    kc, vc = case.k_cache.copy(), case.v_cache.copy()
    oracle.reshape_and_cache(case.new_key, case.new_value, kc, vc, case.slot_mapping, bs, q_dtype,
                             FP8_E4M3, case.k_scale, case.v_scale)
    for part in (0, 64):
        out = run_decode(pa, dc, partition_size=part)
        ref = oracle_decode(case, k_cache=kc, v_cache=vc)
        torch.cuda.synchronize()
        max_abs, _ = assert_close(out, ref, q_dtype, FP8_E4M3, f"fp8 part={part}")
        assert max_abs <= 3e-2, max_abs
    assert dc.debug_err.item() == 0
    assert np.array_equal(host_bits(dc.k_cache), kc)


@pytest.mark.parametrize("Hq,Hkv", [(8, 4), (12, 3), (16, 8), (4, 4)])
def test_fp8_kv_head_pairs(Hq, Hkv):
    """E4M3 caches with 2 or 4 query heads per KV head and an even number of
    KV heads run units of two adjacent KV heads (8 KV heads: 4 units; 4 KV
    heads of 2 query heads each: units of 4 query heads); an odd number of KV
    heads, or one query head per KV head, keeps units of one KV head. Every
    layout matches the oracle, on the library's schedule and the split path."""
    lengths = [1, 15, 16, 17, 100, 333, 1024, 1500]
    case = workloads.fp8_layer(990 + Hq + Hkv, lengths, num_heads=Hq, num_kv_heads=Hkv, head_dim=128,
                               block_size=16, src_dtype=BF16, name=f"fp8_pairs_{Hq}_{Hkv}")
    dc = DeviceCase(case)
    pa.reshape_and_cache(dc.new_key, dc.new_value, dc.k_cache, dc.v_cache, dc.slot_mapping,
                         k_scale=dc.k_scale, v_scale=dc.v_scale, debug_err=dc.debug_err)
    kc, vc = case.k_cache.copy(), case.v_cache.copy()
    oracle.reshape_and_cache(case.new_key, case.new_value, kc, vc, case.slot_mapping, 16, BF16,
                             FP8_E4M3, case.k_scale, case.v_scale)
    ref = oracle_decode(case, k_cache=kc, v_cache=vc)
    for part in (0, 32, 512):
        out = run_decode(pa, dc, partition_size=part)
        torch.cuda.synchronize()
        max_abs, _ = assert_close(out, ref, BF16, FP8_E4M3, f"fp8 pairs part={part}")
        assert max_abs <= 3e-2, max_abs
    assert dc.debug_err.item() == 0


def test_merge_of_eight_head_units_over_many_pairs():
    """Units of 8 query heads (a 256-float4 block per pair) with more pairs
    than one wave of 256-thread merge CTAs holds: the merge runs 128-thread
    CTAs of two elements per thread, whose four warps derive the weights of
    all eight heads. Short random lengths leave most pairs split over two or
    three ranges."""
    g = np.random.default_rng(4242)
    lengths = g.integers(1, 400, size=100)
    for dtype in (BF16, F16):
        case = workloads.paged_case(4243, lengths, 64, 8, 128, 16, dtype, name="wide_merge")
        dc = DeviceCase(case)
        out = run_decode(pa, dc)
        ref = oracle_decode(case)
        torch.cuda.synchronize()
        assert_close(out, ref, dtype, dtype, f"wide merge {dtype}")
        assert dc.debug_err.item() == 0


def test_fp8_q_beyond_f16_range_is_flagged():
    """With an 8-bit cache q is multiplied in f16: a bf16 q value above 65504
    has no f16 counterpart, and the call reports it through debug_err."""
    case = workloads.fp8_layer(860, [40, 70], num_heads=8, num_kv_heads=2, head_dim=128,
                               block_size=16, src_dtype=BF16, name="fp8_big_q")
    dc = DeviceCase(case)
    pa.reshape_and_cache(dc.new_key, dc.new_value, dc.k_cache, dc.v_cache, dc.slot_mapping,
                         k_scale=dc.k_scale, v_scale=dc.v_scale, debug_err=dc.debug_err)
    run_decode(pa, dc)
    torch.cuda.synchronize()
    assert dc.debug_err.item() == 0
    q = dc.q.clone()
    q[1, 3, 17] = 1.0e5
    run_decode(pa, dc, q=q)
    torch.cuda.synchronize()
    assert dc.debug_err.item() & pa.DEVERR_Q_RANGE


@pytest.mark.parametrize("v_sigma,k_sigma", [(0.0125, 1.0), (0.0125, 0.0125), (1e-3, 1.0)])
def test_fp8_kv_decode_small_value_scales(v_sigma, k_sigma):
    """E4M3 caches of activations much smaller than N(0, 1): V drawn with
    sigma 0.0125 (amax about 0.05, V scales about 1e-4) or 1e-3, and K either
    N(0, 1) or as small as V (so the weights are nearly uniform). The kernel
    folds each block's V scale into the softmax weights before they are
    rounded to f16, where such small products are f16 subnormals; the error
    that adds must stay within the 8-bit bound scaled to the size of V
    (3e-2 * amax|V| / 4, i.e. the N(0, 1) bound times sigma)."""
    lengths = [1, 16, 100, 777, 2048]
    case = workloads.fp8_layer(850, lengths, num_heads=32, num_kv_heads=8, head_dim=128,
                               block_size=16, src_dtype=BF16, name="fp8_small_v",
                               k_sigma=k_sigma, v_sigma=v_sigma)
    dc = DeviceCase(case)
    pa.reshape_and_cache(dc.new_key, dc.new_value, dc.k_cache, dc.v_cache, dc.slot_mapping,
                         k_scale=dc.k_scale, v_scale=dc.v_scale, debug_err=dc.debug_err)
    kc, vc = case.k_cache.copy(), case.v_cache.copy()
    oracle.reshape_and_cache(case.new_key, case.new_value, kc, vc, case.slot_mapping, 16, BF16,
                             FP8_E4M3, case.k_scale, case.v_scale)
    ref = oracle_decode(case, k_cache=kc, v_cache=vc)
    for part in (0, 512):
        out = run_decode(pa, dc, partition_size=part)
        torch.cuda.synchronize()
        max_abs, _ = assert_close(out, ref, BF16, FP8_E4M3, f"fp8 small v part={part}",
                                  value_scale=v_sigma)
        # relative to the output's own size the error stays small as well
        assert max_abs <= 1e-2 * np.abs(ref).max() + 2.0 ** -8 * np.abs(ref).max(), max_abs
    assert dc.debug_err.item() == 0


@pytest.mark.parametrize("group", [2, 4, 8])
def test_merges_of_few_and_many_ranges_in_one_batch(group):
    """One auto-schedule call whose pairs are merged from a few ranges (2000
    tokens), from hundreds of static shares and chunks (a 32768-token
    context), or not at all (a 100-token and a one-token pair)."""
    lengths = [32768, 2000, 100, 1]
    case = workloads.paged_case(700 + group, lengths, group * 4, 4, 128, 16, BF16, name=f"merges{group}")
    _check(case)


def test_binding_refuses_strided_views():
    """A strided view passes a pointer whose rows are not where the kernels
    look: the binding refuses it instead of letting the call misread memory."""
    case = workloads.paged_case(870, [20, 33], 8, 2, 64, 16, F16)
    dc = DeviceCase(case)
    q2 = torch.cat([dc.q, dc.q], dim=2)[:, :, ::2]  # right shape, not contiguous
    assert q2.shape == dc.q.shape and not q2.is_contiguous()
    with pytest.raises(ValueError, match="contiguous"):
        pa.decode(torch.empty_like(dc.q), q2, dc.k_cache, dc.v_cache, dc.block_tables,
                  dc.context_lens, case.scale, case.max_context_len)
    with pytest.raises(ValueError, match="contiguous"):
        pa.decode(torch.empty_like(dc.q), dc.q, dc.k_cache, dc.v_cache, dc.block_tables.t().contiguous().t(),
                  dc.context_lens, case.scale, case.max_context_len)
