"""GPU parity of pa_decode_shared_prefix: groups of sequences whose tables
share leading blocks (serving-paged-attention, "공유는 표를 베끼는 일이
된다"), decoded with the shared blocks attended once per group. The result is
the same definition as pa_decode's, so every case is checked against the fp64
oracle's paged_decode, which knows nothing of the groups."""

import numpy as np
import pytest
import torch

import oracle
import workloads
from workloads import BF16, F16
from gpu_helpers import DeviceCase, assert_close, oracle_decode, run_decode, to_f64
import paged_kv_cache_288_gb300 as pa

pytestmark = pytest.mark.gpu


def _run(dc, group_start, group_prefix, max_group_size=None, max_prefix_len=None, debug_err=None):
    c = dc.case
    gs = torch.from_numpy(np.asarray(group_start, np.int32)).cuda()
    gp = torch.from_numpy(np.asarray(group_prefix, np.int32)).cuda()
    sizes = np.diff(np.asarray(group_start))
    mgs = int(sizes.max()) if max_group_size is None and len(sizes) else (max_group_size or 1)
    mpl = int(np.max(group_prefix)) if max_prefix_len is None and len(group_prefix) else (max_prefix_len or 0)
    n = pa.decode_shared_prefix_workspace_size(c.num_seqs, c.num_heads, c.num_kv_heads, c.head_dim,
                                               c.block_size, len(group_prefix), mgs, mpl)
    ws = torch.empty(max(n, 256), dtype=torch.uint8, device="cuda")
    out = torch.full_like(dc.q, float("nan"))
    pa.decode_shared_prefix(out, dc.q, dc.k_cache, dc.v_cache, dc.block_tables, dc.context_lens, c.scale,
                            c.max_context_len, gs, gp, mgs, mpl, ws,
                            debug_err=dc.debug_err if debug_err is None else debug_err)
    return out


GROUPED = [
    # (group sizes, prefix blocks, suffix lo..hi, Hq, Hkv, d, bs, dtype)
    ([5, 1, 9, 3], [4, 0, 17, 1], (0, 70), 8, 2, 128, 16, BF16),
    ([12], [40], (1, 300), 32, 8, 128, 16, F16),
    ([2, 7], [9, 30], (0, 50), 4, 4, 64, 8, BF16),        # group 1 (MHA)
    ([6, 4], [3, 5], (5, 90), 16, 2, 128, 32, F16),        # group 8
    ([3, 3], [2, 6], (0, 130), 32, 1, 128, 64, BF16),      # MQA: 32 query heads, one KV head
    ([40], [12], (0, 20), 16, 4, 128, 16, BF16),           # many members per group
]


@pytest.mark.parametrize("sizes,pblocks,suffix,Hq,Hkv,d,bs,dtype", GROUPED)
def test_shared_prefix_matches_oracle(sizes, pblocks, suffix, Hq, Hkv, d, bs, dtype):
    case, gs, gp = workloads.grouped_prefix_case(sum(sizes) * 7 + bs, sizes, pblocks, suffix[0], suffix[1],
                                                 Hq, Hkv, d, bs, dtype)
    dc = DeviceCase(case)
    out = _run(dc, gs, gp)
    ref = oracle_decode(case)
    torch.cuda.synchronize()
    assert dc.debug_err.item() == 0
    assert_close(out, ref, dtype, dtype, f"shared prefix {sizes}/{pblocks}")
    # and against pa_decode on the same batch, within the same bound
    plain = run_decode(pa, dc)
    a, b = to_f64(out, dtype), to_f64(plain, dtype)
    assert np.all(np.abs(a - b) <= 2e-3 + 1e-2 * np.abs(b))


def test_shared_prefix_serving_batch_copy_on_write_flow():
    """The shared-prefix serving batch at full size: 100 sequences whose 64
    prefix blocks are shared, the partly filled 64th copied per sequence
    before its suffix is written (pa_copy_blocks), then one decode with the
    63 still shared blocks described as one group."""
    case = workloads.shared_prefix()
    dc = DeviceCase(case)
    block_bytes = case.num_kv_heads * case.block_size * case.head_dim * 2
    pa.copy_blocks(pa.pointer_array([dc.k_cache], "cuda"), pa.pointer_array([dc.v_cache], "cuda"),
                   dc.cow_pairs, case.num_blocks, block_bytes, debug_err=dc.debug_err)
    pa.reshape_and_cache(dc.new_key, dc.new_value, dc.k_cache, dc.v_cache, dc.slot_mapping,
                         debug_err=dc.debug_err)
    shared_tokens = (case.meta["prefix_len"] // case.block_size) * case.block_size  # 63 whole blocks
    out = _run(dc, [0, case.num_seqs], [shared_tokens])
    kc, vc = case.k_cache.copy(), case.v_cache.copy()
    oracle.copy_blocks([kc], [vc], case.cow_pairs)
    oracle.reshape_and_cache(case.new_key, case.new_value, kc, vc, case.slot_mapping, 16, F16, F16)
    ref = oracle_decode(case, k_cache=kc, v_cache=vc)
    torch.cuda.synchronize()
    assert dc.debug_err.item() == 0
    max_abs, _ = assert_close(out, ref, F16, F16, "shared-prefix serving batch")
    assert max_abs <= 2e-3, max_abs


def test_shared_prefix_two_calls_and_no_groups():
    """Two calls in a row reuse the workspace; a call with no groups is plain decode."""
    case, gs, gp = workloads.grouped_prefix_case(77, [4, 4], [6, 2], 0, 60, 8, 2, 128, 16, BF16)
    dc = DeviceCase(case)
    ref = oracle_decode(case)
    for _ in range(2):
        out = _run(dc, gs, gp)
        torch.cuda.synchronize()
        assert_close(out, ref, BF16, BF16, "repeat")
    out = _run(dc, [0], np.zeros(0, np.int32), max_group_size=1, max_prefix_len=0)
    torch.cuda.synchronize()
    assert_close(out, ref, BF16, BF16, "no groups")
    assert dc.debug_err.item() == 0


def test_shared_prefix_flags_bad_descriptions():
    """A member whose table differs from its group's in the shared blocks, and
    a group range past the batch, are flagged; every index stays in bounds
    (the kernels clamp), so the calls complete."""
    case, gs, gp = workloads.grouped_prefix_case(78, [3, 2], [4, 2], 1, 30, 8, 2, 128, 16, BF16)
    dc = DeviceCase(case)
    bad_tables = case.block_tables.copy()
    bad_tables[1, 2] = bad_tables[3, 0]  # not the group's shared block
    dc.block_tables = torch.from_numpy(bad_tables).cuda()
    _run(dc, gs, gp)
    torch.cuda.synchronize()
    assert dc.debug_err.item() & pa.DEVERR_PREFIX
    dc2 = DeviceCase(case)
    _run(dc2, [0, 3, 9], gp, max_group_size=6)  # the last group ends past the 5 sequences
    torch.cuda.synchronize()
    assert dc2.debug_err.item() & pa.DEVERR_PREFIX
    dc3 = DeviceCase(case)
    _run(dc3, gs, [64, 40])  # 40 tokens is not a whole number of 16-token blocks
    torch.cuda.synchronize()
    assert dc3.debug_err.item() & pa.DEVERR_PREFIX
