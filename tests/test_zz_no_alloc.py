"""pa_decode_split_noalloc: the split decode for callers that cannot allocate.

Some callers of this library have no way to allocate device memory (a plugin
inside a framework that owns every allocation, or a runtime whose device
memory is fixed at start-up), so they cannot provide the workspace that
pa_decode's split path needs. pa_decode_split_noalloc keeps those partials in
a scratch array built into the library instead. This test calls it through
the C ABI twice in a row, on two different problems, and checks each result
against the fp64 oracle and against pa_decode with a caller-allocated
workspace, within the tolerance of the other decode tests (the output starts
as NaN, so a row the call leaves unwritten fails). It also checks that sizes
beyond the built-in scratch are refused.

The file name sorts last so that a run stopping at the first failure has run
every other test first; the test also passes on its own in a fresh process.
"""

import ctypes

import pytest
import torch

import workloads
from workloads import BF16, F16
from gpu_helpers import DeviceCase, assert_close, oracle_decode, to_f64
import paged_kv_cache_288_gb300 as pa

pytestmark = pytest.mark.gpu

PA_ERR_WORKSPACE = 4


def _noalloc_call(dc, partition_size):
    """pa_decode_split_noalloc through ctypes, on the current stream."""
    c = dc.case
    out = torch.full_like(dc.q, float("nan"))
    L = pa.lib()
    status = L.pa_decode_split_noalloc(
        ctypes.c_void_p(out.data_ptr()), ctypes.c_void_p(dc.q.data_ptr()),
        ctypes.c_void_p(dc.k_cache.data_ptr()), ctypes.c_void_p(dc.v_cache.data_ptr()),
        ctypes.c_void_p(dc.block_tables.data_ptr()), dc.block_tables.shape[1],
        ctypes.c_void_p(dc.context_lens.data_ptr()), c.num_seqs, c.num_heads, c.num_kv_heads,
        c.head_dim, c.block_size, c.num_blocks, c.scale,
        pa.BF16 if c.q_dtype == BF16 else pa.F16, pa.BF16 if c.kv_dtype == BF16 else pa.F16,
        None, None, c.max_context_len, partition_size, ctypes.c_void_p(dc.debug_err.data_ptr()),
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    return status, out


def _with_workspace(dc, partition_size):
    c = dc.case
    n = pa.decode_workspace_size(c.num_seqs, c.num_heads, c.num_kv_heads, c.head_dim,
                                 c.max_context_len, partition_size)
    ws = torch.empty(n, dtype=torch.uint8, device="cuda")
    out = torch.full_like(dc.q, float("nan"))
    pa.decode(out, dc.q, dc.k_cache, dc.v_cache, dc.block_tables, dc.context_lens, c.scale,
              c.max_context_len, partition_size=partition_size, workspace=ws,
              debug_err=dc.debug_err)
    return out


def test_noalloc_matches_workspace_decode_on_two_calls_in_a_row():
    first = workloads.paged_case(9001, [4096, 17, 1000, 2500, 1], 32, 8, 128, 16, BF16,
                                 name="noalloc_a")
    second = workloads.paged_case(9002, [300, 1500, 64], 8, 2, 64, 32, F16, name="noalloc_b")
    for case, part in ((first, 512), (second, 64)):
        dc = DeviceCase(case)
        status, got = _noalloc_call(dc, part)
        assert status == 0, pa.lib().pa_last_error_message()
        ref = _with_workspace(dc, part)
        torch.cuda.synchronize()
        assert dc.debug_err.item() == 0
        assert_close(got, oracle_decode(case), case.q_dtype, case.kv_dtype, case.name + " vs oracle")
        assert_close(got, to_f64(ref, case.q_dtype), case.q_dtype, case.kv_dtype, case.name)


def test_noalloc_refuses_sizes_beyond_its_scratch():
    """256 sequences x 64 heads x 64 partitions of head dim 128 need ~540 MB of partials.

    Every tensor passed is real and every table entry valid, so the refusal is
    the only thing that keeps the call from running.
    """
    B, Hq, Hkv, d, bs, Nb, ctx = 256, 64, 8, 128, 16, 8, 32768
    need = pa.decode_workspace_size(B, Hq, Hkv, d, ctx, 512)
    assert need > (16 << 20)
    q = torch.zeros(B, Hq, d, dtype=torch.bfloat16, device="cuda")
    out = torch.empty_like(q)
    kc = torch.zeros(Nb, Hkv, bs, d, dtype=torch.bfloat16, device="cuda")
    vc = torch.zeros_like(kc)
    tables = (torch.arange(B * (ctx // bs), dtype=torch.int32, device="cuda") % Nb).view(B, -1)
    lens = torch.full((B,), ctx, dtype=torch.int32, device="cuda")
    status = pa.lib().pa_decode_split_noalloc(
        ctypes.c_void_p(out.data_ptr()), ctypes.c_void_p(q.data_ptr()),
        ctypes.c_void_p(kc.data_ptr()), ctypes.c_void_p(vc.data_ptr()),
        ctypes.c_void_p(tables.data_ptr()), tables.shape[1], ctypes.c_void_p(lens.data_ptr()),
        B, Hq, Hkv, d, bs, Nb, 0.1, pa.BF16, pa.BF16, None, None, ctx, 512, None,
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert status == PA_ERR_WORKSPACE
    assert b"scratch" in pa.lib().pa_last_error_message()
