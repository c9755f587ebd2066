"""GPU parity at the full sizes of the five workloads, in the launch
configuration bench.py times (partition_size 0 = the library's own schedule,
512 for the long-context split path)."""

import numpy as np
import pytest
import torch

import oracle
import workloads
from workloads import F16, BF16, FP8_E4M3
from gpu_helpers import DeviceCase, assert_close, host_bits, oracle_decode, run_decode
import paged_kv_cache_288_gb300 as pa

pytestmark = pytest.mark.gpu


def test_llama8b_batch64_step():
    case = workloads.llama8b()
    dc = DeviceCase(case)
    pa.reshape_and_cache(dc.new_key, dc.new_value, dc.k_cache, dc.v_cache, dc.slot_mapping,
                         debug_err=dc.debug_err)
    out = run_decode(pa, dc)
    kc, vc = case.k_cache.copy(), case.v_cache.copy()
    oracle.reshape_and_cache(case.new_key, case.new_value, kc, vc, case.slot_mapping, 16, BF16, BF16)
    torch.cuda.synchronize()
    assert np.array_equal(host_bits(dc.k_cache), kc)
    assert np.array_equal(host_bits(dc.v_cache), vc)
    ref = oracle_decode(case, k_cache=kc, v_cache=vc)
    max_abs, max_rel = assert_close(out, ref, BF16, BF16, "llama8b")
    assert max_abs <= 2e-3, max_abs  # the literal bound holds here as well
    assert dc.debug_err.item() == 0


def test_shared_prefix_copy_on_write_flow():
    case = workloads.shared_prefix()
    dc = DeviceCase(case)
    block_bytes = case.num_kv_heads * case.block_size * case.head_dim * 2
    pa.copy_blocks(pa.pointer_array([dc.k_cache], "cuda"), pa.pointer_array([dc.v_cache], "cuda"),
                   dc.cow_pairs, case.num_blocks, block_bytes, debug_err=dc.debug_err)
    pa.reshape_and_cache(dc.new_key, dc.new_value, dc.k_cache, dc.v_cache, dc.slot_mapping,
                         debug_err=dc.debug_err)
    out = run_decode(pa, dc)
    kc, vc = case.k_cache.copy(), case.v_cache.copy()
    oracle.copy_blocks([kc], [vc], case.cow_pairs)
    oracle.reshape_and_cache(case.new_key, case.new_value, kc, vc, case.slot_mapping, 16, F16, F16)
    torch.cuda.synchronize()
    assert np.array_equal(host_bits(dc.k_cache), kc)
    assert np.array_equal(host_bits(dc.v_cache), vc)
    ref = oracle_decode(case, k_cache=kc, v_cache=vc)
    assert_close(out, ref, F16, F16, "shared prefix")
    assert dc.debug_err.item() == 0


@pytest.mark.parametrize("bs", [8, 16, 32, 64])
def test_long_context_split(bs):
    case = workloads.long_context(bs)
    dc = DeviceCase(case)
    pa.reshape_and_cache(dc.new_key, dc.new_value, dc.k_cache, dc.v_cache, dc.slot_mapping,
                         debug_err=dc.debug_err)
    out = run_decode(pa, dc, partition_size=512)
    kc, vc = case.k_cache.copy(), case.v_cache.copy()
    oracle.reshape_and_cache(case.new_key, case.new_value, kc, vc, case.slot_mapping, bs, BF16, BF16)
    # the oracle on three of the eight sequences (all heads); each is independent
    sample = [0, 3, 7]
    sub = workloads.DecodeCase(**{**case.__dict__, "q": case.q[sample],
                                  "block_tables": case.block_tables[sample],
                                  "context_lens": case.context_lens[sample], "num_seqs": 3})
    ref = oracle_decode(sub, k_cache=kc, v_cache=vc)
    torch.cuda.synchronize()
    assert_close(out[sample], ref, BF16, BF16, f"long context bs{bs}")
    assert dc.debug_err.item() == 0


@pytest.mark.parametrize("layer", [0, 31])
def test_fp8_step_layer(layer):
    case = workloads.fp8_step_layer(layer)
    dc = DeviceCase(case)
    pa.reshape_and_cache(dc.new_key, dc.new_value, dc.k_cache, dc.v_cache, dc.slot_mapping,
                         k_scale=dc.k_scale, v_scale=dc.v_scale, debug_err=dc.debug_err)
    out = run_decode(pa, dc)
    kc, vc = case.k_cache.copy(), case.v_cache.copy()
    oracle.reshape_and_cache(case.new_key, case.new_value, kc, vc, case.slot_mapping, 16, BF16,
                             FP8_E4M3, case.k_scale, case.v_scale)
    torch.cuda.synchronize()
    assert np.array_equal(host_bits(dc.k_cache), kc)
    assert np.array_equal(host_bits(dc.v_cache), vc)
    ref = oracle_decode(case, k_cache=kc, v_cache=vc)
    max_abs, _ = assert_close(out, ref, BF16, FP8_E4M3, f"fp8 layer {layer}")
    assert max_abs <= 3e-2, max_abs  # the literal bound for the 8-bit KV workload
    assert dc.debug_err.item() == 0
