"""Helpers for the GPU parity tests: move a seeded case to the device, run
the library through its binding, and compare with the oracle.

Tolerances, element-wise:
16-bit KV: the allclose form |gpu - ref| <= 2e-3 + 1e-2 * |ref| (the literal
2e-3 alone fails for bf16 outputs of magnitude >= 0.5, whose half ulp is
2^-9); 8-bit KV: the literal |gpu - ref| <= 3e-2, against the oracle run on
the same stored E4M3 codes. For inputs drawn with a smaller spread than
N(0, 1) the 8-bit bound scales with the largest |V| (``value_scale``).
"""

import numpy as np
import torch

import oracle
import workloads

ATOL_16 = 2e-3
RTOL_16 = 1e-2
ATOL_FP8 = 3e-2

_TORCH = {workloads.F16: torch.float16, workloads.BF16: torch.bfloat16,
          workloads.FP8_E4M3: torch.uint8}


def dev(bits, dtype, device="cuda"):
    """Raw-bit numpy array -> device tensor of the storage dtype (bits kept)."""
    a = np.ascontiguousarray(bits)
    if dtype == workloads.FP8_E4M3:
        return torch.from_numpy(a.view(np.uint8)).to(device)
    t = torch.from_numpy(a.view(np.int16)).to(device)
    return t.view(_TORCH[dtype])


def host_bits(t):
    """Device tensor -> raw-bit numpy array (uint16 or uint8)."""
    t = t.detach().cpu()
    if t.dtype in (torch.float16, torch.bfloat16):
        return t.view(torch.int16).numpy().view(np.uint16)
    return t.view(torch.uint8).numpy()


def to_f64(t, dtype):
    return oracle.bits_to_f64(host_bits(t), dtype)


class DeviceCase:
    """Device tensors of a workloads.DecodeCase."""

    def __init__(self, case, device="cuda"):
        self.case = case
        self.q = dev(case.q, case.q_dtype, device)
        self.k_cache = dev(case.k_cache, case.kv_dtype, device) if case.k_cache is not None else None
        self.v_cache = dev(case.v_cache, case.kv_dtype, device) if case.v_cache is not None else None
        self.block_tables = torch.from_numpy(case.block_tables).to(device)
        self.context_lens = torch.from_numpy(case.context_lens).to(device)
        self.k_scale = torch.from_numpy(case.k_scale).to(device) if case.k_scale is not None else None
        self.v_scale = torch.from_numpy(case.v_scale).to(device) if case.v_scale is not None else None
        self.debug_err = torch.zeros(1, dtype=torch.int32, device=device)
        if case.new_key is not None:
            self.new_key = dev(case.new_key, case.src_dtype, device)
            self.new_value = dev(case.new_value, case.src_dtype, device)
            self.slot_mapping = torch.from_numpy(case.slot_mapping).to(device)
        if case.cow_pairs is not None:
            self.cow_pairs = torch.from_numpy(case.cow_pairs).to(device)

    def out_like_q(self):
        return torch.empty_like(self.q)


def run_decode(pa, dc, partition_size=0, workspace=True, k_cache=None, v_cache=None,
               block_tables=None, context_lens=None, q=None):
    c = dc.case
    q = dc.q if q is None else q
    kc = dc.k_cache if k_cache is None else k_cache
    vc = dc.v_cache if v_cache is None else v_cache
    bt = dc.block_tables if block_tables is None else block_tables
    cl = dc.context_lens if context_lens is None else context_lens
    max_ctx = int(cl.max().item()) if cl.numel() else 0
    ws = None
    if workspace:
        n = pa.decode_workspace_size(q.shape[0], q.shape[1], kc.shape[1], q.shape[2], max_ctx,
                                     partition_size)
        ws = torch.empty(max(n, 1), dtype=torch.uint8, device=q.device)
    out = torch.full_like(q, float("nan"))
    pa.decode(out, q, kc, vc, bt, cl, c.scale, max_ctx, k_scale=dc.k_scale, v_scale=dc.v_scale,
              partition_size=partition_size, workspace=ws, debug_err=dc.debug_err)
    return out


def oracle_decode(case, k_cache=None, v_cache=None, context_lens=None, q=None):
    return oracle.paged_decode(
        case.q if q is None else q,
        case.k_cache if k_cache is None else k_cache,
        case.v_cache if v_cache is None else v_cache,
        case.block_tables, case.context_lens if context_lens is None else context_lens,
        case.scale, case.block_size, case.q_dtype, case.kv_dtype, case.k_scale, case.v_scale)


def assert_close(got_t, ref, dtype_out, kv_dtype, what="", value_scale=1.0):
    got = to_f64(got_t, dtype_out)
    if kv_dtype == workloads.FP8_E4M3:
        atol, rtol = ATOL_FP8 * value_scale, 0.0
    else:
        atol, rtol = ATOL_16, RTOL_16
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    err = np.abs(got - ref)
    bad = err > atol + rtol * np.abs(ref)
    if bad.any():
        idx = np.argwhere(bad)[:5]
        raise AssertionError(
            f"{what}: {bad.sum()} of {bad.size} elements out of tolerance; max abs err "
            f"{err.max():.3e}; first bad {idx.tolist()} got {got[tuple(idx[0])]} ref {ref[tuple(idx[0])]}")
    return float(err.max()), float((err / np.maximum(np.abs(ref), 1e-30)).max())
