"""GPU parity of the paged prefill (tcgen05 kernel) against the fp64 oracle."""

import numpy as np
import pytest
import torch

import oracle
import workloads
from workloads import BF16, F16
from gpu_helpers import assert_close, dev

pytestmark = pytest.mark.gpu

import paged_kv_cache_288_gb300 as pa  # noqa: E402


def _run(case, max_query_len=None, err=None):
    q = dev(case.q, case.dtype)
    out = torch.full_like(q, float("nan"))
    err = torch.zeros(1, dtype=torch.int32, device="cuda") if err is None else err
    pa.prefill(out, q, dev(case.k_cache, case.dtype), dev(case.v_cache, case.dtype),
               torch.from_numpy(case.block_tables).cuda(), torch.from_numpy(case.context_lens).cuda(),
               torch.from_numpy(case.query_start).cuda(), case.scale,
               case.max_query_len if max_query_len is None else max_query_len, debug_err=err)
    torch.cuda.synchronize()
    return out, err


def _oracle(case):
    return oracle.paged_prefill(case.q, case.k_cache, case.v_cache, case.block_tables, case.context_lens,
                                case.query_start, case.scale, case.block_size, case.dtype, case.dtype)


# Tolerance. The decode reading (|err| <= 2e-3 + 1e-2 |ref|) plus the one
# rounding prefill adds on the tensor cores: the softmax weights p enter the
# P.V product rounded to the 16-bit type of V (relative error <= u = 2^-9 for
# bf16, 2^-11 for f16) while the normaliser sums the unrounded float32
# weights, so out = sum(p~ v) / sum(p) differs from the exact value by at
# most u * max |v| over the keys the query attends, column by column.
_U = {BF16: 2.0 ** -9, F16: 2.0 ** -11}


def _weight_rounding_bound(case):
    """u * max over the attended keys of |v|, per output element."""
    bound = np.zeros((case.q.shape[0], case.num_heads, case.head_dim))
    G = case.num_heads // case.num_kv_heads
    for i in range(case.num_seqs):
        q0, q1 = int(case.query_start[i]), int(case.query_start[i + 1])
        n, ctx = q1 - q0, int(case.context_lens[i])
        if n == 0:
            continue
        for g in range(case.num_kv_heads):
            V = oracle.gather_sequence(case.v_cache, case.block_tables[i], ctx, case.block_size, g, case.dtype)
            run = np.maximum.accumulate(np.abs(V), axis=0)  # [ctx, d]
            for j in range(n):
                bound[q0 + j, g * G:(g + 1) * G] = run[ctx - n + j]
    return _U[case.dtype] * bound


def _check(out, ref, case, what, rows=slice(None)):
    got = out.double().cpu().numpy()[rows]
    ref = ref[rows]
    tol = 2e-3 + 1e-2 * np.abs(ref) + _weight_rounding_bound(case)[rows]
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    err = np.abs(got - ref)
    bad = err > tol
    assert not bad.any(), (f"{what}: {bad.sum()} of {bad.size} out of tolerance; max err {err.max():.3e}; "
                           f"first bad {np.argwhere(bad)[:3].tolist()}")


@pytest.mark.parametrize("dtype", [BF16, F16])
@pytest.mark.parametrize("G,bs", [(4, 16), (1, 8), (2, 32), (8, 64)])
def test_prefill_matches_oracle(dtype, G, bs):
    """Chunks with and without cached prefixes, ragged against the 128-row
    query tiles and the 128-key tiles; a chunk of one token; an empty chunk."""
    Hkv = 2
    prefix = [0, 5, 130, 0, 300, 17, 64]
    chunk = [1, 40, 77, 128 // G + 3, 0, 200, 129]
    case = workloads.prefill_case(60 + G + bs, prefix, chunk, G * Hkv, Hkv, 128, bs, dtype)
    out, err = _run(case)
    ref = _oracle(case)
    assert err.item() == 0
    _check(out, ref, case, f"prefill G{G} bs{bs}")
    # how often the decode reading alone (2e-3 + 1e-2 |ref|, without the
    # weight-rounding term) would fail: the weight term is needed for a few
    # elements of the early queries of a chunk (few keys, large |v|) only
    got = out.double().cpu().numpy()
    plain_bad = np.abs(got - ref) > 2e-3 + 1e-2 * np.abs(ref)
    frac = float(plain_bad.mean())
    print(f"prefill G{G} bs{bs} {dtype}: {plain_bad.sum()} of {plain_bad.size} elements "
          f"({100 * frac:.3f} %) beyond the decode reading alone")
    assert frac <= 0.02, frac


def test_prefill_single_query_chunks_equal_decode():
    """A chunk of one query is a decode step: both kernels agree with the oracle
    and with each other within rounding."""
    ctx = [1, 16, 17, 300, 1000]
    case = workloads.prefill_case(70, [c - 1 for c in ctx], [1] * len(ctx), 32, 8, 128, 16, BF16)
    out, _ = _run(case)
    dq = dev(case.q, BF16)
    dout = torch.empty_like(dq)
    mx = max(ctx)
    ws = torch.empty(pa.decode_workspace_size(len(ctx), 32, 8, 128, mx, 0), dtype=torch.uint8, device="cuda")
    pa.decode(dout, dq, dev(case.k_cache, BF16), dev(case.v_cache, BF16),
              torch.from_numpy(case.block_tables).cuda(), torch.from_numpy(case.context_lens).cuda(),
              case.scale, mx, workspace=ws)
    torch.cuda.synchronize()
    ref = _oracle(case)
    _check(out, ref, case, "prefill n=1")
    assert_close(dout, ref, BF16, BF16, "decode")


def test_prefill_flags_contexts_shorter_than_the_chunk():
    case = workloads.prefill_case(71, [10, 0], [20, 30], 8, 2, 128, 16, BF16)
    lens = case.context_lens.copy()
    case.context_lens[1] = 12  # shorter than its 30 queries
    out, err = _run(case)
    assert err.item() & pa.DEVERR_CONTEXT_RANGE
    case.context_lens = lens
    ref = _oracle(case)
    q1 = int(case.query_start[1])
    _check(out, ref, case, "the valid sequence", rows=slice(0, q1))


def test_prefill_clamps_query_start_past_num_tokens():
    """query_start entries beyond num_tokens are clamped by the kernel and
    flagged: q and out are views of the first T rows of buffers with 8 guard
    rows after them, the last sequence's query_start claims those 8 rows too,
    and the guard rows of out must stay untouched (NaN) while the rows in
    range still match the oracle. The guard rows exist, so even a missing
    clamp would stay inside the allocation."""
    case = workloads.prefill_case(73, [20, 5], [10, 12], 8, 2, 128, 16, BF16)
    T = case.q.shape[0]
    q_all = dev(np.concatenate([case.q, case.q[:8]]), BF16)
    out_all = torch.full_like(q_all, float("nan"))
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    qs = case.query_start.copy()
    qs[-1] = T + 8  # past num_tokens = T
    pa.prefill(out_all[:T], q_all[:T], dev(case.k_cache, BF16), dev(case.v_cache, BF16),
               torch.from_numpy(case.block_tables).cuda(), torch.from_numpy(case.context_lens).cuda(),
               torch.from_numpy(qs).cuda(), case.scale, int(np.diff(qs).max()), debug_err=err)
    torch.cuda.synchronize()
    assert err.item() & pa.DEVERR_QUERY_START
    assert torch.isnan(out_all[T:].float()).all(), "a guard row past num_tokens was written"
    _check(out_all[:T], _oracle(case), case, "clamped query_start")


@pytest.mark.parametrize("num_seqs", [9, 260])
def test_prefill_work_order_covers_every_sequence(num_seqs):
    """CTAs take the heaviest sequences first (by n (2 ctx - n)) when the batch
    has at most 256 sequences, and launch order beyond that. Sequences of
    equal work (ties, broken by index) and a batch past that limit must each
    still land on their own rows; their data differ, so a swap shows."""
    rng = np.random.default_rng(num_seqs)
    if num_seqs == 9:
        prefix = [40, 40, 40, 0, 300, 40, 7, 300, 0]
        chunk = [33, 33, 33, 1, 70, 33, 90, 70, 1]
    else:
        prefix = rng.integers(0, 40, num_seqs).tolist()
        chunk = rng.integers(0, 4, num_seqs).tolist()
    case = workloads.prefill_case(72 + num_seqs, prefix, chunk, 8, 2, 128, 16, BF16)
    out, err = _run(case)
    assert err.item() == 0
    _check(out, _oracle(case), case, f"{num_seqs} sequences")


def test_prefill_llama8b_shape_sampled():
    """The bench's chunked-prefill batch (16 x 512-token chunks after prefixes
    up to 2048, 32/8/128 bf16): rows sampled across every sequence, checked
    against the oracle computed for those rows only."""
    case = workloads.prefill_llama8b()
    out, err = _run(case)
    assert err.item() == 0
    got = out.float().cpu().numpy()
    rng = np.random.default_rng(5)
    for i in range(case.num_seqs):
        q0, q1 = int(case.query_start[i]), int(case.query_start[i + 1])
        rows = sorted(set([q0, q1 - 1] + list(rng.integers(q0, q1, 3))))
        sub = workloads.PrefillCase(**{**case.__dict__})
        for r in rows:
            j = r - q0
            ctx = int(case.context_lens[i]) - (q1 - q0) + j + 1
            dec = oracle.paged_decode(case.q[r:r + 1], case.k_cache, case.v_cache, case.block_tables[i:i + 1],
                                      np.array([ctx], np.int32), case.scale, 16, BF16, BF16)
            err_abs = np.abs(got[r] - dec[0])
            V = oracle.gather_sequence(case.v_cache, case.block_tables[i], ctx, 16, 0, BF16)
            vmax = np.abs(np.stack([oracle.gather_sequence(case.v_cache, case.block_tables[i], ctx, 16, g, BF16)
                                    for g in range(case.num_kv_heads)])).max(axis=1)  # [Hkv, d]
            bound = _U[BF16] * np.repeat(vmax, case.num_heads // case.num_kv_heads, axis=0)
            del V
            assert np.all(err_abs <= 2e-3 + 1e-2 * np.abs(dec[0]) + bound), (i, j, float(err_abs.max()))
        del sub
