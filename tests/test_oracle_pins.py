"""Pins of the fp64 oracle against what the pages and the mathematics fix.

Nothing here compares the oracle with itself: each check is a value the
pages print (tests/golden/*.json, with their sources), a closed form, an
invariant, a special case that reduces to a textbook result or to a library
routine (torch's scaled_dot_product_attention in float64), or brute force on
tiny inputs written as plain Python loops over a contiguous cache.
"""

import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
from oracle import F16, BF16, FP8_E4M3
import workloads

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


# ----------------------------------------------------------------------------
# memory accounting: the worked examples printed on the pages


def test_kv_size_worked_example():
    g = _golden("kv_size_worked_example.json")
    per_token = oracle.kv_cache_bytes(g["num_layers"], g["num_kv_heads"], g["head_dim"], 1,
                                      g["bytes_per_value_fp16"])
    assert per_token == g["bytes_per_token"] == 128 * 1024
    per_req = oracle.kv_cache_bytes(g["num_layers"], g["num_kv_heads"], g["head_dim"],
                                    g["tokens_per_request"], g["bytes_per_value_fp16"])
    assert per_req == g["bytes_per_request"] == 512 * 1024 * 1024
    free = g["card_bytes"] - g["weight_bytes"]
    assert oracle.max_concurrent_requests(free, per_req) == g["max_requests"]
    # 8-bit values: half the bytes, twice the requests
    per_req8 = oracle.kv_cache_bytes(g["num_layers"], g["num_kv_heads"], g["head_dim"],
                                     g["tokens_per_request"], g["bytes_per_value_8bit"])
    assert 2 * per_req8 == per_req
    assert oracle.max_concurrent_requests(free, per_req8) == g["max_requests_8bit"]


def test_kv_size_is_linear_in_every_factor():
    base = oracle.kv_cache_bytes(3, 5, 7, 11, 2)
    assert base == 2 * 3 * 5 * 7 * 11 * 2
    for i in range(5):
        args = [3, 5, 7, 11, 2]
        args[i] *= 2
        assert oracle.kv_cache_bytes(*args) == 2 * base


def test_naive_waste_example():
    g = _golden("waste_examples.json")["naive"]
    w = oracle.naive_waste_fraction(g["max_len"], g["mean_len"])
    assert abs(w - g["stated_waste_fraction"]) < g["stated_precision"]
    assert w == pytest.approx(1 - 500 / 2048)


def test_paged_tail_waste_bound():
    g = _golden("waste_examples.json")["paged"]
    bs = g["block_size"]
    rng = np.random.default_rng(0)
    wastes = [oracle.paged_tail_waste_tokens(int(n), bs) for n in rng.integers(1, 5000, 2000)]
    assert max(wastes) == g["max_tail_waste_tokens"]
    assert min(wastes) == 0
    assert oracle.paged_tail_waste_tokens(16, 16) == 0
    assert oracle.paged_tail_waste_tokens(17, 16) == 15
    assert oracle.paged_tail_waste_tokens(1, 16) == 15
    assert oracle.paged_tail_waste_tokens(0, 16) == 0


def test_capacity_rule():
    g = _golden("waste_examples.json")["capacity"]
    assert oracle.concurrent_capacity(g["num_blocks"], g["block_size"],
                                      g["mean_request_len"]) == g["concurrent_requests"]


def test_naive_vs_paged_population():
    # 100 users, max 2048, all answers 500 tokens: paged keeps 512 tokens each
    naive, paged = oracle.naive_vs_paged_bytes([500] * 100, 2048, 16, 1)
    assert naive == 100 * 2048
    assert paged == 100 * 512
    # paged never holds more than one partly filled block per request
    rng = np.random.default_rng(1)
    lengths = list(rng.integers(1, 2048, 300))
    naive, paged = oracle.naive_vs_paged_bytes(lengths, 2048, 16, 1)
    assert sum(lengths) <= paged <= sum(lengths) + 15 * len(lengths)


# ----------------------------------------------------------------------------
# E4M3 codec, against the OCP OFP8 definition


def test_e4m3_spec_values():
    g = _golden("ofp8_e4m3_spec_values.json")
    for code, val in g["decode"]:
        got = oracle.e4m3_decode(np.array([int(code, 16)]))[0]
        assert got == val and math.copysign(1, got) == math.copysign(1, val), code
    for code in g["nan_codes"]:
        assert np.isnan(oracle.e4m3_decode(np.array([int(code, 16)]))[0])
    for x, code in g["encode_rne_satfinite"]["cases"]:
        assert int(oracle.e4m3_encode(np.array([x], np.float32))[0]) == int(code, 16), x


def test_e4m3_all_codes_round_trip():
    codes = np.arange(256)
    vals = oracle.e4m3_decode(codes)
    finite = ~np.isnan(vals)
    back = oracle.e4m3_encode(vals[finite].astype(np.float32))
    assert np.array_equal(back, codes[finite].astype(np.uint8))
    assert finite.sum() == 254
    assert np.nanmax(np.abs(vals)) == 448.0


def _nearest_even_brute(x):
    """Nearest finite E4M3 code by exhaustive search; ties go to the even code."""
    vals = oracle.e4m3_decode(np.arange(256))
    best = None
    for c in range(256):
        v = vals[c]
        if np.isnan(v):
            continue
        if v == 0 and c == 0x80 and not np.signbit(x):
            continue
        if v == 0 and c == 0x00 and np.signbit(x):
            continue
        d = abs(v - x)
        if best is None or d < best[0] or (d == best[0] and (c & 1) == 0 and (best[1] & 1) == 1):
            best = (d, c)
    return best[1]


def test_e4m3_encoder_matches_exhaustive_nearest():
    rng = np.random.default_rng(7)
    xs = np.concatenate([
        rng.normal(0, 1, 300), rng.normal(0, 100, 200), rng.uniform(-448, 448, 200),
        rng.uniform(-0.02, 0.02, 200),
        # exact midpoints between neighbouring codes
        [(a + b) / 2 for a, b in zip(np.sort(oracle.e4m3_decode(np.arange(0, 0x7f))),
                                     np.sort(oracle.e4m3_decode(np.arange(0, 0x7f)))[1:])],
    ]).astype(np.float32)
    got = oracle.e4m3_encode(xs)
    for x, c in zip(xs.astype(np.float64), got):
        assert int(c) == _nearest_even_brute(x), x


# ----------------------------------------------------------------------------
# widening of stored codes to float64, against torch's own conversions


_TORCH_VIEW = {F16: torch.float16, BF16: torch.bfloat16, FP8_E4M3: torch.float8_e4m3fn}


def _torch_widen(bits, dtype):
    """Raw codes -> float64 through torch's reinterpretation of the bits, an
    implementation of the formats that shares nothing with the oracle."""
    a = np.ascontiguousarray(bits)
    if dtype == FP8_E4M3:
        t = torch.from_numpy(a.astype(np.uint8)).view(torch.float8_e4m3fn)
    else:
        t = torch.from_numpy(a.astype(np.uint16).view(np.int16)).view(_TORCH_VIEW[dtype])
    return t.double().numpy()


@pytest.mark.parametrize("dtype,ncodes", [(F16, 1 << 16), (BF16, 1 << 16), (FP8_E4M3, 256)])
def test_bits_to_f64_matches_torch_on_every_code(dtype, ncodes):
    """Every 16-bit (f16, bf16) and 8-bit (E4M3) code widens to the value torch
    gives the same bits: same value, same sign of zero, NaN exactly where torch
    has NaN. A wrong shift, a float16 view used for bf16 or a dropped sign
    fails here."""
    codes = np.arange(ncodes, dtype=np.uint16 if ncodes > 256 else np.uint8)
    got = oracle.bits_to_f64(codes, dtype)
    want = _torch_widen(codes, dtype)
    assert np.array_equal(np.isnan(got), np.isnan(want))
    fin = ~np.isnan(want)
    assert np.array_equal(got[fin], want[fin])
    assert np.array_equal(np.signbit(got[fin]), np.signbit(want[fin]))


def test_bits_to_f64_known_codes():
    """A few codes whose values the formats fix: 1.0, -2.0, the largest finite
    value, the smallest subnormal."""
    assert oracle.bits_to_f64(np.array([0x3F80, 0xC000, 0x7F7F, 0x0001]), BF16).tolist() == [
        1.0, -2.0, (2 - 2.0 ** -7) * 2.0 ** 127, 2.0 ** -133]
    assert oracle.bits_to_f64(np.array([0x3C00, 0xC000, 0x7BFF, 0x0001]), F16).tolist() == [
        1.0, -2.0, 65504.0, 2.0 ** -24]


# ----------------------------------------------------------------------------
# scatter and copy


def test_scatter_hand_example():
    """Pool of 3 blocks x 2 KV heads x block size 2 x head dim 2, by hand."""
    key = np.array([[[1, 2], [3, 4]], [[5, 6], [7, 8]], [[9, 10], [11, 12]]], dtype=np.uint16)
    value = key + 100
    kc = np.zeros((3, 2, 2, 2), dtype=np.uint16)
    vc = np.zeros((3, 2, 2, 2), dtype=np.uint16)
    # token 0 -> slot 5 = block 2 offset 1; token 1 skipped; token 2 -> slot 2 = block 1 offset 0
    oracle.reshape_and_cache(key, value, kc, vc, np.array([5, -1, 2]), 2, F16, F16)
    want = np.zeros((3, 2, 2, 2), dtype=np.uint16)
    want[2, 0, 1] = [1, 2]
    want[2, 1, 1] = [3, 4]
    want[1, 0, 0] = [9, 10]
    want[1, 1, 0] = [11, 12]
    assert np.array_equal(kc, want)
    assert np.array_equal(vc, np.where(want > 0, want + 100, 0))


def test_scatter_then_gather_returns_tokens_in_order():
    case = workloads.paged_case(11, [13, 40, 1], 4, 2, 8, 8, F16)
    # write every token of every sequence through its slot, then gather
    kc = np.zeros_like(case.k_cache)
    vc = np.zeros_like(case.v_cache)
    g = torch.Generator().manual_seed(3)
    for i, ctx in enumerate(case.context_lens):
        toks_k = workloads.normal_bits(g, (int(ctx), 2, 8), F16)
        toks_v = workloads.normal_bits(g, (int(ctx), 2, 8), F16)
        slots = np.array([int(case.block_tables[i, p // 8]) * 8 + p % 8 for p in range(int(ctx))])
        oracle.reshape_and_cache(toks_k, toks_v, kc, vc, slots, 8, F16, F16)
        for h in range(2):
            got = oracle.gather_sequence(kc, case.block_tables[i], int(ctx), 8, h, F16)
            assert np.array_equal(got, toks_k[:, h].view(np.float16).astype(np.float64))


def test_scatter_fp8_quantises_with_block_scale():
    key = workloads.normal_bits(torch.Generator().manual_seed(5), (3, 1, 16), BF16)
    value = key.copy()
    kc = np.zeros((2, 1, 4, 16), dtype=np.uint8)
    vc = np.zeros((2, 1, 4, 16), dtype=np.uint8)
    ks = np.array([[0.5], [0.01]], dtype=np.float32)
    vs = np.array([[2.0], [1.0]], dtype=np.float32)
    oracle.reshape_and_cache(key, value, kc, vc, np.array([6, 1, -1]), 4, BF16, FP8_E4M3, ks, vs)
    x0 = (key[0, 0].astype(np.uint32) << 16).view(np.float32)
    # exact division by a power of two, then the spec encoder
    assert np.array_equal(kc[1, 0, 2], oracle.e4m3_encode(x0 / np.float32(0.01)))
    assert np.array_equal(vc[1, 0, 2], oracle.e4m3_encode(x0))
    x1 = (key[1, 0].astype(np.uint32) << 16).view(np.float32)
    assert np.array_equal(kc[0, 0, 1], oracle.e4m3_encode(x1 * np.float32(2.0)))
    assert np.array_equal(vc[0, 0, 1], oracle.e4m3_encode(x1 * np.float32(0.5)))
    # untouched slots stay zero
    assert kc[0, 0, 0].sum() == 0 and kc[1, 0, 3].sum() == 0


def test_copy_blocks_copies_every_layer_and_nothing_else():
    rng = np.random.default_rng(2)
    ks = [rng.integers(0, 65535, (6, 2, 4, 8), dtype=np.uint16) for _ in range(3)]
    vs = [rng.integers(0, 65535, (6, 2, 4, 8), dtype=np.uint16) for _ in range(3)]
    k0 = [k.copy() for k in ks]
    v0 = [v.copy() for v in vs]
    oracle.copy_blocks(ks, vs, [(1, 4), (1, 5), (3, 0)])
    for L in range(3):
        for b, src in ((4, 1), (5, 1), (0, 3)):
            assert np.array_equal(ks[L][b], k0[L][src])
            assert np.array_equal(vs[L][b], v0[L][src])
        for b in (1, 2, 3):
            assert np.array_equal(ks[L][b], k0[L][b])
            assert np.array_equal(vs[L][b], v0[L][b])


def _block_bytes(pool, b):
    """Block b of a pool read through a flat byte view at its byte offset (an
    indexing route independent of the oracle's per-block assignment)."""
    flat = pool.reshape(-1).view(np.uint8)
    n = flat.size // pool.shape[0]
    return flat[b * n:(b + 1) * n]


def test_swap_out_then_in_restores_the_request():
    """Swap-out copies the preempted request's blocks to the host pool byte for
    byte, swap-in brings them back into other device blocks: the round trip is
    the identity on those bytes, and no other block of either pool changes."""
    rng = np.random.default_rng(3)
    L, Nd, Nh = 3, 9, 5
    dk = [rng.integers(0, 65535, (Nd, 2, 4, 8), dtype=np.uint16) for _ in range(L)]
    dv = [rng.integers(0, 65535, (Nd, 2, 4, 8), dtype=np.uint16) for _ in range(L)]
    hk = [rng.integers(0, 65535, (Nh, 2, 4, 8), dtype=np.uint16) for _ in range(L)]
    hv = [rng.integers(0, 65535, (Nh, 2, 4, 8), dtype=np.uint16) for _ in range(L)]
    dk0, dv0 = [x.copy() for x in dk], [x.copy() for x in dv]
    hk0, hv0 = [x.copy() for x in hk], [x.copy() for x in hv]
    out_pairs = [(7, 0), (2, 3), (5, 4)]
    assert oracle.swap_blocks(hk, hv, dk, dv, out_pairs) == []
    for layer in range(L):
        for s, d in out_pairs:
            assert np.array_equal(_block_bytes(hk[layer], d), _block_bytes(dk0[layer], s))
            assert np.array_equal(_block_bytes(hv[layer], d), _block_bytes(dv0[layer], s))
        for b in (1, 2):
            assert np.array_equal(_block_bytes(hk[layer], b), _block_bytes(hk0[layer], b))
        for b in range(Nd):
            assert np.array_equal(_block_bytes(dk[layer], b), _block_bytes(dk0[layer], b))
    in_pairs = [(0, 1), (3, 8), (4, 6)]
    oracle.swap_blocks(dk, dv, hk, hv, in_pairs)
    for layer in range(L):
        for (s, _), (_, d) in zip(out_pairs, in_pairs):
            assert np.array_equal(_block_bytes(dk[layer], d), _block_bytes(dk0[layer], s))
            assert np.array_equal(_block_bytes(dv[layer], d), _block_bytes(dv0[layer], s))
        for b in (0, 2, 3, 4, 5, 7):
            assert np.array_equal(_block_bytes(dk[layer], b), _block_bytes(dk0[layer], b))


def test_swap_skips_pairs_outside_their_pool():
    rng = np.random.default_rng(4)
    dk = [rng.integers(0, 255, (4, 16), dtype=np.uint8)]
    hk = [rng.integers(0, 255, (2, 16), dtype=np.uint8)]
    dv, hv = [dk[0].copy()], [hk[0].copy()]
    h0 = hk[0].copy()
    skipped = oracle.swap_blocks(hk, hv, dk, dv, [(4, 0), (1, 2), (-1, 1), (3, 1)])
    assert skipped == [(4, 0), (1, 2), (-1, 1)]
    assert np.array_equal(hk[0][0], h0[0])
    assert np.array_equal(hk[0][1], dk[0][3])


# ----------------------------------------------------------------------------
# decode


def _brute_force_decode(q, K, V, scale):
    """softmax(q.K^T * scale) V for one query, as plain Python loops."""
    scores = [scale * sum(qc * kc for qc, kc in zip(q, krow)) for krow in K]
    w = [math.exp(s) for s in scores]
    z = sum(w)
    return [sum(wt * vrow[c] for wt, vrow in zip(w, V)) / z for c in range(len(q))]


def _contiguous_case(seed, lengths, Hq, Hkv, d, bs, dtype=F16):
    """Logical contiguous K/V per sequence, then placed block by block in a pool."""
    g = torch.Generator().manual_seed(seed)
    nbs = [-(-n // bs) for n in lengths]
    Nb = sum(nbs) + 3
    perm = torch.randperm(Nb, generator=g).numpy()
    tables = np.zeros((len(lengths), max(nbs)), dtype=np.int32)
    kc = np.full((Nb, Hkv, bs, d), workloads.NAN_BITS[dtype], dtype=np.uint16)
    vc = kc.copy()
    K_log, V_log = [], []
    cur = 0
    for i, n in enumerate(lengths):
        Kl = workloads.normal_bits(g, (nbs[i] * bs, Hkv, d), dtype)
        Vl = workloads.normal_bits(g, (nbs[i] * bs, Hkv, d), dtype)
        Kl[n:] = workloads.NAN_BITS[dtype]
        Vl[n:] = workloads.NAN_BITS[dtype]
        for j in range(nbs[i]):
            pb = perm[cur]
            cur += 1
            tables[i, j] = pb
            # pool block pb, all heads, holds logical rows j*bs..j*bs+bs-1
            kc[pb] = Kl[j * bs:(j + 1) * bs].transpose(1, 0, 2)
            vc[pb] = Vl[j * bs:(j + 1) * bs].transpose(1, 0, 2)
        K_log.append(Kl[:n])
        V_log.append(Vl[:n])
    q = workloads.normal_bits(g, (len(lengths), Hq, d), dtype)
    return q, kc, vc, tables, np.array(lengths, np.int32), K_log, V_log


def _f(bits, dtype=F16):
    return oracle.bits_to_f64(bits, dtype)


@pytest.mark.parametrize("lengths,Hq,Hkv,d,bs", [
    ([5, 17, 1], 4, 2, 8, 4),
    ([9, 3], 6, 2, 4, 8),
    ([7], 2, 2, 6, 2),
])
def test_decode_matches_brute_force_on_contiguous_cache(lengths, Hq, Hkv, d, bs):
    q, kc, vc, tables, ctx, K_log, V_log = _contiguous_case(21, lengths, Hq, Hkv, d, bs)
    scale = 0.37
    out = oracle.paged_decode(q, kc, vc, tables, ctx, scale, bs, F16, F16)
    G = Hq // Hkv
    for i in range(len(lengths)):
        for h in range(Hq):
            # the contiguous cache of vLLM의 핵심 이해 section 2: rows 0..n-1 of this sequence
            K = _f(K_log[i][:, h // G]).tolist()
            V = _f(V_log[i][:, h // G]).tolist()
            want = _brute_force_decode(_f(q[i, h]).tolist(), K, V, scale)
            np.testing.assert_allclose(out[i, h], want, rtol=1e-12, atol=1e-12)


def test_decode_matches_torch_sdpa_float64():
    case = workloads.paged_case(31, [1, 16, 17, 100, 257], 8, 2, 32, 16, BF16)
    out = oracle.paged_decode(case.q, case.k_cache, case.v_cache, case.block_tables,
                              case.context_lens, case.scale, 16, BF16, BF16)
    qf = _torch_widen(case.q, BF16)
    G = 4
    for i, n in enumerate(case.context_lens):
        n = int(n)
        nb = -(-n // 16)
        ids = case.block_tables[i, :nb]
        # [Hkv, nb*bs, d] -> library attention with grouped heads
        # inputs widened by torch itself, so this pin does not lean on bits_to_f64
        K = torch.from_numpy(_torch_widen(case.k_cache[ids], BF16)).permute(1, 0, 2, 3).reshape(2, -1, 32)[:, :n]
        V = torch.from_numpy(_torch_widen(case.v_cache[ids], BF16)).permute(1, 0, 2, 3).reshape(2, -1, 32)[:, :n]
        K = K.repeat_interleave(G, dim=0)
        V = V.repeat_interleave(G, dim=0)
        Q = torch.from_numpy(qf[i]).unsqueeze(1)  # [Hq, 1, d]
        ref = torch.nn.functional.scaled_dot_product_attention(Q, K, V, scale=case.scale)
        np.testing.assert_allclose(out[i], ref[:, 0].numpy(), rtol=1e-11, atol=1e-12)


def test_decode_single_token_returns_its_value():
    case = workloads.paged_case(41, [1, 1, 1], 4, 4, 16, 8, F16)
    out = oracle.paged_decode(case.q, case.k_cache, case.v_cache, case.block_tables,
                              case.context_lens, case.scale, 8, F16, F16)
    for i in range(3):
        blk = case.block_tables[i, 0]
        assert np.array_equal(out[i], _f(case.v_cache[blk, :, 0]))


def test_decode_zero_query_or_equal_keys_average_values():
    case = workloads.paged_case(42, [37, 5], 4, 2, 16, 16, F16)
    q0 = np.zeros_like(case.q)
    out = oracle.paged_decode(q0, case.k_cache, case.v_cache, case.block_tables,
                              case.context_lens, case.scale, 16, F16, F16)
    for i, n in enumerate(case.context_lens):
        for h in range(4):
            V = oracle.gather_sequence(case.v_cache, case.block_tables[i], int(n), 16, h // 2, F16)
            np.testing.assert_allclose(out[i, h], V.mean(axis=0), rtol=1e-13, atol=1e-14)
    # every key of sequence 0 equal (one row copied into all its slots)
    kc = case.k_cache.copy()
    row = kc[case.block_tables[0, 0], :, 0:1, :].copy()
    for j in range(3):
        kc[case.block_tables[0, j]] = row
    out = oracle.paged_decode(case.q, kc, case.v_cache, case.block_tables,
                              case.context_lens, case.scale, 16, F16, F16)
    V = oracle.gather_sequence(case.v_cache, case.block_tables[0], 37, 16, 0, F16)
    np.testing.assert_allclose(out[0, 0], V.mean(axis=0), rtol=1e-13, atol=1e-14)


def test_decode_empty_sequence_gives_zeros():
    case = workloads.paged_case(43, [0, 3], 2, 1, 8, 4, F16)
    out = oracle.paged_decode(case.q, case.k_cache, case.v_cache, case.block_tables,
                              case.context_lens, case.scale, 4, F16, F16)
    assert np.all(out[0] == 0)
    assert np.all(np.isfinite(out[1]))


def test_decode_is_invariant_under_physical_permutation():
    """Where a block lives does not matter, only what the table says."""
    case = workloads.paged_case(44, [30, 64, 9], 4, 2, 16, 8, F16)
    out = oracle.paged_decode(case.q, case.k_cache, case.v_cache, case.block_tables,
                              case.context_lens, case.scale, 8, F16, F16)
    rng = np.random.default_rng(0)
    Nb2 = case.num_blocks + 17
    new_id = rng.permutation(Nb2)[:case.num_blocks]
    kc = np.full((Nb2,) + case.k_cache.shape[1:], 0x7E00, dtype=np.uint16)
    vc = kc.copy()
    kc[new_id] = case.k_cache
    vc[new_id] = case.v_cache
    tables = new_id[case.block_tables].astype(np.int32)
    out2 = oracle.paged_decode(case.q, kc, vc, tables, case.context_lens, case.scale, 8, F16, F16)
    assert np.array_equal(out, out2)


def test_decode_shared_prefix_equals_private_copies():
    case = workloads.shared_prefix(seed=5, num_seqs=3, prefix_len=40, suffix_lo=3, suffix_hi=20,
                                   num_heads=4, num_kv_heads=2, head_dim=8, block_size=16)
    kc, vc = case.k_cache.copy(), case.v_cache.copy()
    oracle.copy_blocks([kc], [vc], case.cow_pairs)
    oracle.reshape_and_cache(case.new_key, case.new_value, kc, vc, case.slot_mapping, 16, F16, F16)
    out_shared = oracle.paged_decode(case.q, kc, vc, case.block_tables, case.context_lens,
                                     case.scale, 16, F16, F16)
    # give every sequence private copies of the shared prefix blocks
    tables = case.block_tables.copy()
    extra = []
    for i in range(3):
        for j, b in enumerate(case.meta["shared_blocks"][:-1]):
            extra.append((int(b), i, j))
    Nb2 = kc.shape[0] + len(extra)
    kc2 = np.concatenate([kc, np.zeros((len(extra),) + kc.shape[1:], np.uint16)])
    vc2 = np.concatenate([vc, np.zeros((len(extra),) + vc.shape[1:], np.uint16)])
    for n, (b, i, j) in enumerate(extra):
        kc2[kc.shape[0] + n] = kc[b]
        vc2[kc.shape[0] + n] = vc[b]
        tables[i, j] = kc.shape[0] + n
    assert Nb2 == kc2.shape[0]
    out_private = oracle.paged_decode(case.q, kc2, vc2, tables, case.context_lens,
                                      case.scale, 16, F16, F16)
    assert np.array_equal(out_shared, out_private)


def test_shared_prefix_copy_on_write_isolates_writers():
    """Writing through one table never changes what another table reads."""
    case = workloads.shared_prefix(seed=6, num_seqs=2, prefix_len=24, suffix_lo=4, suffix_hi=4,
                                   num_heads=2, num_kv_heads=1, head_dim=4, block_size=16)
    kc, vc = case.k_cache.copy(), case.v_cache.copy()
    shared_last = int(case.cow_pairs[0, 0])
    before = kc[shared_last].copy()
    oracle.copy_blocks([kc], [vc], case.cow_pairs)
    oracle.reshape_and_cache(case.new_key, case.new_value, kc, vc, case.slot_mapping, 16, F16, F16)
    assert np.array_equal(kc[shared_last], before)
    for i in range(2):
        own = int(case.cow_pairs[i, 1])
        assert np.array_equal(kc[own, :, :8], before[:, :8])


def test_partitioned_merge_equals_direct():
    case = workloads.paged_case(45, [1, 511, 512, 513, 1500, 2049], 8, 2, 16, 16, BF16)
    direct = oracle.paged_decode(case.q, case.k_cache, case.v_cache, case.block_tables,
                                 case.context_lens, case.scale, 16, BF16, BF16)
    for P in (16, 64, 512):
        split = oracle.paged_decode_partitioned(case.q, case.k_cache, case.v_cache,
                                                case.block_tables, case.context_lens,
                                                case.scale, 16, BF16, BF16, P)
        np.testing.assert_allclose(split, direct, rtol=1e-12, atol=1e-13)


def test_fp8_decode_uses_dequantised_values():
    case = workloads.fp8_layer(46, [3, 20, 33], num_heads=4, num_kv_heads=2, head_dim=16,
                               block_size=8)
    kc, vc = case.k_cache.copy(), case.v_cache.copy()
    oracle.reshape_and_cache(case.new_key, case.new_value, kc, vc, case.slot_mapping, 8,
                             BF16, FP8_E4M3, case.k_scale, case.v_scale)
    out = oracle.paged_decode(case.q, kc, vc, case.block_tables, case.context_lens,
                              case.scale, 8, BF16, FP8_E4M3, case.k_scale, case.v_scale)
    qf = _f(case.q, BF16)
    t0 = 0
    for i, n in enumerate(case.context_lens):
        n = int(n)
        for h in range(4):
            g = h // 2
            K, V = [], []
            for p in range(n):
                b = int(case.block_tables[i, p // 8])
                K.append(oracle.e4m3_decode(kc[b, g, p % 8]) * float(case.k_scale[b, g]))
                V.append(oracle.e4m3_decode(vc[b, g, p % 8]) * float(case.v_scale[b, g]))
            want = _brute_force_decode(qf[i, h].tolist(), K, V, case.scale)
            np.testing.assert_allclose(out[i, h], want, rtol=1e-12, atol=1e-12)
        # a stored value is off by at most half an E4M3 step: 2^-4 relative in
        # the normal range, 2^-10 (times the scale) among the subnormals
        for p in range(n):
            b = int(case.block_tables[i, p // 8])
            src = _f(case.new_key[t0 + p, 0], BF16)
            got = oracle.e4m3_decode(kc[b, 0, p % 8]) * float(case.k_scale[b, 0])
            bound = np.abs(src) / 16 + 2.0 ** -10 * float(case.k_scale[b, 0])
            assert np.all(np.abs(got - src) <= bound * (1 + 1e-6))
        t0 += n


# ----------------------------------------------------------------------------
# planted mistakes: each pin above must catch a plausible slip in the oracle


def test_planted_mistakes_are_caught(monkeypatch):
    q, kc, vc, tables, ctx, K_log, V_log = _contiguous_case(22, [19, 6], 4, 2, 4, 4)
    scale = 0.5

    def max_err():
        out = oracle.paged_decode(q, kc, vc, tables, ctx, scale, 4, F16, F16)
        err = 0.0
        for i in range(2):
            for h in range(4):
                want = _brute_force_decode(_f(q[i, h]).tolist(), _f(K_log[i][:, h // 2]).tolist(),
                                           _f(V_log[i][:, h // 2]).tolist(), scale)
                e = float(np.max(np.abs(out[i, h] - want)))
                err = float("inf") if math.isnan(e) else max(err, e)
        return err

    assert max_err() < 1e-12
    real_gather = oracle.paged_attention.gather_sequence
    mistakes = {
        "skips the first logical block": lambda c, t, n, bs, g, dt, s=None: real_gather(c, t[1:], n, bs, g, dt, s),
        "reads one slot past the context": lambda c, t, n, bs, g, dt, s=None: real_gather(c, t, n + 1, bs, g, dt, s),
        "drops the last token": lambda c, t, n, bs, g, dt, s=None: real_gather(c, t, n - 1, bs, g, dt, s),
        "wrong KV head": lambda c, t, n, bs, g, dt, s=None: real_gather(c, t, n, bs, 1 - g, dt, s),
        "transposed block": lambda c, t, n, bs, g, dt, s=None: real_gather(c.swapaxes(2, 3).copy(), t, n, bs, g, dt, s) if c.shape[2] == c.shape[3] else real_gather(c, t, n, bs, g, dt, s)[:, ::-1],
    }
    for name, fn in mistakes.items():
        monkeypatch.setattr(oracle.paged_attention, "gather_sequence", fn)
        try:
            err = max_err()
        except Exception:
            err = float("inf")
        assert not err < 1e-6, name
        monkeypatch.setattr(oracle.paged_attention, "gather_sequence", real_gather)


# ----------------------------------------------------------------------------
# prefill


def test_prefill_without_prefix_is_causal_sdpa():
    """With no cached prefix the chunk is the whole sequence: torch's causal
    scaled_dot_product_attention (float64) over the gathered K/V."""
    case = workloads.prefill_case(51, [0, 0, 0], [1, 17, 40], 8, 2, 16, 16, BF16)
    out = oracle.paged_prefill(case.q, case.k_cache, case.v_cache, case.block_tables, case.context_lens,
                               case.query_start, case.scale, 16, BF16, BF16)
    qf = _f(case.q, BF16)
    for i, n in enumerate(case.context_lens):
        n = int(n)
        nb = -(-n // 16)
        ids = case.block_tables[i, :nb]
        K = torch.from_numpy(_f(case.k_cache[ids], BF16)).permute(1, 0, 2, 3).reshape(2, -1, 16)[:, :n]
        V = torch.from_numpy(_f(case.v_cache[ids], BF16)).permute(1, 0, 2, 3).reshape(2, -1, 16)[:, :n]
        K, V = K.repeat_interleave(4, dim=0), V.repeat_interleave(4, dim=0)
        q0 = int(case.query_start[i])
        Q = torch.from_numpy(qf[q0:q0 + n]).permute(1, 0, 2)  # [Hq, n, d]
        ref = torch.nn.functional.scaled_dot_product_attention(Q, K, V, is_causal=True, scale=case.scale)
        np.testing.assert_allclose(out[q0:q0 + n], ref.permute(1, 0, 2).numpy(), rtol=1e-11, atol=1e-12)


def test_prefill_query_equals_decode_over_its_prefix():
    """Query j of a chunk after a cached prefix sees exactly the first
    ctx - n + j + 1 tokens: it equals a single-query decode over a context cut
    to that length."""
    case = workloads.prefill_case(52, [0, 5, 16, 33], [3, 12, 1, 20], 4, 2, 8, 8, F16)
    out = oracle.paged_prefill(case.q, case.k_cache, case.v_cache, case.block_tables, case.context_lens,
                               case.query_start, case.scale, 8, F16, F16)
    for i in range(case.num_seqs):
        q0, q1 = int(case.query_start[i]), int(case.query_start[i + 1])
        n, ctx = q1 - q0, int(case.context_lens[i])
        for j in range(n):
            dec = oracle.paged_decode(case.q[q0 + j:q0 + j + 1], case.k_cache, case.v_cache,
                                      case.block_tables[i:i + 1], np.array([ctx - n + j + 1], np.int32),
                                      case.scale, 8, F16, F16)
            np.testing.assert_allclose(out[q0 + j], dec[0], rtol=1e-12, atol=1e-13)


def test_prefill_brute_force_loops():
    case = workloads.prefill_case(53, [2, 9], [4, 3], 2, 1, 4, 4, F16)
    out = oracle.paged_prefill(case.q, case.k_cache, case.v_cache, case.block_tables, case.context_lens,
                               case.query_start, case.scale, 4, F16, F16)
    for i in range(2):
        ctx = int(case.context_lens[i])
        rows = [(int(case.block_tables[i, p // 4]), p % 4) for p in range(ctx)]
        q0, q1 = int(case.query_start[i]), int(case.query_start[i + 1])
        for j in range(q1 - q0):
            last = ctx - (q1 - q0) + j
            for h in range(2):
                qv = list(_f(case.q[q0 + j, h], F16))
                K = [list(_f(case.k_cache[b, 0, o], F16)) for b, o in rows[:last + 1]]
                V = [list(_f(case.v_cache[b, 0, o], F16)) for b, o in rows[:last + 1]]
                ref = _brute_force_decode(qv, K, V, case.scale)
                np.testing.assert_allclose(out[q0 + j, h], ref, rtol=1e-12, atol=1e-14)
