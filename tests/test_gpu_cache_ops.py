"""GPU parity of the cache writes: slot scatter and block copy, bit for bit."""

import numpy as np
import pytest
import torch

import oracle
import workloads
from workloads import F16, BF16, FP8_E4M3
from gpu_helpers import DeviceCase, dev, host_bits

pytestmark = pytest.mark.gpu

import paged_kv_cache_288_gb300 as pa  # noqa: E402


def _random_pool(seed, Nb, Hkv, bs, d, dtype):
    g = torch.Generator().manual_seed(seed)
    if dtype == FP8_E4M3:
        return torch.randint(0, 256, (Nb, Hkv, bs, d), generator=g, dtype=torch.int32).numpy().astype(np.uint8)
    return workloads.normal_bits(g, (Nb, Hkv, bs, d), dtype)


@pytest.mark.parametrize("dtype", [F16, BF16])
@pytest.mark.parametrize("Hkv,d,bs", [(2, 64, 16), (8, 128, 16), (1, 256, 8), (4, 128, 64)])
def test_reshape_and_cache_16bit_bit_exact(dtype, Hkv, d, bs):
    Nb, T = 37, 50
    g = torch.Generator().manual_seed(Hkv * 1000 + d + bs)
    kc = _random_pool(1, Nb, Hkv, bs, d, dtype)
    vc = _random_pool(2, Nb, Hkv, bs, d, dtype)
    key = workloads.normal_bits(g, (T, Hkv, d), dtype)
    value = workloads.normal_bits(g, (T, Hkv, d), dtype)
    slots = torch.randperm(Nb * bs, generator=g)[:T].numpy().astype(np.int64)
    slots[::7] = -1  # padding tokens
    k_d, v_d = dev(kc, dtype), dev(vc, dtype)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    pa.reshape_and_cache(dev(key, dtype), dev(value, dtype), k_d, v_d,
                         torch.from_numpy(slots).cuda(), debug_err=err)
    oracle.reshape_and_cache(key, value, kc, vc, slots, bs, dtype, dtype)
    torch.cuda.synchronize()
    assert np.array_equal(host_bits(k_d), kc)
    assert np.array_equal(host_bits(v_d), vc)
    assert err.item() == 0


@pytest.mark.parametrize("src", [F16, BF16])
@pytest.mark.parametrize("bs", [8, 16, 32])
def test_reshape_and_cache_fp8_bit_exact(src, bs):
    ctx = [1, 15, 16, 17, 100, 333]
    case = workloads.fp8_layer(77 + bs, ctx, num_heads=8, num_kv_heads=4, head_dim=128,
                               block_size=bs, src_dtype=src)
    dc = DeviceCase(case)
    pa.reshape_and_cache(dc.new_key, dc.new_value, dc.k_cache, dc.v_cache, dc.slot_mapping,
                         k_scale=dc.k_scale, v_scale=dc.v_scale, debug_err=dc.debug_err)
    kc, vc = case.k_cache.copy(), case.v_cache.copy()
    oracle.reshape_and_cache(case.new_key, case.new_value, kc, vc, case.slot_mapping, bs, src,
                             FP8_E4M3, case.k_scale, case.v_scale)
    torch.cuda.synchronize()
    assert np.array_equal(host_bits(dc.k_cache), kc)
    assert np.array_equal(host_bits(dc.v_cache), vc)
    assert dc.debug_err.item() == 0


def test_reshape_and_cache_fp8_ties_saturation_and_signed_zero():
    """Values at exact E4M3 midpoints, beyond 448, and tiny negatives."""
    src = BF16
    codes = np.arange(0, 0x7E)
    vals = np.sort(oracle.e4m3_decode(codes))
    mids = (vals[:-1] + vals[1:]) / 2
    special = np.array([448.0, 464.0, 480.0, 1e4, -1e4, -1e-6, 1e-6, 0.0, -0.0,
                        2.0 ** -10, -(2.0 ** -10), 3 * 2.0 ** -11])
    x = np.concatenate([mids, -mids, special]).astype(np.float32)
    # bf16 must hold them exactly: keep those that survive the rounding to bf16
    xb = torch.from_numpy(x).to(torch.bfloat16)
    keep = xb.float().numpy() == x
    x = x[keep]
    n = (len(x) + 127) // 128 * 128
    x = np.concatenate([x, np.zeros(n - len(x), np.float32)])
    T = n // 128
    key = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16).reshape(T, 1, 128)
    bs = 8
    Nb = (T + bs - 1) // bs
    kc = np.zeros((Nb, 1, bs, 128), np.uint8)
    vc = kc.copy()
    scale = np.ones((Nb, 1), np.float32)
    scale[0, 0] = 0.5  # an exact power of two keeps the midpoints exact
    slots = np.arange(T, dtype=np.int64)
    k_d, v_d = dev(kc, FP8_E4M3), dev(vc, FP8_E4M3)
    pa.reshape_and_cache(dev(key, src), dev(key, src), k_d, v_d, torch.from_numpy(slots).cuda(),
                         k_scale=torch.from_numpy(scale).cuda(), v_scale=torch.from_numpy(scale).cuda())
    oracle.reshape_and_cache(key, key, kc, vc, slots, bs, src, FP8_E4M3, scale, scale)
    torch.cuda.synchronize()
    got = host_bits(k_d)
    assert np.array_equal(got, kc), np.argwhere(got != kc)[:5]


def test_reshape_and_cache_rejects_out_of_range_slots():
    Nb, Hkv, bs, d = 4, 2, 16, 64
    kc = _random_pool(3, Nb, Hkv, bs, d, F16)
    g = torch.Generator().manual_seed(9)
    key = workloads.normal_bits(g, (3, Hkv, d), F16)
    slots = np.array([Nb * bs, 5, 10 ** 12], dtype=np.int64)
    k_d, v_d = dev(kc, F16), dev(kc, F16)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    pa.reshape_and_cache(dev(key, F16), dev(key, F16), k_d, v_d, torch.from_numpy(slots).cuda(),
                         debug_err=err)
    want = kc.copy()
    oracle.reshape_and_cache(key[1:2], key[1:2], want, want.copy(), slots[1:2], bs, F16, F16)
    torch.cuda.synchronize()
    assert err.item() & pa.DEVERR_SLOT_RANGE
    assert np.array_equal(host_bits(k_d), want)


@pytest.mark.parametrize("dtype", [F16, FP8_E4M3])
def test_copy_blocks_bit_exact_all_layers(dtype):
    L, Nb, Hkv, bs, d = 3, 20, 8, 16, 128
    ks = [_random_pool(10 + i, Nb, Hkv, bs, d, dtype) for i in range(L)]
    vs = [_random_pool(20 + i, Nb, Hkv, bs, d, dtype) for i in range(L)]
    kd = [dev(k, dtype) for k in ks]
    vd = [dev(v, dtype) for v in vs]
    pairs = np.array([[3, 7], [3, 8], [11, 0], [19, 1]], dtype=np.int64)
    block_bytes = Hkv * bs * d * (1 if dtype == FP8_E4M3 else 2)
    pa.copy_blocks(pa.pointer_array(kd, "cuda"), pa.pointer_array(vd, "cuda"),
                   torch.from_numpy(pairs).cuda(), Nb, block_bytes)
    oracle.copy_blocks(ks, vs, pairs)
    torch.cuda.synchronize()
    for i in range(L):
        assert np.array_equal(host_bits(kd[i]), ks[i])
        assert np.array_equal(host_bits(vd[i]), vs[i])


def test_copy_blocks_flags_out_of_range_pairs():
    Nb, Hkv, bs, d = 6, 2, 8, 64
    k = _random_pool(30, Nb, Hkv, bs, d, BF16)
    kd, vd = dev(k, BF16), dev(k, BF16)
    pairs = np.array([[0, 6], [-1, 2], [1, 2]], dtype=np.int64)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    pa.copy_blocks(pa.pointer_array([kd], "cuda"), pa.pointer_array([vd], "cuda"),
                   torch.from_numpy(pairs).cuda(), Nb, Hkv * bs * d * 2, debug_err=err)
    want = k.copy()
    want[2] = k[1]
    torch.cuda.synchronize()
    assert err.item() & pa.DEVERR_BLOCK_RANGE
    assert np.array_equal(host_bits(kd), want)


# ----------------------------------------------------------------------------
# swap to and from pinned host memory


def _pinned(bits, dtype):
    """Raw-bit numpy array -> pinned host tensor of the storage dtype."""
    return dev(bits, dtype, device="cpu").pin_memory()


@pytest.mark.parametrize("dtype,L", [(BF16, 1), (F16, 3), (FP8_E4M3, 2)])
@pytest.mark.parametrize("map_on_host", [False, True])
def test_swap_out_then_in_bit_exact(dtype, L, map_on_host):
    """A preempted request's blocks go to a pinned host pool and come back into
    other device blocks; every byte of both pools matches the oracle."""
    Nd, Nh, Hkv, bs, d = 24, 10, 8, 16, 128
    dk = [_random_pool(40 + i, Nd, Hkv, bs, d, dtype) for i in range(L)]
    dv = [_random_pool(50 + i, Nd, Hkv, bs, d, dtype) for i in range(L)]
    hk = [_random_pool(60 + i, Nh, Hkv, bs, d, dtype) for i in range(L)]
    hv = [_random_pool(70 + i, Nh, Hkv, bs, d, dtype) for i in range(L)]
    dkt, dvt = [dev(x, dtype) for x in dk], [dev(x, dtype) for x in dv]
    hkt, hvt = [_pinned(x, dtype) for x in hk], [_pinned(x, dtype) for x in hv]

    def mapping(pairs):
        t = torch.from_numpy(np.array(pairs, dtype=np.int64).reshape(-1, 2))
        return t.pin_memory() if map_on_host else t.cuda()

    out_pairs = [[17, 0], [3, 9], [4, 5], [23, 2]]
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    m_out = mapping(out_pairs)
    pa.swap_blocks(hkt, hvt, dkt, dvt, m_out, debug_err=err)
    oracle.swap_blocks(hk, hv, dk, dv, out_pairs)
    torch.cuda.synchronize()
    for i in range(L):
        assert np.array_equal(host_bits(hkt[i]), hk[i])
        assert np.array_equal(host_bits(hvt[i]), hv[i])

    in_pairs = [[0, 1], [9, 20], [5, 17], [2, 3]]
    m_in = mapping(in_pairs)
    pa.swap_blocks(dkt, dvt, hkt, hvt, m_in, debug_err=err)
    oracle.swap_blocks(dk, dv, hk, hv, in_pairs)
    torch.cuda.synchronize()
    assert err.item() == 0
    for i in range(L):
        assert np.array_equal(host_bits(dkt[i]), dk[i])
        assert np.array_equal(host_bits(dvt[i]), dv[i])


def test_swap_flags_out_of_range_pairs():
    Nd, Nh, Hkv, bs, d = 6, 3, 2, 8, 64
    dk = _random_pool(80, Nd, Hkv, bs, d, BF16)
    hk = _random_pool(81, Nh, Hkv, bs, d, BF16)
    dkt, hkt, hvt = dev(dk, BF16), _pinned(hk, BF16), _pinned(hk, BF16)
    pairs = [[6, 0], [1, 3], [-1, 1], [2, 1]]
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    pa.swap_blocks([hkt], [hvt], [dkt], [dkt], torch.tensor(pairs, dtype=torch.int64).cuda(), debug_err=err)
    want = hk.copy()
    skipped = oracle.swap_blocks([want], [hk.copy()], [dk], [dk], pairs)
    torch.cuda.synchronize()
    assert skipped == [(6, 0), (1, 3), (-1, 1)]
    assert err.item() & pa.DEVERR_BLOCK_RANGE
    assert np.array_equal(host_bits(hkt), want)


def test_swap_refuses_pageable_host_memory():
    """Host memory the device cannot address is refused before any launch."""
    dk = _random_pool(82, 4, 2, 8, 64, BF16)
    dkt = dev(dk, BF16)
    pageable = dev(dk, BF16, device="cpu")
    assert not pageable.is_pinned()
    n0 = pa.lib().pa_kernel_launch_count()
    with pytest.raises(pa.PaError) as e:
        pa.swap_blocks([pageable], [pageable], [dkt], [dkt], torch.tensor([[0, 1]], dtype=torch.int64).cuda())
    assert e.value.status == 1
    with pytest.raises(pa.PaError):
        pa.swap_blocks([dkt], [dkt], [dkt], [dkt], torch.tensor([[0, 1]], dtype=torch.int64))
    assert pa.lib().pa_kernel_launch_count() == n0


def test_swap_all_layers_at_the_limit():
    L, Nd, Nh, Hkv, bs, d = pa.SWAP_MAX_LAYERS, 3, 2, 1, 8, 64
    dk = [_random_pool(100 + i, Nd, Hkv, bs, d, F16) for i in range(L)]
    hk = [_random_pool(200 + i, Nh, Hkv, bs, d, F16) for i in range(L)]
    dkt = [dev(x, F16) for x in dk]
    hkt = [_pinned(x, F16) for x in hk]
    pairs = [[2, 1], [0, 0]]
    pa.swap_blocks(hkt, hkt, dkt, dkt, torch.tensor(pairs, dtype=torch.int64).cuda())
    oracle.swap_blocks(hk, hk, dk, dk, pairs)
    torch.cuda.synchronize()
    for i in range(L):
        assert np.array_equal(host_bits(hkt[i]), hk[i])
    with pytest.raises(pa.PaError) as e:
        pa.swap_blocks(hkt + hkt[:1], hkt + hkt[:1], dkt + dkt[:1], dkt + dkt[:1],
                       torch.tensor(pairs, dtype=torch.int64).cuda())
    assert e.value.status == 2
