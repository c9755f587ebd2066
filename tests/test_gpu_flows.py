"""GPU parity of the sharing flows the host pool drives: fork for beam search
(table copy + reference counts, copy-on-write when a beam writes into a
shared block) and prefix caching (full blocks of a common prompt found by
their chained keys and shared). Each step runs the library's kernels on the
device and the oracle on host copies of the same pools, through the same
tables."""

import numpy as np
import pytest
import torch

import oracle
import workloads
from workloads import BF16, F16
from gpu_helpers import assert_close, dev, host_bits

pytestmark = pytest.mark.gpu

import paged_kv_cache_288_gb300 as pa  # noqa: E402
from paged_kv_cache_288_gb300 import BlockPool, PrefixCache  # noqa: E402


class Pools:
    """One layer's K/V pools on the device and as host oracle copies."""

    def __init__(self, seed, Nb, Hkv, bs, d, dtype):
        g = torch.Generator().manual_seed(seed)
        self.kc = workloads.normal_bits(g, (Nb, Hkv, bs, d), dtype)
        self.vc = workloads.normal_bits(g, (Nb, Hkv, bs, d), dtype)
        self.kd, self.vd = dev(self.kc, dtype), dev(self.vc, dtype)
        self.dtype, self.bs, self.Nb = dtype, bs, Nb
        self.block_bytes = Hkv * bs * d * 2
        self.err = torch.zeros(1, dtype=torch.int32, device="cuda")

    def copy(self, pairs):
        if not pairs:
            return
        m = torch.tensor(pairs, dtype=torch.int64).cuda()
        pa.copy_blocks(pa.pointer_array([self.kd], "cuda"), pa.pointer_array([self.vd], "cuda"), m,
                       self.Nb, self.block_bytes, debug_err=self.err)
        oracle.copy_blocks([self.kc], [self.vc], pairs)

    def write(self, key, value, slots):
        s = np.asarray(slots, dtype=np.int64)
        pa.reshape_and_cache(dev(key, self.dtype), dev(value, self.dtype), self.kd, self.vd,
                             torch.from_numpy(s).cuda(), debug_err=self.err)
        oracle.reshape_and_cache(key, value, self.kc, self.vc, s, self.bs, self.dtype, self.dtype)

    def decode(self, q, tables, lens, scale):
        B, Hq, d = q.shape
        out = torch.empty(B, Hq, d, dtype=dev(q, self.dtype).dtype, device="cuda")
        mx = int(lens.max())
        ws = torch.empty(max(1, pa.decode_workspace_size(B, Hq, self.kd.shape[1], d, mx, 0)),
                         dtype=torch.uint8, device="cuda")
        pa.decode(out, dev(q, self.dtype), self.kd, self.vd, torch.from_numpy(tables).cuda(),
                  torch.from_numpy(lens).cuda(), scale, mx, workspace=ws, debug_err=self.err)
        ref = oracle.paged_decode(q, self.kc, self.vc, tables, lens, scale, self.bs, self.dtype,
                                  self.dtype)
        return out, ref

    def check_pools(self):
        torch.cuda.synchronize()
        assert np.array_equal(host_bits(self.kd), self.kc)
        assert np.array_equal(host_bits(self.vd), self.vc)
        assert self.err.item() == 0


@pytest.mark.parametrize("dtype,bs", [(BF16, 16), (F16, 8)])
def test_beam_search_fork_and_copy_on_write(dtype, bs):
    """A prompt forks into 4 beams; each step every beam appends a token
    (copying its shared last block first), all beams decode, the worst beam is
    dropped and the best is forked in its place."""
    Hq, Hkv, d, Nb = 8, 2, 64, 160
    rng = np.random.default_rng(11)
    g = torch.Generator().manual_seed(12)
    P = Pools(13, Nb, Hkv, bs, d, dtype)
    pool = BlockPool(Nb, bs)
    prompt = 3 * bs + 5
    slots = pool.add_sequence("root", prompt)
    P.write(workloads.normal_bits(g, (prompt, Hkv, d), dtype),
            workloads.normal_bits(g, (prompt, Hkv, d), dtype), slots)
    beams = [f"b{i}" for i in range(4)]
    for b in beams:
        pool.fork("root", b)
    pool.free_sequence("root")
    root_blocks = list(pool.tables["b0"])
    before = P.kc[root_blocks].copy()
    n_copies = 0
    for step in range(6):
        for b in beams:
            s, cow = pool.append(b, 1)
            P.copy(cow)
            n_copies += len(cow)
            P.write(workloads.normal_bits(g, (1, Hkv, d), dtype),
                    workloads.normal_bits(g, (1, Hkv, d), dtype), s)
        tables = pool.block_table_array(beams, width=16, pad=0)
        lens = pool.context_lens(beams)
        q = workloads.normal_bits(g, (4, Hq, d), dtype)
        out, ref = P.decode(q, tables, lens, 1.0 / np.sqrt(d))
        torch.cuda.synchronize()
        assert_close(out, ref, dtype, dtype, f"beam step {step}")
        worst, best = beams[rng.integers(4)], beams[rng.integers(4)]
        if worst != best:
            pool.free_sequence(worst)
            pool.fork(best, worst)
    P.check_pools()
    assert n_copies >= 4
    # the full prompt blocks every beam still shares were never written
    full = prompt // bs
    assert np.array_equal(P.kc[root_blocks[:full]], before[:full])


def _prefix_kv(tokens, Hkv, d, dtype):
    """K/V of each token as a function of the token ids up to and including it,
    so that equal prefixes have equal K/V (as a model's would)."""
    k = np.empty((len(tokens), Hkv, d), dtype=np.uint16)
    v = np.empty_like(k)
    for i in range(len(tokens)):
        seed = int.from_bytes(pa.block_key(b"", tokens[:i + 1])[:8], "little") & 0x7FFFFFFF
        g = torch.Generator().manual_seed(seed)
        k[i] = workloads.normal_bits(g, (Hkv, d), dtype)
        v[i] = workloads.normal_bits(g, (Hkv, d), dtype)
    return k, v


def test_prefix_cache_sharing_matches_private_copies():
    """Requests whose prompts share a prefix read its full blocks from the
    blocks the first request filled; their outputs equal attention over
    private contiguous copies of their own K/V."""
    dtype, bs, Hq, Hkv, d, Nb = BF16, 16, 8, 2, 64, 96
    rng = np.random.default_rng(21)
    system = rng.integers(0, 32000, 70)
    prompts = [np.concatenate([system, rng.integers(0, 32000, n)]) for n in (9, 30, 0, 51)]
    P = Pools(22, Nb, Hkv, bs, d, dtype)
    pool = BlockPool(Nb, bs)
    cache = PrefixCache(pool)
    kv = []
    for i, t in enumerate(prompts):
        k, v = _prefix_kv(t, Hkv, d, dtype)
        kv.append((k, v))
        cached, slots = cache.add_sequence(i, t)
        assert cached == (0 if i == 0 else (70 // bs) * bs)
        P.write(k[cached:], v[cached:], slots)
    ids = list(range(len(prompts)))
    tables = pool.block_table_array(ids, width=8, pad=0)
    assert all((tables[i, :4] == tables[0, :4]).all() for i in ids)
    lens = pool.context_lens(ids)
    g = torch.Generator().manual_seed(23)
    q = workloads.normal_bits(g, (len(ids), Hq, d), dtype)
    out, ref = P.decode(q, tables, lens, 0.125)
    # the same attention over private contiguous copies of each request's K/V
    for i in ids:
        k, v = kv[i]
        n = len(prompts[i])
        nbk = -(-n // bs)
        kc = np.zeros((nbk, Hkv, bs, d), dtype=np.uint16)
        vc = np.zeros_like(kc)
        for t in range(n):
            kc[t // bs, :, t % bs] = k[t]
            vc[t // bs, :, t % bs] = v[t]
        own = oracle.paged_decode(q[i:i + 1], kc, vc, np.arange(nbk, dtype=np.int32)[None],
                                  np.array([n], dtype=np.int32), 0.125, bs, dtype, dtype)
        assert np.allclose(own[0], ref[i], rtol=0, atol=1e-12)
    torch.cuda.synchronize()
    assert_close(out, ref, dtype, dtype, "prefix-cache decode")
    # the sharing the prefix cache set up, found from the tables, read once:
    # one group of the four requests over the 4 whole blocks of the prompt
    from paged_kv_cache_288_gb300.block_pool import shared_prefix_groups
    gs, gp = shared_prefix_groups(tables, lens, bs)
    assert gs.tolist() == [0, 4] and gp.tolist() == [64]
    B, mx = len(ids), int(lens.max())
    n = pa.decode_shared_prefix_workspace_size(B, Hq, Hkv, d, bs, len(gp), 4, int(gp.max()))
    ws = torch.empty(n, dtype=torch.uint8, device="cuda")
    grouped = torch.full((B, Hq, d), float("nan"), dtype=torch.bfloat16, device="cuda")
    pa.decode_shared_prefix(grouped, dev(q, dtype), P.kd, P.vd, torch.from_numpy(tables).cuda(),
                            torch.from_numpy(lens).cuda(), 0.125, mx, torch.from_numpy(gs).cuda(),
                            torch.from_numpy(gp).cuda(), 4, int(gp.max()), ws, debug_err=P.err)
    torch.cuda.synchronize()
    assert_close(grouped, ref, dtype, dtype, "prefix-cache decode, shared blocks read once")
    P.check_pools()
