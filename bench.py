"""Benchmark of the paged-KV decode step on GB300.

One step is the whole hot path over one batch: the new token of every
sequence is written into the paged cache (pa_reshape_and_cache), then every
sequence's query attends over its paged KV (pa_decode). The default workload
is the Llama-8B-shaped batch: 64 sequences, 32 query / 8 KV heads, head dim
128, bf16, 16-token blocks, context lengths uniform in [128, 4096], blocks
shuffled over a pool 1.25x the need. Other workloads (--workload) are the
shared-prefix, long-context and fp8 cases.

Prints one JSON line (rank 0). ``value`` is whole-job KV GB/s: algorithmic
bytes of all ranks' steps / max-over-ranks time, where the algorithmic bytes
of a step are the KV rows of real tokens read by the decode, plus q, out,
block-table entries and context lengths, plus the new tokens read and written
by the cache write. Timing: CUDA events around every step on the launching
stream; between steps, outside the events, the L2 is flushed by writing a
256 MiB buffer and reading it back (so no dirty flush lines are written back
during a timed step).

``--impl reference`` times the fp64 CPU oracle on the same workload instead.
"""

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

import workloads  # noqa: E402

METRIC = "pa_decode KV GB/s and decode tokens/s per layer; % of GB300 HBM roofline"
L2_FLUSH_BYTES = 256 << 20
# DRAM bytes of one pa_decode call measured by ncu, valid while these
# sources are unchanged (their hash is stored beside the numbers)
TRAFFIC_PATH = os.path.join(ROOT, "profiles", "traffic.json")
TRAFFIC_SOURCES = ("paged_kv_cache_288_gb300/csrc/decode_tc.cu",
                   "paged_kv_cache_288_gb300/csrc/decode_prefix.cu",
                   "paged_kv_cache_288_gb300/csrc/decode_simt.cu",
                   "paged_kv_cache_288_gb300/csrc/ptx.cuh",
                   "paged_kv_cache_288_gb300/csrc/common.cuh")


def kernel_sources_hash():
    h = hashlib.sha256()
    for rel in TRAFFIC_SOURCES:
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()


def recorded_traffic(workload, partition_size):
    """ncu DRAM bytes (read + write) per pa_decode call, or None when no capture
    of the current kernel sources exists for this workload."""
    try:
        with open(TRAFFIC_PATH) as f:
            rec = json.load(f)
    except (OSError, ValueError):
        return None
    if rec.get("sources_sha256") != kernel_sources_hash():
        return None
    w = rec.get("workloads", {}).get(f"{workload}/p{partition_size}")
    return None if w is None else int(w["bytes_per_call"])


# ----------------------------------------------------------------------------
# workloads and their algorithmic bytes


def rank_seed(base, rank):
    """Each rank runs its own replica batch of the same shape."""
    return base + 10007 * rank


def make_case(name, rank):
    if name == "tiny":
        # the pool before the append, with the appended token of each
        # sequence as the step's cache write and the lengths after it
        before, step = workloads.tiny()
        return workloads.DecodeCase(**{**step.__dict__, "k_cache": before.k_cache,
                                       "v_cache": before.v_cache})
    if name == "llama8b":
        return workloads.llama8b(seed=rank_seed(1002, rank))
    if name == "llama8b_mha":
        # the Llama-8B-shaped batch with one KV head per query head (MHA, group 1)
        ctx = workloads.llama8b_lengths(rank_seed(1002, rank))
        return workloads.paged_case(rank_seed(1102, rank), ctx, 32, 32, 128, 16, workloads.BF16,
                                    table_width=256, name="llama8b_mha", append=True)
    if name == "llama8b_mqa":
        # the same batch with one KV head shared by all 32 query heads (MQA)
        ctx = workloads.llama8b_lengths(rank_seed(1002, rank))
        return workloads.paged_case(rank_seed(1202, rank), ctx, 32, 1, 128, 16, workloads.BF16,
                                    table_width=256, name="llama8b_mqa", append=True)
    if name == "shared_prefix":
        return workloads.shared_prefix(seed=rank_seed(1003, rank))
    if name.startswith("long_context"):
        bs = int(name.split("bs")[-1]) if "bs" in name else 16
        return workloads.long_context(bs, seed=rank_seed(1004, rank))
    if name in ("fp8_layer", "fp8_step"):
        return workloads.fp8_step_layer(0, seed=rank_seed(1005, rank))
    if name == "prefix_cache":
        return prefix_cache_case(rank_seed(1007, rank))
    raise ValueError(name)


def prefix_cache_case(seed, num_seqs=100, prefix_len=1016, suffix_lo=32, suffix_hi=512,
                      num_heads=32, num_kv_heads=8, head_dim=128, block_size=16):
    """The shared-prefix shape with the sharing found by the prefix cache.

    num_seqs requests open with one prefix_len-token system prompt and go on
    with a private suffix of suffix_lo..suffix_hi tokens (token ids are seeded
    random). Each request is admitted through the prefix cache, which finds
    the system prompt's full blocks from the token ids; its last token is the
    one written and decoded in the timed step. Pool contents are random bf16,
    block ids shuffled; host admission time is kept in ``meta``.
    """
    from paged_kv_cache_288_gb300.block_pool import BlockPool, PrefixCache

    g = workloads._gen(seed)
    bs = block_size
    system = torch.randint(0, 32000, (prefix_len,), generator=g).numpy()
    suffix = torch.randint(suffix_lo, suffix_hi + 1, (num_seqs,), generator=g).numpy()
    prompts = [np.concatenate([system, torch.randint(0, 32000, (int(n),), generator=g).numpy()])
               for n in suffix]
    full = prefix_len // bs
    need = full + sum(-(-len(t) // bs) - full for t in prompts)
    num_blocks = int(math.ceil(1.25 * need)) + 1
    pool = BlockPool(num_blocks - 1, bs)
    cache = PrefixCache(pool)
    t0 = time.perf_counter()
    cached = [cache.add_sequence(i, t)[0] for i, t in enumerate(prompts)]
    host_s = time.perf_counter() - t0
    perm = torch.randperm(num_blocks, generator=g).numpy().astype(np.int32)
    poison = int(perm[-1])
    ctx = np.array([len(t) for t in prompts], dtype=np.int64)
    width = int(max(-(-c // bs) for c in ctx))
    tables = np.full((num_seqs, width), poison, dtype=np.int32)
    for i in range(num_seqs):
        tables[i, :len(pool.tables[i])] = perm[np.asarray(pool.tables[i])]
    dtype = workloads.BF16
    shape = (num_blocks, num_kv_heads, bs, head_dim)
    kc = workloads.normal_bits(g, shape, dtype)
    vc = workloads.normal_bits(g, shape, dtype)
    kc[poison] = workloads.NAN_BITS[dtype]
    vc[poison] = workloads.NAN_BITS[dtype]
    workloads._poison_tails(kc, tables, ctx, bs, dtype)
    workloads._poison_tails(vc, tables, ctx, bs, dtype)
    slots = np.array([int(tables[i, (c - 1) // bs]) * bs + (c - 1) % bs for i, c in enumerate(ctx)],
                     dtype=np.int64)
    return workloads.DecodeCase(
        name="prefix_cache", num_seqs=num_seqs, num_heads=num_heads, num_kv_heads=num_kv_heads,
        head_dim=head_dim, block_size=bs, num_blocks=num_blocks, q_dtype=dtype, kv_dtype=dtype,
        scale=1.0 / math.sqrt(head_dim), q=workloads.normal_bits(g, (num_seqs, num_heads, head_dim), dtype),
        k_cache=kc, v_cache=vc, block_tables=tables, context_lens=ctx.astype(np.int32),
        poison_block=poison, new_key=workloads.normal_bits(g, (num_seqs, num_kv_heads, head_dim), dtype),
        new_value=workloads.normal_bits(g, (num_seqs, num_kv_heads, head_dim), dtype),
        slot_mapping=slots, src_dtype=dtype,
        meta={"prefix_cache": {"requests": num_seqs, "cached_tokens": int(sum(cached)),
                               "hit_blocks": cache.hits, "miss_blocks": cache.misses,
                               "host_admission_us_per_request": round(1e6 * host_s / num_seqs, 1),
                               "blocks_in_use": pool.used_blocks(),
                               "blocks_without_sharing": int(sum(-(-c // bs) for c in ctx))}})


def job_throughput_gbs(bytes_per_step, steps, world, max_total_ms):
    """Whole-job GB/s: every rank's bytes over the slowest rank's time."""
    return world * bytes_per_step * steps / (max_total_ms / 1e3) / 1e9


def elem(dtype):
    return workloads.elem_bytes(dtype)


def decode_bytes(case):
    """Algorithmic bytes of one pa_decode: real KV rows, scales, q, out, tables, lengths."""
    ctx = case.context_lens.astype(np.int64)
    eb = elem(case.kv_dtype)
    kv = int(ctx.sum()) * case.num_kv_heads * 2 * case.head_dim * eb
    nblocks = int(sum(-(-int(c) // case.block_size) for c in ctx if c > 0))
    scales = nblocks * case.num_kv_heads * 2 * 4 if case.kv_dtype == workloads.FP8_E4M3 else 0
    qo = 2 * case.num_seqs * case.num_heads * case.head_dim * elem(case.q_dtype)
    return kv + scales + qo + nblocks * 4 + case.num_seqs * 4


def write_bytes(case):
    """Algorithmic bytes of one pa_reshape_and_cache: sources read, cache rows written, slots."""
    if case.new_key is None:
        return 0
    T = case.new_key.shape[0]
    src = 2 * T * case.num_kv_heads * case.head_dim * elem(case.src_dtype)
    dst = 2 * T * case.num_kv_heads * case.head_dim * elem(case.kv_dtype)
    return src + dst + 8 * T


# ----------------------------------------------------------------------------
# clocks


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons while the GPU works."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu_index = gpu_index
        self.lines = []
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100", "-i", str(self.gpu_index)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except OSError:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self, t0, t1):
        rows = [l for t, l in self.lines if t0 - 0.25 <= t <= t1 + 0.25] or [l for _, l in self.lines]
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            f = [x.strip() for x in r.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = float(f[2])
            except ValueError:
                continue
            for name, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


# ----------------------------------------------------------------------------
# the oracle on the host (cpu_baseline and --impl reference)


def oracle_worker_code(workload, rank, sel, reps, barrier_dir, index, workers):
    """Source of one single-threaded oracle process: it builds the case, waits
    until every worker is ready (a file barrier), then times `reps` runs of
    the fp64 oracle decode over the sequences `sel`."""
    return f"""
import os, sys, time, json
sys.path.insert(0, {ROOT!r})
import numpy as np
import bench, workloads, oracle
case = bench.make_case({workload!r}, {rank})
sel = {list(sel)!r}
kc, vc = case.k_cache, case.v_cache
if case.kv_dtype == workloads.FP8_E4M3:
    kc, vc = kc.copy(), vc.copy()
    oracle.reshape_and_cache(case.new_key, case.new_value, kc, vc, case.slot_mapping,
                             case.block_size, case.src_dtype, case.kv_dtype, case.k_scale, case.v_scale)
open(os.path.join({barrier_dir!r}, "ready_{index}"), "w").close()
deadline = time.time() + 600
while len(os.listdir({barrier_dir!r})) < {workers} and time.time() < deadline:
    time.sleep(0.005)
times = []
for r in range({reps}):
    t = time.perf_counter()
    oracle.paged_decode(case.q[sel], kc, vc, case.block_tables[sel], case.context_lens[sel],
                        case.scale, case.block_size, case.q_dtype, case.kv_dtype,
                        case.k_scale, case.v_scale)
    times.append(time.perf_counter() - t)
print(json.dumps(times))
"""


def host_cores():
    try:
        return max(1, len(os.sched_getaffinity(0)))
    except AttributeError:
        return max(1, os.cpu_count() or 1)


def oracle_seconds(workload, seqs, reps, rank=0, workers=None):
    """Run the fp64 oracle decode on the first `seqs` sequences, `reps` times.

    The sequences are dealt round robin to one single-threaded process per
    host core (fresh interpreters, so this is safe after CUDA has been used in
    the calling process); all processes start timing together, and a run's
    time is that of the slowest process. Returns (times, processes used)."""
    import tempfile
    workers = max(1, min(workers or host_cores(), seqs))
    env = dict(os.environ)
    for k in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS", "NUMEXPR_NUM_THREADS"):
        env[k] = "1"
    env["CUDA_VISIBLE_DEVICES"] = ""
    with tempfile.TemporaryDirectory() as barrier_dir:
        procs = []
        for i in range(workers):
            code = oracle_worker_code(workload, rank, range(i, seqs, workers), reps, barrier_dir, i, workers)
            procs.append(subprocess.Popen([sys.executable, "-c", code], stdout=subprocess.PIPE,
                                          stderr=subprocess.PIPE, text=True, env=env, cwd=ROOT))
        per = []
        for pr in procs:
            out, err = pr.communicate()
            if pr.returncode != 0:
                raise RuntimeError(err[-2000:])
            per.append(json.loads(out.strip().splitlines()[-1]))
    return [max(t[r] for t in per) for r in range(reps)], workers


def sample_case(case, seqs):
    return workloads.DecodeCase(**{**case.__dict__, "q": case.q[:seqs],
                                   "block_tables": case.block_tables[:seqs],
                                   "context_lens": case.context_lens[:seqs], "num_seqs": seqs})


def cpu_baseline(workload, case, target_s=12.0):
    """The oracle on the whole batch, repeated to about target_s seconds of CPU work."""
    probe = oracle_seconds(workload, case.num_seqs, 1)[0][0]
    reps = max(1, min(50, int(math.ceil(target_s / max(probe, 1e-3)))))
    if probe > target_s:
        seqs = max(1, int(case.num_seqs * target_s / probe))
        reps = 1
    else:
        seqs = case.num_seqs
    times, cores = oracle_seconds(workload, seqs, reps)
    sub = sample_case(case, seqs)
    gbs = decode_bytes(sub) * len(times) / sum(times) / 1e9
    return {"value": round(gbs, 4), "unit": "GB/s", "cores": cores, "kind": "oracle",
            "sample": f"fp64 numpy oracle pa_decode over {seqs} of {case.num_seqs} sequences, "
                      f"{len(times)} repetitions, {sum(times):.1f} s of wall time, {cores} "
                      f"single-threaded processes (one per host core)"}


# ----------------------------------------------------------------------------
# the GPU arm


def setup_dist():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x, world, device):
    if world == 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def peak_hbm():
    """(GB/s, source) of the roofline denominator."""
    peaks_path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(peaks_path):
        return json.load(open(peaks_path))["hbm_gbs"], "measured"
    return 6800.0, "fallback"


def shared_groups_of(case):
    """Groups of sequences sharing leading whole blocks, from the tables the
    decode reads (the shared-prefix workload's tables after its copy-on-write
    of the partly filled last prefix block)."""
    from paged_kv_cache_288_gb300.block_pool import shared_prefix_groups
    return shared_prefix_groups(case.block_tables, case.context_lens, case.block_size)


def unique_decode_bytes(case):
    """Algorithmic bytes of one pa_decode counting each physical block's KV
    once: a block that several tables share (a common prefix) need come from
    HBM only once, so this is the call's HBM floor. Table entries are still
    counted per sequence."""
    bs = case.block_size
    used = {}
    nb_total = 0
    for i, c in enumerate(case.context_lens):
        c = int(c)
        nb = -(-c // bs) if c > 0 else 0
        nb_total += nb
        for j in range(nb):
            b = int(case.block_tables[i, j])
            used[b] = max(used.get(b, 0), min(bs, c - j * bs))
    eb = elem(case.kv_dtype)
    kv = sum(used.values()) * case.num_kv_heads * 2 * case.head_dim * eb
    scales = len(used) * case.num_kv_heads * 2 * 4 if case.kv_dtype == workloads.FP8_E4M3 else 0
    qo = 2 * case.num_seqs * case.num_heads * case.head_dim * elem(case.q_dtype)
    return kv + scales + qo + nb_total * 4 + case.num_seqs * 4


class DeviceDecode:
    """One decode workload on the device: pool, tables, q, the step's new
    tokens (one per sequence, written before the decode) and a workspace for
    the chosen schedule. Setup that the workload's flow needs before its
    steps (copy-on-write copies, the suffix or history tokens) is done once
    here, outside any timing."""

    def __init__(self, pa, case, device, part, groups=None):
        self.pa, self.case, self.part = pa, case, part
        self.groups = groups

        def to_dev(bits, dtype):
            a = np.ascontiguousarray(bits)
            if dtype == workloads.FP8_E4M3:
                return torch.from_numpy(a.view(np.uint8)).to(device)
            t = torch.from_numpy(a.view(np.int16)).to(device)
            return t.view(torch.float16 if dtype == workloads.F16 else torch.bfloat16)

        self.to_dev = to_dev
        self.q = to_dev(case.q, case.q_dtype)
        self.kc = to_dev(case.k_cache, case.kv_dtype)
        self.vc = to_dev(case.v_cache, case.kv_dtype)
        self.tables = torch.from_numpy(case.block_tables).to(device)
        self.lens = torch.from_numpy(case.context_lens).to(device)
        self.ks = torch.from_numpy(case.k_scale).to(device) if case.k_scale is not None else None
        self.vs = torch.from_numpy(case.v_scale).to(device) if case.v_scale is not None else None
        self.err = torch.zeros(1, dtype=torch.int32, device=device)
        nk = to_dev(case.new_key, case.src_dtype)
        nv = to_dev(case.new_value, case.src_dtype)
        slots = torch.from_numpy(case.slot_mapping).to(device)
        if case.cow_pairs is not None:
            # the copy-on-write of the shared, partly filled block, once
            block_bytes = case.num_kv_heads * case.block_size * case.head_dim * elem(case.kv_dtype)
            pa.copy_blocks(pa.pointer_array([self.kc], device), pa.pointer_array([self.vc], device),
                           torch.from_numpy(case.cow_pairs).to(device), case.num_blocks, block_bytes,
                           debug_err=self.err)
        T = nk.shape[0]
        if T > case.num_seqs:
            # the history (fp8: the empty pool; shared prefix: the private
            # suffixes) is written once; a step then writes each sequence's
            # last token again
            pa.reshape_and_cache(nk, nv, self.kc, self.vc, slots, k_scale=self.ks, v_scale=self.vs,
                                 debug_err=self.err)
            last = np.cumsum(case.context_lens.astype(np.int64)) - 1
            if case.cow_pairs is not None:
                start = np.concatenate([[0], np.cumsum(case.context_lens.astype(np.int64)
                                                       - int(case.meta["prefix_len"]))])
                last = start[1:] - 1
            idx = torch.from_numpy(last).to(device)
            nk, nv, slots = nk[idx].contiguous(), nv[idx].contiguous(), slots[idx].contiguous()
            case.new_key, case.new_value = case.new_key[last], case.new_value[last]
            case.slot_mapping = case.slot_mapping[last]
        self.nk, self.nv, self.slots = nk, nv, slots
        self.out = torch.empty_like(self.q)
        self.max_ctx = int(case.context_lens.max())
        ws_bytes = pa.decode_workspace_size(case.num_seqs, case.num_heads, case.num_kv_heads,
                                            case.head_dim, self.max_ctx, part)
        if groups is not None:
            # sequences sharing leading blocks, attended once per group
            gs, gp = groups
            self.gs = torch.from_numpy(np.asarray(gs, np.int32)).to(device)
            self.gp = torch.from_numpy(np.asarray(gp, np.int32)).to(device)
            self.mgs = int(np.diff(gs).max())
            self.mpl = int(np.max(gp))
            ws_bytes = pa.decode_shared_prefix_workspace_size(
                case.num_seqs, case.num_heads, case.num_kv_heads, case.head_dim, case.block_size,
                len(gp), self.mgs, self.mpl)
        self.ws = torch.empty(max(ws_bytes, 256), dtype=torch.uint8, device=device)

    def write(self, nk=None, nv=None, slots=None):
        self.pa.reshape_and_cache(self.nk if nk is None else nk, self.nv if nv is None else nv,
                                  self.kc, self.vc, self.slots if slots is None else slots,
                                  k_scale=self.ks, v_scale=self.vs, debug_err=self.err)

    def decode(self, q=None, tables=None, lens=None):
        c = self.case
        if self.groups is not None:
            self.pa.decode_shared_prefix(
                self.out, self.q if q is None else q, self.kc, self.vc,
                self.tables if tables is None else tables, self.lens if lens is None else lens,
                c.scale, self.max_ctx, self.gs, self.gp, self.mgs, self.mpl, self.ws,
                debug_err=self.err)
            return
        self.pa.decode(self.out, self.q if q is None else q, self.kc, self.vc,
                       self.tables if tables is None else tables, self.lens if lens is None else lens,
                       c.scale, self.max_ctx, k_scale=self.ks, v_scale=self.vs,
                       partition_size=self.part, workspace=self.ws, debug_err=self.err)


class PackedH2D:
    """One pinned host staging buffer and one device buffer that hold several
    input tensors, each at a 256-byte boundary: a step's inputs cross the host
    link in a single copy, and the library's calls read device views into it."""

    def __init__(self, tensors, device):
        offs, n = [], 0
        for t in tensors:
            offs.append(n)
            n += (t.numel() * t.element_size() + 255) // 256 * 256
        self.host = torch.empty(max(n, 256), dtype=torch.uint8).pin_memory()
        self.dev = torch.empty(max(n, 256), dtype=torch.uint8, device=device)
        self.views = []
        for t, o in zip(tensors, offs):
            nb = t.numel() * t.element_size()
            self.host[o:o + nb].copy_(t.detach().cpu().contiguous().view(-1).view(torch.uint8))
            self.views.append(self.dev[o:o + nb].view(t.dtype).view(t.shape))

    @property
    def nbytes(self):
        return self.dev.numel()

    def h2d(self):
        self.dev.copy_(self.host, non_blocking=True)


def make_flush(device):
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=device)

    def flush_l2():
        # write a buffer twice the L2 size, then read it back: the lines left in
        # L2 are clean, so no write-back of the flush lands inside a timed step
        flush.zero_()
        flush.sum()

    return flush_l2


def time_write_decode(dd, K, W, flush_l2, stream, world=1):
    """K timed steps (cache write, then decode) after W untimed ones; CUDA
    events on the launching stream around both parts. Returns per-step
    (step ms, decode ms) lists and the launches of the timed steps."""
    for _ in range(W):
        flush_l2()
        dd.write()
        dd.decode()
    torch.cuda.synchronize()
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(K)]
    barrier(world)
    torch.cuda.synchronize()
    n0 = dd.pa.lib().pa_kernel_launch_count()
    for k in range(K):
        flush_l2()
        ev[k][0].record(stream)
        dd.write()
        ev[k][1].record(stream)
        dd.decode()
        ev[k][2].record(stream)
    torch.cuda.synchronize()
    barrier(world)
    n1 = dd.pa.lib().pa_kernel_launch_count()
    return ([ev[k][0].elapsed_time(ev[k][2]) for k in range(K)],
            [ev[k][1].elapsed_time(ev[k][2]) for k in range(K)], n1 - n0)


def decode_result(case, step_ms, dec_ms, launches, part, peak, peak_src, workload, extra=None,
                  traffic_key=None):
    """A per-workload bench record: decode call and step throughput and the
    HBM roofline fraction of the decode call."""
    K = len(step_ms)
    dbytes = decode_bytes(case)
    sbytes = dbytes + write_bytes(case)
    dec_mean = statistics.mean(dec_ms)
    step_mean = statistics.mean(step_ms)
    achieved = dbytes / (dec_mean / 1e3) / 1e9
    rec = {
        "workload": workload, "partition_size": part, "steps": K,
        "num_seqs": case.num_seqs, "num_heads": case.num_heads, "num_kv_heads": case.num_kv_heads,
        "head_dim": case.head_dim, "block_size": case.block_size,
        "kv_dtype": case.kv_dtype, "context_tokens": int(case.context_lens.sum()),
        "decode_us": round(dec_mean * 1e3, 2), "step_us": round(step_mean * 1e3, 2),
        "decode_bytes": dbytes, "step_bytes": sbytes,
        "decode_gbs": round(achieved, 1), "step_gbs": round(sbytes / (step_mean / 1e3) / 1e9, 1),
        "tokens_per_s_per_layer": round(case.num_seqs / (step_mean / 1e3), 1),
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak,
                     "peak_source": peak_src, "unit": "GB/s", "frac": round(achieved / peak, 4),
                     "traffic": recorded_traffic(traffic_key or workload, part),
                     "kernel": "pa_decode (every kernel of the call)"},
        "gpu_launches": launches,
    }
    if extra:
        rec.update(extra)
    return rec


def run_config_suite(pa, device, stream, flush_l2, K, W, peak, peak_src):
    """The other workloads' decode numbers, timed in the same run as the
    headline line: the tiny case (latency), the shared-prefix serving batch
    (logical and unique-byte rooflines; per-sequence decode and the shared
    blocks read once per group), the long-context batch at every block size
    (512-token split path and the library's schedule) and the 32-layer E4M3
    decode step."""
    out = {}

    def one(name, case, parts, extra_fn=None, groups=None, key=None):
        for part in parts:
            dd = DeviceDecode(pa, case, device, part, groups)
            step_ms, dec_ms, launches = time_write_decode(dd, K, W, flush_l2, stream)
            torch.cuda.synchronize()
            if dd.err.item() != 0:
                raise RuntimeError(f"{name}: device error word {dd.err.item():#x}")
            extra = extra_fn(case, statistics.mean(dec_ms)) if extra_fn else None
            out[key or f"{name}/p{part}"] = decode_result(
                case, step_ms, dec_ms, launches, part, peak, peak_src, name, extra,
                traffic_key=name + ("_grouped" if groups is not None else ""))
            del dd
            torch.cuda.empty_cache()

    def shared_extra(case, dec_ms):
        ub = unique_decode_bytes(case)
        a = ub / (dec_ms / 1e3) / 1e9
        return {"unique_decode_bytes": ub, "unique_gbs": round(a, 1),
                "roofline_unique": {"bound": "hbm", "achieved": round(a, 1), "peak": peak,
                                    "peak_source": peak_src, "unit": "GB/s", "frac": round(a / peak, 4),
                                    "note": "each shared block's KV counted once"}}

    one("tiny", make_case("tiny", 0), [0])
    one("shared_prefix", workloads.shared_prefix(), [0], shared_extra)
    sp = workloads.shared_prefix()
    one("shared_prefix", sp, [0], shared_extra, groups=shared_groups_of(sp), key="shared_prefix/grouped")
    for bs in (8, 16, 32, 64):
        one(f"long_context_bs{bs}", workloads.long_context(bs), [512, 0])
    out["fp8_step"] = run_fp8_step(pa, device, stream, flush_l2, K, W, peak, peak_src)
    return out


FP8_STEP_LAYERS = 32


def run_fp8_step(pa, device, stream, flush_l2, K, W, peak, peak_src, layers=FP8_STEP_LAYERS):
    """The full 8-bit decode step: for each of 32 layers, one
    pa_reshape_and_cache of the new token of each of 256 sequences, then one
    pa_decode over that layer's pool (E4M3 K/V, one float32 scale per block
    and KV head). Every layer owns its pool; the pools hold the same history
    (filled once from layer 0's tokens through the library, then copied on
    the device), the block tables are shared by all layers as a model's are,
    and q is drawn per layer."""
    base = workloads.fp8_step_layer(0)
    dd = DeviceDecode(pa, base, device, 0)
    case = dd.case
    g = workloads._gen(4242)
    pools = [(dd.kc, dd.vc)] + [(dd.kc.clone(), dd.vc.clone()) for _ in range(layers - 1)]
    qs = [dd.q] + [dd.to_dev(workloads.normal_bits(g, case.q.shape, case.q_dtype), case.q_dtype)
                   for _ in range(layers - 1)]

    def step():
        for l in range(layers):
            dd.kc, dd.vc = pools[l]
            dd.write()
            dd.decode(q=qs[l])

    for _ in range(W):
        flush_l2()
        step()
    torch.cuda.synchronize()
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2 * layers + 1)] for _ in range(K)]
    n0 = pa.lib().pa_kernel_launch_count()
    for k in range(K):
        flush_l2()
        ev[k][0].record(stream)
        for l in range(layers):
            dd.kc, dd.vc = pools[l]
            dd.write()
            ev[k][2 * l + 1].record(stream)
            dd.decode(q=qs[l])
            ev[k][2 * l + 2].record(stream)
    torch.cuda.synchronize()
    n1 = pa.lib().pa_kernel_launch_count()
    if dd.err.item() != 0:
        raise RuntimeError(f"fp8 step: device error word {dd.err.item():#x}")
    step_ms = [ev[k][0].elapsed_time(ev[k][2 * layers]) for k in range(K)]
    dec_ms = [sum(ev[k][2 * l + 1].elapsed_time(ev[k][2 * l + 2]) for l in range(layers)) for k in range(K)]
    dbytes = layers * decode_bytes(case)
    sbytes = layers * (decode_bytes(case) + write_bytes(case))
    step_mean, dec_mean = statistics.mean(step_ms), statistics.mean(dec_ms)
    achieved = dbytes / (dec_mean / 1e3) / 1e9
    step_gbs = sbytes / (step_mean / 1e3) / 1e9
    del pools, qs, dd
    torch.cuda.empty_cache()
    return {
        "workload": "fp8_step", "layers": layers, "steps": K, "num_seqs": case.num_seqs,
        "num_heads": case.num_heads, "num_kv_heads": case.num_kv_heads, "head_dim": case.head_dim,
        "block_size": case.block_size, "kv_dtype": case.kv_dtype,
        "context_tokens_per_layer": int(case.context_lens.sum()),
        "step_ms": round(step_mean, 4), "decode_ms_per_step": round(dec_mean, 4),
        "decode_us_per_layer": round(1e3 * dec_mean / layers, 2),
        "step_bytes": sbytes, "decode_bytes_per_step": dbytes,
        "step_gbs": round(step_gbs, 1), "decode_gbs": round(achieved, 1),
        "tokens_per_s_per_layer": round(case.num_seqs * layers / (step_mean / 1e3), 1),
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "peak_source": peak_src,
                     "unit": "GB/s", "frac": round(achieved / peak, 4),
                     "traffic": recorded_traffic("fp8_layer", 0),
                     "kernel": "pa_decode (every kernel of the call), summed over the 32 layers"},
        "roofline_step": {"bound": "hbm", "achieved": round(step_gbs, 1), "peak": peak,
                          "peak_source": peak_src, "unit": "GB/s", "frac": round(step_gbs / peak, 4),
                          "kernel": "the whole step: 32 x (pa_reshape_and_cache + pa_decode)"},
        "gpu_launches": n1 - n0,
    }


def run_ours(args, world, rank, local):
    import paged_kv_cache_288_gb300 as pa
    from paged_kv_cache_288_gb300 import build

    build.build_library()
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    stream = torch.cuda.current_stream(device)
    flush_l2 = make_flush(device)
    peak, peak_src = peak_hbm()
    if args.workload == "fp8_step":
        sampler = ClockSampler(local)
        sampler.start()
        time.sleep(0.3)
        t0 = time.time()
        rec = run_fp8_step(pa, device, stream, flush_l2, args.steps, args.warmup, peak, peak_src)
        t1 = time.time()
        sampler.stop()
        if rank != 0:
            return None
        return {"metric": METRIC, "value": rec["step_gbs"], "unit": "GB/s", "n_gpus": world,
                "steps": args.steps, "warmup": args.warmup, "ms_per_step": rec["step_ms"],
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
                "dtype": "fp8_e4m3 KV, bf16 q, f32 accumulate", "data": "synthetic",
                "config": {"workload": "fp8_step", "l2": "flushed between steps"},
                "roofline": rec["roofline"], "fp8_step": rec, "clocks": sampler.summary(t0, t1),
                "gpu_launches": rec["gpu_launches"]}
    case = make_case(args.workload, rank)
    part = args.partition_size
    groups = None
    if args.shared_groups:
        # the sharing in the tables (after any copy-on-write), found on the host
        groups = shared_groups_of(case)
    dd = DeviceDecode(pa, case, device, part, groups)
    case = dd.case

    K = args.steps
    sampler = ClockSampler(local)
    sampler.start()
    time.sleep(0.3)
    t0 = time.time()
    step_ms, dec_ms, launches = time_write_decode(dd, K, args.warmup, flush_l2, stream, world)
    t1 = time.time()
    sampler.stop()
    total_ms = max_over_ranks(sum(step_ms), world, device)
    dec_mean_ms = statistics.mean(dec_ms)
    if dd.err.item() != 0:
        raise RuntimeError(f"device error word {dd.err.item():#x}")

    # end to end through the public API with host buffers: the step's inputs
    # (q, the new token's K/V, its slots, the tables, the lengths) cross in one
    # copy from a pinned staging buffer, the output comes back
    packed = PackedH2D([dd.q, dd.nk, dd.nv, dd.slots, dd.tables, dd.lens], device)
    d_q, d_nk, d_nv, d_slots, d_tables, d_lens = packed.views
    h_out = torch.empty(dd.out.shape, dtype=dd.out.dtype).pin_memory()
    h2d = packed.nbytes
    d2h = h_out.numel() * h_out.element_size()
    Ke = max(1, min(K, 200))
    eev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(Ke)]
    barrier(world)
    torch.cuda.synchronize()
    for k in range(Ke):
        flush_l2()
        eev[k][0].record(stream)
        packed.h2d()
        dd.write(d_nk, d_nv, d_slots)
        dd.decode(q=d_q, tables=d_tables, lens=d_lens)
        h_out.copy_(dd.out, non_blocking=True)
        eev[k][1].record(stream)
    torch.cuda.synchronize()
    barrier(world)
    e2e_ms = max_over_ranks(sum(eev[k][0].elapsed_time(eev[k][1]) for k in range(Ke)), world,
                            device)

    bytes_step = decode_bytes(case) + write_bytes(case)
    value = job_throughput_gbs(bytes_step, K, world, total_ms)
    e2e_value = job_throughput_gbs(bytes_step, Ke, world, e2e_ms)
    dbytes = decode_bytes(case)
    achieved = dbytes / (dec_mean_ms / 1e3) / 1e9
    del dd
    torch.cuda.empty_cache()
    configs = None
    if args.workload == "llama8b" and not args.no_configs and world == 1:
        configs = run_config_suite(pa, device, stream, flush_l2, K, args.warmup, peak, peak_src)
    if rank != 0:
        return None
    line = {
        "metric": METRIC,
        "value": round(value, 2),
        "unit": "GB/s",
        "n_gpus": world,
        "steps": K,
        "warmup": args.warmup,
        "ms_per_step": round(total_ms / K, 5),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16" if case.kv_dtype == workloads.BF16 else (
            "f16" if case.kv_dtype == workloads.F16 else "fp8_e4m3 KV, bf16 q, f32 accumulate"),
        "data": "synthetic (seeded N(0,1) K/V/q, shuffled physical blocks)",
        "config": {
            "workload": args.workload,
            "num_seqs": case.num_seqs, "num_heads": case.num_heads,
            "num_kv_heads": case.num_kv_heads, "head_dim": case.head_dim,
            "block_size": case.block_size, "num_blocks": case.num_blocks,
            "context_tokens": int(case.context_lens.sum()),
            "max_context_len": dd_max_ctx(case), "partition_size": part,
            "shared_groups": groups is not None,
            "l2": "flushed between steps: 256 MiB written then read back, outside the timed events",
            "parallelism": f"{world} independent replica(s), one per GPU",
        },
        "tokens_per_s_per_layer": round(world * case.num_seqs * K / (total_ms / 1e3), 1),
        "decode_us": round(dec_mean_ms * 1e3, 2),
        "decode_bytes": dbytes,
        "step_bytes": bytes_step,
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak,
                     "peak_source": peak_src, "unit": "GB/s", "frac": round(achieved / peak, 4),
                     "traffic": recorded_traffic(args.workload + ("_grouped" if groups is not None else ""),
                                                 part),
                     "kernel": "pa_decode (every kernel of the call)"},
        "e2e": {"value": round(e2e_value, 2), "unit": "GB/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "steps": Ke},
        "clocks": sampler.summary(t0, t1),
        "gpu_launches": launches,
        "launches_per_step": launches / K,
    }
    if args.workload == "shared_prefix":
        ub = unique_decode_bytes(case)
        a = ub / (dec_mean_ms / 1e3) / 1e9
        line["roofline_unique"] = {"bound": "hbm", "achieved": round(a, 1), "peak": peak,
                                   "peak_source": peak_src, "unit": "GB/s", "frac": round(a / peak, 4),
                                   "note": "each shared block's KV counted once"}
    if case.meta and "prefix_cache" in case.meta:
        line["prefix_cache"] = case.meta["prefix_cache"]
    if configs is not None:
        line["configs"] = configs
    if not args.no_cpu_baseline and world == 1:
        line["cpu_baseline"] = cpu_baseline(args.workload, case)
    return line


def dd_max_ctx(case):
    return int(case.context_lens.max()) if case.num_seqs else 0


# ----------------------------------------------------------------------------
# chunked prefill (pa_reshape_and_cache of the chunks + pa_prefill)

PREFILL_METRIC = "pa_prefill TFLOP/s (causal chunked prefill over the paged cache)"


def prefill_flops(case):
    """Algorithmic FLOPs of one pa_prefill: per query at position p and head,
    2*d*(p+1) for q.K and as many for P.V."""
    total = 0
    for i in range(case.num_seqs):
        n = int(case.query_start[i + 1] - case.query_start[i])
        ctx = int(case.context_lens[i])
        keys = n * (ctx - n) + n * (n + 1) // 2  # sum over j of (ctx - n + j + 1)
        total += 4 * case.head_dim * keys * case.num_heads
    return total


def run_prefill(args, world, rank, local):
    import paged_kv_cache_288_gb300 as pa
    from paged_kv_cache_288_gb300 import build

    build.build_library()
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    case = workloads.prefill_llama8b(seed=rank_seed(1011, rank))

    def to_dev(bits):
        return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to(device).view(torch.bfloat16)

    q, kc, vc = to_dev(case.q), to_dev(case.k_cache), to_dev(case.v_cache)
    nk, nv = to_dev(case.new_key), to_dev(case.new_value)
    slots = torch.from_numpy(case.slot_mapping).to(device)
    tables = torch.from_numpy(case.block_tables).to(device)
    lens = torch.from_numpy(case.context_lens).to(device)
    qs = torch.from_numpy(case.query_start).to(device)
    out = torch.empty_like(q)
    err = torch.zeros(1, dtype=torch.int32, device=device)
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=device)
    stream = torch.cuda.current_stream(device)
    mq = case.max_query_len

    def step():
        pa.reshape_and_cache(nk, nv, kc, vc, slots, debug_err=err)
        pa.prefill(out, q, kc, vc, tables, lens, qs, case.scale, mq, debug_err=err)

    for _ in range(args.warmup):
        flush.zero_()
        flush.sum()
        step()
    torch.cuda.synchronize()
    K = args.steps
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(K)]
    sampler = ClockSampler(local)
    sampler.start()
    time.sleep(0.3)
    barrier(world)
    torch.cuda.synchronize()
    n0 = pa.lib().pa_kernel_launch_count()
    t0 = time.time()
    for k in range(K):
        flush.zero_()
        flush.sum()
        ev[k][0].record(stream)
        pa.reshape_and_cache(nk, nv, kc, vc, slots, debug_err=err)
        ev[k][1].record(stream)
        pa.prefill(out, q, kc, vc, tables, lens, qs, case.scale, mq, debug_err=err)
        ev[k][2].record(stream)
    torch.cuda.synchronize()
    t1 = time.time()
    barrier(world)
    n1 = pa.lib().pa_kernel_launch_count()
    sampler.stop()
    assert err.item() == 0, "a kernel flagged an out-of-range index"
    step_ms = [ev[k][0].elapsed_time(ev[k][2]) for k in range(K)]
    pf_ms = statistics.mean(ev[k][1].elapsed_time(ev[k][2]) for k in range(K))
    total_ms = max_over_ranks(sum(step_ms), world, device)
    flops = prefill_flops(case)
    value = world * flops * K / (total_ms / 1e3) / 1e12
    achieved = flops / (pf_ms / 1e3) / 1e12

    # end to end: queries and the chunks' K/V from pinned host memory, output back
    h_q, h_nk, h_nv = q.cpu().pin_memory(), nk.cpu().pin_memory(), nv.cpu().pin_memory()
    h_out = torch.empty_like(out, device="cpu").pin_memory()
    Ke = min(K, 50)
    eev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(Ke)]
    for k in range(Ke):
        flush.zero_()
        flush.sum()
        eev[k][0].record(stream)
        q.copy_(h_q, non_blocking=True)
        nk.copy_(h_nk, non_blocking=True)
        nv.copy_(h_nv, non_blocking=True)
        step()
        h_out.copy_(out, non_blocking=True)
        eev[k][1].record(stream)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(sum(eev[k][0].elapsed_time(eev[k][1]) for k in range(Ke)), world, device)
    if rank != 0:
        return None
    peaks_path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    peaks = json.load(open(peaks_path)) if os.path.exists(peaks_path) else {}
    peak = peaks.get("bf16_tflops", 1900.0)
    line = {
        "metric": PREFILL_METRIC, "value": round(value, 2), "unit": "TFLOP/s", "n_gpus": world,
        "steps": K, "warmup": args.warmup, "ms_per_step": round(total_ms / K, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded N(0,1) K/V/q, shuffled physical blocks)",
        "config": {"workload": args.workload, "num_seqs": case.num_seqs, "num_heads": case.num_heads,
                   "num_kv_heads": case.num_kv_heads, "head_dim": case.head_dim,
                   "block_size": case.block_size, "chunk_tokens": int(case.query_start[-1]),
                   "context_tokens": int(case.context_lens.sum()),
                   "l2": "flushed between steps: 256 MiB written then read back, outside the timed events",
                   "parallelism": f"{world} independent replica(s), one per GPU"},
        "prefill_us": round(pf_ms * 1e3, 1),
        "flops_per_step": flops,
        "roofline": {"bound": "tensor", "achieved": round(achieved, 1), "peak": peak,
                     "peak_source": "measured" if "bf16_tflops" in peaks else "fallback",
                     "unit": "TFLOP/s", "frac": round(achieved / peak, 4), "traffic": None,
                     "kernel": "prefill_tc_kernel"},
        "e2e": {"value": round(world * flops * Ke / (e2e_ms / 1e3) / 1e12, 2), "unit": "TFLOP/s",
                "h2d_bytes_per_step": 3 * 0 + (h_q.numel() + h_nk.numel() + h_nv.numel()) * 2,
                "d2h_bytes_per_step": h_out.numel() * 2, "steps": Ke},
        "clocks": sampler.summary(t0, t1), "gpu_launches": n1 - n0, "launches_per_step": (n1 - n0) / K,
    }
    if not args.no_cpu_baseline and world == 1:
        line["cpu_baseline"] = prefill_cpu_baseline(case)
    return line


def prefill_oracle_tflops(case, seqs, target_s):
    """The oracle on the first rows of a few sequences' chunks, about target_s."""
    import oracle
    flops, t_used, rows_done = 0, 0.0, 0
    for i in range(seqs):
        q0 = int(case.query_start[i])
        for rows in (1, 2, 4, 8, 16, 32, 64, 128):
            sub = workloads.PrefillCase(**{**case.__dict__})
            sub.num_seqs = 1
            sub.block_tables = case.block_tables[i:i + 1]
            n = int(case.query_start[i + 1] - case.query_start[i])
            rows = min(rows, n)
            # the first `rows` queries of the chunk: a chunk of `rows` at the same place
            sub.context_lens = np.array([int(case.context_lens[i]) - n + rows], np.int32)
            sub.query_start = np.array([0, rows], np.int32)
            sub.q = case.q[q0:q0 + rows]
            t = time.perf_counter()
            oracle.paged_prefill(sub.q, case.k_cache, case.v_cache, sub.block_tables, sub.context_lens,
                                 sub.query_start, case.scale, case.block_size, case.dtype, case.dtype)
            dt = time.perf_counter() - t
            flops += prefill_flops(sub)
            t_used += dt
            rows_done += rows
            if t_used > target_s:
                return flops / t_used / 1e12, rows_done, t_used
    return flops / t_used / 1e12, rows_done, t_used


def prefill_cpu_baseline(case):
    value, rows, secs = prefill_oracle_tflops(case, case.num_seqs, 10.0)
    return {"value": round(value, 6), "unit": "TFLOP/s", "cores": 1, "kind": "oracle",
            "sample": f"fp64 numpy oracle pa_prefill on {rows} query rows (chunk starts of the batch's "
                      f"sequences), {secs:.1f} s, 1 thread"}


def run_prefill_reference(args, world, rank):
    if rank != 0:
        return None
    case = workloads.prefill_llama8b(seed=rank_seed(1011, 0))
    value, rows, secs = prefill_oracle_tflops(case, case.num_seqs, 2.0 * (args.steps + args.warmup) / 10)
    return {"impl": "reference", "metric": PREFILL_METRIC, "value": round(value, 6), "unit": "TFLOP/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(1e3 * secs / max(1, args.steps + args.warmup), 2),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64 (oracle)",
            "data": "synthetic", "config": {"workload": args.workload, "sample_rows": rows},
            "cpu_baseline": {"value": round(value, 6), "unit": "TFLOP/s", "cores": 1, "kind": "oracle",
                             "sample": f"fp64 numpy oracle on {rows} query rows, {secs:.1f} s, 1 thread"},
            "e2e": {"value": round(value, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}


# ----------------------------------------------------------------------------
# beam search: fork + copy-on-write + decode


def beam_plan(steps, seed, requests=16, beams=4, prompt_lo=1536, prompt_hi=2560, block_size=16):
    """Host bookkeeping of a beam-search decode, planned ahead of the GPU run.

    ``requests`` prompts (lengths uniform in [prompt_lo, prompt_hi]) each fork
    into ``beams`` beams that share the prompt's blocks. Every step each beam
    appends one token (copying a shared, partly filled last block first), all
    beams decode, and in every request the lowest-ranked beam is dropped and
    a random surviving beam forked in its place (ranks are seeded random:
    there is no model). Returns the pool size and per step the copy pairs,
    new-token slots, tables and context lengths.
    """
    from paged_kv_cache_288_gb300.block_pool import BlockPool

    rng = np.random.default_rng(seed)
    bs = block_size
    prompts = rng.integers(prompt_lo, prompt_hi + 1, requests)
    max_len = int(prompts.max()) + steps + 1
    num_blocks = requests * (-(-int(prompts.max()) // bs)) + requests * beams * (-(-(steps + 1) // bs) + 2) + 1
    pool = BlockPool(num_blocks, bs)
    names = [[(r, b) for b in range(beams)] for r in range(requests)]
    for r in range(requests):
        pool.add_sequence(("p", r), int(prompts[r]))
        for n in names[r]:
            pool.fork(("p", r), n)
        pool.free_sequence(("p", r))
    order = [n for group in names for n in group]
    width = -(-max_len // bs)
    plan = []
    for _ in range(steps):
        pairs, slots = [], []
        for n in order:
            sl, cow = pool.append(n, 1)
            pairs += cow
            slots += sl
        plan.append({"pairs": np.array(pairs, dtype=np.int64).reshape(-1, 2),
                     "slots": np.array(slots, dtype=np.int64),
                     "tables": pool.block_table_array(order, width=width, pad=0),
                     "lens": pool.context_lens(order)})
        for r in range(requests):
            worst, best = rng.choice(beams, 2, replace=False)
            pool.free_sequence(names[r][worst])
            pool.fork(names[r][best], names[r][worst])
    return num_blocks, width, plan


def run_beam_reference(args, world, rank):
    """The oracle on the beam-search plan: copies, cache writes and the decode
    of a sample of beams per step, on host pools."""
    if rank != 0:
        return None
    import oracle
    H, Hkv, d, bs, sample = 32, 8, 128, 16, 4
    num_blocks, width, plan = beam_plan(args.warmup + args.steps, rank_seed(1008, 0))
    g = workloads._gen(1010)
    kc = workloads.normal_bits(g, (num_blocks, Hkv, bs, d), workloads.BF16)
    vc = workloads.normal_bits(g, (num_blocks, Hkv, bs, d), workloads.BF16)
    B = plan[0]["lens"].shape[0]
    q = workloads.normal_bits(g, (B, H, d), workloads.BF16)
    nk = workloads.normal_bits(g, (B, Hkv, d), workloads.BF16)
    secs, nbytes = [], []
    for st in plan:
        t = time.perf_counter()
        oracle.copy_blocks([kc], [vc], st["pairs"])
        oracle.reshape_and_cache(nk, nk, kc, vc, st["slots"], bs, workloads.BF16, workloads.BF16)
        oracle.paged_decode(q[:sample], kc, vc, st["tables"][:sample], st["lens"][:sample],
                            1.0 / math.sqrt(d), bs, workloads.BF16, workloads.BF16)
        secs.append(time.perf_counter() - t)
        nbytes.append(int(st["lens"][:sample].astype(np.int64).sum()) * Hkv * 2 * d * 2)
    W = args.warmup
    value = sum(nbytes[W:]) / sum(secs[W:]) / 1e9
    return {"impl": "reference", "metric": METRIC + " (beam search step: copy-on-write + cache write + "
            "decode, logical KV bytes)", "value": round(value, 4), "unit": "GB/s", "n_gpus": world,
            "steps": args.steps, "warmup": W, "ms_per_step": round(1e3 * sum(secs[W:]) / args.steps, 2),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64 (oracle)",
            "data": "synthetic", "config": {"workload": args.workload, "sample_beams_per_step": sample},
            "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": 1, "kind": "oracle",
                             "sample": f"fp64 numpy oracle: every step's copies and cache writes, the "
                                       f"decode of {sample} of {B} beams, 1 thread"},
            "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}


def run_beam(args, world, rank, local):
    import paged_kv_cache_288_gb300 as pa
    from paged_kv_cache_288_gb300 import build

    build.build_library()
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    H, Hkv, d, bs = 32, 8, 128, 16
    W, K = args.warmup, args.steps
    num_blocks, width, plan = beam_plan(W + K, rank_seed(1008, rank))
    B = plan[0]["lens"].shape[0]
    shape = (num_blocks, Hkv, bs, d)
    kc = torch.empty(shape, dtype=torch.bfloat16, device=device).normal_()
    vc = torch.empty(shape, dtype=torch.bfloat16, device=device).normal_()
    kptr, vptr = pa.pointer_array([kc], device), pa.pointer_array([vc], device)
    block_bytes = Hkv * bs * d * 2
    g = torch.Generator(device="cpu").manual_seed(rank_seed(1009, rank))
    dev_plan = []
    for st in plan:
        dev_plan.append({
            "pairs": torch.from_numpy(st["pairs"]).to(device),
            "slots": torch.from_numpy(st["slots"]).to(device),
            "tables": torch.from_numpy(st["tables"]).to(device),
            "lens": torch.from_numpy(st["lens"]).to(device),
            "max": int(st["lens"].max())})
    q = torch.randn(B, H, d, generator=g).to(torch.bfloat16).to(device)
    nk = torch.randn(B, Hkv, d, generator=g).to(torch.bfloat16).to(device)
    nv = torch.randn(B, Hkv, d, generator=g).to(torch.bfloat16).to(device)
    out = torch.empty_like(q)
    ws = torch.empty(pa.decode_workspace_size(B, H, Hkv, d, max(st["max"] for st in dev_plan), 0),
                     dtype=torch.uint8, device=device)
    err = torch.zeros(1, dtype=torch.int32, device=device)
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=device)
    stream = torch.cuda.current_stream(device)

    def step(st):
        if st["pairs"].shape[0]:
            pa.copy_blocks(kptr, vptr, st["pairs"], num_blocks, block_bytes, debug_err=err)
        pa.reshape_and_cache(nk, nv, kc, vc, st["slots"], debug_err=err)
        pa.decode(out, q, kc, vc, st["tables"], st["lens"], 1.0 / math.sqrt(d), st["max"],
                  workspace=ws, debug_err=err)

    for k in range(W):
        flush.zero_()
        flush.sum()
        step(dev_plan[k])
    torch.cuda.synchronize()
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(K)]
    sampler = ClockSampler(local)
    sampler.start()
    time.sleep(0.3)
    barrier(world)
    torch.cuda.synchronize()
    n0 = pa.lib().pa_kernel_launch_count()
    t0 = time.time()
    for k in range(K):
        flush.zero_()
        flush.sum()
        ev[k][0].record(stream)
        step(dev_plan[W + k])
        ev[k][1].record(stream)
    torch.cuda.synchronize()
    t1 = time.time()
    barrier(world)
    n1 = pa.lib().pa_kernel_launch_count()
    sampler.stop()
    assert err.item() == 0, "a kernel flagged an out-of-range index"
    # end to end through the public API: each step's plan (pairs, slots,
    # tables, lengths) and new tokens come from pinned host memory, the
    # output goes back to pinned host memory
    Ke = min(K, 100)
    host_plan = [{k: torch.from_numpy(v).pin_memory() for k, v in st.items()} for st in plan[W:W + Ke]]
    h_nk, h_nv, h_out = nk.cpu().pin_memory(), nv.cpu().pin_memory(), torch.empty_like(out, device="cpu").pin_memory()
    eev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(Ke)]
    h2d = d2h = 0
    for k in range(Ke):
        st, hp = dev_plan[W + k], host_plan[k]
        flush.zero_()
        flush.sum()
        eev[k][0].record(stream)
        for key in ("pairs", "slots", "tables", "lens"):
            st[key].copy_(hp[key], non_blocking=True)
        nk.copy_(h_nk, non_blocking=True)
        nv.copy_(h_nv, non_blocking=True)
        step(st)
        h_out.copy_(out, non_blocking=True)
        eev[k][1].record(stream)
        h2d += sum(hp[key].numel() * hp[key].element_size() for key in ("pairs", "slots", "tables", "lens"))
        h2d += 2 * h_nk.numel() * 2
        d2h += h_out.numel() * 2
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(sum(eev[k][0].elapsed_time(eev[k][1]) for k in range(Ke)), world, device)
    ms = [ev[k][0].elapsed_time(ev[k][1]) for k in range(K)]
    total_ms = max_over_ranks(sum(ms), world, device)
    timed = plan[W:]
    kv_bytes = [int(st["lens"].astype(np.int64).sum()) * Hkv * 2 * d * 2 for st in timed]
    copies = [st["pairs"].shape[0] for st in timed]
    step_bytes = [kvb + 2 * B * H * d * 2 + 2 * c * 2 * block_bytes + 2 * B * Hkv * d * 2 * 2
                  for kvb, c in zip(kv_bytes, copies)]
    value = world * sum(step_bytes) / (total_ms / 1e3) / 1e9
    if rank != 0:
        return None
    peaks_path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    peak = json.load(open(peaks_path))["hbm_gbs"] if os.path.exists(peaks_path) else 6800.0
    return {
        "metric": METRIC + " (beam search step: copy-on-write + cache write + decode, logical KV bytes)",
        "value": round(value, 2), "unit": "GB/s", "n_gpus": world, "steps": K, "warmup": W,
        "ms_per_step": round(total_ms / K, 5), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (random pools, seeded beam ranks)",
        "config": {"workload": args.workload, "requests": 16, "beams": 4, "num_seqs": B,
                   "num_heads": H, "num_kv_heads": Hkv, "head_dim": d, "block_size": bs,
                   "prompt_tokens": "uniform 1536..2560", "num_blocks": num_blocks,
                   "l2": "flushed between steps: 256 MiB written then read back, outside the timed events",
                   "parallelism": f"{world} independent replica(s), one per GPU"},
        "tokens_per_s_per_layer": round(world * B * K / (total_ms / 1e3), 1),
        "copies_per_step": round(statistics.mean(copies), 2),
        "roofline": {"bound": "hbm", "achieved": round(value, 1), "peak": peak, "unit": "GB/s",
                     "frac": round(value / peak, 4), "traffic": None,
                     "kernel": "copy_blocks + reshape_and_cache + pa_decode (logical bytes: "
                               "beams re-read their shared prompt blocks, mostly from L2)"},
        "e2e": {"value": round(world * sum(step_bytes[:Ke]) / (e2e_ms / 1e3) / 1e9, 2), "unit": "GB/s",
                "h2d_bytes_per_step": h2d // Ke, "d2h_bytes_per_step": d2h // Ke, "steps": Ke},
        "clocks": sampler.summary(t0, t1), "gpu_launches": n1 - n0,
        "launches_per_step": (n1 - n0) / K,
        **({} if args.no_cpu_baseline or world != 1 else {"cpu_baseline": beam_cpu_baseline()}),
    }


def beam_cpu_baseline():
    """The oracle arm on about 10 s of steps."""
    ns = argparse.Namespace(warmup=0, steps=200, workload="beam_llama8b")
    ref = run_beam_reference(ns, 1, 0)
    return ref["cpu_baseline"]


# ----------------------------------------------------------------------------
# swap: preemption of one request by moving its blocks to pinned host memory
# and back (pa_swap_blocks)

SWAP_METRIC = "pa_swap_blocks host-link GB/s (swap-out + swap-in of one preempted request)"


def swap_shape():
    """The Llama-8B-shaped pool (32 layers, 8 KV heads, d 128, bf16, 16-token
    blocks) with the longest request of the decode batch (4096 tokens, 256
    blocks per layer) preempted."""
    return dict(layers=32, kv_heads=8, block_size=16, head_dim=128, elem=2, request_blocks=256,
                device_blocks=512)


def run_swap(args, world, rank, local):
    import paged_kv_cache_288_gb300 as pa
    from paged_kv_cache_288_gb300 import build

    build.build_library()
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    sh = swap_shape()
    L, nb, nd = sh["layers"], sh["request_blocks"], sh["device_blocks"]
    blk_elems = sh["kv_heads"] * sh["block_size"] * sh["head_dim"]
    block_bytes = blk_elems * sh["elem"]
    g = torch.Generator(device="cpu").manual_seed(rank_seed(1006, rank))
    dk = [torch.empty(nd, blk_elems, dtype=torch.bfloat16, device=device).normal_() for _ in range(L)]
    dv = [torch.empty(nd, blk_elems, dtype=torch.bfloat16, device=device).normal_() for _ in range(L)]
    hk = [torch.empty(nb, blk_elems, dtype=torch.bfloat16).pin_memory() for _ in range(L)]
    hv = [torch.empty(nb, blk_elems, dtype=torch.bfloat16).pin_memory() for _ in range(L)]
    # the request's blocks are scattered over the device pool; it comes back
    # into other free blocks
    perm = torch.randperm(nd, generator=g)
    out_map = torch.stack([perm[:nb], torch.arange(nb)], 1).to(torch.int64)
    in_map = torch.stack([torch.arange(nb), perm[nb:2 * nb]], 1).to(torch.int64)
    out_d, in_d = out_map.to(device), in_map.to(device)
    err = torch.zeros(1, dtype=torch.int32, device=device)
    stream = torch.cuda.current_stream(device)
    moved = 2 * L * nb * block_bytes  # K and V, all layers, one direction

    def swap_out():
        pa.swap_blocks(hk, hv, dk, dv, out_d, debug_err=err)

    def swap_in():
        pa.swap_blocks(dk, dv, hk, hv, in_d, debug_err=err)

    # the host link's copy-engine rate for the same number of bytes, one
    # contiguous cudaMemcpyAsync per direction: the roofline denominator
    dbuf = torch.empty(moved, dtype=torch.uint8, device=device)
    hbuf = torch.empty(moved, dtype=torch.uint8).pin_memory()
    for _ in range(args.warmup):
        swap_out()
        swap_in()
        hbuf.copy_(dbuf, non_blocking=True)
        dbuf.copy_(hbuf, non_blocking=True)
    torch.cuda.synchronize()
    K = args.steps
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(K)]
    cev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(K)]
    sampler = ClockSampler(local)
    sampler.start()
    time.sleep(0.3)
    barrier(world)
    torch.cuda.synchronize()
    n0 = pa.lib().pa_kernel_launch_count()
    t0 = time.time()
    for k in range(K):
        ev[k][0].record(stream)
        swap_out()
        ev[k][1].record(stream)
        swap_in()
        ev[k][2].record(stream)
    torch.cuda.synchronize()
    t1 = time.time()
    barrier(world)
    n1 = pa.lib().pa_kernel_launch_count()
    sampler.stop()
    for k in range(K):
        cev[k][0].record(stream)
        hbuf.copy_(dbuf, non_blocking=True)
        cev[k][1].record(stream)
        dbuf.copy_(hbuf, non_blocking=True)
        cev[k][2].record(stream)
    torch.cuda.synchronize()
    out_ms = statistics.mean(ev[k][0].elapsed_time(ev[k][1]) for k in range(K))
    in_ms = statistics.mean(ev[k][1].elapsed_time(ev[k][2]) for k in range(K))
    total_ms = max_over_ranks(sum(ev[k][0].elapsed_time(ev[k][2]) for k in range(K)), world, device)
    d2h_ms = statistics.mean(cev[k][0].elapsed_time(cev[k][1]) for k in range(K))
    h2d_ms = statistics.mean(cev[k][1].elapsed_time(cev[k][2]) for k in range(K))
    value = job_throughput_gbs(2 * moved, K, world, total_ms)
    peak = 2 * moved / ((d2h_ms + h2d_ms) / 1e3) / 1e9
    achieved = 2 * moved / ((out_ms + in_ms) / 1e3) / 1e9

    # end to end through the public API: the mapping comes from pinned host
    # memory each step and the error flag is read back
    h_out, h_in = out_map.pin_memory(), in_map.pin_memory()
    h_err = torch.zeros(1, dtype=torch.int32).pin_memory()
    Ke = min(K, 50)
    eev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(Ke)]
    torch.cuda.synchronize()
    for k in range(Ke):
        eev[k][0].record(stream)
        out_d.copy_(h_out, non_blocking=True)
        swap_out()
        in_d.copy_(h_in, non_blocking=True)
        swap_in()
        h_err.copy_(err, non_blocking=True)
        eev[k][1].record(stream)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(sum(eev[k][0].elapsed_time(eev[k][1]) for k in range(Ke)), world, device)
    assert int(h_err.item()) == 0, "swap flagged an out-of-range block"
    if rank != 0:
        return None
    line = {
        "metric": SWAP_METRIC,
        "value": round(value, 2),
        "unit": "GB/s",
        "n_gpus": world,
        "steps": K,
        "warmup": args.warmup,
        "ms_per_step": round(total_ms / K, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16 (bytes moved as is)",
        "data": "synthetic (seeded N(0,1) pools, shuffled request blocks)",
        "config": {"workload": args.workload, "layers": L, "num_kv_heads": sh["kv_heads"],
                   "block_size": sh["block_size"], "head_dim": sh["head_dim"],
                   "request_blocks": nb, "device_blocks": nd, "block_bytes": block_bytes,
                   "bytes_per_direction": moved,
                   "l2": "not flushed: each direction moves 512 MiB, four times the L2",
                   "parallelism": f"{world} independent replica(s), one per GPU"},
        "swap_out_us": round(out_ms * 1e3, 1),
        "swap_in_us": round(in_ms * 1e3, 1),
        "swap_out_gbs": round(moved / (out_ms / 1e3) / 1e9, 1),
        "swap_in_gbs": round(moved / (in_ms / 1e3) / 1e9, 1),
        "roofline": {"bound": "host_link", "achieved": round(achieved, 1), "peak": round(peak, 1),
                     "peak_source": "measured in this run: one contiguous cudaMemcpyAsync of the "
                                    "same bytes per direction over the same link",
                     "unit": "GB/s", "frac": round(achieved / peak, 4), "traffic": None,
                     "kernel": "swap_blocks_kernel",
                     "copy_engine_d2h_gbs": round(moved / (d2h_ms / 1e3) / 1e9, 1),
                     "copy_engine_h2d_gbs": round(moved / (h2d_ms / 1e3) / 1e9, 1)},
        "e2e": {"value": round(job_throughput_gbs(2 * moved, Ke, world, e2e_ms), 2), "unit": "GB/s",
                "h2d_bytes_per_step": int(out_map.numel() * 8 + in_map.numel() * 8),
                "d2h_bytes_per_step": 4, "steps": Ke},
        "clocks": sampler.summary(t0, t1),
        "gpu_launches": n1 - n0,
        "launches_per_step": (n1 - n0) / K,
    }
    if not args.no_cpu_baseline and world == 1:
        line["cpu_baseline"] = swap_cpu_baseline()
    return line


def swap_oracle_gbs(layers, blocks, reps):
    """The oracle's swap (numpy byte copies) on host arrays of the swap shape."""
    import oracle
    sh = swap_shape()
    n = sh["kv_heads"] * sh["block_size"] * sh["head_dim"]
    rng = np.random.default_rng(7)
    src = [rng.integers(0, 65535, (2 * blocks, n), dtype=np.uint16) for _ in range(2 * layers)]
    dst = [np.zeros((blocks, n), dtype=np.uint16) for _ in range(2 * layers)]
    pairs = [(2 * i + 1, i) for i in range(blocks)]
    t = time.perf_counter()
    for _ in range(reps):
        oracle.swap_blocks(dst[:layers], dst[layers:], src[:layers], src[layers:], pairs)
    dt = time.perf_counter() - t
    return 2 * layers * blocks * n * 2 * reps / dt / 1e9, dt


def swap_cpu_baseline():
    """The oracle on host arrays, repeated for about 10 s."""
    value, dt = swap_oracle_gbs(32, 256, 1)
    reps = max(1, int(10.0 / max(dt, 1e-3)))
    value, dt = swap_oracle_gbs(32, 256, reps)
    return {"value": round(value, 3), "unit": "GB/s", "cores": 1, "kind": "oracle",
            "sample": f"numpy oracle swap of the full request (32 layers x 256 blocks, K and V) "
                      f"between host arrays, {reps} repetitions, {dt:.1f} s, 1 thread"}


def run_reference(args, world, rank):
    if rank != 0:
        return None
    case = make_case(args.workload, 0)
    # at least one sequence per host core, so every core works as in cpu_baseline
    want = args.reference_seqs if args.reference_seqs > 0 else max(8, host_cores())
    seqs = max(1, min(case.num_seqs, want))
    times, cores = oracle_seconds(args.workload, seqs, args.warmup + args.steps)
    timed = times[args.warmup:]
    sub = sample_case(case, seqs)
    value = decode_bytes(sub) * len(timed) / sum(timed) / 1e9
    return {
        "impl": "reference",
        "metric": METRIC,
        "value": round(value, 5),
        "unit": "GB/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(1e3 * sum(timed) / len(timed), 3),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f64 (oracle)",
        "data": "synthetic (seeded N(0,1) K/V/q, shuffled physical blocks)",
        "config": {"workload": args.workload, "num_seqs": case.num_seqs,
                   "sample_seqs_per_step": seqs},
        "cpu_baseline": {"value": round(value, 5), "unit": "GB/s", "cores": cores, "kind": "oracle",
                         "sample": f"fp64 numpy oracle pa_decode over {seqs} of {case.num_seqs} "
                                   f"sequences per step, {cores} single-threaded processes"},
        "e2e": {"value": round(value, 5), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


def run_swap_reference(args, world, rank):
    if rank != 0:
        return None
    secs = []
    value = 0.0
    for _ in range(args.warmup + args.steps):
        v, dt = swap_oracle_gbs(32, 32, 1)
        secs.append(dt)
        value = v
    timed = secs[args.warmup:]
    sh = swap_shape()
    moved = 2 * 32 * 32 * sh["kv_heads"] * sh["block_size"] * sh["head_dim"] * sh["elem"]  # K and V
    value = moved * len(timed) / sum(timed) / 1e9
    return {
        "impl": "reference", "metric": SWAP_METRIC, "value": round(value, 3), "unit": "GB/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(1e3 * sum(timed) / len(timed), 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bytes (oracle)",
        "data": "synthetic host arrays", "config": {"workload": args.workload,
                                                    "sample_blocks_per_layer": 32},
        "cpu_baseline": {"value": round(value, 3), "unit": "GB/s", "cores": 1, "kind": "oracle",
                         "sample": "numpy oracle swap of 32 of the request's 256 blocks per layer, "
                                   "32 layers, K and V, 1 thread"},
        "e2e": {"value": round(value, 3), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=500)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="llama8b")
    ap.add_argument("--partition-size", type=int, default=0)
    ap.add_argument("--reference-seqs", type=int, default=0,
                    help="sequences per reference step (0: one per host core, at least 8)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--shared-groups", action="store_true",
                    help="shared_prefix / prefix_cache: decode with pa_decode_shared_prefix")
    ap.add_argument("--no-configs", action="store_true",
                    help="time only --workload (the llama8b line otherwise adds the other workloads)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("at least 3 warm-up steps")
    world, rank, local = setup_dist()
    swap = args.workload.startswith("swap")
    beam = args.workload.startswith("beam")
    prefill = args.workload.startswith("prefill")
    if prefill:
        line = (run_prefill_reference(args, world, rank) if args.impl == "reference"
                else run_prefill(args, world, rank, local))
    elif args.impl == "reference":
        if beam:
            line = run_beam_reference(args, world, rank)
        else:
            line = run_swap_reference(args, world, rank) if swap else run_reference(args, world, rank)
    elif beam:
        line = run_beam(args, world, rank, local)
    else:
        line = run_swap(args, world, rank, local) if swap else run_ours(args, world, rank, local)
    if line is not None:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
