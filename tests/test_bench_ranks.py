"""The multi-rank logic of bench.py on CPU: two gloo ranks agree on the
slowest rank's time, each runs its own replica of the same workload shape,
and the whole-job throughput counts every rank's bytes."""

import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    os.environ.update(RANK=str(rank), LOCAL_RANK=str(rank), WORLD_SIZE=str(world),
                      MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    import bench
    import torch.distributed as dist

    w, r, _ = bench.setup_dist()
    assert (w, r) == (world, rank)
    assert dist.get_backend() == "gloo"
    local_ms = 10.0 + 5.0 * rank
    worst = bench.max_over_ranks(local_ms, w, "cpu")
    bench.barrier(w)
    q.put((rank, worst, bench.rank_seed(1002, rank)))
    dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_time():
    pytest.importorskip("torch.distributed")
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(2))
    assert [g[1] for g in got] == [15.0, 15.0]
    assert got[0][2] != got[1][2]  # different seeds, same shape


def test_job_throughput_counts_every_rank():
    import bench

    one = bench.job_throughput_gbs(1e9, 10, 1, 1000.0)
    two = bench.job_throughput_gbs(1e9, 10, 2, 1000.0)
    assert one == pytest.approx(10.0) and two == pytest.approx(20.0)


def test_replica_workloads_share_shape():
    import workloads
    import bench

    a = workloads.llama8b_lengths(bench.rank_seed(1002, 0), num_seqs=8)
    b = workloads.llama8b_lengths(bench.rank_seed(1002, 1), num_seqs=8)
    assert a.shape == b.shape and not (a == b).all()


def test_oracle_timing_spreads_sequences_over_processes():
    """The host oracle baseline runs one single-threaded process per worker,
    never more workers than sequences, and reports one time per repetition."""
    import bench
    times, workers = bench.oracle_seconds("tiny", 4, 2, workers=2)
    assert workers == 2 and len(times) == 2 and all(t > 0 for t in times)
    times, workers = bench.oracle_seconds("tiny", 1, 1, workers=4)
    assert workers == 1 and len(times) == 1


def test_unique_bytes_count_shared_blocks_once():
    """Two sequences sharing their first block: the logical bytes count it
    twice, the unique bytes once; a private tail block counts its used
    tokens only."""
    import numpy as np
    import bench
    import workloads

    case = workloads.paged_case(5, [20, 20], 4, 2, 8, 16, workloads.F16)
    per_tok = case.num_kv_heads * 2 * case.head_dim * 2
    case.block_tables[1, 0] = case.block_tables[0, 0]
    fixed = 2 * 2 * 4 * 8 * 2 + 4 * 4 + 2 * 4  # q + out, 4 table entries, 2 lengths
    assert bench.decode_bytes(case) == 40 * per_tok + fixed
    assert bench.unique_decode_bytes(case) == (16 + 4 + 4) * per_tok + fixed
    del np
