"""The bench's multi-GPU host logic on CPU: two gloo ranks (processes) each
draw their own batch, the job's time is the maximum over the ranks, and the
job's throughput counts both ranks' tokens.  (The GPU path itself runs one
process per GPU with no data-path collective.)"""
import multiprocessing as mp
import os
import socket

import numpy as np

import bench
import synth


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, times, q):
    import torch
    import torch.distributed as dist
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=world)
    try:
        cfg = bench.rank_config(synth.CONFIGS["pr1"], rank)
        x = synth.make_ffn_inputs(cfg)["X"]
        got = bench.max_over_ranks(times[rank], world, torch.device("cpu"))
        q.put((rank, cfg.seed, int(x[:4, :4].astype(np.int64).sum()), got))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_max_and_distinct_batches():
    world, port = 2, _free_port()
    times = [[0.50, 0.90], [0.70, 0.80]]   # per rank: step ms, end-to-end ms
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank, args=(r, world, port, times, q)) for r in range(world)]
    for p in procs:
        p.start()
    out = [q.get(timeout=120) for _ in range(world)]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    out.sort()
    # the slowest rank's time, element-wise, on every rank
    assert out[0][3] == [0.70, 0.90] and out[1][3] == [0.70, 0.90]
    # each rank drew its own batch
    assert out[0][1] != out[1][1] and out[0][2] != out[1][2]
    assert out[0][1] == synth.CONFIGS["pr1"].seed
    # whole-job throughput: both ranks' tokens over the slowest time
    assert bench.job_throughput(2, 4096, 0.70) == 2 * 4096 / 0.70e-3


def test_single_rank_passthrough():
    assert bench.max_over_ranks([1.5, 2.5], 1, None) == [1.5, 2.5]
    assert bench.rank_config(synth.CONFIGS["1b"], 0) is synth.CONFIGS["1b"]


def test_single_thread_oracle_line():
    """The bench's single-thread CPU figure: the oracle over the whole small
    layer in a child process limited to one OpenMP thread."""
    line = bench.cpu_single_thread_pr1()
    assert line["cores"] == 1 and line["kind"] == "oracle" and line["unit"] == bench.UNIT
    assert line["value"] > 0 and "one thread" in line["sample"]
