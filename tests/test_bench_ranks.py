"""The bench's multi-GPU host logic on CPU, with two gloo ranks (processes):
each rank draws its own batch, the job's time is the maximum over the ranks,
the job's throughput counts both ranks' tokens, and the training step's one
exchange -- a sum of the weight gradients over the ranks -- gives the
gradients of the two batches taken together."""
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
        inp = bench.rank_inputs(synth.CONFIGS["pr1"], rank)
        x = inp["X"]
        got = bench.max_over_ranks(times[rank], world, torch.device("cpu"))
        q.put((rank, int(inp["W_inT"][:4, :4].astype(np.int64).sum()), int(x[:4, :4].astype(np.int64).sum()), got))
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
    # each rank drew its own batch of the same layer; rank 0's is the config's
    assert out[0][1] == out[1][1] and out[0][2] != out[1][2]
    assert out[0][2] == int(synth.make_ffn_inputs(synth.CONFIGS["pr1"])["X"][:4, :4].astype(np.int64).sum())
    # whole-job throughput: both ranks' tokens over the slowest time
    assert bench.job_throughput(2, 4096, 0.70) == 2 * 4096 / 0.70e-3


def _grad_rank(rank, world, port, q):
    import torch
    import torch.distributed as dist
    import oracle
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=world)
    try:
        cfg = _DP_CFG
        inp = bench.rank_inputs(cfg, rank)
        dY = synth.make_grad_output(cfg.n_rows, cfg.d_model, seed=cfg.seed + 77 + rank)
        _, H = oracle.hidden(inp["X"], inp["W_inT"], inp["b"])
        grads = [torch.from_numpy(np.ascontiguousarray(g)) for g in
                 oracle.grad_weights(inp["X"], inp["W_down"], H, dY, cfg.l1_lambda)]
        bench.allreduce_grads(grads, world)
        q.put((rank, [g.numpy() for g in grads]))
    finally:
        dist.destroy_process_group()


# a small layer: every rank holds the same weights and its own batch
_DP_CFG = synth.FFNConfig("dp", 96, 128, 512, 64, 8, seed=11, row_spread="lognormal", forced_frac_rows=0.03,
                          l1_lambda=1e-3)


def test_two_gloo_ranks_allreduce_weight_gradients():
    """Each rank's oracle gradients on its own batch, summed by the exchange,
    equal the oracle's gradients on both batches as one batch (up to fp32
    reassociation of the sums over rows)."""
    import oracle
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_grad_rank, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    out = dict(q.get(timeout=300) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    cfg = _DP_CFG
    inps = [bench.rank_inputs(cfg, r) for r in range(world)]
    for k in ("W_inT", "W_down", "b"):
        assert np.array_equal(inps[0][k], inps[1][k])
    X = np.concatenate([i["X"] for i in inps])
    dY = np.concatenate([synth.make_grad_output(cfg.n_rows, cfg.d_model, seed=cfg.seed + 77 + r)
                         for r in range(world)])
    _, H = oracle.hidden(X, inps[0]["W_inT"], inps[0]["b"])
    want = oracle.grad_weights(X, inps[0]["W_down"], H, dY, cfg.l1_lambda)
    for r in range(world):
        for g, w in zip(out[r], want):
            assert np.allclose(g, w, rtol=1e-5, atol=1e-5 * np.abs(w).max())
    assert all(np.array_equal(a, b) for a, b in zip(out[0], out[1]))   # every rank holds the same sum


def test_single_rank_passthrough():
    assert bench.max_over_ranks([1.5, 2.5], 1, None) == [1.5, 2.5]
    inp = bench.rank_inputs(synth.CONFIGS["pr1"], 0)
    assert np.array_equal(inp["X"], synth.make_ffn_inputs(synth.CONFIGS["pr1"])["X"])


def test_single_thread_oracle_line():
    """The bench's single-thread CPU figure: the oracle over the whole small
    layer in a child process limited to one OpenMP thread."""
    line = bench.cpu_single_thread_pr1()
    assert line["cores"] == 1 and line["kind"] == "oracle" and line["unit"] == bench.UNIT
    assert line["value"] > 0 and "one thread" in line["sample"]
