#!/usr/bin/env python3
"""Throughput of the TwELL activation-sparse FFN layer on one GB300.

One step = the whole layer: twell_ffn_fwd (tensor-core up-projection with the
fused bias/ReLU/TwELL-pack epilogue, hybrid routing, dense fallback rows on the
tensor cores, gather-SpMM down-projection) followed by twell_ffn_bwd (SDDMM
with the L1 term, dX gather, unit-major weight gradients), on the 1B-model FFN
shape N=4096, d_model=2048, d_ff=8192, T=128, C=8 with synthetic seeded inputs.

With N GPUs (torchrun, one rank per GPU; `--gpus N` starts the ranks itself)
every rank holds the same layer and runs its own batch of the same shape (weak
scaling); the step ends with the data-parallel exchange, an all-reduce (sum)
of dW_in^T, dW_down and db.  The job's time per step is the slowest rank's
and `value` counts the tokens of all ranks.

Prints one JSON line.  `value` is tokens/s of the step with inputs resident in
HBM (L2 flushed between steps by writing a 2x-L2 buffer); `e2e` is the same
step through the same C-ABI calls with X and dY copied in from pinned host
memory and Y and dX copied back inside the timed region.  `--impl reference`
times the CPU oracle on a bounded sample of the same workload instead.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "sparse-FFN tokens/s (TwELL fwd/bwd, 99% sparse) + % of HBM/tensor roofline"
UNIT = "tokens/s"
PEAKS_FALLBACK = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def workload_name(cfg) -> str:
    """The bench line's workload: what the step is, with its sizes and input recipe."""
    rows = "lognormal row activity (mean 1%)" if cfg.row_spread == "lognormal" else "uniform row activity"
    forced = (f", {round(100 * cfg.forced_frac_rows)}% rows at {round(100 * cfg.forced_activity)}%"
              if cfg.forced_frac_rows else "")
    lam = f", lambda {cfg.l1_lambda:g}" if cfg.l1_lambda else ""
    return (f"{'1B-scale' if cfg.name == '1b' else cfg.name} FFN fwd+bwd: N={cfg.n_rows} d_model={cfg.d_model} "
            f"d_ff={cfg.d_ff} T={cfg.tile} C={cfg.cap}, {rows}{forced}{lam}")


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as fh:
            d = json.load(fh)
        return d, "measured"
    return dict(PEAKS_FALLBACK), "fallback"


def rank_inputs(cfg, rank: int) -> dict:
    """Weak scaling: every rank holds the same layer (the configuration's
    weights and bias) and its own batch of the same shape (batch seed shifted
    by 1000 x rank); rank 0 keeps the configuration's own batch."""
    import synth
    return synth.make_ffn_inputs(cfg) if rank == 0 else synth.make_ffn_inputs(cfg, batch_seed=cfg.seed + 1000 * rank)


def max_over_ranks(values, world: int, device):
    """Element-wise maximum over the ranks: the slowest rank sets the job's time."""
    if world <= 1:
        return [float(v) for v in values]
    import torch
    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return [float(x) for x in t]


def job_throughput(world: int, n_rows: int, ms: float) -> float:
    """Tokens per second of the whole job: every rank's batch, the slowest rank's time."""
    return world * n_rows / (ms * 1e-3)


def dist_info():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def allreduce_grads(grads, world: int) -> None:
    """The data-parallel exchange of a training step: every rank's weight
    gradients (dW_in^T, dW_down, db) summed over the ranks, in place.  Each
    rank's batch is its own, so the sum is the gradient of the whole job's
    batch."""
    if world <= 1:
        return
    import torch
    for g in grads:
        torch.distributed.all_reduce(g, op=torch.distributed.ReduceOp.SUM)


def relaunch_with_ranks(n: int) -> int:
    """`bench.py --gpus N` outside torchrun: start N ranks on this node (one per
    GPU) through torch.distributed.run and return its exit status."""
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", f"--nproc-per-node={n}",
           "--master-addr", "127.0.0.1", "--master-port", os.environ.get("MASTER_PORT", "29533"),
           os.path.abspath(__file__)] + sys.argv[1:]
    return subprocess.call(cmd, env=dict(os.environ, TWELL_BENCH_CHILD="1"))


class ClockSampler:
    """nvidia-smi clocks and throttle reasons of one GPU sampled every 50 ms."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "50"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        if self.thread:
            self.thread.join(timeout=2)
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for name, val in zip(names, parts[5:9]):
                if val.lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "sm_mhz_min": min(sm) if sm else None, "reasons": sorted(reasons), "samples": len(sm)}


class EnergyCounter:
    """The GPU's cumulative energy counter (NVML total energy consumption, mJ),
    read through the NVML C library.  Read-only: nothing on the GPU is set."""

    def __init__(self, device_index: int):
        import ctypes
        self.ok = False
        try:
            self.nvml = ctypes.CDLL("libnvidia-ml.so.1")
        except OSError:
            return
        if self.nvml.nvmlInit_v2() != 0:
            return
        self.handle = ctypes.c_void_p()
        uuid = None
        try:
            import torch
            uuid = str(torch.cuda.get_device_properties(device_index).uuid)
        except Exception:
            uuid = None
        rc = -1
        if uuid:
            rc = self.nvml.nvmlDeviceGetHandleByUUID(("GPU-" + uuid if not uuid.startswith("GPU-") else uuid).encode(),
                                                     ctypes.byref(self.handle))
        if rc != 0:
            rc = self.nvml.nvmlDeviceGetHandleByIndex_v2(ctypes.c_uint(device_index), ctypes.byref(self.handle))
        self.ok = rc == 0 and self.read_mj() is not None

    def read_mj(self):
        import ctypes
        v = ctypes.c_ulonglong(0)
        if self.nvml.nvmlDeviceGetTotalEnergyConsumption(self.handle, ctypes.byref(v)) != 0:
            return None
        return int(v.value)


def kernel_work(N, d, f, T, C, nnz_tw, n_fb):
    """Algorithmic work of one launch (group) of each kernel of the step at one
    layer shape: FLOPs for the tensor-core products; for the rest the bytes a
    kernel must move through HBM at least (every input read once, every output
    written once), and beside them the bytes its gathers pull from L2 (one
    d_model-wide bf16 row per stored entry and gathered matrix)."""
    nt = f // T
    cells = N * nt
    packed = cells * C * 2 + cells * C + cells          # values, idx, counts
    fb_rows = n_fb * f * 2
    row = d * 2                                          # one gathered bf16 row
    return {
        "up_pack": {"bound": "tensor", "flops": 2.0 * N * d * f, "bytes": N * d * 2 + f * d * 2 + packed,
                    "what": "tcgen05 up-projection + bias/ReLU/TwELL-pack epilogue"},
        "spmm": {"bound": "hbm", "bytes": packed + f * d * 2 + N * d * 2, "l2_gather_bytes": nnz_tw * row,
                 "what": "standalone TwELL gather-SpMM (Y)"},
        "fb_down": {"bound": "tensor", "flops": 2.0 * n_fb * d * f,
                    "what": "dense fallback rows' down-projection (split-K tcgen05) + ordered reduction"},
        "sddmm": {"bound": "tensor", "flops": 2.0 * N * d * f,
                  "what": "tcgen05 dY.W_down^T with the pattern-sampling + L1 epilogue"},
        "dx": {"bound": "hbm", "bytes": cells * C * 4 + cells * C + cells + f * d * 2 + N * d * 2,
               "l2_gather_bytes": nnz_tw * row,
               "what": "dX gather of the TwELL rows (fp32 dZ entries x W_in^T rows)"},
        # the lists hold per entry its row (int32), h (bf16 bits) and dZ (fp32)
        "dw": {"bound": "hbm", "bytes": 2 * N * d * 2 + 2 * f * d * 4 + nnz_tw * 10 + f * 4,
               "l2_gather_bytes": 2 * nnz_tw * row,
               "what": "unit-major walk: the TwELL rows' dW_down, dW_in^T (fp32, added to the fallback share "
                       "stored before it) and db"},
        "dw_fallback": {"bound": "tensor", "flops": 2.0 * 3 * n_fb * d * f,
                        "what": "the fallback rows' dW_down and dW_in^T (store GEMMs; dZ as two bf16 parts) "
                                "and db, on the second stream"},
        "dx_fallback": {"bound": "tensor", "flops": 2.0 * 2 * n_fb * d * f,
                        "what": "the fallback rows' dX (split-K GEMM over the two bf16 parts of dZ) and its "
                                "ordered reduction, on the second stream"},
        "pack": {"bound": "hbm", "bytes": N * f * 2 + packed + N * 4 + fb_rows,
                 "what": "standalone dense -> TwELL (twell_pack)"},
        "unpack": {"bound": "hbm", "bytes": packed + N * 4 + fb_rows + N * f * 2,
                   "what": "standalone TwELL -> dense (twell_unpack)"},
    }


def roofline_entry(work, us, peaks, peak_src):
    """achieved / peak of one kernel group from its algorithmic work per step
    (or per call) and its CUDA-event time per step (the sum of its launches)."""
    sec = us * 1e-6
    if work["bound"] == "tensor":
        ach = work["flops"] / sec / 1e12
        e = {"bound": "tensor", "achieved": round(ach, 1), "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
             "frac": round(ach / peaks["bf16_tflops"], 4),
             "frac_of_sustained": round(ach / peaks.get("bf16_tflops_sustained", peaks["bf16_tflops"]), 4),
             "algorithmic_per_step": work["flops"], "us_per_step": round(us, 2),
             "peak_source": f"{peak_src} bf16 dense (cuBLAS burst; frac_of_sustained against the sustained loop)"}
    else:
        ach = work["bytes"] / sec / 1e9
        e = {"bound": "hbm", "achieved": round(ach, 1), "peak": peaks["hbm_gbs"], "unit": "GB/s",
             "frac": round(ach / peaks["hbm_gbs"], 4), "algorithmic_per_step": work["bytes"],
             "us_per_step": round(us, 2), "peak_source": f"{peak_src} HBM copy bandwidth"}
    if "l2_gather_bytes" in work:
        e["l2_gather_bytes"] = work["l2_gather_bytes"]
        e["l2_gather_tbs"] = round(work["l2_gather_bytes"] / sec / 1e12, 2)
    e["kernel"] = work["what"]
    return e


def _code_lines(text: str):
    """The lines of a C/CUDA source with // comments and blank lines left out
    (a // inside a string literal is kept)."""
    for line in text.splitlines():
        out, in_str, i = [], False, 0
        while i < len(line):
            ch = line[i]
            if ch == '"' and (i == 0 or line[i - 1] != "\\"):
                in_str = not in_str
            elif not in_str and line.startswith("//", i):
                break
            out.append(ch)
            i += 1
        code = "".join(out).rstrip()
        if code:
            yield code


def source_digest(name: str) -> str:
    """First 16 hex digits of the sha256 of a kernel source file's code
    (csrc/<name>, comments and blank lines left out), so that a capture stays
    tied to the code it measured across edits of the comments."""
    import hashlib
    with open(os.path.join(ROOT, "activation_sparse_transformer_gb300", "csrc", name)) as fh:
        code = "\n".join(_code_lines(fh.read()))
    return hashlib.sha256(code.encode()).hexdigest()[:16]


def ncu_traffic(kernel: str, workload: str):
    """DRAM bytes per launch of a kernel recorded by an ncu capture
    (profiles/ncu_traffic.txt: kernel, workload, source file, its digest at the
    capture, bytes, the summary that shows the capture), or None with a note
    when the kernel's source has changed since."""
    path = os.path.join(ROOT, "profiles", "ncu_traffic.txt")
    if not os.path.exists(path):
        return None, None
    with open(path) as fh:
        for line in fh:
            parts = line.split()
            if len(parts) >= 6 and parts[0] == kernel and parts[1] == workload:
                if source_digest(parts[2]) == parts[3]:
                    return float(parts[4]), parts[5]
                return None, "stale: kernel changed since the capture"
    return None, None


def bench_ours(args, rank, world, local):
    import numpy as np
    import torch

    import activation_sparse_transformer_gb300 as tw
    import synth

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    tw.load_library()
    cfg = synth.CONFIGS[args.config]
    # every rank draws its own batch (weak scaling: per-GPU work is fixed)
    base = rank_inputs(cfg, rank)
    N, d, f, T, C, fb = cfg.n_rows, cfg.d_model, cfg.d_ff, cfg.tile, cfg.cap, cfg.fallback_capacity
    lam = cfg.l1_lambda or 1e-4
    dY_np = synth.make_grad_output(N, d, seed=cfg.seed + 77 + rank)

    def dt(a):
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(dev).view(torch.bfloat16)

    X, Wi, b, Wd, dY = dt(base["X"]), dt(base["W_inT"]), dt(base["b"]), dt(base["W_down"]), dt(dY_np)
    packed = tw.alloc_packed(N, f, T, C, fb, dev)
    Y = torch.empty((N, d), dtype=torch.bfloat16, device=dev)
    dX = torch.empty((N, d), dtype=torch.bfloat16, device=dev)
    dWi = torch.empty((f, d), dtype=torch.float32, device=dev)
    dWd = torch.empty((f, d), dtype=torch.float32, device=dev)
    db = torch.empty((f,), dtype=torch.float32, device=dev)
    # one workspace serves the forward and the backward (nothing in the
    # forward's outlives its call)
    ws_bytes = max(tw.fwd_workspace_bytes(N, d, f, T, C, fb), tw.bwd_workspace_bytes(N, d, f, T, C, fb))
    wsf = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
    wsb = wsf
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    flush = torch.empty(max(2 * l2, 256 << 20), dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)

    def fwd():
        tw.twell_ffn_fwd(X, Wi, b, Wd, packed, Y, wsf, stream)

    def exchange():
        # data-parallel training: the one exchange of the step
        allreduce_grads((dWi, dWd, db), world)

    def step():
        fwd()
        tw.twell_ffn_bwd(X, Wi, Wd, packed, dY, lam, dX, dWi, dWd, db, wsb, stream)
        exchange()

    # correctness of the routing on this batch (status word, fallback count)
    step()
    rc = tw.twell_read_status(packed, stream)
    if rc != 0:
        raise RuntimeError(f"layer status {rc}: {tw.status_string(rc)}")
    n_fb = int(packed.n_fb[0].item())
    counts = packed.counts.to(torch.int32)
    nnz_tw = int(counts.sum().item())
    nnz_fb = int((packed.fb_dense[:n_fb].view(torch.int16) & 0x7FFF).ne(0).sum().item()) if n_fb else 0
    density = (nnz_tw + nnz_fb) / float(N * f)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()

    if args.timeline:
        timelines = []
        for _ in range(3):
            flush.zero_()
            torch.cuda.synchronize()
            tw.twell_profile_reset()
            tw.twell_profile_enable(True)
            step()
            tw.twell_profile_enable(False)
            timelines.append(tw.twell_profile_timeline())
            tw.twell_profile_reset()
        main_stream = int(stream.cuda_stream)
        for tl in timelines:
            for e in tl:
                e["stream"] = "main" if e["stream"] == main_stream else "second"
                e["start_ms"] = round(e["start_ms"], 4)
                e["end_ms"] = round(e["end_ms"], 4)
        return {"timeline": timelines, "config": {"workload": workload_name(cfg), "n_rows": N},
                "note": "one fwd + bwd step, three times; times relative to each step's first launch"}

    def timed(fn, k, profile=False, warm=False):
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(k)]
        if profile:
            tw.twell_profile_reset()
            tw.twell_profile_enable(True)
        for i in range(k):
            if not warm:
                flush.zero_()
            ev[i][0].record(stream)
            fn()
            ev[i][1].record(stream)
        torch.cuda.synchronize()
        if profile:
            tw.twell_profile_enable(False)
        return [a.elapsed_time(bb) for a, bb in ev]

    def med(v):
        return statistics.median(v)

    # ---- the timed region: K steps, L2 scrubbed between steps, CUDA events on
    # the launching stream.  The K-step loop is repeated until the region spans
    # at least --min-window seconds, so the clock record covers the timed work;
    # the reported time is the median over repeats of each repeat's median step.
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    clocks = ClockSampler(local)
    clocks.start()
    launches0 = tw.twell_launch_count()
    t_wall = time.perf_counter()
    rep_ms, reps = [], 0
    while True:
        rep_ms.append(med(timed(step, args.steps)))
        reps += 1
        if time.perf_counter() - t_wall >= args.min_window or reps >= 1000:
            break
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    wall = time.perf_counter() - t_wall
    launches = (tw.twell_launch_count() - launches0) // reps
    clk = clocks.stop()

    # per-kernel breakdown from a separate pass with an event pair around every
    # launch (kept out of the timed steps above); a kernel group may launch
    # several kernels per step, so its time per step is the sum of its launches
    prof_steps = min(args.steps, 20)
    timed(step, prof_steps, profile=True)
    per_kernel = {}
    for name in tw.KERNELS:
        n, ms = tw.twell_profile_read(name)
        if n:
            per_kernel[name] = {"launches_per_step": round(n / prof_steps, 2), "avg_us": 1000.0 * ms / n,
                                "us_per_step": 1000.0 * ms / prof_steps, "share": 0.0}
    tot = sum(v["us_per_step"] for v in per_kernel.values()) or 1.0
    for v in per_kernel.values():
        v["share"] = round(v["us_per_step"] / tot, 4)
        v["avg_us"] = round(v["avg_us"], 2)
        v["us_per_step"] = round(v["us_per_step"], 2)

    # forward alone (the layer's inference path) and the dense comparator
    fwd_ms = timed(fwd, max(args.steps, 50))
    tw.twell_profile_reset()
    tw.twell_profile_enable(True)
    timed(fwd, prof_steps)
    tw.twell_profile_enable(False)
    fwd_kernels = {}
    for name in tw.KERNELS:
        n, ms = tw.twell_profile_read(name)
        if n:
            fwd_kernels[name] = {"launches_per_call": round(n / prof_steps, 2),
                                 "us_per_call": round(1000.0 * ms / prof_steps, 2)}
    # the same calls back to back without the L2 scrub (warm L2: the weights stay resident)
    warm_step_ms = timed(step, min(args.steps, 50), warm=True)
    warm_fwd_ms = timed(fwd, min(args.steps, 50), warm=True)
    # the same fwd + bwd calls captured once in a CUDA graph and replayed: the
    # same kernels on the same buffers, without the host launch path between them
    graph_step_ms = None
    if world == 1:
        graph = torch.cuda.CUDAGraph()
        torch.cuda.synchronize()
        with torch.cuda.graph(graph):
            cap = torch.cuda.current_stream(dev)
            tw.twell_ffn_fwd(X, Wi, b, Wd, packed, Y, wsf, cap)
            tw.twell_ffn_bwd(X, Wi, Wd, packed, dY, lam, dX, dWi, dWd, db, wsb, cap)
        for _ in range(3):
            graph.replay()
        torch.cuda.synchronize()
        graph_step_ms = timed(graph.replay, args.steps)
        del graph
    Hbuf = torch.empty((N, f), dtype=torch.bfloat16, device=dev)

    def dense():
        tw.twell_dense_ffn_fwd(X, Wi, b, Wd, Hbuf, Y, stream)

    dense()
    dense_ms = timed(dense, max(3, args.steps // 2))

    # ---- the standalone format conversions on the dense H of this layer
    # (67 MB at the 1B shape): TwELL -> dense, then dense -> TwELL
    packed2 = tw.alloc_packed(N, f, T, C, fb, dev)
    tw.twell_unpack(packed, Hbuf, stream)
    tw.twell_pack(Hbuf, packed2, stream)
    torch.cuda.synchronize()
    conv = {}
    for name, fn in (("unpack", lambda: tw.twell_unpack(packed, Hbuf, stream)),
                     ("pack", lambda: tw.twell_pack(Hbuf, packed2, stream))):
        ms_list = timed(fn, max(args.steps, 20))
        tw.twell_profile_reset()
        tw.twell_profile_enable(True)
        timed(fn, prof_steps)
        tw.twell_profile_enable(False)
        n_l, k_ms = tw.twell_profile_read(name)
        conv[name] = {"call_ms": round(med(ms_list), 4), "kernel_us_per_call": round(1000.0 * k_ms / prof_steps, 2),
                      "launches_per_call": round(n_l / prof_steps, 2)}
    same = all(torch.equal(getattr(packed, k), getattr(packed2, k)) for k in ("values", "idx", "counts"))
    # plain torch streams over the same bytes as dense H, under the same scrub:
    # on this GPU a write-only stream runs at about half the copy bandwidth, so
    # unpack (67 MB written) is compared with a fill and pack (67 MB read) with
    # a reduction
    red = torch.empty((), dtype=torch.float32, device=dev)
    hwords = Hbuf.view(-1).view(torch.float32)  # finite: pairs of non-negative finite bf16
    stream_ref = {"write_stream_us": round(1000.0 * med(timed(lambda: Hbuf.zero_(), max(args.steps, 20))), 2),
                  "read_stream_us": round(1000.0 * med(timed(lambda: torch.amax(hwords, dim=0, out=red),
                                                             max(args.steps, 20))), 2),
                  "bytes": int(Hbuf.numel() * Hbuf.element_size())}
    conv["unpack"]["vs_write_stream"] = round(stream_ref["write_stream_us"] / conv["unpack"]["kernel_us_per_call"], 3)
    conv["pack"]["vs_read_stream"] = round(stream_ref["read_stream_us"] / conv["pack"]["kernel_us_per_call"], 3)
    del packed2, Hbuf

    # ---- energy per token: the GPU's cumulative energy counter (NVML, mJ)
    # differenced over a back-to-back loop of >= 2 s of each call, after a
    # warm-up loop of ~0.5 s so the power has settled (warm L2, no scrub
    # writes, so the scrub's own energy is not counted)
    energy_out = None
    if not args.no_energy:
        meter = EnergyCounter(local)

        def energy(fn, ms_each, tokens):
            if not meter.ok:
                return None
            warm_iters = max(20, int(500.0 / max(ms_each, 1e-3)))
            iters = max(50, int(2000.0 / max(ms_each, 1e-3)))
            for _ in range(warm_iters):
                fn()
            torch.cuda.synchronize()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            j0 = meter.read_mj()
            e0.record(stream)
            for _ in range(iters):
                fn()
            e1.record(stream)
            torch.cuda.synchronize()
            j1 = meter.read_mj()
            loop_ms = e0.elapsed_time(e1)
            joules = (j1 - j0) * 1e-3
            return {"j_per_token": joules / (iters * tokens), "avg_power_w": round(joules / (loop_ms * 1e-3), 1),
                    "ms_per_call": round(loop_ms / iters, 4), "loop_s": round(loop_ms * 1e-3, 2)}

        Hbuf = torch.empty((N, f), dtype=torch.bfloat16, device=dev)
        energy_out = {"fwd_bwd_step": [energy(step, med(rep_ms), N) for _ in range(2)],
                      "fwd": [energy(fwd, med(fwd_ms), N) for _ in range(2)],
                      "dense_fwd": [energy(dense, med(dense_ms), N) for _ in range(2)],
                      "how": "NVML total-energy counter of this GPU differenced over a >= 2 s back-to-back loop "
                             "after a ~0.5 s warm-up loop (warm L2), / tokens; each measured twice; the GPU "
                             "sits in a shared machine" if meter.ok else "NVML energy counter unavailable"}
        del Hbuf

    # end to end through the C ABI with host buffers (pinned): every step
    # uploads its X and dY and downloads its Y and dX inside the timed loop.
    # The copies run on their own streams, one step ahead / behind the
    # compute (double buffering as a training loop would), over 4 rotating
    # device buffer sets (134 MB of inputs > L2).
    hX = torch.from_numpy(base["X"].view(np.int16)).view(torch.bfloat16).pin_memory()
    hdY = torch.from_numpy(dY_np.view(np.int16)).view(torch.bfloat16).pin_memory()
    hY = torch.empty((N, d), dtype=torch.bfloat16).pin_memory()
    hdX = torch.empty((N, d), dtype=torch.bfloat16).pin_memory()
    SETS = 4
    bufs = [dict(X=torch.empty_like(X), dY=torch.empty_like(dY), Y=torch.empty_like(Y), dX=torch.empty_like(dX))
            for _ in range(SETS)]
    up_s, down_s = torch.cuda.Stream(dev), torch.cuda.Stream(dev)

    def e2e_loop(k):
        ev_up = [torch.cuda.Event() for _ in range(SETS)]
        ev_done = [torch.cuda.Event() for _ in range(SETS)]
        used = [False] * SETS
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        t0.record(stream)
        up_s.wait_event(t0)
        down_s.wait_event(t0)

        def upload(i):
            bs = bufs[i % SETS]
            with torch.cuda.stream(up_s):
                if used[i % SETS]:
                    up_s.wait_event(ev_done[i % SETS])   # step i - SETS is done with this set
                bs["X"].copy_(hX, non_blocking=True)
                bs["dY"].copy_(hdY, non_blocking=True)
                ev_up[i % SETS].record(up_s)

        upload(0)
        for i in range(k):
            if i + 1 < k:
                upload(i + 1)
            bs = bufs[i % SETS]
            stream.wait_event(ev_up[i % SETS])
            tw.twell_ffn_fwd(bs["X"], Wi, b, Wd, packed, bs["Y"], wsf, stream)
            tw.twell_ffn_bwd(bs["X"], Wi, Wd, packed, bs["dY"], lam, bs["dX"], dWi, dWd, db, wsb, stream)
            exchange()
            ev_done[i % SETS].record(stream)
            used[i % SETS] = True
            with torch.cuda.stream(down_s):
                down_s.wait_event(ev_done[i % SETS])
                hY.copy_(bs["Y"], non_blocking=True)
                hdX.copy_(bs["dX"], non_blocking=True)
        stream.wait_stream(down_s)
        stream.wait_stream(up_s)
        t1.record(stream)
        torch.cuda.synchronize()
        return t0.elapsed_time(t1) / k

    e2e_loop(max(3, args.warmup))
    e2e_m_loop = e2e_loop(args.steps)
    h2d = hX.numel() * 2 + hdY.numel() * 2
    d2h = hY.numel() * 2 + hdX.numel() * 2

    ms, e2e_m = max_over_ranks([med(rep_ms), e2e_m_loop], world, dev)
    del bufs, hX, hdY, hY, hdX

    # ---- rooflines: every kernel group against its own bound; the dominant
    # one (the largest share of the step's kernel time) is the headline's
    peaks, peak_src = load_peaks()
    work = kernel_work(N, d, f, T, C, nnz_tw, n_fb)
    roofs = {}
    for name, v in per_kernel.items():
        if name in work:
            roofs[name] = roofline_entry(work[name], v["us_per_step"], peaks, peak_src)
            roofs[name]["share_of_step"] = v["share"]
    for name in ("pack", "unpack"):
        roofs[name] = roofline_entry(work[name], conv[name]["kernel_us_per_call"], peaks, peak_src)
    dominant = max((k for k in roofs if k in per_kernel), key=lambda k: per_kernel[k]["share"], default=None)
    roof = dict(roofs[dominant]) if dominant else None
    for name, r in roofs.items():
        traffic, note = ncu_traffic(name, args.config)
        r["traffic"] = traffic
        if note:
            r["traffic_note"] = note
    if roof is not None:
        roof["name"] = dominant
        roof["traffic"] = roofs[dominant]["traffic"]
        if "traffic_note" in roofs[dominant]:
            roof["traffic_note"] = roofs[dominant]["traffic_note"]
    fwd_m = med(fwd_ms)
    packed_bytes = (packed.values.numel() * 2 + packed.idx.numel() + packed.counts.numel() + packed.row_fb.numel() * 4
                    + packed.fb_rows.numel() * 4 + packed.fb_dense.numel() * 2)
    roof_fwd_us = max(2.0 * N * d * f / (peaks["bf16_tflops"] * 1e12),
                      (N * d * 2 * 2 + f * d * 2 * 2 + N * (f // T) * (3 * C + 1)) / (peaks["hbm_gbs"] * 1e9)) * 1e6
    sm_mhz = clk.get("sm_mhz")
    clk["time_x_median_mhz"] = round(ms * sm_mhz, 1) if sm_mhz else None
    result = {
        "metric": METRIC, "value": round(job_throughput(world, N, ms), 1), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic (seeded, see synth/)",
        "config": {"workload": workload_name(cfg), "n_rows": N, "d_model": d, "d_ff": f, "tile": T, "cap": C,
                   "fb_cap": fb, "l1_lambda": lam, "l2": "flushed between steps (2x L2 write)",
                   "parallelism": (f"data parallel x{world}: each rank its own batch, weight gradients "
                                   "all-reduced (NCCL sum) inside the step") if world > 1 else "single GPU"},
        "timed_repeats": {"repeats": reps, "steps_each": args.steps,
                          "rep_ms_min": round(min(rep_ms), 4), "rep_ms_max": round(max(rep_ms), 4),
                          "note": "the K-step timed loop repeated until the timed window spans >= "
                                  f"{args.min_window} s; ms_per_step is the median over repeats"},
        "roofline": roof,
        "roofline_kernels": roofs,
        "fwd": {"tokens_per_s": round(world * N / (fwd_m * 1e-3), 1), "ms": round(fwd_m, 4),
                "roofline_us": round(roof_fwd_us, 2), "roofline_frac": round(roof_fwd_us / (fwd_m * 1e3), 4),
                "kernels": fwd_kernels,
                "roofline_note": "max(up-projection FLOPs at the measured bf16 burst peak, X + W_in^T + W_down + "
                                 "packed H + Y bytes at the measured HBM peak)"},
        "graph": ({"ms_per_step": round(med(graph_step_ms), 4),
                   "tokens_per_s": round(job_throughput(world, N, med(graph_step_ms)), 1),
                   "note": "the same fwd + bwd calls captured once in a CUDA graph and replayed, L2 flushed "
                           "between replays"} if graph_step_ms else None),
        "warm_l2": {"ms_per_step": round(med(warm_step_ms), 4), "fwd_ms": round(med(warm_fwd_ms), 4),
                    "tokens_per_s": round(job_throughput(world, N, med(warm_step_ms)), 1),
                    "note": "no L2 scrub between calls; the headline value scrubs L2 (cold)"},
        "dense_ffn_fwd": {"tokens_per_s": round(world * N / (med(dense_ms) * 1e-3), 1), "ms": round(med(dense_ms), 4),
                          "note": "same tcgen05 GEMM, no sparsity: reported baseline"},
        "format_conversion": {**conv, "round_trip_identical": bool(same), "torch_streams": {
            **stream_ref, "how": "torch fill (Hbuf.zero_) and fp32 max-reduction over a dense-H-sized buffer, L2 "
                                 "scrubbed before each; vs_*_stream = that stream's time / the conversion's kernel "
                                 "time"},
                              "note": "twell_unpack of this layer's packed H into dense bf16 [N, d_ff], then "
                                      "twell_pack of that dense H; L2 scrubbed between calls"},
        "kernels": per_kernel,
        "layer": {"n_fb": n_fb, "density": round(density, 5), "sparsity": round(1 - density, 5),
                  "twell_entries": nnz_tw,
                  "packed_h_bytes": int(packed.values.numel() * 2 + packed.idx.numel() + packed.counts.numel()
                                        + fb * f * 2),
                  "dense_h_bytes": N * f * 2},
        "e2e": {"value": round(job_throughput(world, N, e2e_m), 1), "unit": UNIT, "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": round(e2e_m, 4),
                "how": "through the C ABI; each step uploads X, dY from pinned host memory and downloads Y, "
                       "dX, on two copy streams one step ahead / behind the compute; 4 rotating device buffer "
                       "sets (134 MB of inputs, more than L2); one event pair around all K steps"},
        "gpu_launches": int(launches),
        "clocks": clk,
        "timed_wall_s": round(wall, 3),
        "energy": energy_out,
    }
    if world == 1 and not args.no_memory:
        result["train_memory"] = bench_train_memory(tw, dev, args)
        result["gated_train"] = bench_gated_train(tw, dev, args)
    return result


def bench_gated_train(tw, dev, args):
    """One training step of the gated layer (twell_gated_ffn_fwd_train, then
    twell_gated_ffn_bwd) at its training shape: median time with L2 scrubbed
    before each step, the per-kernel device times, the allocator's peak over a
    step (inputs, weights and dY allocated before and not counted), and the
    tensor-core floor of the GEMM work the step does densely."""
    import numpy as np
    import torch

    import synth
    cfg = synth.CONFIGS["gated_train"]
    inp = synth.make_ffn_inputs(cfg)
    N, d, f, T, C, fb = cfg.n_rows, cfg.d_model, cfg.d_ff, cfg.tile, cfg.cap, cfg.fallback_capacity
    lam = cfg.l1_lambda
    peaks, peak_src = load_peaks()

    def dt(a):
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(dev).view(torch.bfloat16)

    X, Wg, Wu, b, Wd = (dt(inp[k]) for k in ("X", "W_inT", "W_uT", "b", "W_down"))
    dY = dt(synth.make_grad_output(N, d, seed=cfg.seed + 77))
    flush = torch.empty(max(2 * torch.cuda.get_device_properties(dev).L2_cache_size, 256 << 20),
                        dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    base = torch.cuda.memory_allocated(dev)
    torch.cuda.reset_peak_memory_stats(dev)
    packed = tw.alloc_packed(N, f, T, C, fb, dev)
    gu = torch.empty((N, f // T, C, 2), dtype=torch.float32, device=dev)
    Y = torch.empty((N, d), dtype=torch.bfloat16, device=dev)
    dX = torch.empty((N, d), dtype=torch.bfloat16, device=dev)
    dW = [torch.empty((f, d), dtype=torch.float32, device=dev) for _ in range(3)]
    db = torch.empty((f,), dtype=torch.float32, device=dev)
    ws = torch.empty(max(tw.fwd_workspace_bytes(N, d, f, T, C, fb), tw.gated_bwd_workspace_bytes(N, d, f, T, C, fb)),
                     dtype=torch.uint8, device=dev)

    def step():
        tw.twell_gated_ffn_fwd_train(X, Wg, Wu, b, Wd, packed, Y, gu, ws, stream)
        tw.twell_gated_ffn_bwd(X, Wg, Wu, b, Wd, packed, gu, dY, lam, dX, dW[0], dW[1], dW[2], db, ws, stream)

    step()
    torch.cuda.synchronize()
    peak = torch.cuda.max_memory_allocated(dev) - base
    rc = tw.twell_read_status(packed, stream)
    if rc != 0:
        raise RuntimeError(f"gated training step: status {rc}")
    n_fb = int(packed.n_fb[0].item())
    nnz = int(packed.counts.to(torch.int64).sum().item())
    for _ in range(args.warmup):
        step()
    k = max(10, min(args.steps, 100))
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(k)]
    for e0, e1 in ev:
        flush.zero_()
        e0.record(stream)
        step()
        e1.record(stream)
    torch.cuda.synchronize()
    ms = statistics.median(a.elapsed_time(bb) for a, bb in ev)
    tw.twell_profile_reset()
    tw.twell_profile_enable(True)
    for _ in range(10):
        flush.zero_()
        step()
    torch.cuda.synchronize()
    tw.twell_profile_enable(False)
    kernels = {}
    for name in tw.KERNELS:
        n_l, k_ms = tw.twell_profile_read(name)
        if n_l:
            kernels[name] = {"launches": n_l, "avg_us": round(1000.0 * k_ms / n_l, 2)}
    # dense GEMM work on the tensor cores: gate and up (4 N d f), the SDDMM's dY.W_down^T (2 N d f)
    floor_us = 6.0 * N * d * f / (peaks["bf16_tflops"] * 1e12) * 1e6
    dense_floor_us = 18.0 * N * d * f / (peaks["bf16_tflops"] * 1e12) * 1e6
    kept = packed.values.numel() * 2 + packed.idx.numel() + packed.counts.numel() + fb * f * 2 + gu.numel() * 4
    out = {
        "workload": (f"gated layer training step fwd+bwd: N={N} d_model={d} d_ff={f} T={T} C={C}, lognormal rows, "
                     f"1% rows at 20%, lambda {lam}"),
        "ms_per_step": round(ms, 4), "tokens_per_s": round(N / (ms * 1e-3), 1),
        "peak_bytes": int(peak),
        "kept_for_backward_bytes": int(kept),
        "dense_h_bytes": N * f * 2,
        "layer": {"n_fb": n_fb, "twell_entries": nnz},
        "kernels": kernels,
        "roofline": {"bound": "tensor (gate + up GEMM and the SDDMM's GEMM)", "time_us": round(floor_us, 2),
                     "frac": round(floor_us / (ms * 1e3), 4), "peak_source": peak_src,
                     "dense_step_floor_us": round(dense_floor_us, 2)},
        "how": ("median of scrubbed steps; kept_for_backward = the packed H and the (g, u) pairs of its stored "
                "slots (dense_h_bytes: one dense bf16 [N, d_ff] for scale); dense_step_floor_us = 18 N d f at the same peak, the GEMM work of a dense gated fwd+bwd (not "
                "run)"),
    }
    del X, Wg, Wu, b, Wd, dY, packed, gu, Y, dX, dW, db, ws, flush
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    return out


def bench_train_memory(tw, dev, args):
    """Peak device memory of one training step (forward + backward) at the
    training shape, TwELL against the dense comparator, measured with the
    allocator's peak counter: the inputs, weights and upstream gradient are
    allocated first and left out; everything the step allocates -- the
    activations kept for the backward, the workspace, the outputs and the
    weight gradients -- is counted.  Each step is also timed (L2 scrubbed)."""
    import numpy as np
    import torch

    import synth
    cfg = synth.CONFIGS["train"]
    inp = synth.make_ffn_inputs(cfg)
    N, d, f, T, C, fb = cfg.n_rows, cfg.d_model, cfg.d_ff, cfg.tile, cfg.cap, cfg.fallback_capacity
    lam = cfg.l1_lambda

    def dt(a):
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(dev).view(torch.bfloat16)

    X, Wi, b, Wd, dY = dt(inp["X"]), dt(inp["W_inT"]), dt(inp["b"]), dt(inp["W_down"]), dt(inp["dY"])
    flush = torch.empty(max(2 * torch.cuda.get_device_properties(dev).L2_cache_size, 256 << 20),
                        dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)

    def measure(alloc, run):
        torch.cuda.synchronize()
        torch.cuda.empty_cache()
        base = torch.cuda.memory_allocated(dev)
        torch.cuda.reset_peak_memory_stats(dev)
        bufs = alloc()
        run(bufs)
        torch.cuda.synchronize()
        peak = torch.cuda.max_memory_allocated(dev) - base
        for _ in range(3):
            run(bufs)
        ms = []
        for _ in range(max(10, args.steps)):
            flush.zero_()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            run(bufs)
            e1.record(stream)
            ms.append((e0, e1))
        torch.cuda.synchronize()
        t = statistics.median(a.elapsed_time(bb) for a, bb in ms)
        del bufs
        torch.cuda.synchronize()
        torch.cuda.empty_cache()
        return peak, t

    def grads():
        return dict(dX=torch.empty((N, d), dtype=torch.bfloat16, device=dev),
                    dWi=torch.empty((f, d), dtype=torch.float32, device=dev),
                    dWd=torch.empty((f, d), dtype=torch.float32, device=dev),
                    db=torch.empty((f,), dtype=torch.float32, device=dev),
                    Y=torch.empty((N, d), dtype=torch.bfloat16, device=dev))

    def twell_alloc():
        g = grads()
        g["H"] = tw.alloc_packed(N, f, T, C, fb, dev)
        g["ws"] = torch.empty(max(tw.fwd_workspace_bytes(N, d, f, T, C, fb), tw.bwd_workspace_bytes(N, d, f, T, C, fb)),
                              dtype=torch.uint8, device=dev)
        return g

    def twell_run(g):
        tw.twell_ffn_fwd(X, Wi, b, Wd, g["H"], g["Y"], g["ws"], stream)
        tw.twell_ffn_bwd(X, Wi, Wd, g["H"], dY, lam, g["dX"], g["dWi"], g["dWd"], g["db"], g["ws"], stream)

    def dense_alloc():
        g = grads()
        g["H"] = torch.empty((N, f), dtype=torch.bfloat16, device=dev)
        g["ws"] = torch.empty(tw.dense_bwd_workspace_bytes(N, d, f), dtype=torch.uint8, device=dev)
        return g

    def dense_run(g):
        tw.twell_dense_ffn_fwd(X, Wi, b, Wd, g["H"], g["Y"], stream)
        tw.twell_dense_ffn_bwd(X, Wi, Wd, g["H"], dY, lam, g["dX"], g["dWi"], g["dWd"], g["db"], g["ws"], stream)

    tw_peak, tw_ms = measure(twell_alloc, twell_run)
    de_peak, de_ms = measure(dense_alloc, dense_run)
    grads_bytes = N * d * 2 * 2 + 2 * f * d * 4 + f * 4
    return {
        "workload": "training step fwd+bwd: N=8192 d_model=2048 d_ff=8192 T=128 C=8, lognormal rows, 1% rows at "
                    "20%, lambda 1e-4",
        "twell": {"peak_bytes": int(tw_peak), "ms_per_step": round(tw_ms, 4),
                  "tokens_per_s": round(N / (tw_ms * 1e-3), 1)},
        "dense": {"peak_bytes": int(de_peak), "ms_per_step": round(de_ms, 4),
                  "tokens_per_s": round(N / (de_ms * 1e-3), 1)},
        "peak_ratio": round(tw_peak / de_peak, 4),
        "activation_and_scratch_bytes": {"twell": int(tw_peak - grads_bytes), "dense": int(de_peak - grads_bytes)},
        "how": "torch.cuda.max_memory_allocated over one step minus the memory allocated before it; inputs, "
               "weights and dY allocated before and not counted; Y, dX, dW_in^T, dW_down, db (fp32) counted in "
               "both (activation_and_scratch_bytes leaves them out)",
    }


def next_shapes(args, steps):
    """Forward-only measurements of the next shapes, one result dict each (a
    generator): the gated (Llama-style) layer, the decode-shaped sweep and the
    1B forward with row- and tile-granular fallback, `steps` timed calls each."""
    import numpy as np
    import torch

    import activation_sparse_transformer_gb300 as tw
    import synth

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(0)
    tw.load_library()
    peaks, peak_src = load_peaks()
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    flush = torch.empty(max(2 * l2, 256 << 20), dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)

    def dt(a):
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(dev).view(torch.bfloat16)

    def timed(fn, k, rotate=None):
        """Median event time of k calls.  With `rotate` (a list of calls on
        separate copies of the layer's weights, together larger than L2) the
        calls take the copies in turn and nothing is flushed; otherwise L2 is
        scrubbed before every call."""
        fns = rotate or [fn]
        for _ in range(args.warmup):
            for g in fns:
                g()
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(k)]
        for i in range(k):
            if not rotate:
                flush.zero_()
            ev[i][0].record(stream)
            fns[i % len(fns)]()
            ev[i][1].record(stream)
        torch.cuda.synchronize()
        return statistics.median(a.elapsed_time(b) for a, b in ev)

    import dataclasses
    # the 1B forward with row-granular and tile-granular fallback, same inputs
    cfgs = ([synth.CONFIGS["gated"]] + synth.decode_sweep() +
            [dataclasses.replace(synth.CONFIGS["1b"], name="1b_rows"),
             dataclasses.replace(synth.CONFIGS["1b"], name="1b_tiles")])
    if args.only:
        cfgs = [c for c in cfgs if c.name in args.only.split(",")]
    for cfg in cfgs:
        inp = synth.make_ffn_inputs(cfg)
        N, d, f, T, C = cfg.n_rows, cfg.d_model, cfg.d_ff, cfg.tile, cfg.cap
        fb = cfg.fallback_capacity if not cfg.name.startswith("decode") else N
        X, Wi, b, Wd = dt(inp["X"]), dt(inp["W_inT"]), dt(inp["b"]), dt(inp["W_down"])
        hybrid = tw.HYBRID_TILES if cfg.name.endswith("_tiles") else tw.HYBRID_ROWS
        packed = tw.alloc_packed(N, f, T, C, fb, dev, hybrid=hybrid)
        Y = torch.empty((N, d), dtype=torch.bfloat16, device=dev)
        ws = torch.empty(tw.fwd_workspace_bytes(N, d, f, T, C, fb), dtype=torch.uint8, device=dev)
        if cfg.gated:
            Wu = dt(inp["W_uT"])
            fn = lambda: tw.twell_gated_ffn_fwd(X, Wi, Wu, b, Wd, packed, Y, ws, stream)
        else:
            fn = lambda: tw.twell_ffn_fwd(X, Wi, b, Wd, packed, Y, ws, stream)
        fn()
        rc = tw.twell_read_status(packed, stream)
        if rc != 0:
            raise RuntimeError(f"{cfg.name}: status {rc}")
        n_fb = int(packed.n_fb[0].item())
        cnts = packed.counts.to(torch.int64)
        nnz = int(cnts[cnts != tw.DENSE_TILE].sum().item())   # entries stored in TwELL cells
        # Decode is bound by streaming the weights: scrubbing L2 by writing a
        # buffer leaves ~L2-size of dirty lines whose write-back then competes
        # with that stream, so these shapes instead take three device copies of
        # the layer (as consecutive layers of a model would: 3 x 234 MB, more
        # than L2) in turn, with no scrub.  The scrubbed time is reported beside.
        decode = cfg.name.startswith("decode")
        copies, rot = [], None
        if decode:
            copies = [tuple(t.clone() for t in (X, Wi, b, Wd)) for _ in range(3)]
            rot = [(lambda c=c: tw.twell_ffn_fwd(c[0], c[1], c[2], c[3], packed, Y, ws, stream)) for c in copies]
        ms_flush = timed(fn, steps)
        ms = timed(fn, steps, rotate=rot) if decode else ms_flush
        tw.twell_profile_reset()
        tw.twell_profile_enable(True)
        timed(fn, min(steps, 20), rotate=rot)
        tw.twell_profile_enable(False)
        kernels = {}
        for name in tw.KERNELS:
            n_l, k_ms = tw.twell_profile_read(name)
            if n_l:
                kernels[name] = {"launches": n_l, "avg_us": round(1000.0 * k_ms / n_l, 2)}
        # the same call captured once in a CUDA graph and replayed (no host
        # launch overhead per kernel): what a decode loop would run
        graphs = []
        for c in (copies or [(X, Wi, b, Wd)]):
            graph = torch.cuda.CUDAGraph()
            torch.cuda.synchronize()
            with torch.cuda.graph(graph):
                cap = torch.cuda.current_stream(dev)
                if cfg.gated:
                    tw.twell_gated_ffn_fwd(X, Wi, Wu, b, Wd, packed, Y, ws, cap)
                else:
                    tw.twell_ffn_fwd(c[0], c[1], c[2], c[3], packed, Y, ws, cap)
            graphs.append(graph)
        ms_graph = timed(graphs[0].replay, steps, rotate=[g.replay for g in graphs] if decode else None)
        roof_wo_us = None
        if cfg.gated:
            flops = 2.0 * 2 * N * d * f
            roof_us = flops / (peaks["bf16_tflops"] * 1e12) * 1e6
            bound = "tensor (gate and up GEMMs)"
        elif cfg.name.startswith("1b"):
            roof_us = 2.0 * N * d * f / (peaks["bf16_tflops"] * 1e12) * 1e6
            bound = "tensor (up GEMM)"
        else:
            H = torch.empty((N, f), dtype=torch.bfloat16, device=dev)
            tw.twell_unpack(packed, H)
            used = int((H.view(torch.int16) & 0x7FFF).ne(0).any(dim=0).sum().item())
            byts = f * d * 2 + used * d * 2 + 2 * N * d * 2 + packed.values.numel() * 3
            roof_us = byts / (peaks["hbm_gbs"] * 1e9) * 1e6
            bound = f"hbm (W_in^T + {used} active W_down rows)"
            # the layer specification's byte list leaves W_in^T out; reported beside the honest count
            roof_wo_us = (byts - f * d * 2) / (peaks["hbm_gbs"] * 1e9) * 1e6
            del H
        yield {
            "metric": f"sparse-FFN forward tokens/s ({cfg.name})", "value": round(N / (ms * 1e-3), 1),
            "unit": "tokens/s", "ms": round(ms, 4), "ms_graph": round(ms_graph, 4),
            "ms_l2_scrubbed": round(ms_flush, 4),
            "tokens_per_s_graph": round(N / (ms_graph * 1e-3), 1), "n_gpus": 1, "steps": steps,
            "warmup": args.warmup,
            "dtype": "bf16", "data": "synthetic (seeded, see synth/)",
            "config": {"workload": cfg.name, "n_rows": N, "d_model": d, "d_ff": f, "tile": T, "cap": C,
                       "sparsity_target": cfg.sparsity, "gated": cfg.gated,
                       "l2": ("inputs larger than L2: 3 device copies of the layer's weights used in turn, "
                              "no scrub" if decode else "flushed between steps (2x L2 write)")},
            "layer": {"n_fb": n_fb, "twell_entries": nnz,
                      "hybrid": "tiles" if hybrid == tw.HYBRID_TILES else "rows",
                      "fallback_bytes": n_fb * (T if hybrid == tw.HYBRID_TILES else f) * 2},
            "kernels": kernels,
            "roofline": {"bound": bound, "time_us": round(roof_us, 2), "frac": round(roof_us / (ms * 1e3), 4),
                         "frac_graph": round(roof_us / (ms_graph * 1e3), 4), "peak_source": peak_src,
                         "time_us_without_w_in": round(roof_wo_us, 2) if roof_wo_us else None},
        }
        del X, Wi, b, Wd, packed, Y, ws, graph, graphs, copies, rot
        torch.cuda.empty_cache()


def bench_next(args):
    """`--next`: one JSON line per next shape."""
    for res in next_shapes(args, args.steps):
        print(json.dumps(res), flush=True)


def next_summary(args, steps=50):
    """The next shapes in brief, for the main bench line."""
    out = {}
    for res in next_shapes(args, steps):
        r = res["roofline"]
        out[res["config"]["workload"]] = {"ms": res["ms"], "ms_graph": res["ms_graph"], "roofline_us": r["time_us"],
                                          "bound": r["bound"], "frac": r["frac"], "frac_graph": r["frac_graph"]}
    out["how"] = (f"forward only, {steps} timed calls each (median); decode shapes rotate 3 device copies of the "
                  "weights with no scrub, the others scrub L2; frac_graph = the call replayed as a CUDA graph; "
                  "full lines with `bench.py --next`")
    return out


def synth_configs():
    import synth
    return synth.CONFIGS


def cpu_sample_rows(default):
    return int(os.environ.get("TWELL_CPU_SAMPLE_ROWS", default))


def oracle_step(base, dY, rows, cfg, lam):
    """One fwd+bwd of the oracle on the first `rows` tokens treated as a batch."""
    import oracle
    X = base["X"][:rows]
    Z, H = oracle.hidden(X, base["W_inT"], base["b"])
    packed = oracle.pack(H, cfg.tile, cfg.cap, max(1, rows))
    oracle.down_packed(packed, base["W_down"])
    _, dZ = oracle.grad_hidden(dY[:rows], base["W_down"], H, lam)
    oracle.grad_input(dZ, base["W_inT"])
    oracle.grad_weights(X, base["W_down"], H, dY[:rows], lam)


def cpu_baseline(config="1b", rows=None):
    import oracle
    import synth
    cfg = synth.CONFIGS[config]
    base = synth.make_ffn_inputs(cfg)
    dY = synth.make_grad_output(cfg.n_rows, cfg.d_model, seed=cfg.seed + 77)
    rows = rows or cpu_sample_rows(1536)  # ~10-15 s of the oracle on the host cores
    oracle.build()
    t = time.perf_counter()
    oracle_step(base, dY, rows, cfg, cfg.l1_lambda or 1e-4)
    el = time.perf_counter() - t
    cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
    return {"value": round(rows / el, 3), "unit": UNIT, "cores": cores, "kind": "oracle",
            "sample": f"fwd+bwd of the first {rows} tokens of the {cfg.name} layer as one batch "
                      f"(plain C fp32 loops, OpenMP over {cores} threads), {el:.1f} s"}


def time_pr1_oracle() -> None:
    """Prints the seconds of one oracle fwd + bwd of the whole small layer
    (N 256, d_model 256, d_ff 1024, T 64, C 8) as one JSON number."""
    import oracle
    import synth
    cfg = synth.CONFIGS["pr1"]
    base = synth.make_ffn_inputs(cfg)
    dY = synth.make_grad_output(cfg.n_rows, cfg.d_model, seed=cfg.seed + 77)
    oracle.build()
    t = time.perf_counter()
    oracle_step(base, dY, cfg.n_rows, cfg, cfg.l1_lambda or 1e-4)
    print(json.dumps(time.perf_counter() - t))


def cpu_single_thread_pr1():
    """The oracle on one host thread over the whole small layer, in a fresh
    process: the OpenMP runtime reads OMP_NUM_THREADS once, when it loads."""
    import synth
    n = synth.CONFIGS["pr1"].n_rows
    env = dict(os.environ, OMP_NUM_THREADS="1")
    out = subprocess.run([sys.executable, "-c", "import bench; bench.time_pr1_oracle()"], cwd=ROOT, env=env,
                         capture_output=True, text=True, timeout=600, check=True)
    el = float(out.stdout.strip().splitlines()[-1])
    return {"value": round(n / el, 3), "unit": UNIT, "cores": 1, "kind": "oracle",
            "sample": f"fwd+bwd of the whole small layer (N={n}, d_model=256, d_ff=1024, T=64, C=8), "
                      f"one thread, {el:.2f} s"}


def bench_reference(args, rank, world):
    if rank != 0:
        return None
    import oracle
    import synth
    cfg = synth.CONFIGS[args.config]
    base = synth.make_ffn_inputs(cfg)
    dY = synth.make_grad_output(cfg.n_rows, cfg.d_model, seed=cfg.seed + 77)
    lam = cfg.l1_lambda or 1e-4
    rows = cpu_sample_rows(32)
    oracle.build()
    for _ in range(args.warmup):
        oracle_step(base, dY, rows, cfg, lam)
    times = []
    for _ in range(args.steps):
        t = time.perf_counter()
        oracle_step(base, dY, rows, cfg, lam)
        times.append(time.perf_counter() - t)
    s = statistics.median(times)
    cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
    value = round(rows / s, 3)
    return {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(1000 * s, 2),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
            "data": "synthetic (seeded, see synth/)",
            "config": {"workload": workload_name(cfg), "sample_rows": rows},
            "step": f"one step = fwd+bwd of the first {rows} tokens of the layer (ms_per_step is its measured "
                    "median time)",
            "extrapolated_ms_per_full_batch": round(1000 * s * cfg.n_rows / rows, 1),
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                             "sample": f"each step: fwd+bwd of the first {rows} tokens as one batch"},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    # the main step times the plain layer; the gated layer is timed by the
    # gated_train block of the line and by --next
    ap.add_argument("--config", default="1b",
                    choices=sorted(k for k, c in synth_configs().items() if not c.gated))
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-energy", action="store_true",
                    help="skip the energy loops (e.g. to keep an ncu launch list to the timed steps)")
    ap.add_argument("--only", default="",
                    help="with --next: comma-separated workload names to run (default: all)")
    ap.add_argument("--next", action="store_true",
                    help="forward-only lines for the gated layer and the decode sweep instead of the main step")
    ap.add_argument("--no-memory", action="store_true",
                    help="skip the training-shape peak-memory comparison against the dense step and the gated "
                         "layer's training step")
    ap.add_argument("--no-next", action="store_true",
                    help="leave the next shapes' summary (gated layer, decode sweep, tile routing) out of the line")
    ap.add_argument("--min-window", type=float, default=1.0,
                    help="repeat the K-step timed loop until the timed window spans this many seconds")
    ap.add_argument("--timeline", action="store_true",
                    help="print the launch timeline of one fwd + bwd step (L2 scrubbed before it) instead of "
                         "the bench line")
    args = ap.parse_args()
    args.warmup = max(3, args.warmup)
    rank, world, local = dist_info()
    if args.gpus > 1 and "WORLD_SIZE" not in os.environ and not os.environ.get("TWELL_BENCH_CHILD"):
        sys.exit(relaunch_with_ranks(args.gpus))
    if world != args.gpus:
        sys.exit(f"bench.py: --gpus {args.gpus} but WORLD_SIZE={world}: run one rank per GPU")
    if args.impl == "reference":
        res = bench_reference(args, rank, world)
        if res is not None:
            print(json.dumps(res), flush=True)
        return
    if args.next:
        if rank == 0:
            bench_next(args)
        return
    if world > 1:
        import torch
        torch.distributed.init_process_group("nccl")
    res = bench_ours(args, rank, world, local)
    if rank == 0 and args.timeline:
        print(json.dumps(res), flush=True)
    elif rank == 0:
        if not args.no_cpu_baseline:
            res["cpu_baseline"] = cpu_baseline(args.config)
            try:
                res["cpu_baseline"]["single_thread_pr1"] = cpu_single_thread_pr1()
            except (subprocess.SubprocessError, ValueError, IndexError) as exc:
                res["cpu_baseline"]["single_thread_pr1"] = {"unavailable": f"{type(exc).__name__}: {exc}"[:200]}
        if not args.no_next and world == 1 and args.config == "1b":
            res["next_shapes"] = next_summary(args)
        print(json.dumps(res), flush=True)
    if world > 1:
        import torch
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
