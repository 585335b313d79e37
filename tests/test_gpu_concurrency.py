"""Callers on different streams share nothing in the library: two host
threads run training steps (forward + backward) of two different layers on
two streams at the same time, while a third thread captures a third layer's
step into a CUDA graph on a third stream and replays it.  Every result --
Y, the packed activations, dX, dW_in^T, dW_down, db -- is bit-identical to the
same calls run one after another on one stream (the layer's outputs are
deterministic, so any cross-talk between callers would show)."""
import threading

import numpy as np
import pytest

import synth
from twell_check import to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def tw():
    import __graft_entry__ as g
    g.build()
    import activation_sparse_transformer_gb300 as m
    return m


class Layer:
    def __init__(self, tw, torch, cfg, dev):
        inp = synth.make_ffn_inputs(cfg)
        self.tw = tw
        self.lam = cfg.l1_lambda or 1e-4
        self.X, self.Wi, self.b, self.Wd = (to_dev(inp[k], torch) for k in ("X", "W_inT", "b", "W_down"))
        self.dY = to_dev(synth.make_grad_output(cfg.n_rows, cfg.d_model, seed=cfg.seed + 3), torch)
        N, d, f, T, C, fb = cfg.n_rows, cfg.d_model, cfg.d_ff, cfg.tile, cfg.cap, cfg.fallback_capacity
        self.H = tw.alloc_packed(N, f, T, C, fb, dev)
        self.Y = torch.empty((N, d), dtype=torch.bfloat16, device=dev)
        self.dX = torch.empty((N, d), dtype=torch.bfloat16, device=dev)
        self.dWi = torch.empty((f, d), dtype=torch.float32, device=dev)
        self.dWd = torch.empty((f, d), dtype=torch.float32, device=dev)
        self.db = torch.empty((f,), dtype=torch.float32, device=dev)
        self.ws = torch.empty(max(tw.fwd_workspace_bytes(N, d, f, T, C, fb), tw.bwd_workspace_bytes(N, d, f, T, C, fb)),
                              dtype=torch.uint8, device=dev)

    def step(self, stream):
        self.tw.twell_ffn_fwd(self.X, self.Wi, self.b, self.Wd, self.H, self.Y, self.ws, stream)
        self.tw.twell_ffn_bwd(self.X, self.Wi, self.Wd, self.H, self.dY, self.lam, self.dX, self.dWi, self.dWd,
                              self.db, self.ws, stream)

    def outputs(self):
        n_fb = int(self.H.n_fb[0].item())   # only the used fallback rows are written
        out = [self.Y, self.dX, self.dWi, self.dWd, self.db, self.H.values, self.H.idx, self.H.counts,
               self.H.row_fb, self.H.fb_dense[:n_fb], self.H.n_fb]
        return [t.cpu().clone() for t in out]

    def poison(self):
        for t in (self.Y, self.dX, self.dWi, self.dWd, self.db, self.H.values, self.H.fb_dense):
            t.view(torch_int_view(t)).fill_(0x3333)


def torch_int_view(t):
    import torch
    return {2: torch.int16, 4: torch.int32, 1: torch.uint8}[t.element_size()]


def test_three_callers_on_three_streams_match_serial(tw):
    import torch
    dev = torch.device("cuda")
    cfgs = [synth.FFNConfig("ca", 384, 256, 1024, 64, 8, seed=31, row_spread="lognormal", forced_frac_rows=0.03,
                            l1_lambda=1e-3),
            synth.FFNConfig("cb", 512, 512, 2048, 128, 8, seed=32, row_spread="lognormal", forced_frac_rows=0.02),
            synth.FFNConfig("cc", 300, 256, 1536, 128, 16, seed=33, row_spread="lognormal", forced_frac_rows=0.03)]
    layers = [Layer(tw, torch, c, dev) for c in cfgs]
    main = torch.cuda.current_stream()
    ref = []
    for L in layers:
        L.step(main)
        torch.cuda.synchronize()
        assert tw.twell_read_status(L.H) == 0
        assert int(L.H.n_fb[0].item()) > 0      # the second stream (fallback rows) takes part
        ref.append(L.outputs())
        L.poison()
    torch.cuda.synchronize()

    streams = [torch.cuda.Stream(dev) for _ in range(3)]
    errors = []
    graph_box = {}

    def loop(L, s, iters):
        try:
            with torch.cuda.stream(s):
                for _ in range(iters):
                    L.step(s)
            s.synchronize()
        except Exception as exc:  # noqa: BLE001 - reported below
            errors.append(exc)

    def capture(L, s):
        try:
            with torch.cuda.stream(s):
                L.step(s)               # first use of this stream outside the capture
            s.synchronize()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=s, capture_error_mode="thread_local"):
                L.step(torch.cuda.current_stream())
            L.poison()
            torch.cuda.synchronize(dev)
            for _ in range(3):
                g.replay()
            torch.cuda.synchronize(dev)
            graph_box["g"] = g
        except Exception as exc:  # noqa: BLE001 - reported below
            errors.append(exc)

    threads = [threading.Thread(target=loop, args=(layers[0], streams[0], 12)),
               threading.Thread(target=loop, args=(layers[1], streams[1], 12)),
               threading.Thread(target=capture, args=(layers[2], streams[2]))]
    for t in threads:
        t.start()
    for t in threads:
        t.join(timeout=300)
    assert not errors, errors
    torch.cuda.synchronize()
    names = ["Y", "dX", "dW_inT", "dW_down", "db", "values", "idx", "counts", "row_fb", "fb_dense", "n_fb"]
    for L, want in zip(layers, ref):
        assert tw.twell_read_status(L.H) == 0
        for name, a, b in zip(names, L.outputs(), want):
            assert torch.equal(a, b), (L.Y.shape, name)


class GatedLayer(Layer):
    """The gated layer's training step (forward keeping (g, u), gated backward)."""

    def __init__(self, tw, torch, cfg, dev):
        super().__init__(tw, torch, cfg, dev)
        inp = synth.make_ffn_inputs(cfg)
        N, d, f, T, C, fb = cfg.n_rows, cfg.d_model, cfg.d_ff, cfg.tile, cfg.cap, cfg.fallback_capacity
        self.Wu = to_dev(inp["W_uT"], torch)
        self.gu = torch.empty((N, f // T, C, 2), dtype=torch.float32, device=dev)
        self.dWu = torch.empty((f, d), dtype=torch.float32, device=dev)
        self.ws = torch.empty(max(tw.fwd_workspace_bytes(N, d, f, T, C, fb),
                                  tw.gated_bwd_workspace_bytes(N, d, f, T, C, fb)), dtype=torch.uint8, device=dev)

    def step(self, stream):
        self.tw.twell_gated_ffn_fwd_train(self.X, self.Wi, self.Wu, self.b, self.Wd, self.H, self.Y, self.gu,
                                          self.ws, stream)
        self.tw.twell_gated_ffn_bwd(self.X, self.Wi, self.Wu, self.b, self.Wd, self.H, self.gu, self.dY, self.lam,
                                    self.dX, self.dWi, self.dWu, self.dWd, self.db, self.ws, stream)

    def outputs(self):
        return super().outputs() + [self.dWu.cpu().clone()]

    def poison(self):
        super().poison()
        self.dWu.view(torch_int_view(self.dWu)).fill_(0x3333)


def test_gated_callers_and_graph_capture_match_serial(tw):
    """The same with gated layers: one gated and one plain caller on two
    streams while a third thread captures a gated layer's training step
    (which also forks the second stream a second time, beside its SDDMM) into
    a CUDA graph and replays it."""
    import torch
    dev = torch.device("cuda")
    mk = lambda name, seed, gated: synth.FFNConfig(name, 320, 256, 1024, 64, 8, seed=seed, gated=gated,
                                                  row_spread="lognormal", forced_frac_rows=0.03, l1_lambda=1e-3)
    layers = [GatedLayer(tw, torch, mk("ga", 51, True), dev), Layer(tw, torch, mk("pa", 52, False), dev),
              GatedLayer(tw, torch, mk("gc", 53, True), dev)]
    main = torch.cuda.current_stream()
    ref = []
    for L in layers:
        L.step(main)
        torch.cuda.synchronize()
        assert tw.twell_read_status(L.H) == 0
        assert int(L.H.n_fb[0].item()) > 0
        ref.append(L.outputs())
        L.poison()
    torch.cuda.synchronize()
    streams = [torch.cuda.Stream(dev) for _ in range(3)]
    errors = []

    def loop(L, s, iters):
        try:
            with torch.cuda.stream(s):
                for _ in range(iters):
                    L.step(s)
            s.synchronize()
        except Exception as exc:  # noqa: BLE001 - reported below
            errors.append(exc)

    def capture(L, s):
        try:
            with torch.cuda.stream(s):
                L.step(s)
            s.synchronize()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=s, capture_error_mode="thread_local"):
                L.step(torch.cuda.current_stream())
            L.poison()
            torch.cuda.synchronize(dev)
            for _ in range(3):
                g.replay()
            torch.cuda.synchronize(dev)
        except Exception as exc:  # noqa: BLE001 - reported below
            errors.append(exc)

    threads = [threading.Thread(target=loop, args=(layers[0], streams[0], 8)),
               threading.Thread(target=loop, args=(layers[1], streams[1], 8)),
               threading.Thread(target=capture, args=(layers[2], streams[2]))]
    for t in threads:
        t.start()
    for t in threads:
        t.join(timeout=300)
    assert not errors, errors
    torch.cuda.synchronize()
    names = ["Y", "dX", "dW_gT", "dW_down", "db", "values", "idx", "counts", "row_fb", "fb_dense", "n_fb", "dW_uT"]
    for L, want in zip(layers, ref):
        assert tw.twell_read_status(L.H) == 0
        for name, a, b in zip(names, L.outputs(), want):
            assert torch.equal(a, b), (L.Y.shape, name)
