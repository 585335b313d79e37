"""Backward on the GPU (SDDMM at the TwELL pattern with the L1 term, dX gather,
unit-major dW_down / dW_in / db) against the oracle's dense fp32 loops, using
the H the GPU's forward produced (so both sides share the pattern)."""
import numpy as np
import pytest

import oracle
import synth
from twell_check import assert_close, from_dev_bits, from_dev_f32, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def tw():
    import __graft_entry__ as g
    g.build()
    import activation_sparse_transformer_gb300 as m
    return m


def run(tw, torch, cfg, inp, dY, lam):
    dev = torch.device("cuda")
    T, C, fb = cfg.tile, cfg.cap, cfg.fallback_capacity
    X, Wi, b, Wd = (to_dev(inp[k], torch) for k in ("X", "W_inT", "b", "W_down"))
    N, d = inp["X"].shape
    f = inp["W_inT"].shape[0]
    p = tw.alloc_packed(N, f, T, C, fb, dev)
    Y = torch.empty((N, d), dtype=torch.bfloat16, device=dev)
    ws = torch.empty(tw.fwd_workspace_bytes(N, d, f, T, C, fb), dtype=torch.uint8, device=dev)
    tw.twell_ffn_fwd(X, Wi, b, Wd, p, Y, ws)
    assert tw.twell_read_status(p) == 0
    H = torch.empty((N, f), dtype=torch.bfloat16, device=dev)
    tw.twell_unpack(p, H)
    dYd = to_dev(dY, torch)
    dX = torch.full((N, d), 5.0, dtype=torch.bfloat16, device=dev)
    dWi = torch.full((f, d), 5.0, dtype=torch.float32, device=dev)
    dWd = torch.full((f, d), 5.0, dtype=torch.float32, device=dev)
    db = torch.full((f,), 5.0, dtype=torch.float32, device=dev)
    wsb = torch.full((tw.bwd_workspace_bytes(N, d, f, T, C, fb),), 0x5A, dtype=torch.uint8, device=dev)
    tw.twell_ffn_bwd(X, Wi, Wd, p, dYd, lam, dX, dWi, dWd, db, wsb)
    torch.cuda.synchronize()
    return from_dev_bits(H), from_dev_f32(dX), dWi.cpu().numpy(), dWd.cpu().numpy(), db.cpu().numpy()


@pytest.mark.parametrize("name,N,d,T,C,lam", [("pr1", 256, 256, 64, 8, 1e-4), ("ragged", 301, 256, 128, 8, 1e-2),
                                                ("t32", 160, 256, 32, 4, 0.0),
                                                # wider rows (2048 and 4096 columns)
                                                ("wide", 300, 2048, 128, 8, 1e-4),
                                                ("wide16", 200, 4096, 64, 16, 1e-3),
                                                # 256-wide tiles (the unit lists' largest shared-memory
                                                # case) at C = 8 and 16, and a decode-sized batch whose
                                                # forward takes the small-batch path
                                                ("t256c8", 130, 256, 256, 8, 0.0),
                                                ("t256c16", 200, 512, 256, 16, 1e-3),
                                                ("small", 16, 256, 64, 8, 1e-4),
                                                ("c32", 160, 256, 64, 32, 1e-3)])
def test_bwd_matches_oracle(tw, name, N, d, T, C, lam):
    import torch
    cfg = synth.FFNConfig(name, N, d, 1024, T, C, seed=N + 7, row_spread="lognormal", forced_frac_rows=0.03,
                          fb_cap=N // 4)
    inp = synth.make_ffn_inputs(cfg)
    dY = synth.make_grad_output(N, d, seed=N)
    H, dX, dWi, dWd, db = run(tw, torch, cfg, inp, dY, lam)
    _, dZ = oracle.grad_hidden(dY, inp["W_down"], H, lam)
    assert_close(dX, oracle.grad_input(dZ, inp["W_inT"]), "dX")
    rWi, rWd, rdb = oracle.grad_weights(inp["X"], inp["W_down"], H, dY, lam)
    assert_close(dWi, rWi, "dW_inT")
    assert_close(dWd, rWd, "dW_down")
    assert_close(db, rdb, "db")


def test_repeat_calls_bit_identical(tw):
    # one workspace shared by forward and backward, each called twice: the
    # gathers hand out rows from counters that every call re-zeroes, and each
    # output is summed by one thread in a fixed order, so repeated calls give
    # the same bits
    import torch
    cfg = synth.FFNConfig("rep", 300, 2048, 1024, 128, 8, seed=41, row_spread="lognormal", forced_frac_rows=0.03,
                          fb_cap=64)
    inp = synth.make_ffn_inputs(cfg)
    N, d, f, T, C, fb = cfg.n_rows, cfg.d_model, cfg.d_ff, cfg.tile, cfg.cap, cfg.fallback_capacity
    dev = torch.device("cuda")
    X, Wi, b, Wd = (to_dev(inp[k], torch) for k in ("X", "W_inT", "b", "W_down"))
    dY = to_dev(synth.make_grad_output(N, d, seed=5), torch)
    ws = torch.full((max(tw.fwd_workspace_bytes(N, d, f, T, C, fb), tw.bwd_workspace_bytes(N, d, f, T, C, fb)),),
                    0x5A, dtype=torch.uint8, device=dev)
    outs = []
    for _ in range(2):
        p = tw.alloc_packed(N, f, T, C, fb, dev)
        Y = torch.empty((N, d), dtype=torch.bfloat16, device=dev)
        tw.twell_ffn_fwd(X, Wi, b, Wd, p, Y, ws)
        assert tw.twell_read_status(p) == 0
        assert int(p.n_fb[0].item()) > 0
        dX = torch.empty((N, d), dtype=torch.bfloat16, device=dev)
        dWi = torch.empty((f, d), dtype=torch.float32, device=dev)
        dWd = torch.empty((f, d), dtype=torch.float32, device=dev)
        db = torch.empty((f,), dtype=torch.float32, device=dev)
        tw.twell_ffn_bwd(X, Wi, Wd, p, dY, 1e-4, dX, dWi, dWd, db, ws)
        torch.cuda.synchronize()
        outs.append([from_dev_bits(Y), from_dev_bits(dX), dWi.cpu().numpy().view(np.uint32),
                     dWd.cpu().numpy().view(np.uint32), db.cpu().numpy().view(np.uint32)])
    for a, c in zip(*outs):
        assert np.array_equal(a, c)


def test_bwd_zero_upstream_closed_form(tw):
    # dY = 0: dZ = lambda exactly on the pattern, so db = lambda * active count,
    # dW_down = 0 and dX = lambda * sum of active W_in^T rows (integer weights:
    # exact in fp32).
    import torch
    N, d, f = 192, 128, 512
    inp = synth.make_integer_inputs(N, d, f, seed=8, sparsity=0.95)
    cfg = synth.FFNConfig("z", N, d, f, 64, 8, seed=0, fb_cap=N)
    lam = 0.5
    H, dX, dWi, dWd, db = run(tw, torch, cfg, inp, np.zeros((N, d), np.uint16), lam)
    act = synth.bf16_bits_to_f32(H) > 0
    assert not dWd.any()
    assert np.array_equal(db, (lam * act.sum(0)).astype(np.float32))
    Wi = synth.bf16_bits_to_f32(inp["W_inT"]).astype(np.float64)
    ref_dx = lam * (act.astype(np.float64) @ Wi)
    assert np.array_equal(dX, synth.bf16_bits_to_f32(synth.f32_to_bf16_bits(ref_dx.astype(np.float32))))
    X = synth.bf16_bits_to_f32(inp["X"]).astype(np.float64)
    assert np.array_equal(dWi, (lam * (act.T.astype(np.float64) @ X)).astype(np.float32))


def test_bwd_1b_full_size_sampled(tw):
    import torch
    cfg = synth.CONFIGS["1b"]
    inp = synth.make_ffn_inputs(cfg)
    dY = synth.make_grad_output(cfg.n_rows, cfg.d_model, seed=77)
    lam = 1e-4
    H, dX, dWi, dWd, db = run(tw, torch, cfg, inp, dY, lam)
    rng = np.random.default_rng(5)
    rows = np.sort(rng.choice(cfg.n_rows, size=192, replace=False)).astype(np.int32)
    fbrows = np.nonzero(oracle.pack(H, cfg.tile, cfg.cap, cfg.fallback_capacity)["row_fb"] >= 0)[0][:16]
    rows = np.unique(np.concatenate([rows, fbrows])).astype(np.int32)
    _, dZ = oracle.grad_hidden(dY, inp["W_down"], H[rows], lam, rows=rows)
    assert_close(dX[rows], oracle.grad_input(dZ, inp["W_inT"]), "dX")
    cols = np.sort(rng.choice(cfg.d_ff, size=96, replace=False)).astype(np.int32)
    rWi, rWd, rdb = oracle.grad_weights(inp["X"], inp["W_down"], H, dY, lam, cols=cols)
    assert_close(dWi[cols], rWi, "dW_inT")
    assert_close(dWd[cols], rWd, "dW_down")
    assert_close(db[cols], rdb, "db")


def test_train_shape_full_size_sampled(tw):
    """The training configuration (N = 8192, 1% forced-dense rows, lambda 1e-4)
    in the launch configuration the bench times, checked on sampled rows and
    hidden units plus fallback rows."""
    import torch
    cfg = synth.CONFIGS["train"]
    inp = synth.make_ffn_inputs(cfg)
    dY = inp["dY"]
    lam = cfg.l1_lambda
    H, dX, dWi, dWd, db = run(tw, torch, cfg, inp, dY, lam)
    rng = np.random.default_rng(9)
    rows = np.sort(rng.choice(cfg.n_rows, size=128, replace=False)).astype(np.int32)
    fbrows = np.nonzero(oracle.pack(H, cfg.tile, cfg.cap, cfg.fallback_capacity)["row_fb"] >= 0)[0][:8]
    rows = np.unique(np.concatenate([rows, fbrows])).astype(np.int32)
    _, dZ = oracle.grad_hidden(dY, inp["W_down"], H[rows], lam, rows=rows)
    assert_close(dX[rows], oracle.grad_input(dZ, inp["W_inT"]), "dX")
    cols = np.sort(rng.choice(cfg.d_ff, size=48, replace=False)).astype(np.int32)
    rWi, rWd, rdb = oracle.grad_weights(inp["X"], inp["W_down"], H, dY, lam, cols=cols)
    assert_close(dWi[cols], rWi, "dW_inT")
    assert_close(dWd[cols], rWd, "dW_down")
    assert_close(db[cols], rdb, "db")


@pytest.mark.parametrize("N,d,f,T,C,sp,lam", [(256, 128, 512, 64, 8, 0.92, 1.0), (200, 256, 1024, 128, 16, 0.9, 0.0),
                                              (130, 128, 512, 32, 4, 0.9, 2.0),
                                              # a small batch: its forward takes the small-batch path
                                              (16, 256, 1024, 64, 8, 0.9, 1.0),
                                              # wide rows, most of them routed to the fallback
                                              (300, 2048, 1024, 128, 8, 0.95, 1.0),
                                              # the widest tile (the unit lists' largest shared memory)
                                              (200, 256, 1024, 256, 16, 0.95, 1.0)])
def test_bwd_integer_bit_exact(tw, N, d, f, T, C, sp, lam):
    """Integer layer, integer dY and lambda: every dZ, every product and every
    partial sum is an exact fp32 integer (the fallback rows' dZ fit the 16 bits
    of their high + low bf16 parts), so dX, dW_in^T, dW_down and db equal the
    oracle's bit for bit, TwELL rows and fallback rows alike."""
    import torch
    dev = torch.device("cuda")
    inp = synth.make_integer_inputs(N, d, f, seed=N + f + 5, lo=-1, hi=1, sparsity=sp)
    rng = np.random.default_rng(N + 1)
    dY = synth.f32_to_bf16_bits(rng.integers(-1, 2, size=(N, d)).astype(np.float32))
    X, Wi, b, Wd = (to_dev(inp[k], torch) for k in ("X", "W_inT", "b", "W_down"))
    p = tw.alloc_packed(N, f, T, C, N, dev)
    Y = torch.empty((N, d), dtype=torch.bfloat16, device=dev)
    ws = torch.empty(max(tw.fwd_workspace_bytes(N, d, f, T, C, N), tw.bwd_workspace_bytes(N, d, f, T, C, N)),
                     dtype=torch.uint8, device=dev)
    tw.twell_ffn_fwd(X, Wi, b, Wd, p, Y, ws)
    assert tw.twell_read_status(p) == 0
    assert int(p.n_fb[0].item()) > 0
    dX = torch.full((N, d), 5.0, dtype=torch.bfloat16, device=dev)
    dWi = torch.full((f, d), 5.0, dtype=torch.float32, device=dev)
    dWd = torch.full((f, d), 5.0, dtype=torch.float32, device=dev)
    db = torch.full((f,), 5.0, dtype=torch.float32, device=dev)
    tw.twell_ffn_bwd(X, Wi, Wd, p, to_dev(dY, torch), lam, dX, dWi, dWd, db, ws)
    torch.cuda.synchronize()
    _, H = oracle.hidden(inp["X"], inp["W_inT"], inp["b"])
    Hg = torch.empty((N, f), dtype=torch.bfloat16, device=dev)
    tw.twell_unpack(p, Hg)
    assert np.array_equal(from_dev_bits(Hg), H)
    _, dZ = oracle.grad_hidden(dY, inp["W_down"], H, lam)
    assert np.abs(dZ).max() < 2 ** 15
    rdX = oracle.grad_input(dZ, inp["W_inT"])
    rWi, rWd, rdb = oracle.grad_weights(inp["X"], inp["W_down"], H, dY, lam)
    for a in (rdX, rWi, rWd, rdb):
        assert np.abs(a).max() < 2 ** 24
    assert np.array_equal(from_dev_bits(dX), oracle.round_bf16(rdX))
    assert np.array_equal(dWi.cpu().numpy(), rWi)
    assert np.array_equal(dWd.cpu().numpy(), rWd)
    assert np.array_equal(db.cpu().numpy(), rdb)
