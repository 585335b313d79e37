"""The tile-granular hybrid on the GPU (only over-full tiles leave TwELL, for a
pool of dense tiles numbered in (row, tile) order) against the oracle:
standalone pack / unpack bit-exact, the fused forward bit-exact on integer
layers and within tolerance on random ones, pool overflow reported, the
backward (through its row view) equal to the row-routed backward of the same
layer and within tolerance of the oracle, and the calls that do not take this
variant refusing it."""
import ctypes

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


def check_tiles_packing(p, ref, T):
    """GPU packed buffers of the tile variant == the oracle's, bit for bit."""
    k = min(ref["n_fb"], ref["pool_cap"])
    assert int(p.n_fb[0].item()) == ref["n_fb"]
    assert np.array_equal(from_dev_bits(p.values).reshape(ref["values"].shape), ref["values"])
    assert np.array_equal(from_dev_bits(p.idx), ref["idx"])
    assert np.array_equal(from_dev_bits(p.counts), ref["counts"])
    assert np.array_equal(from_dev_bits(p.row_fb)[:p.n_rows], ref["row_fb"])
    pool = from_dev_bits(p.fb_dense).reshape(-1, T)
    assert np.array_equal(pool[:k], ref["pool"][:k])


@pytest.mark.parametrize("T,C", [(64, 4), (128, 8), (32, 2), (256, 16)])
def test_pack_tiles_bit_exact(tw, T, C):
    import torch
    N, f = 300, 2048
    H = synth.make_dense_h(N, f, seed=T + C, activity=0.02, dense_rows=np.arange(5, N, 37), dense_activity=0.2)
    fb_cap = 16
    p = tw.alloc_packed(N, f, T, C, fb_cap, "cuda", hybrid=tw.HYBRID_TILES)
    p.values.view(torch.int16).fill_(0x7777)
    p.idx.fill_(0xAB)
    p.counts.fill_(0xCD)
    Hd = to_dev(H, torch)
    tw.twell_pack(Hd, p)
    assert tw.twell_read_status(p) == 0
    ref = oracle.pack_tiles(H, T, C, fb_cap * (f // T))
    assert ref["n_fb"] > 0
    check_tiles_packing(p, ref, T)
    out = torch.empty((N, f), dtype=torch.bfloat16, device="cuda")
    tw.twell_unpack(p, out)
    torch.cuda.synchronize()
    assert np.array_equal(from_dev_bits(out), H)


def test_pack_tiles_pool_overflow(tw):
    import torch
    N, f, T, C = 64, 1024, 64, 4
    H = synth.make_dense_h(N, f, seed=9, activity=0.02, dense_rows=np.arange(0, N, 4), dense_activity=0.3)
    fb_cap = 1                                 # a pool of f / T = 16 tiles
    ref = oracle.pack_tiles(H, T, C, fb_cap * (f // T))
    assert ref["n_fb"] > 16
    p = tw.alloc_packed(N, f, T, C, fb_cap, "cuda", hybrid=tw.HYBRID_TILES)
    tw.twell_pack(to_dev(H, torch), p)
    assert tw.twell_read_status(p) == -6
    check_tiles_packing(p, ref, T)


INT_CASES = [
    # N, d, f, T, C, sparsity, seed (sparsities low enough that many tiles overflow)
    (256, 256, 1024, 64, 4, 0.95, 21),
    (200, 128, 1152, 128, 8, 0.93, 22),
    (130, 128, 512, 32, 2, 0.9, 23),
]


@pytest.mark.parametrize("N,d,f,T,C,sp,seed", INT_CASES)
def test_fwd_tiles_integer_bit_exact(tw, N, d, f, T, C, sp, seed):
    import torch
    inp = synth.make_integer_inputs(N, d, f, seed=seed, sparsity=sp)
    fb_cap = N
    ref = oracle.forward(inp["X"], inp["W_inT"], inp["b"], inp["W_down"], T, C, fb_cap, hybrid="tiles")
    assert ref["packed"]["n_fb"] > 0
    X, Wi, b, Wd = (to_dev(inp[k], torch) for k in ("X", "W_inT", "b", "W_down"))
    p = tw.alloc_packed(N, f, T, C, fb_cap, "cuda", hybrid=tw.HYBRID_TILES)
    Y = torch.full((N, d), 3.0, dtype=torch.bfloat16, device="cuda")
    ws = torch.empty(tw.fwd_workspace_bytes(N, d, f, T, C, fb_cap), dtype=torch.uint8, device="cuda")
    tw.twell_ffn_fwd(X, Wi, b, Wd, p, Y, ws)
    assert tw.twell_read_status(p) == 0
    check_tiles_packing(p, ref["packed"], T)
    assert np.array_equal(from_dev_bits(Y), ref["Y_bf16"])


def test_fwd_tiles_random_layer_and_row_variant_agree(tw):
    import torch
    cfg = synth.FFNConfig("t", 333, 256, 1024, 64, 8, seed=31, row_spread="lognormal", forced_frac_rows=0.05,
                          fb_cap=64)
    inp = synth.make_ffn_inputs(cfg)
    N, d, f, T, C = cfg.n_rows, cfg.d_model, cfg.d_ff, cfg.tile, cfg.cap
    X, Wi, b, Wd = (to_dev(inp[k], torch) for k in ("X", "W_inT", "b", "W_down"))
    ws = torch.empty(tw.fwd_workspace_bytes(N, d, f, T, C, cfg.fb_cap), dtype=torch.uint8, device="cuda")
    pt = tw.alloc_packed(N, f, T, C, cfg.fb_cap, "cuda", hybrid=tw.HYBRID_TILES)
    Yt = torch.empty((N, d), dtype=torch.bfloat16, device="cuda")
    tw.twell_ffn_fwd(X, Wi, b, Wd, pt, Yt, ws)
    assert tw.twell_read_status(pt) == 0
    Ht = torch.empty((N, f), dtype=torch.bfloat16, device="cuda")
    tw.twell_unpack(pt, Ht)
    pr = tw.alloc_packed(N, f, T, C, cfg.fb_cap, "cuda")
    Yr = torch.empty((N, d), dtype=torch.bfloat16, device="cuda")
    tw.twell_ffn_fwd(X, Wi, b, Wd, pr, Yr, ws)
    assert tw.twell_read_status(pr) == 0
    Hr = torch.empty((N, f), dtype=torch.bfloat16, device="cuda")
    tw.twell_unpack(pr, Hr)
    torch.cuda.synchronize()
    Hg = from_dev_bits(Ht)
    # the same up-projection: both variants hold the same H
    assert np.array_equal(Hg, from_dev_bits(Hr))
    ref = oracle.pack_tiles(Hg, T, C, cfg.fb_cap * (f // T))
    assert ref["n_fb"] >= len(inp["forced_rows"])
    check_tiles_packing(pt, ref, T)
    Z, Ho = oracle.hidden(inp["X"], inp["W_inT"], inp["b"])
    mism = (Hg != 0) != (Ho != 0)
    assert not mism.any() or np.abs(Z[mism]).max() < 1e-3
    Yo = oracle.down_dense(Ho, inp["W_down"])
    assert_close(from_dev_f32(Yt), Yo, "Y tiles")
    assert_close(from_dev_f32(Yr), Yo, "Y rows")


def test_fwd_tiles_1b_sampled(tw):
    import torch
    cfg = synth.CONFIGS["1b"]
    inp = synth.make_ffn_inputs(cfg)
    N, d, f, T, C, fb = cfg.n_rows, cfg.d_model, cfg.d_ff, cfg.tile, cfg.cap, cfg.fallback_capacity
    X, Wi, b, Wd = (to_dev(inp[k], torch) for k in ("X", "W_inT", "b", "W_down"))
    p = tw.alloc_packed(N, f, T, C, fb, "cuda", hybrid=tw.HYBRID_TILES)
    Y = torch.empty((N, d), dtype=torch.bfloat16, device="cuda")
    ws = torch.empty(tw.fwd_workspace_bytes(N, d, f, T, C, fb), dtype=torch.uint8, device="cuda")
    tw.twell_ffn_fwd(X, Wi, b, Wd, p, Y, ws)
    assert tw.twell_read_status(p) == 0
    H = torch.empty((N, f), dtype=torch.bfloat16, device="cuda")
    tw.twell_unpack(p, H)
    torch.cuda.synchronize()
    Hg = from_dev_bits(H)
    check_tiles_packing(p, oracle.pack_tiles(Hg, T, C, fb * (f // T)), T)
    rows = np.unique(np.concatenate([np.random.default_rng(1).choice(N, 128, replace=False), inp["forced_rows"]]))
    rows = rows.astype(np.int32)
    Z, Ho = oracle.hidden(inp["X"], inp["W_inT"], inp["b"], rows=rows)
    mism = (Hg[rows] != 0) != (Ho != 0)
    assert not mism.any() or np.abs(Z[mism]).max() < 1e-3
    assert_close(from_dev_f32(Y)[rows], oracle.down_dense(Ho, inp["W_down"]), "Y")


def test_tiles_refused_where_not_built(tw):
    """The plain layer's small-batch forward refuses the variant; the backward
    asks for its own workspace size."""
    import torch
    lib = tw.load_library()
    N, d, f, T, C = 64, 128, 256, 64, 4
    inp = synth.make_integer_inputs(N, d, f, seed=2, sparsity=0.9)
    X, Wi, b, Wd = (to_dev(inp[k], torch) for k in ("X", "W_inT", "b", "W_down"))
    p = tw.alloc_packed(N, f, T, C, 8, "cuda", hybrid=tw.HYBRID_TILES)
    st = p.struct()
    ws = torch.empty(max(tw.fwd_workspace_bytes(N, d, f, T, C, 8), tw.bwd_workspace_bytes(N, d, f, T, C, 8)),
                     dtype=torch.uint8, device="cuda")
    dY = torch.zeros((N, d), dtype=torch.bfloat16, device="cuda")
    dX = torch.empty((N, d), dtype=torch.bfloat16, device="cuda")
    dWi = torch.empty((f, d), dtype=torch.float32, device="cuda")
    dWd = torch.empty((f, d), dtype=torch.float32, device="cuda")
    db = torch.empty((f,), dtype=torch.float32, device="cuda")
    # the backward takes the variant, with the larger workspace its row view needs
    rc = lib.twell_ffn_bwd(X.data_ptr(), Wi.data_ptr(), Wd.data_ptr(), ctypes.byref(st), d, dY.data_ptr(),
                           ctypes.c_float(0.0), dX.data_ptr(), dWi.data_ptr(), dWd.data_ptr(), db.data_ptr(),
                           ws.data_ptr(), tw.bwd_workspace_bytes(N, d, f, T, C, 8, hybrid=tw.HYBRID_TILES) - 256,
                           None)
    assert rc == -5   # TWELL_ERR_WORKSPACE
    Y = torch.empty((N, d), dtype=torch.bfloat16, device="cuda")
    small = tw.alloc_packed(8, f, T, C, 8, "cuda", hybrid=tw.HYBRID_TILES)
    ss = small.struct()
    rc = lib.twell_ffn_fwd(X.data_ptr(), Wi.data_ptr(), b.data_ptr(), Wd.data_ptr(), 8, d, f, ctypes.byref(ss),
                           Y.data_ptr(), ws.data_ptr(), ws.numel(), None)
    assert rc == -3


def _fwd_bwd(tw, torch, inp, dY, lam, T, C, fb_cap, hybrid):
    dev = torch.device("cuda")
    X, Wi, b, Wd = (to_dev(inp[k], torch) for k in ("X", "W_inT", "b", "W_down"))
    N, d = inp["X"].shape
    f = inp["W_inT"].shape[0]
    p = tw.alloc_packed(N, f, T, C, fb_cap, dev, hybrid=hybrid)
    Y = torch.empty((N, d), dtype=torch.bfloat16, device=dev)
    ws = torch.empty(tw.fwd_workspace_bytes(N, d, f, T, C, fb_cap), dtype=torch.uint8, device=dev)
    tw.twell_ffn_fwd(X, Wi, b, Wd, p, Y, ws)
    assert tw.twell_read_status(p) == 0
    H = torch.empty((N, f), dtype=torch.bfloat16, device=dev)
    tw.twell_unpack(p, H)
    counts = from_dev_bits(p.counts).copy()
    dX = torch.full((N, d), 5.0, dtype=torch.bfloat16, device=dev)
    dWi = torch.full((f, d), 5.0, dtype=torch.float32, device=dev)
    dWd = torch.full((f, d), 5.0, dtype=torch.float32, device=dev)
    db = torch.full((f,), 5.0, dtype=torch.float32, device=dev)
    wsb = torch.full((tw.bwd_workspace_bytes(N, d, f, T, C, fb_cap, hybrid=hybrid),), 0x5A, dtype=torch.uint8,
                     device=dev)
    tw.twell_ffn_bwd(X, Wi, Wd, p, to_dev(dY, torch), lam, dX, dWi, dWd, db, wsb)
    assert tw.twell_read_status(p) == 0
    torch.cuda.synchronize()
    # the backward leaves the layout as it was
    assert np.array_equal(from_dev_bits(p.counts), counts)
    return (from_dev_bits(H), from_dev_bits(dX).copy(), dWi.cpu().numpy(), dWd.cpu().numpy(), db.cpu().numpy(),
            int(p.n_fb[0].item()))


@pytest.mark.parametrize("N,d,f,T,C,lam,seed", [(301, 256, 1024, 64, 8, 1e-3, 1), (200, 512, 2048, 128, 8, 1e-4, 2),
                                               (160, 256, 1024, 32, 4, 0.0, 3)])
def test_tiles_backward(tw, N, d, f, T, C, lam, seed):
    """The tile variant's backward computes the gradients of the same h as
    the row-routed layer: bit for bit the row-routed backward's outputs (the
    rows holding a dense tile are exactly the rows routed whole), and within
    the stated tolerance of the oracle."""
    import torch
    cfg = synth.FFNConfig("tb", N, d, f, T, C, seed=seed, row_spread="lognormal", forced_frac_rows=0.04,
                          l1_lambda=lam)
    inp = synth.make_ffn_inputs(cfg)
    dY = synth.make_grad_output(N, d, seed=seed + 5)
    fb = cfg.fallback_capacity
    rows = _fwd_bwd(tw, torch, inp, dY, lam, T, C, fb, tw.HYBRID_ROWS)
    tiles = _fwd_bwd(tw, torch, inp, dY, lam, T, C, fb, tw.HYBRID_TILES)
    assert rows[5] > 0 and tiles[5] > 0          # fallback rows / dense tiles present
    assert np.array_equal(rows[0], tiles[0])     # the same h
    for a, b, name in zip(rows[1:5], tiles[1:5], ("dX", "dW_inT", "dW_down", "db")):
        assert np.array_equal(a, b), name
    H = tiles[0]
    _, dZ = oracle.grad_hidden(dY, inp["W_down"], H, lam)
    assert_close(synth.bf16_bits_to_f32(tiles[1]), oracle.grad_input(dZ, inp["W_inT"]), "dX")
    rWi, rWd, rdb = oracle.grad_weights(inp["X"], inp["W_down"], H, dY, lam)
    assert_close(tiles[2], rWi, "dW_inT")
    assert_close(tiles[3], rWd, "dW_down")
    assert_close(tiles[4], rdb, "db")
