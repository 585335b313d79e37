"""Training path of the gated (Llama-style) layer on the GPU, against the
oracle: the forward that keeps (g, u) at the stored slots, and the backward
(dG = dh u, dU = dh g at the pattern h != 0, both dX gathers, the unit-major
walk with three outputs, the fallback rows' recomputed g and u and their
tensor-core shares), using the H the GPU's forward produced so both sides share
the pattern."""
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


def _fwd_train(tw, torch, inp, T, C, fb_cap, train=True, hybrid=None):
    dev = torch.device("cuda")
    X, Wg, Wu, b, Wd = (to_dev(inp[k], torch) for k in ("X", "W_inT", "W_uT", "b", "W_down"))
    N, d = inp["X"].shape
    f = inp["W_inT"].shape[0]
    p = tw.alloc_packed(N, f, T, C, fb_cap, dev, hybrid=tw.HYBRID_ROWS if hybrid is None else hybrid)
    Y = torch.full((N, d), 3.0, dtype=torch.bfloat16, device=dev)
    gu = torch.full((N, f // T, C, 2), 7.0, dtype=torch.float32, device=dev)
    ws = torch.empty(tw.fwd_workspace_bytes(N, d, f, T, C, fb_cap), dtype=torch.uint8, device=dev)
    if train:
        tw.twell_gated_ffn_fwd_train(X, Wg, Wu, b, Wd, p, Y, gu, ws)
    else:
        tw.twell_gated_ffn_fwd(X, Wg, Wu, b, Wd, p, Y, ws)
    assert tw.twell_read_status(p) == 0
    return p, Y, gu, (X, Wg, Wu, b, Wd)


def _bwd(tw, torch, p, gu, dev_inp, dY, lam):
    dev = torch.device("cuda")
    X, Wg, Wu, b, Wd = dev_inp
    N, d = X.shape
    f, T, C, fb = p.d_ff, p.tile, p.cap, p.fb_cap
    H = torch.empty((N, f), dtype=torch.bfloat16, device=dev)
    tw.twell_unpack(p, H)
    dX = torch.full((N, d), 5.0, dtype=torch.bfloat16, device=dev)
    outs = [torch.full((f, d), 5.0, dtype=torch.float32, device=dev) for _ in range(3)]
    db = torch.full((f,), 5.0, dtype=torch.float32, device=dev)
    wsb = torch.full((tw.gated_bwd_workspace_bytes(N, d, f, T, C, fb, hybrid=p.hybrid),), 0x5A, dtype=torch.uint8,
                     device=dev)
    tw.twell_gated_ffn_bwd(X, Wg, Wu, b, Wd, p, gu, to_dev(dY, torch), lam, dX, outs[0], outs[1], outs[2], db, wsb)
    assert tw.twell_read_status(p) == 0
    torch.cuda.synchronize()
    return (from_dev_bits(H), from_dev_bits(dX), outs[0].cpu().numpy(), outs[1].cpu().numpy(),
            outs[2].cpu().numpy(), db.cpu().numpy())


def _integer_dy(N, d, seed):
    rng = np.random.default_rng(seed)
    return synth.f32_to_bf16_bits(rng.integers(-1, 2, size=(N, d)).astype(np.float32))


@pytest.mark.parametrize("N,d,f,T,C,sp", [(256, 128, 512, 64, 8, 0.95), (200, 256, 1024, 128, 16, 0.97),
                                          (130, 128, 512, 32, 4, 0.9)])
def test_fwd_train_keeps_gate_and_up(tw, N, d, f, T, C, sp):
    """(g, u) at every stored slot of a TwELL row equal the oracle's g (bias
    applied) and u = X.W_u (integer layer: exact in fp32); the layout and Y are
    those of the plain gated forward."""
    import torch
    inp = synth.make_integer_inputs(N, d, f, seed=N + f, lo=-1, hi=1, sparsity=sp, gated=True)
    p, Y, gu, _ = _fwd_train(tw, torch, inp, T, C, N)
    p0, Y0, _, _ = _fwd_train(tw, torch, inp, T, C, N, train=False)
    n_fb = int(p.n_fb[0].item())
    assert n_fb == int(p0.n_fb[0].item())
    # fb_dense rows past n_fb are never written
    for a, b in ((p.values, p0.values), (p.idx, p0.idx), (p.counts, p0.counts), (p.row_fb, p0.row_fb),
                 (p.fb_dense[:n_fb], p0.fb_dense[:n_fb]), (Y, Y0)):
        assert np.array_equal(from_dev_bits(a), from_dev_bits(b))
    Zg, Hr = oracle.hidden_gated(inp["X"], inp["W_inT"], inp["W_uT"], inp["b"])
    U = synth.bf16_bits_to_f32(inp["X"]) @ synth.bf16_bits_to_f32(inp["W_uT"]).T
    ref = oracle.pack(Hr, T, C, N)
    gu = gu.cpu().numpy()
    counts = ref["counts"]
    idx = ref["idx"].astype(np.int64)
    n, t, s = np.nonzero(np.arange(C)[None, None, :] < counts[:, :, None])
    assert len(n) > 0
    assert (ref["row_fb"][n] < 0).all()       # fallback rows have empty cells
    j = t * T + idx[n, t, s]
    assert np.array_equal(gu[n, t, s, 0], Zg[n, j])
    assert np.array_equal(gu[n, t, s, 1], U[n, j].astype(np.float32))
    assert (Zg[n, j] > 0).all()


@pytest.mark.parametrize("N,d,f,T,C,sp,lam", [(256, 128, 512, 64, 8, 0.92, 1.0),
                                              (200, 256, 1024, 128, 16, 0.9, 0.0),
                                              # no fallback rows
                                              (200, 256, 1024, 128, 16, 0.97, 1.0),
                                              (130, 128, 512, 32, 4, 0.9, 2.0),
                                              # d_ff a multiple of 128 but not of 256: the
                                              # SDDMM on 128-wide tiles
                                              (200, 128, 1152, 64, 8, 0.93, 1.0),
                                              # a small batch (one M tile, zero-filled)
                                              (16, 256, 1024, 64, 8, 0.9, 1.0),
                                              # the epilogue's largest capacity (C = 32), and C = T,
                                              # where no tile can overflow
                                              (160, 128, 512, 64, 32, 0.6, 1.0),
                                              (160, 128, 512, 32, 32, 0.5, 1.0)])
def test_gated_bwd_integer_bit_exact(tw, N, d, f, T, C, sp, lam):
    """Integer layer and integer dY, lambda an integer: dG, dU and every sum are
    exact in fp32 (the fallback rows' dG and dU fit the 16 bits of their high +
    low bf16 parts), so the GPU's gradients equal the oracle's bit for bit."""
    import torch
    inp = synth.make_integer_inputs(N, d, f, seed=N + f + 1, lo=-1, hi=1, sparsity=sp, gated=True)
    dY = _integer_dy(N, d, seed=N)
    p, Y, gu, dev_inp = _fwd_train(tw, torch, inp, T, C, N)
    H, dX, dWg, dWu, dWd, db = _bwd(tw, torch, p, gu, dev_inp, dY, lam)
    _, Hr = oracle.hidden_gated(inp["X"], inp["W_inT"], inp["W_uT"], inp["b"])
    assert np.array_equal(H, Hr)
    n_fb = int(p.n_fb[0].item())
    assert (n_fb > 0) == (sp < 0.97 and C < T)
    dG, dU = oracle.grad_hidden_gated(inp["X"], inp["W_inT"], inp["W_uT"], inp["b"], dY, inp["W_down"], H, lam)
    assert np.abs(np.concatenate([dG, dU])).max() < 2 ** 15
    rdX = oracle.grad_input_gated(dG, dU, inp["W_inT"], inp["W_uT"])
    rWg, rWu, rWd, rdb = oracle.grad_weights_gated(inp["X"], inp["W_inT"], inp["W_uT"], inp["b"], inp["W_down"], H,
                                                   dY, lam)
    for a in (rdX, rWg, rWu, rWd, rdb):
        assert np.abs(a).max() < 2 ** 24
    assert np.array_equal(dX, oracle.round_bf16(rdX))
    assert np.array_equal(dWg, rWg)
    assert np.array_equal(dWu, rWu)
    assert np.array_equal(dWd, rWd)
    assert np.array_equal(db, rdb)


def test_gated_dx_in_passes_integer_bit_exact(tw):
    """W_g and W_u rows larger than the dX gather's L2 budget (2 x 59 MB at
    d_model 2048, d_ff 14336) make it run in passes over tile ranges, with the
    fp32 sums carried between passes: on an integer layer dX (and db) are
    still the oracle's bits."""
    import torch
    N, d, f, T, C, sp, lam = 200, 2048, 14336, 128, 16, 0.95, 1.0
    inp = synth.make_integer_inputs(N, d, f, seed=77, lo=-1, hi=1, sparsity=sp, gated=True)
    dY = _integer_dy(N, d, seed=78)
    p, Y, gu, dev_inp = _fwd_train(tw, torch, inp, T, C, N)
    H, dX, dWg, dWu, dWd, db = _bwd(tw, torch, p, gu, dev_inp, dY, lam)
    assert int(p.n_fb[0].item()) > 0
    dG, dU = oracle.grad_hidden_gated(inp["X"], inp["W_inT"], inp["W_uT"], inp["b"], dY, inp["W_down"], H, lam)
    assert np.abs(np.concatenate([dG, dU])).max() < 2 ** 15
    rdX = oracle.grad_input_gated(dG, dU, inp["W_inT"], inp["W_uT"])
    assert np.abs(rdX).max() < 2 ** 24
    assert np.array_equal(dX, oracle.round_bf16(rdX))
    assert np.array_equal(db, dG.sum(axis=0, dtype=np.float64).astype(np.float32))


def test_gated_bwd_random_layer(tw):
    import torch
    cfg = synth.FFNConfig("g", 384, 512, 2048, 128, 16, seed=23, gated=True, fb_cap=96, row_spread="lognormal",
                          forced_frac_rows=0.03)
    inp = synth.make_ffn_inputs(cfg)
    dY = synth.make_grad_output(cfg.n_rows, cfg.d_model, seed=3)
    lam = 1e-2
    p, Y, gu, dev_inp = _fwd_train(tw, torch, inp, cfg.tile, cfg.cap, cfg.fallback_capacity)
    assert int(p.n_fb[0].item()) > 0
    H, dX, dWg, dWu, dWd, db = _bwd(tw, torch, p, gu, dev_inp, dY, lam)
    dG, dU = oracle.grad_hidden_gated(inp["X"], inp["W_inT"], inp["W_uT"], inp["b"], dY, inp["W_down"], H, lam)
    assert_close(synth.bf16_bits_to_f32(dX), oracle.grad_input_gated(dG, dU, inp["W_inT"], inp["W_uT"]), "dX")
    rWg, rWu, rWd, rdb = oracle.grad_weights_gated(inp["X"], inp["W_inT"], inp["W_uT"], inp["b"], inp["W_down"], H,
                                                   dY, lam)
    assert_close(dWg, rWg, "dW_gT")
    assert_close(dWu, rWu, "dW_uT")
    assert_close(dWd, rWd, "dW_down")
    assert_close(db, rdb, "db")


def test_gated_bwd_full_size_sampled(tw):
    """The gated layer's training shape (N = 4096, d_model 4096, d_ff 14336,
    T 128, C 16, 1% forced-dense rows) checked on sampled rows (dX, with
    fallback rows among them) and sampled hidden units (dW_g, dW_u, dW_down, db
    over all rows)."""
    import torch
    cfg = synth.CONFIGS["gated_train"]
    inp = synth.make_ffn_inputs(cfg)
    dY = synth.make_grad_output(cfg.n_rows, cfg.d_model, seed=78)
    lam = cfg.l1_lambda
    p, Y, gu, dev_inp = _fwd_train(tw, torch, inp, cfg.tile, cfg.cap, cfg.fallback_capacity)
    H, dX, dWg, dWu, dWd, db = _bwd(tw, torch, p, gu, dev_inp, dY, lam)
    rng = np.random.default_rng(6)
    rows = rng.choice(cfg.n_rows, size=24, replace=False)
    fbrows = np.nonzero(from_dev_bits(p.row_fb)[:cfg.n_rows] >= 0)[0][:8]
    assert len(fbrows) > 0
    rows = np.unique(np.concatenate([rows, fbrows])).astype(np.int32)
    dG, dU = oracle.grad_hidden_gated(inp["X"], inp["W_inT"], inp["W_uT"], inp["b"], dY, inp["W_down"], H, lam,
                                      rows=rows)
    assert_close(synth.bf16_bits_to_f32(dX[rows]), oracle.grad_input_gated(dG, dU, inp["W_inT"], inp["W_uT"]), "dX")
    cols = np.sort(rng.choice(cfg.d_ff, size=24, replace=False)).astype(np.int32)
    rWg, rWu, rWd, rdb = oracle.grad_weights_gated(inp["X"], inp["W_inT"], inp["W_uT"], inp["b"], inp["W_down"], H,
                                                   dY, lam, cols=cols)
    assert_close(dWg[cols], rWg, "dW_gT")
    assert_close(dWu[cols], rWu, "dW_uT")
    assert_close(dWd[cols], rWd, "dW_down")
    assert_close(db[cols], rdb, "db")


def test_gated_bwd_refuses(tw):
    """A short workspace is refused before any launch, for either layout
    (the tile-granular one needs room for its row view as well)."""
    import torch
    dev = torch.device("cuda")
    N, d, f, T, C, fb = 64, 128, 512, 64, 8, 16
    X = torch.zeros((N, d), dtype=torch.bfloat16, device=dev)
    W = torch.zeros((f, d), dtype=torch.bfloat16, device=dev)
    b = torch.zeros((f,), dtype=torch.bfloat16, device=dev)
    gu = torch.zeros((N, f // T, C, 2), dtype=torch.float32, device=dev)
    dX = torch.empty((N, d), dtype=torch.bfloat16, device=dev)
    o = [torch.empty((f, d), dtype=torch.float32, device=dev) for _ in range(3)]
    db = torch.empty((f,), dtype=torch.float32, device=dev)
    lib = tw.load_library()
    need = tw.gated_bwd_workspace_bytes(N, d, f, T, C, fb)
    assert need > tw.bwd_workspace_bytes(N, d, f, T, C, fb)
    ws = torch.empty((need,), dtype=torch.uint8, device=dev)
    need_tiles = tw.gated_bwd_workspace_bytes(N, d, f, T, C, fb, hybrid=tw.HYBRID_TILES)
    assert need_tiles > need
    ws = torch.empty((need_tiles,), dtype=torch.uint8, device=dev)
    for hybrid, nbytes, want in ((tw.HYBRID_ROWS, need - 256, -5), (tw.HYBRID_TILES, need_tiles - 256, -5)):
        p = tw.alloc_packed(N, f, T, C, fb, dev, hybrid=hybrid)
        st = p.struct()
        rc = lib.twell_gated_ffn_bwd(X.data_ptr(), W.data_ptr(), W.data_ptr(), b.data_ptr(), W.data_ptr(),
                                     tw.ctypes.byref(st), gu.data_ptr(), d, X.data_ptr(), 0.0, dX.data_ptr(),
                                     o[0].data_ptr(), o[1].data_ptr(), o[2].data_ptr(), db.data_ptr(), ws.data_ptr(),
                                     nbytes, None)
        assert rc == want, tw.status_string(rc)


def test_bwd_empty_batch_zero_weight_gradients(tw):
    """No rows: both backward calls succeed and store zero weight gradients
    (the outputs are overwritten, not accumulated); X, dY and dX have no rows
    and are never dereferenced."""
    import ctypes
    import torch
    dev = torch.device("cuda")
    d, f, T, C, fb = 128, 512, 64, 8, 4
    lib = tw.load_library()
    W = torch.ones((f, d), dtype=torch.bfloat16, device=dev)
    b = torch.ones((f,), dtype=torch.bfloat16, device=dev)
    fake = 0x100   # 256-byte aligned, not null: a row pointer of a zero-row tensor
    ws = torch.empty(max(tw.bwd_workspace_bytes(0, d, f, T, C, fb), tw.gated_bwd_workspace_bytes(0, d, f, T, C, fb),
                         256), dtype=torch.uint8, device=dev)
    p = tw.alloc_packed(0, f, T, C, fb, dev)
    st = p.struct()
    o = [torch.full((f, d), 5.0, dtype=torch.float32, device=dev) for _ in range(3)]
    db = torch.full((f,), 5.0, dtype=torch.float32, device=dev)
    rc = lib.twell_ffn_bwd(fake, W.data_ptr(), W.data_ptr(), ctypes.byref(st), d, fake, 0.5, fake, o[0].data_ptr(),
                           o[1].data_ptr(), db.data_ptr(), ws.data_ptr(), ws.numel(), None)
    torch.cuda.synchronize()
    assert rc == 0, tw.status_string(rc)
    assert not o[0].any() and not o[1].any() and not db.any()
    for t in o + [db]:
        t.fill_(5.0)
    gu = torch.empty((16,), dtype=torch.float32, device=dev)
    rc = lib.twell_gated_ffn_bwd(fake, W.data_ptr(), W.data_ptr(), b.data_ptr(), W.data_ptr(), ctypes.byref(st),
                                 gu.data_ptr(), d, fake, 0.5, fake, o[0].data_ptr(), o[1].data_ptr(), o[2].data_ptr(),
                                 db.data_ptr(), ws.data_ptr(), ws.numel(), None)
    torch.cuda.synchronize()
    assert rc == 0, tw.status_string(rc)
    assert not o[0].any() and not o[1].any() and not o[2].any() and not db.any()


def test_gated_repeat_calls_bit_identical(tw):
    """Forward and backward twice on one workspace (fallback rows present):
    every output has the same bits, as each is summed by one thread in a fixed
    order (no atomics on outputs)."""
    import torch
    cfg = synth.FFNConfig("grep", 300, 512, 2048, 128, 16, seed=29, gated=True, fb_cap=64, row_spread="lognormal",
                          forced_frac_rows=0.03)
    inp = synth.make_ffn_inputs(cfg)
    dY = synth.make_grad_output(cfg.n_rows, cfg.d_model, seed=8)
    outs = []
    for _ in range(2):
        p, Y, gu, dev_inp = _fwd_train(tw, torch, inp, cfg.tile, cfg.cap, cfg.fallback_capacity)
        assert int(p.n_fb[0].item()) > 0
        H, dX, dWg, dWu, dWd, db = _bwd(tw, torch, p, gu, dev_inp, dY, 1e-3)
        outs.append([from_dev_bits(Y), H, dX, dWg.view(np.uint32), dWu.view(np.uint32), dWd.view(np.uint32),
                     db.view(np.uint32)])
    for a, c in zip(*outs):
        assert np.array_equal(a, c)


@pytest.mark.parametrize("N,d,f,T,C,sp", [(256, 128, 512, 64, 8, 0.9), (200, 256, 1024, 128, 16, 0.9),
                                          # a small batch: the gated layer has no separate path for it
                                          (16, 256, 1024, 64, 8, 0.9)])
def test_gated_tiles_forward_integer_bit_exact(tw, N, d, f, T, C, sp):
    """The gated forward on the tile-granular layout: packing (cells, dense
    tiles of the pool in (row, tile) order) and Y equal the oracle's tile
    packer and packed product of the oracle's gated h, bit for bit."""
    import torch
    inp = synth.make_integer_inputs(N, d, f, seed=N + f + 3, lo=-1, hi=1, sparsity=sp, gated=True)
    _, Hr = oracle.hidden_gated(inp["X"], inp["W_inT"], inp["W_uT"], inp["b"])
    fb_cap = N
    ref = oracle.pack_tiles(Hr, T, C, fb_cap * (f // T))
    assert ref["n_fb"] > 0
    Yr = oracle.down_packed(ref, inp["W_down"])
    assert np.abs(Yr).max() < 2 ** 24
    p, Y, gu, _ = _fwd_train(tw, torch, inp, T, C, fb_cap, hybrid=tw.HYBRID_TILES)
    k = min(ref["n_fb"], ref["pool_cap"])
    assert int(p.n_fb[0].item()) == ref["n_fb"]
    assert np.array_equal(from_dev_bits(p.values).reshape(ref["values"].shape), ref["values"])
    assert np.array_equal(from_dev_bits(p.idx), ref["idx"])
    assert np.array_equal(from_dev_bits(p.counts), ref["counts"])
    assert np.array_equal(from_dev_bits(p.fb_dense).reshape(-1, T)[:k], ref["pool"][:k])
    assert np.array_equal(from_dev_bits(Y), oracle.round_bf16(Yr))


def test_gated_tiles_backward_equals_rows(tw):
    """The gated backward of a tile-granular layout runs on its row view: the
    rows holding a dense tile are exactly the rows row routing sends whole, so
    every gradient equals the row-routed layout's bit for bit, and both are
    within tolerance of the oracle."""
    import torch
    cfg = synth.FFNConfig("gt", 301, 256, 1024, 64, 8, seed=41, gated=True, row_spread="lognormal",
                          forced_frac_rows=0.04)
    inp = synth.make_ffn_inputs(cfg)
    dY = synth.make_grad_output(cfg.n_rows, cfg.d_model, seed=12)
    lam = 1e-3
    outs = {}
    for name, hybrid in (("rows", tw.HYBRID_ROWS), ("tiles", tw.HYBRID_TILES)):
        p, Y, gu, dev_inp = _fwd_train(tw, torch, inp, cfg.tile, cfg.cap, cfg.fallback_capacity, hybrid=hybrid)
        assert int(p.n_fb[0].item()) > 0
        counts = from_dev_bits(p.counts).copy()
        outs[name] = _bwd(tw, torch, p, gu, dev_inp, dY, lam)
        assert np.array_equal(from_dev_bits(p.counts), counts)   # the layout is left as it was
    for a, c, what in zip(outs["rows"], outs["tiles"], ("H", "dX", "dW_gT", "dW_uT", "dW_down", "db")):
        assert np.array_equal(a, c), what
    H, dX, dWg, dWu, dWd, db = outs["tiles"]
    dG, dU = oracle.grad_hidden_gated(inp["X"], inp["W_inT"], inp["W_uT"], inp["b"], dY, inp["W_down"], H, lam)
    assert_close(synth.bf16_bits_to_f32(dX), oracle.grad_input_gated(dG, dU, inp["W_inT"], inp["W_uT"]), "dX")
    rWg, rWu, rWd, rdb = oracle.grad_weights_gated(inp["X"], inp["W_inT"], inp["W_uT"], inp["b"], inp["W_down"], H,
                                                   dY, lam)
    assert_close(dWg, rWg, "dW_gT")
    assert_close(dWu, rWu, "dW_uT")
    assert_close(dWd, rWd, "dW_down")
    assert_close(db, rdb, "db")
