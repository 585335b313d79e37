"""Fused forward on the GPU (tcgen05 up-projection with the TwELL-pack
epilogue, routing, dense-fallback recompute, gather-SpMM) against the oracle.

* integer inputs: every sum is exact, so the GPU must match bit for bit;
* random bf16 layers: the packed output is exactly the oracle's packing of the
  H the GPU computed; H agrees with the oracle's except where |z| < 1e-3;
  Y is within the stated tolerance;
* the 1B-scale layer in the bench's launch configuration, checked on sampled
  rows plus every fallback row.
"""
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


def run_fwd(tw, torch, inp, T, C, fb_cap):
    dev = torch.device("cuda")
    X, Wi, b, Wd = (to_dev(inp[k], torch) for k in ("X", "W_inT", "b", "W_down"))
    N, d = inp["X"].shape
    f = inp["W_inT"].shape[0]
    p = tw.alloc_packed(N, f, T, C, fb_cap, dev)
    p.values.view(torch.int16).fill_(0x7777)
    p.idx.fill_(0xAB)
    p.counts.fill_(0xCD)
    Y = torch.full((N, d), 3.0, dtype=torch.bfloat16, device=dev)
    ws = torch.empty(tw.fwd_workspace_bytes(N, d, f, T, C, fb_cap), dtype=torch.uint8, device=dev)
    tw.twell_ffn_fwd(X, Wi, b, Wd, p, Y, ws)
    rc = tw.twell_read_status(p)
    return p, Y, rc


def gpu_h(tw, torch, p):
    H = torch.empty((p.n_rows, p.d_ff), dtype=torch.bfloat16, device="cuda")
    tw.twell_unpack(p, H)
    torch.cuda.synchronize()
    return from_dev_bits(H)


def check_packing_of(p, H, T, C, fb_cap):
    ref = oracle.pack(H, T, C, fb_cap)
    assert int(p.n_fb[0].item()) == ref["n_fb"]
    assert np.array_equal(from_dev_bits(p.values).reshape(ref["values"].shape), ref["values"])
    assert np.array_equal(from_dev_bits(p.idx), ref["idx"])
    assert np.array_equal(from_dev_bits(p.counts), ref["counts"])
    assert np.array_equal(from_dev_bits(p.row_fb)[:H.shape[0]], ref["row_fb"])
    k = min(ref["n_fb"], fb_cap)
    assert np.array_equal(from_dev_bits(p.fb_rows)[:k], ref["fb_rows"][:k])
    assert np.array_equal(from_dev_bits(p.fb_dense)[:k], ref["fb_dense"][:k])
    return ref


INT_CASES = [
    # N, d, f, T, C, sparsity, seed
    (256, 256, 1024, 64, 8, 0.97, 1),
    (200, 128, 1152, 128, 8, 0.95, 2),    # ragged N, d_ff % 256 == 128 (128-wide N tiles)
    (130, 128, 512, 32, 4, 0.9, 3),       # K = two 64-wide steps, many overflow rows
    (384, 512, 2048, 256, 16, 0.98, 4),
    # wide rows: each stored entry's W_down row spans 8, 16 and 32 of the
    # gather's 256-column blocks
    (300, 2048, 1024, 128, 8, 0.97, 5),
    (200, 4096, 1024, 64, 16, 0.95, 6),
    (136, 8192, 512, 128, 8, 0.97, 7),
    # the largest capacity (C = 32), and C = T, where no tile can overflow
    (200, 256, 1024, 64, 32, 0.8, 8),
    (130, 128, 512, 32, 32, 0.5, 9),
    # W_down (73 MB) above the gather's L2 budget per pass: two tile-range
    # passes with fp32 sums carried between them
    (200, 2560, 14336, 128, 16, 0.97, 10),
]


@pytest.mark.parametrize("N,d,f,T,C,sp,seed", INT_CASES)
def test_fwd_integer_bit_exact(tw, N, d, f, T, C, sp, seed):
    import torch
    inp = synth.make_integer_inputs(N, d, f, seed=seed, sparsity=sp)
    fb_cap = N
    ref = oracle.forward(inp["X"], inp["W_inT"], inp["b"], inp["W_down"], T, C, fb_cap)
    assert np.abs(ref["Y"]).max() < 2 ** 24
    p, Y, rc = run_fwd(tw, torch, inp, T, C, fb_cap)
    assert rc == 0, tw.status_string(rc)
    H = gpu_h(tw, torch, p)
    assert np.array_equal(H, ref["H"])
    check_packing_of(p, ref["H"], T, C, fb_cap)
    assert np.array_equal(from_dev_bits(Y), ref["Y_bf16"])


def _check_random_layer(tw, torch, cfg, inp, rows=None):
    T, C, fb = cfg.tile, cfg.cap, cfg.fallback_capacity
    p, Y, rc = run_fwd(tw, torch, inp, T, C, fb)
    assert rc == 0, tw.status_string(rc)
    Hg = gpu_h(tw, torch, p)
    ref_pack = check_packing_of(p, Hg, T, C, fb)
    if rows is None:
        rows = np.arange(cfg.n_rows, dtype=np.int32)
    rows = np.unique(np.concatenate([rows, np.nonzero(ref_pack["row_fb"] >= 0)[0]])).astype(np.int32)
    Z, Hr = oracle.hidden(inp["X"], inp["W_inT"], inp["b"], rows=rows)
    # the pattern (ReLU mask) may differ only where the pre-activation is tiny;
    # values may differ by bf16 rounding of a differently ordered fp32 sum
    mism = (Hg[rows] != 0) != (Hr != 0)
    if mism.any():
        assert np.abs(Z[mism]).max() < 1e-3, np.abs(Z[mism]).max()
        assert mism.mean() < 1e-4
    assert_close(synth.bf16_bits_to_f32(Hg[rows]), synth.bf16_bits_to_f32(Hr), "H")
    Yr = oracle.down_dense(Hr, inp["W_down"])
    assert_close(from_dev_f32(Y)[rows], Yr, "Y")
    return p, ref_pack


def test_fwd_pr1(tw):
    import torch
    cfg = synth.CONFIGS["pr1"]
    inp = synth.make_ffn_inputs(cfg)
    _check_random_layer(tw, torch, cfg, inp)


@pytest.mark.parametrize("N,T,C", [(333, 64, 8), (129, 128, 8), (513, 32, 4), (64, 256, 16)])
def test_fwd_ragged_lognormal(tw, N, T, C):
    import torch
    cfg = synth.FFNConfig("t", N, 256, 1024, T, C, seed=N, row_spread="lognormal", forced_frac_rows=0.03,
                          fb_cap=N // 4 + 4)
    inp = synth.make_ffn_inputs(cfg)
    p, ref = _check_random_layer(tw, torch, cfg, inp)
    assert ref["n_fb"] >= 1


def test_fwd_1b_full_size_sampled(tw):
    import torch
    cfg = synth.CONFIGS["1b"]
    inp = synth.make_ffn_inputs(cfg)
    rows = np.random.default_rng(0).choice(cfg.n_rows, size=256, replace=False)
    rows = np.concatenate([rows, [0, cfg.n_rows - 1]])
    p, ref = _check_random_layer(tw, torch, cfg, inp, rows=rows)
    assert ref["n_fb"] >= len(inp["forced_rows"])
    assert set(inp["forced_rows"].tolist()) <= set(np.nonzero(ref["row_fb"] >= 0)[0].tolist())


def test_fwd_every_row_fallback(tw):
    # C = 1 at ~20% activity: every row overflows, so no row reaches the gather
    # and Y comes whole from the dense-fallback path (integer layer: exact)
    import torch
    N, d, f, T, C = 160, 256, 1024, 64, 1
    inp = synth.make_integer_inputs(N, d, f, seed=12, sparsity=0.8)
    ref = oracle.forward(inp["X"], inp["W_inT"], inp["b"], inp["W_down"], T, C, N)
    assert ref["packed"]["n_fb"] == N
    assert np.abs(ref["Y"]).max() < 2 ** 24
    p, Y, rc = run_fwd(tw, torch, inp, T, C, N)
    assert rc == 0, tw.status_string(rc)
    check_packing_of(p, ref["H"], T, C, N)
    assert np.array_equal(from_dev_bits(Y), ref["Y_bf16"])


def test_fwd_rows_without_entries(tw):
    # rows whose input is zero have z = b <= 0 everywhere: no stored entry, a
    # zero Y row written by the gather (integer layer: exact)
    import torch
    N, d, f, T, C = 200, 256, 1024, 64, 8
    inp = synth.make_integer_inputs(N, d, f, seed=13, sparsity=0.97)
    empty = np.unique(np.concatenate([np.arange(0, 50), np.arange(50, N, 3)]))
    inp["X"][empty] = 0
    ref = oracle.forward(inp["X"], inp["W_inT"], inp["b"], inp["W_down"], T, C, N)
    assert not ref["H"][empty].any()
    p, Y, rc = run_fwd(tw, torch, inp, T, C, N)
    assert rc == 0, tw.status_string(rc)
    check_packing_of(p, ref["H"], T, C, N)
    Yg = from_dev_bits(Y)
    assert np.array_equal(Yg, ref["Y_bf16"])
    assert not Yg[empty].any()


def test_fwd_fallback_overflow_status(tw):
    import torch
    cfg = synth.FFNConfig("t", 256, 256, 1024, 64, 8, seed=3, row_spread="lognormal", forced_frac_rows=0.1,
                          fb_cap=4)
    inp = synth.make_ffn_inputs(cfg)
    p, Y, rc = run_fwd(tw, torch, inp, 64, 8, 4)
    assert rc == -6
    assert int(p.n_fb[0].item()) > 4


def test_fwd_empty_batch(tw):
    import torch
    inp = synth.make_integer_inputs(16, 128, 256, seed=1, sparsity=0.9)
    dev = torch.device("cuda")
    p = tw.alloc_packed(0, 256, 64, 8, 4, dev)
    ws = torch.empty(tw.fwd_workspace_bytes(0, 128, 256, 64, 8, 4), dtype=torch.uint8, device=dev)
    Wi, b, Wd = (to_dev(inp[k], torch) for k in ("W_inT", "b", "W_down"))
    # zero rows: a no-op that still validates its arguments
    st = p.struct()
    lib = tw.load_library()
    import ctypes
    rc = lib.twell_ffn_fwd(0x100, Wi.data_ptr(), b.data_ptr(), Wd.data_ptr(), 0, 128, 256, ctypes.byref(st),
                           0x100, ws.data_ptr(), ws.numel(), None)
    assert rc == 0


def test_dense_comparator_integer_exact(tw):
    # N-major B operand (W_down read as [K][N]) through the tensor cores
    import torch
    inp = synth.make_integer_inputs(200, 256, 1536, seed=6, sparsity=0.97)
    dev = torch.device("cuda")
    X, Wi, b, Wd = (to_dev(inp[k], torch) for k in ("X", "W_inT", "b", "W_down"))
    Hb = torch.empty((200, 1536), dtype=torch.bfloat16, device=dev)
    Y = torch.empty((200, 256), dtype=torch.bfloat16, device=dev)
    tw.twell_dense_ffn_fwd(X, Wi, b, Wd, Hb, Y)
    torch.cuda.synchronize()
    ref = oracle.forward(inp["X"], inp["W_inT"], inp["b"], inp["W_down"], 64, 8, 200)
    assert np.array_equal(from_dev_bits(Hb), ref["H"])
    assert np.array_equal(from_dev_bits(Y), oracle.round_bf16(oracle.down_dense(ref["H"], inp["W_down"])))


def test_dense_comparator(tw):
    import torch
    cfg = synth.CONFIGS["pr1"]
    inp = synth.make_ffn_inputs(cfg)
    dev = torch.device("cuda")
    X, Wi, b, Wd = (to_dev(inp[k], torch) for k in ("X", "W_inT", "b", "W_down"))
    Hb = torch.empty((cfg.n_rows, cfg.d_ff), dtype=torch.bfloat16, device=dev)
    Y = torch.empty((cfg.n_rows, cfg.d_model), dtype=torch.bfloat16, device=dev)
    tw.twell_dense_ffn_fwd(X, Wi, b, Wd, Hb, Y)
    torch.cuda.synchronize()
    Z, Hr = oracle.hidden(inp["X"], inp["W_inT"], inp["b"])
    Hg = from_dev_bits(Hb)
    mism = (Hg != 0) != (Hr != 0)
    assert not mism.any() or np.abs(Z[mism]).max() < 1e-3
    assert_close(from_dev_f32(Y), oracle.down_dense(Hr, inp["W_down"]), "dense Y")


def test_profile_timeline_of_a_forward(tw):
    # the launch timeline of one forward: launch order, streams and device times
    import torch
    cfg = synth.CONFIGS["pr1"]
    inp = synth.make_ffn_inputs(cfg)
    dev = torch.device("cuda")
    X, Wi, b, Wd = (to_dev(inp[k], torch) for k in ("X", "W_inT", "b", "W_down"))
    N, d, f, T, C, fb = cfg.n_rows, cfg.d_model, cfg.d_ff, cfg.tile, cfg.cap, cfg.fallback_capacity
    p = tw.alloc_packed(N, f, T, C, fb, dev)
    Y = torch.empty((N, d), dtype=torch.bfloat16, device=dev)
    ws = torch.empty(tw.fwd_workspace_bytes(N, d, f, T, C, fb), dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    tw.twell_ffn_fwd(X, Wi, b, Wd, p, Y, ws, stream)
    torch.cuda.synchronize()
    tw.twell_profile_reset()
    tw.twell_profile_enable(True)
    tw.twell_ffn_fwd(X, Wi, b, Wd, p, Y, ws, stream)
    tw.twell_profile_enable(False)
    tl = tw.twell_profile_timeline()
    tw.twell_profile_reset()
    assert [e["kernel"] for e in tl] == ["up_pack", "route", "fb_assemble", "fb_down", "fb_down", "spmm"]
    main = int(stream.cuda_stream)
    # routing and the fallback rows on the second stream, the gather-SpMM on the caller's
    assert [e["stream"] == main for e in tl] == [True, False, False, False, False, True]
    assert tl[0]["start_ms"] == 0.0
    for e in tl:
        assert e["end_ms"] >= e["start_ms"] >= 0.0
    for s in (True, False):   # launches on one stream run in order
        seq = [e for e in tl if (e["stream"] == main) == s]
        assert all(a["end_ms"] <= c["start_ms"] + 1e-6 for a, c in zip(seq, seq[1:]))
    assert tl[1]["start_ms"] >= tl[0]["end_ms"] - 1e-6          # routing after the up-projection
    assert tl[2]["start_ms"] >= tl[1]["end_ms"] - 1e-6          # assembly after routing
    assert tl[5]["start_ms"] >= tl[0]["end_ms"] - 1e-6          # the SpMM after the up-projection only
