"""Gated (Llama-style) forward on the GPU -- H = ReLU(X.W_g + b) * (X.W_u) in
one tcgen05 GEMM whose B stage stacks gate and up rows, packed in its
epilogue -- against the oracle (hidden_gated + scalar packer + packed
down-projection)."""
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


def run_gated(tw, torch, inp, T, C, fb_cap):
    dev = torch.device("cuda")
    X, Wg, Wu, b, Wd = (to_dev(inp[k], torch) for k in ("X", "W_inT", "W_uT", "b", "W_down"))
    N, d = inp["X"].shape
    f = inp["W_inT"].shape[0]
    p = tw.alloc_packed(N, f, T, C, fb_cap, dev)
    p.values.view(torch.int16).fill_(0x7777)
    p.idx.fill_(0xAB)
    p.counts.fill_(0xCD)
    Y = torch.full((N, d), 3.0, dtype=torch.bfloat16, device=dev)
    ws = torch.empty(tw.fwd_workspace_bytes(N, d, f, T, C, fb_cap), dtype=torch.uint8, device=dev)
    tw.twell_gated_ffn_fwd(X, Wg, Wu, b, Wd, p, Y, ws)
    rc = tw.twell_read_status(p)
    H = torch.empty((N, f), dtype=torch.bfloat16, device=dev)
    tw.twell_unpack(p, H)
    torch.cuda.synchronize()
    return p, from_dev_bits(H), Y, rc


def check_pack(p, H, T, C, fb_cap):
    ref = oracle.pack(H, T, C, fb_cap)
    assert int(p.n_fb[0].item()) == ref["n_fb"]
    assert np.array_equal(from_dev_bits(p.values).reshape(ref["values"].shape), ref["values"])
    assert np.array_equal(from_dev_bits(p.idx), ref["idx"])
    assert np.array_equal(from_dev_bits(p.counts), ref["counts"])
    assert np.array_equal(from_dev_bits(p.row_fb)[:H.shape[0]], ref["row_fb"])
    return ref


@pytest.mark.parametrize("N,d,f,T,C,sp", [(256, 128, 512, 64, 8, 0.95), (200, 128, 1024, 128, 16, 0.97),
                                          (130, 256, 512, 32, 4, 0.9),
                                          # small batches: one zero-filled M tile, the SpMM split into ranges
                                          (16, 256, 1024, 64, 8, 0.9), (32, 512, 1024, 128, 16, 0.95)])
def test_gated_integer_bit_exact(tw, N, d, f, T, C, sp):
    import torch
    inp = synth.make_integer_inputs(N, d, f, seed=N + f, lo=-1, hi=1, sparsity=sp, gated=True)
    Zg, Hr = oracle.hidden_gated(inp["X"], inp["W_inT"], inp["W_uT"], inp["b"])
    ref = oracle.pack(Hr, T, C, N)
    Yr = oracle.down_packed(ref, inp["W_down"])
    assert np.abs(Yr).max() < 2 ** 24
    p, H, Y, rc = run_gated(tw, torch, inp, T, C, N)
    assert rc == 0, tw.status_string(rc)
    assert np.array_equal(H, Hr)
    check_pack(p, Hr, T, C, N)
    assert np.array_equal(from_dev_bits(Y), oracle.round_bf16(Yr))
    assert (synth.bf16_bits_to_f32(Hr) < 0).any()   # negative products are stored too


def _random_gated(tw, torch, cfg, rows=None):
    inp = synth.make_ffn_inputs(cfg)
    T, C, fb = cfg.tile, cfg.cap, cfg.fallback_capacity
    p, Hg, Y, rc = run_gated(tw, torch, inp, T, C, fb)
    assert rc == 0, tw.status_string(rc)
    ref = check_pack(p, Hg, T, C, fb)
    if rows is None:
        rows = np.arange(cfg.n_rows, dtype=np.int32)
    rows = np.unique(np.concatenate([rows, np.nonzero(ref["row_fb"] >= 0)[0][:32]])).astype(np.int32)
    Zg, Hr = oracle.hidden_gated(inp["X"], inp["W_inT"], inp["W_uT"], inp["b"], rows=rows)
    mism = (Hg[rows] != 0) != (Hr != 0)
    if mism.any():
        assert np.abs(Zg[mism]).max() < 1e-3
    assert_close(synth.bf16_bits_to_f32(Hg[rows]), synth.bf16_bits_to_f32(Hr), "H")
    assert_close(from_dev_f32(Y)[rows], oracle.down_dense(Hr, inp["W_down"]), "Y")
    return ref


def test_gated_random_layer(tw):
    import torch
    cfg = synth.FFNConfig("g", 384, 512, 2048, 128, 16, seed=22, gated=True, fb_cap=64)
    _random_gated(tw, torch, cfg)


def test_gated_full_size_sampled(tw):
    import torch
    cfg = synth.CONFIGS["gated"]
    rows = np.random.default_rng(2).choice(cfg.n_rows, size=48, replace=False).astype(np.int32)
    _random_gated(tw, torch, cfg, rows=rows)
