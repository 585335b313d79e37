"""The dense comparator's backward (twell_dense_ffn_bwd: the layer's
gradients with no sparsity used, the training step the TwELL step is measured
against) against the oracle's gradients.

* a small-integer layer: every product and partial sum is an exact fp32
  integer and every dZ fits bf16 exactly, so the results match bit for bit;
* a random bf16 layer: within the stated tolerance (dZ is kept in bf16)."""
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


def _dense_step(tw, torch, inp, dY, lam):
    dev = torch.device("cuda")
    X, Wi, b, Wd, dYd = (to_dev(a, torch) for a in (inp["X"], inp["W_inT"], inp["b"], inp["W_down"], dY))
    N, d = inp["X"].shape
    f = inp["W_inT"].shape[0]
    Hb = torch.empty((N, f), dtype=torch.bfloat16, device=dev)
    Y = torch.empty((N, d), dtype=torch.bfloat16, device=dev)
    tw.twell_dense_ffn_fwd(X, Wi, b, Wd, Hb, Y)
    dX = torch.full((N, d), 7.0, dtype=torch.bfloat16, device=dev)
    dWi = torch.full((f, d), 7.0, dtype=torch.float32, device=dev)
    dWd = torch.full((f, d), 7.0, dtype=torch.float32, device=dev)
    db = torch.full((f,), 7.0, dtype=torch.float32, device=dev)
    ws = torch.empty(tw.dense_bwd_workspace_bytes(N, d, f), dtype=torch.uint8, device=dev)
    tw.twell_dense_ffn_bwd(X, Wi, Wd, Hb, dYd, lam, dX, dWi, dWd, db, ws)
    torch.cuda.synchronize()
    return from_dev_bits(Hb), from_dev_bits(dX), dWi.cpu().numpy(), dWd.cpu().numpy(), db.cpu().numpy()


@pytest.mark.parametrize("N,d,f,seed", [(256, 128, 512, 1), (200, 256, 768, 2), (136, 128, 1024, 3)])
def test_dense_bwd_integer_bit_exact(tw, N, d, f, seed):
    import torch
    inp = synth.make_integer_inputs(N, d, f, seed=seed, lo=-1, hi=1, sparsity=0.9)
    dY = synth.f32_to_bf16_bits(np.random.default_rng(seed + 9).integers(-1, 2, size=(N, d)).astype(np.float32))
    lam = 1.0
    H, dX, dWi, dWd, db = _dense_step(tw, torch, inp, dY, lam)
    _, Href = oracle.hidden(inp["X"], inp["W_inT"], inp["b"])
    assert np.array_equal(H, Href)
    _, dZ = oracle.grad_hidden(dY, inp["W_down"], Href, lam)
    assert np.abs(dZ).max() <= 256                       # exact in bf16
    assert np.array_equal(dX, oracle.round_bf16(oracle.grad_input(dZ, inp["W_inT"])))
    wi, wd, bb = oracle.grad_weights(inp["X"], inp["W_down"], Href, dY, lam)
    assert np.array_equal(dWi, wi) and np.array_equal(dWd, wd) and np.array_equal(db, bb)


def test_dense_bwd_random_layer(tw):
    import torch
    cfg = synth.FFNConfig("dense_bwd", 300, 256, 1024, 64, 8, seed=5, row_spread="lognormal",
                          forced_frac_rows=0.03, l1_lambda=1e-3)
    inp = synth.make_ffn_inputs(cfg)
    dY = synth.make_grad_output(cfg.n_rows, cfg.d_model, seed=17)
    H, dX, dWi, dWd, db = _dense_step(tw, torch, inp, dY, cfg.l1_lambda)
    # the gradients of the H this forward computed (its pattern may differ from
    # the oracle's only where |z| is tiny)
    Z, Href = oracle.hidden(inp["X"], inp["W_inT"], inp["b"])
    mism = (H != 0) != (Href != 0)
    assert not mism.any() or np.abs(Z[mism]).max() < 1e-3
    _, dZ = oracle.grad_hidden(dY, inp["W_down"], H, cfg.l1_lambda)
    assert_close(synth.bf16_bits_to_f32(dX), oracle.grad_input(dZ, inp["W_inT"]), "dense dX")
    wi, wd, bb = oracle.grad_weights(inp["X"], inp["W_down"], H, dY, cfg.l1_lambda)
    assert_close(dWi, wi, "dense dW_in^T")
    assert_close(dWd, wd, "dense dW_down")
    assert_close(db, bb, "dense db")


def test_dense_bwd_checks_arguments(tw):
    import ctypes
    import torch
    lib = tw.load_library()
    dev = torch.device("cuda")
    a = torch.zeros(1 << 20, dtype=torch.uint8, device=dev)
    p = a.data_ptr()
    need = tw.dense_bwd_workspace_bytes(64, 128, 256)
    assert need >= 64 * 256 * 2
    # a workspace one byte short, a misaligned one, a d_model outside the tiling
    assert lib.twell_dense_ffn_bwd(p, p, p, p, 64, 128, 256, p, ctypes.c_float(0.0), p, p, p, p, p, need - 1,
                                   None) == -5
    assert lib.twell_dense_ffn_bwd(p, p, p, p, 64, 128, 256, p, ctypes.c_float(0.0), p, p, p, p, p + 16, need,
                                   None) == -2
    assert lib.twell_dense_ffn_bwd(p, p, p, p, 64, 192, 256, p, ctypes.c_float(0.0), p, p, p, p, p, need,
                                   None) == -3
