"""Small batches (decode-sized, up to 32 tokens) take their own forward path:
the up-projection with the operands swapped (hidden units on the 128-row MMA
side, tokens as the 16/32-wide N side, K split over the SMs), a CUDA-core pass
that adds the K-split partial sums, biases, rounds and packs, and the
gather-SpMM with each row's tiles cut into ranges.  Checked against the
oracle across the 32-token boundary where the regular path takes over.
"""
import numpy as np
import pytest

import oracle
import synth
from test_gpu_fwd import _check_random_layer, check_packing_of, gpu_h, run_fwd
from twell_check import from_dev_bits

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def tw():
    import __graft_entry__ as g
    g.build()
    import activation_sparse_transformer_gb300 as m
    return m


# N, d, f, T, C, sparsity, seed; N <= 32 runs the small-batch path, 33 the regular one
SMALL_INT_CASES = [
    (1, 256, 1024, 64, 8, 0.95, 11),
    (7, 128, 1152, 128, 8, 0.9, 12),     # ragged token count, d_ff % 256 == 128
    (16, 512, 2048, 128, 16, 0.97, 13),
    (17, 256, 1024, 32, 4, 0.9, 14),     # 32-wide N tile with 15 zero-filled token rows
    (32, 256, 2048, 256, 16, 0.95, 15),
    (33, 256, 1024, 64, 8, 0.95, 16),
]


@pytest.mark.parametrize("N,d,f,T,C,sp,seed", SMALL_INT_CASES)
def test_small_batch_integer_bit_exact(tw, N, d, f, T, C, sp, seed):
    import torch
    inp = synth.make_integer_inputs(N, d, f, seed=seed, sparsity=sp)
    fb_cap = N
    ref = oracle.forward(inp["X"], inp["W_inT"], inp["b"], inp["W_down"], T, C, fb_cap)
    assert np.abs(ref["Y"]).max() < 2 ** 24
    p, Y, rc = run_fwd(tw, torch, inp, T, C, fb_cap)
    assert rc == 0, tw.status_string(rc)
    assert np.array_equal(gpu_h(tw, torch, p), ref["H"])
    check_packing_of(p, ref["H"], T, C, fb_cap)
    assert np.array_equal(from_dev_bits(Y), ref["Y_bf16"])


@pytest.mark.parametrize("N", [3, 16, 24])
def test_small_batch_random_layer(tw, N):
    import torch
    # bias from a calibration batch, as in the decode configuration; a few
    # rows forced dense so the fallback copy and its down-projection run
    cfg = synth.FFNConfig("t", N, 512, 2048, 128, 8, seed=40 + N, sparsity=0.99, calib_rows=1024,
                          row_spread="lognormal", forced_frac_rows=0.2, fb_cap=N)
    inp = synth.make_ffn_inputs(cfg)
    p, ref = _check_random_layer(tw, torch, cfg, inp)
    assert ref["n_fb"] >= 1


def test_small_batch_fallback_overflow_status(tw):
    import torch
    cfg = synth.FFNConfig("t", 8, 256, 1024, 64, 4, seed=5, sparsity=0.9, calib_rows=1024, fb_cap=2)
    inp = synth.make_ffn_inputs(cfg)
    p, Y, rc = run_fwd(tw, torch, inp, 64, 4, 2)
    assert rc == -6
    assert int(p.n_fb[0].item()) > 2


def test_small_batch_overflow_rows_keep_their_y(tw):
    """More fallback rows than fb_cap in a small batch (integer layer, exact
    sums): the status reports the overflow, the packed layout is the
    oracle's packing with that capacity (rows past fb_cap stored nowhere, their
    cells empty), and every row of Y -- those past fb_cap included, which the
    small-batch gather takes from the dense h -- is the exact product."""
    import torch
    N, d, f, T, C, fb_cap = 16, 256, 1024, 64, 4, 2
    inp = synth.make_integer_inputs(N, d, f, seed=21, sparsity=0.85)
    full = oracle.forward(inp["X"], inp["W_inT"], inp["b"], inp["W_down"], T, C, N)
    assert np.abs(full["Y"]).max() < 2 ** 24
    p, Y, rc = run_fwd(tw, torch, inp, T, C, fb_cap)
    assert rc == -6, tw.status_string(rc)   # TWELL_ERR_FALLBACK_OVERFLOW
    ref = check_packing_of(p, full["H"], T, C, fb_cap)
    assert ref["n_fb"] > fb_cap
    past = [r for r in range(N) if ref["row_fb"][r] >= fb_cap]
    assert past and all(not from_dev_bits(p.counts)[r].any() for r in past)
    assert np.array_equal(from_dev_bits(Y), full["Y_bf16"])
