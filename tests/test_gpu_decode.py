"""Decode-shaped forward (16 tokens, d_model 4096, d_ff 14336, T 128, C 16,
bias calibrated on a separate batch) at the sweep's sparsity levels, against
the oracle.  At 90% most rows overflow C and take the dense fallback."""
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


@pytest.mark.parametrize("cfg", synth.decode_sweep(), ids=lambda c: c.name)
def test_decode_sweep(tw, cfg):
    import torch
    inp = synth.make_ffn_inputs(cfg)
    dev = torch.device("cuda")
    X, Wi, b, Wd = (to_dev(inp[k], torch) for k in ("X", "W_inT", "b", "W_down"))
    N, d, f, T, C, fb = cfg.n_rows, cfg.d_model, cfg.d_ff, cfg.tile, cfg.cap, cfg.n_rows
    p = tw.alloc_packed(N, f, T, C, fb, dev)
    Y = torch.empty((N, d), dtype=torch.bfloat16, device=dev)
    ws = torch.empty(tw.fwd_workspace_bytes(N, d, f, T, C, fb), dtype=torch.uint8, device=dev)
    tw.twell_ffn_fwd(X, Wi, b, Wd, p, Y, ws)
    assert tw.twell_read_status(p) == 0
    H = torch.empty((N, f), dtype=torch.bfloat16, device=dev)
    tw.twell_unpack(p, H)
    torch.cuda.synchronize()
    Hg = from_dev_bits(H)
    ref = oracle.forward(inp["X"], inp["W_inT"], inp["b"], inp["W_down"], T, C, fb)
    mism = (Hg != 0) != (ref["H"] != 0)
    assert not mism.any() or np.abs(ref["Z"][mism]).max() < 1e-3
    mine = oracle.pack(Hg, T, C, fb)
    assert np.array_equal(from_dev_bits(p.counts), mine["counts"])
    assert np.array_equal(from_dev_bits(p.row_fb)[:N], mine["row_fb"])
    assert_close(from_dev_f32(Y), ref["Y"], "Y")
    if cfg.sparsity <= 0.9:
        assert mine["n_fb"] >= N // 2
