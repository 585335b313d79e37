"""twell_ffn_fwd_noalloc: the forward pass for callers that cannot allocate
device memory (they own no allocator, e.g. inside another framework's pool or
a host application that controls every cudaMalloc).  It must give the same
results as twell_ffn_fwd with a caller-provided workspace, call after call,
and refuse sizes its fixed scratch array cannot hold.  This file is collected
last on purpose."""
import ctypes

import numpy as np
import pytest

import synth
from twell_check import from_dev_bits, from_dev_f32, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def tw():
    import __graft_entry__ as g
    g.build()
    import activation_sparse_transformer_gb300 as m
    return m


def _inputs(torch):
    cfg = synth.FFNConfig("noalloc", 300, 256, 1024, 64, 8, seed=42, row_spread="lognormal",
                          forced_frac_rows=0.05, fb_cap=64)
    inp = synth.make_ffn_inputs(cfg)
    return cfg, [to_dev(inp[k], torch) for k in ("X", "W_inT", "b", "W_down")]


def _snapshot(p, Y):
    return {k: from_dev_bits(getattr(p, k)).copy() for k in ("values", "idx", "counts", "row_fb", "fb_rows",
                                                            "fb_dense", "n_fb")} | {"Y": from_dev_f32(Y)}


def test_noalloc_matches_workspace_call_twice(tw):
    import torch
    lib = tw.load_library()
    cfg, (X, Wi, b, Wd) = _inputs(torch)
    N, d, f, T, C, fb = cfg.n_rows, cfg.d_model, cfg.d_ff, cfg.tile, cfg.cap, cfg.fallback_capacity
    dev = torch.device("cuda")

    ref = tw.alloc_packed(N, f, T, C, fb, dev)
    Yref = torch.empty((N, d), dtype=torch.bfloat16, device=dev)
    ws = torch.empty(tw.fwd_workspace_bytes(N, d, f, T, C, fb), dtype=torch.uint8, device=dev)
    tw.twell_ffn_fwd(X, Wi, b, Wd, ref, Yref, ws)
    assert tw.twell_read_status(ref) == 0
    want = _snapshot(ref, Yref)
    assert want["n_fb"][0] > 0          # the fallback path (which uses the scratch) runs

    stream = torch.cuda.current_stream().cuda_stream
    for call in range(2):
        p = tw.alloc_packed(N, f, T, C, fb, dev)
        p.values.view(torch.int16).fill_(0x7777)
        Y = torch.full((N, d), 9.0, dtype=torch.bfloat16, device=dev)
        st = p.struct()
        rc = lib.twell_ffn_fwd_noalloc(X.data_ptr(), Wi.data_ptr(), b.data_ptr(), Wd.data_ptr(), N, d, f,
                                       ctypes.byref(st), Y.data_ptr(), stream)
        assert rc == 0, tw.status_string(rc)
        assert tw.twell_read_status(p) == 0
        got = _snapshot(p, Y)
        nfb = int(want["n_fb"][0])
        for k in ("values", "idx", "counts", "row_fb"):
            assert np.array_equal(got[k], want[k]), (call, k)
        assert np.array_equal(got["fb_rows"][:nfb], want["fb_rows"][:nfb])
        assert np.array_equal(got["fb_dense"][:nfb], want["fb_dense"][:nfb])
        # the same kernels in the same order on the same inputs: the same bits
        assert np.array_equal(got["Y"], want["Y"]), f"Y call {call}"


def test_noalloc_rejects_sizes_beyond_its_scratch(tw):
    import torch
    lib = tw.load_library()
    cap = int(lib.twell_ffn_fwd_noalloc_max_scratch())
    assert cap == 4 << 20
    cfg, (X, Wi, b, Wd) = _inputs(torch)
    N, d, f, T, C = cfg.n_rows, cfg.d_model, cfg.d_ff, cfg.tile, cfg.cap
    # a fallback capacity whose spill tiles (fb_cap x d_ff bf16) alone exceed the array
    fb_too_many = cap // (f * 2) + 1
    assert tw.fwd_workspace_bytes(N, d, f, T, C, fb_too_many) > cap
    p = tw.alloc_packed(N, f, T, C, fb_too_many, torch.device("cuda"))
    Y = torch.empty((N, d), dtype=torch.bfloat16, device="cuda")
    before = tw.twell_launch_count()
    st = p.struct()
    rc = lib.twell_ffn_fwd_noalloc(X.data_ptr(), Wi.data_ptr(), b.data_ptr(), Wd.data_ptr(), N, d, f,
                                   ctypes.byref(st), Y.data_ptr(), None)
    assert rc == -5 and "workspace" in tw.status_string(rc)
    assert tw.twell_launch_count() == before   # nothing launched
