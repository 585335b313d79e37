"""Failure detection without a GPU fault: the bounded mbarrier wait that
guards every pipeline stage of the GEMM and SpMM kernels is run on a barrier
nothing arrives on.  The wait must give up after its limit, set the status
word to TWELL_ERR_WAIT_TIMEOUT, and leave the context usable for the next
call."""
import time

import numpy as np
import pytest

import oracle
import synth
from twell_check import from_dev_bits, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def tw():
    import __graft_entry__ as g
    g.build()
    import activation_sparse_transformer_gb300 as m
    return m


def test_bounded_wait_reports_timeout_and_context_survives(tw):
    import torch
    status = torch.zeros((4,), dtype=torch.int32, device="cuda")
    t0 = time.perf_counter()
    tw.twell_selftest_wait_timeout(status, 2_000_000)   # 2 ms of GPU time
    torch.cuda.synchronize()
    elapsed = time.perf_counter() - t0
    assert int(status[0].item()) == -7
    assert elapsed < 5.0
    # the context is still usable: an integer layer, bit-exact against the oracle
    inp = synth.make_integer_inputs(128, 128, 512, seed=4, sparsity=0.95)
    X, Wi, b, Wd = (to_dev(inp[k], torch) for k in ("X", "W_inT", "b", "W_down"))
    p = tw.alloc_packed(128, 512, 64, 8, 128, "cuda")
    Y = torch.empty((128, 128), dtype=torch.bfloat16, device="cuda")
    ws = torch.empty(tw.fwd_workspace_bytes(128, 128, 512, 64, 8, 128), dtype=torch.uint8, device="cuda")
    tw.twell_ffn_fwd(X, Wi, b, Wd, p, Y, ws)
    assert tw.twell_read_status(p) == 0
    ref = oracle.forward(inp["X"], inp["W_inT"], inp["b"], inp["W_down"], 64, 8, 128)
    assert np.array_equal(from_dev_bits(Y), ref["Y_bf16"])


def test_wait_timeout_argument_checks(tw):
    import torch
    status = torch.zeros((4,), dtype=torch.int32, device="cuda")
    lib = tw.load_library()
    assert lib.twell_selftest_wait_timeout(None, 1000, None) == -1
    assert lib.twell_selftest_wait_timeout(status.data_ptr(), 0, None) == -1
    assert lib.twell_selftest_wait_timeout(status.data_ptr(), 20_000_000_000, None) == -1
