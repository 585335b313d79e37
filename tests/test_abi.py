"""The C-ABI library loads and exports every entry point include/twell.h
declares; host-side argument checks return their codes without a GPU."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    with open(os.path.join(ROOT, "include", "twell.h")) as fh:
        src = fh.read()
    return sorted(set(re.findall(r"TWELL_API\s+[\w\s\*]+?\b(twell_\w+)\s*\(", src)))


@pytest.fixture(scope="module")
def lib():
    import __graft_entry__ as g
    g.build()
    import activation_sparse_transformer_gb300 as tw
    return tw.load_library()


def test_header_declares_the_four_layer_calls():
    names = _declared()
    for n in ("twell_pack", "twell_unpack", "twell_ffn_fwd", "twell_ffn_bwd"):
        assert n in names
    assert len(names) >= 13


def test_every_declared_symbol_is_exported(lib):
    import activation_sparse_transformer_gb300 as tw
    for n in _declared():
        assert hasattr(lib, n), n
    assert sorted(tw.EXPORTED) == _declared()


def test_status_strings(lib):
    import activation_sparse_transformer_gb300 as tw
    for code in range(0, -10, -1):
        s = tw.status_string(code)
        assert s and s != "unknown status"
    assert tw.status_string(-100) == "unknown status"


def test_host_argument_checks_without_gpu(lib):
    import activation_sparse_transformer_gb300 as tw
    L = tw.twell_t(16, 1024, 64, 8, 4, 0, 0x1000, 0x2000, 0x3000, 0x4000, 0x5000, 0x6000, 0x7000, 0x8000)
    # null layout
    assert lib.twell_pack(ctypes.c_void_p(0x10000), 1024, None, None) == -1
    # bad tile
    bad = tw.twell_t(16, 1024, 48, 8, 4, 0, 0x1000, 0x2000, 0x3000, 0x4000, 0x5000, 0x6000, 0x7000, 0x8000)
    assert lib.twell_pack(ctypes.c_void_p(0x10000), 1024, ctypes.byref(bad), None) == -1
    # capacity above T
    bad = tw.twell_t(16, 1024, 32, 33, 4, 0, 0x1000, 0x2000, 0x3000, 0x4000, 0x5000, 0x6000, 0x7000, 0x8000)
    assert lib.twell_pack(ctypes.c_void_p(0x10000), 1024, ctypes.byref(bad), None) == -1
    # misaligned pointer in the layout
    bad = tw.twell_t(16, 1024, 64, 8, 4, 0, 0x1001, 0x2000, 0x3000, 0x4000, 0x5000, 0x6000, 0x7000, 0x8000)
    assert lib.twell_pack(ctypes.c_void_p(0x10000), 1024, ctypes.byref(bad), None) == -2
    # d_ff not a multiple of 128 (but of T)
    bad = tw.twell_t(16, 960, 64, 8, 4, 0, 0x1000, 0x2000, 0x3000, 0x4000, 0x5000, 0x6000, 0x7000, 0x8000)
    assert lib.twell_pack(ctypes.c_void_p(0x10000), 1024, ctypes.byref(bad), None) == -3
    # unknown hybrid variant; tile pool too large for 24-bit slots
    bad = tw.twell_t(16, 1024, 64, 8, 4, 7, 0x1000, 0x2000, 0x3000, 0x4000, 0x5000, 0x6000, 0x7000, 0x8000)
    assert lib.twell_pack(ctypes.c_void_p(0x10000), 1024, ctypes.byref(bad), None) == -1
    bad = tw.twell_t(16, 1024, 64, 8, 1 << 21, tw.HYBRID_TILES, 0x1000, 0x2000, 0x3000, 0x4000, 0x5000, 0x6000,
                     0x7000, 0x8000)
    assert lib.twell_pack(ctypes.c_void_p(0x10000), 1024, ctypes.byref(bad), None) == -3
    # the wait self-test checks its arguments on the host
    assert lib.twell_selftest_wait_timeout(None, 1000, None) == -1
    assert lib.twell_selftest_wait_timeout(ctypes.c_void_p(0x10000), 0, None) == -1
    # the format check wants an aligned result word
    assert lib.twell_check_format(None, ctypes.c_void_p(0x10000), None) == -1
    assert lib.twell_check_format(ctypes.byref(L), None, None) == -1
    assert lib.twell_check_format(ctypes.byref(L), ctypes.c_void_p(0x10002), None) == -2
    assert lib.twell_check_format(ctypes.byref(bad), ctypes.c_void_p(0x10000), None) == -3
    # the launch timeline: a negative count, or entries asked for without the arrays
    assert lib.twell_profile_timeline(-1, None, None, None, None) == -1
    assert lib.twell_profile_timeline(4, None, None, None, None) == -1
    # a well-formed call reaches the device check and stops there on a CPU-only host
    rc = lib.twell_pack(ctypes.c_void_p(0x10000), 1024, ctypes.byref(L), None)
    try:
        import torch
        gpu = torch.cuda.is_available()
    except Exception:
        gpu = False
    if not gpu:
        assert rc == -8
    # workspace sizes are pure host arithmetic
    # forward: spilled dense tiles (fb_cap * n_tiles tiles of T bf16), a counter,
    # and K-split partial sums of the fallback rows' down-projection
    ws = tw.fwd_workspace_bytes(4096, 2048, 8192, 128, 8, 512)
    assert ws >= 512 * 64 * 128 * 2 + 512 * 2048 * 4
    assert ws % 256 == 0
    assert tw.fwd_workspace_bytes(4096, 2048, 8192, 128, 8, 0) > 0
    assert tw.bwd_workspace_bytes(4096, 2048, 8192, 128, 8, 512) > 4096 * 64 * 8 * 4


def test_missing_library_fails_loudly(monkeypatch, tmp_path):
    # no CPU or eager fallback: without libtwell.so every call raises
    import pytest

    import activation_sparse_transformer_gb300 as tw
    monkeypatch.setattr(tw, "_lib_handle", None)
    monkeypatch.setattr(tw, "LIB_PATH", str(tmp_path / "libtwell.so"))
    with pytest.raises(RuntimeError):
        tw.load_library()
    with pytest.raises(RuntimeError):
        tw.fwd_workspace_bytes(16, 128, 256, 64, 8, 4)


def test_binding_rejects_short_buffers(lib):
    """The C ABI receives bare pointers, so the binding refuses a tensor with
    fewer bytes than the call reads or writes through it; correctly sized CPU
    tensors are then refused as not on the device (there is no CPU path)."""
    import torch
    import activation_sparse_transformer_gb300 as tw
    N, d, f, T, C = 16, 128, 256, 64, 4
    bf = dict(dtype=torch.bfloat16)
    p = tw.alloc_packed(N, f, T, C, 2, "cpu")
    X, Wi, Wd = torch.empty((N, d), **bf), torch.empty((f, d), **bf), torch.empty((f, d), **bf)
    b, ws = torch.empty(f, **bf), torch.empty(64, dtype=torch.uint8)
    with pytest.raises(ValueError, match="^Y: "):
        tw.twell_ffn_fwd(X, Wi, b, Wd, p, torch.empty((N, d - 8), **bf), ws)
    with pytest.raises(ValueError, match="^b: "):
        tw.twell_ffn_fwd(X, Wi, b[: f - 1], Wd, p, torch.empty((N, d), **bf), ws)
    with pytest.raises(ValueError, match="CUDA"):
        tw.twell_ffn_fwd(X, Wi, b, Wd, p, torch.empty((N, d), **bf), ws)
    # a gradient buffer of bf16 where fp32 is written is too short
    dX, db = torch.empty((N, d), **bf), torch.empty(f, dtype=torch.float32)
    dWd = torch.empty((f, d), dtype=torch.float32)
    with pytest.raises(ValueError, match="^dW_inT: "):
        tw.twell_ffn_bwd(X, Wi, Wd, p, X, 0.0, dX, torch.empty((f, d), **bf), dWd, db, ws)
    # the packed layout's own buffers
    short = tw.alloc_packed(N, f, T, C, 2, "cpu")
    short.values = short.values[: N - 1]
    with pytest.raises(ValueError, match="^values: "):
        tw.twell_unpack(short, torch.empty((N, f), **bf))
    with pytest.raises(ValueError, match="^H: "):
        tw.twell_pack(torch.empty((N - 1, f), **bf), p)
    with pytest.raises(ValueError, match="^violations: "):
        tw.twell_check_format(p, torch.empty(0, dtype=torch.int32))


def test_gated_host_argument_checks_without_gpu(lib):
    """The gated calls refuse bad arguments on the host, before any launch:
    no up matrix, no or misaligned (g, u) buffer, a tile wider than the gated
    GEMM's 128-unit halves, a short or misaligned workspace."""
    import activation_sparse_transformer_gb300 as tw
    P = ctypes.c_void_p
    a = P(0x10000)   # aligned fake device pointers, never dereferenced
    N, d, f = 16, 128, 1024
    L = tw.twell_t(N, f, 64, 8, 4, 0, 0x1000, 0x2000, 0x3000, 0x4000, 0x5000, 0x6000, 0x7000, 0x8000)
    ws = 1 << 30
    # forward: no W_u, no (g, u), misaligned (g, u), T = 256
    assert lib.twell_gated_ffn_fwd(a, a, None, a, a, N, d, f, ctypes.byref(L), a, a, ws, None) == -1
    assert lib.twell_gated_ffn_fwd_train(a, a, a, a, a, N, d, f, ctypes.byref(L), a, None, a, ws, None) == -1
    assert lib.twell_gated_ffn_fwd_train(a, a, a, a, a, N, d, f, ctypes.byref(L), a, P(0x10008), a, ws,
                                         None) == -2
    wide = tw.twell_t(N, f, 256, 8, 4, 0, 0x1000, 0x2000, 0x3000, 0x4000, 0x5000, 0x6000, 0x7000, 0x8000)
    assert lib.twell_gated_ffn_fwd(a, a, a, a, a, N, d, f, ctypes.byref(wide), a, a, ws, None) == -3

    def bwd(layout, gu, workspace, nbytes):
        return lib.twell_gated_ffn_bwd(a, a, a, a, a, ctypes.byref(layout), gu, d, a, ctypes.c_float(0.0), a, a, a,
                                       a, a, workspace, nbytes, None)

    need = tw.gated_bwd_workspace_bytes(N, d, f, 64, 8, 4)
    assert need > tw.bwd_workspace_bytes(N, d, f, 64, 8, 4)
    assert tw.gated_bwd_workspace_bytes(N, d, f, 64, 8, 4, hybrid=tw.HYBRID_TILES) > need
    assert bwd(L, None, a, need) == -1
    assert bwd(L, P(0x10004), a, need) == -2
    assert bwd(L, a, a, need - 256) == -5
    assert bwd(L, a, None, need) == -5
    assert bwd(L, a, P(0x10010), need) == -2
    tiles = tw.twell_t(N, f, 64, 8, 4, tw.HYBRID_TILES, 0x1000, 0x2000, 0x3000, 0x4000, 0x5000, 0x6000, 0x7000,
                       0x8000)
    assert bwd(tiles, a, a, need) == -5   # the row view needs room beyond the row layout's workspace
