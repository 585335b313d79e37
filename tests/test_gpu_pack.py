"""Standalone dense -> TwELL and TwELL -> dense on the GPU, bit-exact against
the oracle's scalar packer given the same bf16 H (padding bytes, counts,
fallback routing and fallback order included)."""
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


def _pack_on_gpu(tw, torch, H, T, C, fb_cap, ldh=None):
    N, f = H.shape
    dev = torch.device("cuda")
    if ldh is None or ldh == f:
        Hd = to_dev(H, torch)
    else:
        wide = np.zeros((N, ldh), np.uint16)
        wide[:, :f] = H
        wide[:, f:] = 0x3F80  # junk past d_ff must be ignored
        Hd = to_dev(wide, torch)
    p = tw.alloc_packed(N, f, T, C, fb_cap, dev)
    # poison the outputs so that every byte the call owes is checked
    p.values.view(torch.int16).fill_(0x7777)
    p.idx.fill_(0xAB)
    p.counts.fill_(0xCD)
    tw.twell_pack(Hd, p)
    rc = tw.twell_read_status(p)
    return p, rc, Hd


def _compare(p, ref, fb_cap):
    assert int(p.n_fb[0].item()) == ref["n_fb"]
    assert np.array_equal(from_dev_bits(p.values).reshape(ref["values"].shape), ref["values"])
    assert np.array_equal(from_dev_bits(p.idx), ref["idx"])
    assert np.array_equal(from_dev_bits(p.counts), ref["counts"])
    assert np.array_equal(from_dev_bits(p.row_fb)[:ref["row_fb"].shape[0]], ref["row_fb"])
    k = min(ref["n_fb"], fb_cap)
    assert np.array_equal(from_dev_bits(p.fb_rows)[:k], ref["fb_rows"][:k])
    assert np.array_equal(from_dev_bits(p.fb_dense)[:k], ref["fb_dense"][:k])


CASES = [
    # N, f, T, C, activity, seed
    (256, 1024, 64, 8, 0.01, 0),
    (253, 1024, 64, 8, 0.02, 1),       # ragged row count
    (300, 1536, 128, 8, 0.013, 2),     # d_ff not a multiple of 256
    (128, 2048, 256, 16, 0.01, 3),
    (96, 512, 32, 4, 0.03, 4),
    (64, 1024, 128, 32, 0.05, 5),      # largest capacity
    (40, 768, 64, 1, 0.01, 6),         # capacity 1
    (72, 768, 64, 24, 0.25, 7),        # C = 24: cells read as three 8-slot vectors
    (50, 1280, 256, 8, 0.02, 8),       # d_ff = 5 x 256: a 1024-column chunk and a partial one
]


@pytest.mark.parametrize("N,f,T,C,act,seed", CASES)
def test_pack_bit_exact(tw, N, f, T, C, act, seed):
    import torch
    dense_rows = np.arange(3, N, 17)
    H = synth.make_dense_h(N, f, seed=seed, activity=act, dense_rows=dense_rows)
    fb_cap = max(4, oracle.pack(H, T, C, N)["n_fb"] + 3)
    ref = oracle.pack(H, T, C, fb_cap)
    assert ref["n_fb"] >= len(dense_rows) // 2
    p, rc, Hd = _pack_on_gpu(tw, torch, H, T, C, fb_cap)
    assert rc == 0, tw.status_string(rc)
    _compare(p, ref, fb_cap)
    out = torch.empty_like(Hd).fill_(7.0)
    tw.twell_unpack(p, out)
    torch.cuda.synchronize()
    assert np.array_equal(from_dev_bits(out), H)


def test_pack_with_leading_dimension(tw):
    import torch
    H = synth.make_dense_h(130, 1024, seed=9, activity=0.02, dense_rows=[5, 77])
    ref = oracle.pack(H, 64, 8, 8)
    p, rc, _ = _pack_on_gpu(tw, torch, H, 64, 8, 8, ldh=1152)
    assert rc == 0
    _compare(p, ref, 8)


def test_pack_edge_cases(tw):
    import torch
    # all zero: no fallback, all counts 0, canonical padding
    H = np.zeros((77, 512), np.uint16)
    ref = oracle.pack(H, 64, 8, 4)
    p, rc, _ = _pack_on_gpu(tw, torch, H, 64, 8, 4)
    assert rc == 0
    _compare(p, ref, 4)
    # negative zeros are zeros; negative values are non-zeros
    H = synth.make_dense_h(64, 512, seed=2, activity=0.05)
    H[::3, ::5] = 0x8000
    H[1, 3] = 0xBF80  # -1.0
    ref = oracle.pack(H, 64, 8, 8)
    p, rc, _ = _pack_on_gpu(tw, torch, H, 64, 8, 8)
    _compare(p, ref, 8)
    # exactly C fits, C + 1 overflows
    H = np.zeros((3, 256), np.float32)
    H[0, :8] = 1.0
    H[1, 64:73] = 2.0
    H[2, 200] = 3.0
    Hb = synth.f32_to_bf16_bits(H)
    ref = oracle.pack(Hb, 64, 8, 2)
    p, rc, _ = _pack_on_gpu(tw, torch, Hb, 64, 8, 2)
    assert rc == 0 and ref["row_fb"].tolist() == [-1, 0, -1]
    _compare(p, ref, 2)
    # C = T: nothing overflows even when dense
    Hd = synth.make_dense_h(32, 256, seed=4, activity=1.0)
    ref = oracle.pack(Hd, 32, 32, 1)
    p, rc, _ = _pack_on_gpu(tw, torch, Hd, 32, 32, 1)
    assert rc == 0 and ref["n_fb"] == 0
    _compare(p, ref, 1)


def test_pack_fallback_overflow_status(tw):
    import torch
    H = synth.make_dense_h(64, 512, seed=5, activity=0.01, dense_rows=np.arange(0, 64, 4))
    ref = oracle.pack(H, 64, 8, 6)
    assert ref["n_fb"] == 16
    p, rc, _ = _pack_on_gpu(tw, torch, H, 64, 8, 6)
    assert rc == -6
    assert int(p.n_fb[0].item()) == 16
    # the first fb_cap fallback rows are still stored in order
    _compare(p, ref, 6)
    # unpacking the overflowed layout: rows past fb_cap are stored nowhere and
    # come back as zeros, as the oracle's unpack gives them
    out = torch.full((64, 512), 5.0, dtype=torch.bfloat16, device="cuda")
    tw.twell_unpack(p, out)
    torch.cuda.synchronize()
    want = oracle.unpack(ref, 512)
    assert not want[ref["row_fb"] >= 6].any()
    assert np.array_equal(from_dev_bits(out), want)


def test_pack_full_size_1b(tw):
    import torch
    cfg = synth.CONFIGS["1b"]
    N, f = cfg.n_rows, cfg.d_ff
    rng = np.random.default_rng(1)
    dense_rows = np.sort(rng.choice(N, size=82, replace=False))
    H = synth.make_dense_h(N, f, seed=11, activity=0.01, dense_rows=dense_rows)
    ref = oracle.pack(H, cfg.tile, cfg.cap, cfg.fallback_capacity)
    p, rc, Hd = _pack_on_gpu(tw, torch, H, cfg.tile, cfg.cap, cfg.fallback_capacity)
    assert rc == 0
    _compare(p, ref, cfg.fallback_capacity)
    out = torch.empty_like(Hd)
    tw.twell_unpack(p, out)
    torch.cuda.synchronize()
    assert np.array_equal(from_dev_bits(out), H)
    assert oracle.check_format({**ref, "values": from_dev_bits(p.values).reshape(ref["values"].shape)}, f) == 0
