"""twell_check_format on the GPU against the oracle's format checker: layouts
from the oracle's packers (and from twell_pack), each with planted violations
of one rule.  The device reports a mask of every broken rule, the oracle the
first rule it meets, so the two agree when the mask is empty exactly when the
oracle returns 0 and the oracle's rule is in the mask; where a mutation breaks
one rule only, the mask is that rule's bit alone."""
import numpy as np
import pytest

import oracle
import synth
from twell_check import to_dev

pytestmark = pytest.mark.gpu

BAD_FORMAT = -9


@pytest.fixture(scope="module")
def tw():
    import __graft_entry__ as g
    g.build()
    import activation_sparse_transformer_gb300 as m
    return m


def _upload(tw, d, f, fb_cap):
    """Device copy of an oracle layout dict (rows or tiles variant)."""
    import torch
    tiles = d.get("hybrid") == "tiles"
    N = d["counts"].shape[0]
    p = tw.alloc_packed(N, f, d["T"], d["C"], fb_cap, "cuda", hybrid=tw.HYBRID_TILES if tiles else tw.HYBRID_ROWS)
    p.values.copy_(to_dev(d["values"], torch))
    p.idx.copy_(torch.from_numpy(np.ascontiguousarray(d["idx"])).cuda())
    p.counts.copy_(torch.from_numpy(np.ascontiguousarray(d["counts"])).cuda())
    if N:
        p.row_fb.copy_(torch.from_numpy(np.ascontiguousarray(d["row_fb"])).cuda())
    if fb_cap:
        dense = d["pool"].reshape(fb_cap, f) if tiles else d["fb_dense"]
        p.fb_dense.copy_(to_dev(dense, torch))
        if not tiles:
            p.fb_rows.copy_(torch.from_numpy(np.ascontiguousarray(d["fb_rows"])).cuda())
    p.n_fb[0] = int(d["n_fb"])
    p.status.zero_()
    return p


def _device_mask(tw, p):
    import torch
    v = torch.full((4,), 0x5A5A, dtype=torch.int32, device="cuda")  # the call zeroes it first
    tw.twell_check_format(p, v)
    torch.cuda.synchronize()
    # the raw status word (twell_read_status would also report an overflowed n_fb)
    return int(v[0].item()), int(p.status[0].item())


def _copy(d):
    return {k: (v.copy() if isinstance(v, np.ndarray) else v) for k, v in d.items()}


def _agree(tw, d, f, fb_cap, exact=None):
    code = oracle.check_format(d, f)
    mask, status = _device_mask(tw, _upload(tw, d, f, fb_cap))
    assert (mask == 0) == (code == 0), (code, bin(mask))
    if code:
        assert mask >> code & 1, (code, bin(mask))
        assert status == BAD_FORMAT
    else:
        assert status == 0
    if exact is not None:
        assert code == exact and mask == 1 << exact, (code, bin(mask))
    return code, mask


def test_rows_variant_each_rule(tw):
    N, f, T, C, fb_cap = 40, 256, 64, 4, 8
    H = synth.make_dense_h(N, f, seed=2, activity=0.02, dense_rows=[3, 17])
    good = oracle.pack(H, T, C, fb_cap)
    assert _agree(tw, good, f, fb_cap)[0] == 0
    fbr = [int(r) for r in np.flatnonzero(good["row_fb"] >= 0)]
    assert len(fbr) >= 2 and good["n_fb"] == len(fbr) < 7
    r, t = next((r, t) for r in range(N) for t in range(f // T)
                if good["counts"][r, t] >= 2 and good["row_fb"][r] < 0)
    r0, t0 = next((r, t) for r in range(N) for t in range(f // T)
                  if good["counts"][r, t] < C and good["row_fb"][r] < 0)
    tw_row = next(r for r in range(N) if good["row_fb"][r] < 0 and good["counts"][r].any())

    def case(fn, exact=None, expect=None):
        d = _copy(good)
        fn(d)
        code, _ = _agree(tw, d, f, fb_cap, exact)
        if expect is not None:
            assert code == expect

    case(lambda d: d["counts"].__setitem__((r, t), C + 1), exact=1)
    case(lambda d: d["counts"].__setitem__((fbr[0], 0), 1), expect=2)
    case(lambda d: d["idx"].__setitem__((r, t, 0), T), expect=3)
    case(lambda d: d["idx"].__setitem__((r, t, 1), d["idx"][r, t, 0]), exact=4)
    case(lambda d: d["values"].__setitem__((r, t, 0), 0), exact=5)
    case(lambda d: d["values"].__setitem__((r, t, 0), 0x8000), exact=5)        # -0.0 is zero
    case(lambda d: d["idx"].__setitem__((r0, t0, C - 1), 1), exact=6)
    case(lambda d: d["values"].__setitem__((r0, t0, C - 1), 0x3F80), exact=6)
    case(lambda d: d["row_fb"].__setitem__(tw_row, 1), expect=7)
    case(lambda d: d["row_fb"].__setitem__(0, -2), exact=7)
    case(lambda d: d["fb_rows"].__setitem__(0, fbr[0] + 1), exact=7)

    def renumber(d):
        d["row_fb"][fbr[-1]] = 7
        d["fb_rows"][7] = fbr[-1]
    case(renumber, exact=8)

    def swap_slots(d):
        d["row_fb"][fbr[0]], d["row_fb"][fbr[1]] = 1, 0
        d["fb_rows"][:2] = [fbr[1], fbr[0]]
    case(swap_slots, exact=8)
    case(lambda d: d.__setitem__("n_fb", 1), exact=9)
    case(lambda d: d.__setitem__("n_fb", len(fbr) + 1))             # also reads an unset fb_rows entry
    # a NaN compares unequal to zero: a legal stored value
    case(lambda d: d["values"].__setitem__((r, t, 0), 0x7FC0), expect=0)


def test_rows_variant_overflow_and_edges(tw):
    N, f, T, C = 40, 256, 64, 4
    H = synth.make_dense_h(N, f, seed=2, activity=0.02, dense_rows=[3, 17])
    over = oracle.pack(H, T, C, 1)
    assert over["n_fb"] > 1
    assert _agree(tw, over, f, 1)[0] == 0                 # rows past fb_cap keep their numbers
    no_fb = oracle.pack(H, T, C, 0)
    assert _agree(tw, no_fb, f, 0)[0] == 0
    empty = oracle.pack(np.zeros((0, f), np.uint16), T, C, 4)
    assert _agree(tw, empty, f, 4)[0] == 0
    bad = _copy(empty)
    bad["n_fb"] = 1
    assert _agree(tw, bad, f, 4, exact=9)[0] == 9


def test_rows_variant_many_passes_and_device_pack(tw):
    import torch
    N, f, T, C, fb_cap = 3000, 2048, 128, 8, 256
    H = synth.make_dense_h(N, f, seed=31, activity=0.01, dense_rows=np.arange(7, N, 23), dense_activity=0.2)
    good = oracle.pack(H, T, C, fb_cap)
    fbr = [int(r) for r in np.flatnonzero(good["row_fb"] >= 0)]
    assert 100 < len(fbr) < fb_cap - 1 and fbr[-1] > 2048   # the scan takes several 1024-row passes
    assert _agree(tw, good, f, fb_cap)[0] == 0
    d = _copy(good)
    k = len(fbr) - 1
    d["row_fb"][fbr[k]] = k + 1
    d["fb_rows"][k + 1] = fbr[k]
    _agree(tw, d, f, fb_cap, exact=8)
    # the library's own pack output passes
    p = tw.alloc_packed(N, f, T, C, fb_cap, "cuda")
    tw.twell_pack(to_dev(H, torch), p)
    assert tw.twell_read_status(p) == 0
    assert _device_mask(tw, p) == (0, 0)


def test_tiles_variant_each_rule(tw):
    N, f, T, C, fb_cap = 64, 1024, 64, 4, 16
    nt = f // T
    H = synth.make_dense_h(N, f, seed=9, activity=0.02, dense_rows=np.arange(0, N, 8), dense_activity=0.3)
    good = oracle.pack_tiles(H, T, C, fb_cap * nt)
    assert 2 < good["n_fb"] < fb_cap * nt
    assert _agree(tw, good, f, fb_cap)[0] == 0
    dense = [(r, t) for r in range(N) for t in range(nt) if good["counts"][r, t] == 255]
    (ra, ta), (rb, tb) = dense[0], dense[1]

    def case(fn, exact=None, expect=None):
        d = _copy(good)
        fn(d)
        code, _ = _agree(tw, d, f, fb_cap, exact)
        if expect is not None:
            assert code == expect

    case(lambda d: d["values"].__setitem__((ra, ta, 0), 1), exact=10)          # first dense tile names slot 1
    case(lambda d: d["idx"].__setitem__((rb, tb, 0), 1), exact=10)             # slot 1 + 2^16: past the pool
    case(lambda d: d["counts"].__setitem__((ra, ta), 200), expect=1)
    case(lambda d: d["row_fb"].__setitem__(5, 0), exact=7)
    case(lambda d: d["idx"].__setitem__((ra, ta, 1), 3), exact=6)
    case(lambda d: d["pool"].__setitem__((0, slice(C, None)), 0), exact=12)     # at most C non-zeros left
    case(lambda d: d.__setitem__("n_fb", good["n_fb"] + 1), exact=11)
    r, t = next((r, t) for r in range(N) for t in range(nt) if 2 <= good["counts"][r, t] <= C)
    case(lambda d: d["idx"].__setitem__((r, t, 0), d["idx"][r, t, 1]), exact=4)


def test_tiles_variant_overflow_and_many_passes(tw):
    import torch
    N, f, T, C = 64, 1024, 64, 4
    H = synth.make_dense_h(N, f, seed=9, activity=0.02, dense_rows=np.arange(0, N, 4), dense_activity=0.3)
    over = oracle.pack_tiles(H, T, C, 1 * (f // T))
    assert over["n_fb"] > 16
    assert _agree(tw, over, f, 1)[0] == 0
    # 3000 x 16 cells: the dense-tile numbering takes ~47 passes of the scan
    N, f, T, C, fb_cap = 3000, 2048, 128, 8, 128
    H = synth.make_dense_h(N, f, seed=33, activity=0.01, dense_rows=np.arange(5, N, 29), dense_activity=0.2)
    good = oracle.pack_tiles(H, T, C, fb_cap * (f // T))
    assert 100 < good["n_fb"] < fb_cap * (f // T)
    assert _agree(tw, good, f, fb_cap)[0] == 0
    cells = np.argwhere(good["counts"] == 255)
    r, t = (int(x) for x in cells[-1])
    assert r * (f // T) + t > 1024
    d = _copy(good)
    d["values"][r, t, 0] += 1
    d["pool"][d["values"][r, t, 0]] = d["pool"][d["values"][r, t, 0] - 1]  # keep the named tile dense
    _agree(tw, d, f, fb_cap, exact=10)
    p = tw.alloc_packed(N, f, T, C, fb_cap, "cuda", hybrid=tw.HYBRID_TILES)
    tw.twell_pack(to_dev(H, torch), p)
    assert tw.twell_read_status(p) == 0
    assert _device_mask(tw, p) == (0, 0)
