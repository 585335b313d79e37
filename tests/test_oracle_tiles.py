"""Pins for the oracle's tile-granular hybrid (a tile with more than C
non-zeros is kept densely in a pool instead of sending its whole row to the
dense fallback).  Each test ties it to something other than itself: a
hand-worked example, brute force over every pattern of an 8-column tile
against the row-granular packer's own brute-force pin, the dense H (exact
round trip), the dense product, and planted format violations.
"""
import numpy as np
import pytest

import oracle
import synth

DENSE = 255


def test_tiles_hand_example():
    # H, 2 rows x 8 columns, T = 4, C = 1 (bf16 bit patterns):
    #   row 0: [0, 1.0, 0, 0 | 2.0, 3.0, 0, 0]
    #   row 1: [0.5, 4.0, 1.5, 0 | 0, 0, 0, 0.25]
    # Worked by hand: row 0 tile 0 holds one non-zero (1.0 at index 1);
    # row 0 tile 1 holds two > C, so it is dense and takes pool slot 0; row 1
    # tile 0 holds three, dense, pool slot 1; row 1 tile 1 holds 0.25 at index 3.
    a, b, c, d, e, f, g = 0x3F80, 0x4000, 0x4040, 0x3F00, 0x4080, 0x3FC0, 0x3E80
    H = np.array([[0, a, 0, 0, b, c, 0, 0],
                  [d, e, f, 0, 0, 0, 0, g]], dtype=np.uint16)
    p = oracle.pack_tiles(H, T=4, C=1, pool_cap=4)
    assert p["n_fb"] == 2
    assert p["counts"].tolist() == [[1, DENSE], [DENSE, 1]]
    assert p["values"][:, :, 0].tolist() == [[a, 0], [1, g]]   # slot numbers 0 and 1 in dense cells
    assert p["idx"][:, :, 0].tolist() == [[1, 0], [0, 3]]
    assert p["row_fb"].tolist() == [-1, -1]
    assert p["pool"][:2].tolist() == [[b, c, 0, 0], [d, e, f, 0]]
    assert not p["pool"][2:].any()
    # pool of one slot: the second dense tile is stored nowhere, its cell empty
    q = oracle.pack_tiles(H, T=4, C=1, pool_cap=1)
    assert q["n_fb"] == 2
    assert q["counts"].tolist() == [[1, DENSE], [0, 1]]
    assert q["values"][1, 0, 0] == 0 and q["idx"][1, 0, 0] == 0
    assert q["pool"][0].tolist() == [b, c, 0, 0]


@pytest.mark.parametrize("C", list(range(1, 9)))
def test_tiles_brute_force_all_patterns(C):
    # Every sparsity pattern of one 8-column tile: with <= C non-zeros the cell
    # is the row packer's cell (itself pinned by brute force); with more the
    # cell is dense, slot 0, and the pool tile is the row itself.
    vals = np.array([0x3F80 + 0x10 * k for k in range(8)], dtype=np.uint16)
    for m in range(256):
        row = np.where([(m >> k) & 1 for k in range(8)], vals, 0).astype(np.uint16)[None, :]
        t = oracle.pack_tiles(row, T=8, C=C, pool_cap=1)
        nz = bin(m).count("1")
        if nz <= C:
            r = oracle.pack(row, T=8, C=C, fb_cap=1)
            assert t["n_fb"] == 0
            assert np.array_equal(t["values"], r["values"]) and np.array_equal(t["idx"], r["idx"])
            assert np.array_equal(t["counts"], r["counts"])
        else:
            assert t["n_fb"] == 1
            assert t["counts"][0, 0] == DENSE
            assert t["values"][0, 0, 0] == 0 and t["idx"][0, 0, 0] == 0
            assert not t["values"][0, 0, 1:].any() and not t["idx"][0, 0, 1:].any()
            assert np.array_equal(t["pool"][0], row[0])
        assert oracle.check_format(t, 8) == 0


def _random_h():
    dense_rows = np.array([3, 17, 18, 40])
    return synth.make_dense_h(64, 1024, seed=7, activity=0.02, dense_rows=dense_rows, dense_activity=0.2)


@pytest.mark.parametrize("T,C", [(64, 4), (128, 8), (32, 2), (256, 16)])
def test_tiles_roundtrip_order_and_row_relation(T, C):
    H = _random_h()
    N, f = H.shape
    nt = f // T
    t = oracle.pack_tiles(H, T, C, pool_cap=N * nt)
    r = oracle.pack(H, T, C, fb_cap=N)
    assert oracle.check_format(t, f) == 0
    assert np.array_equal(oracle.unpack(t, f), H)
    # a row the row-granular hybrid keeps in TwELL is packed identically
    twell_rows = r["row_fb"] < 0
    assert np.array_equal(t["values"][twell_rows], r["values"][twell_rows])
    assert np.array_equal(t["counts"][twell_rows], r["counts"][twell_rows])
    # dense tiles are exactly H's over-full tiles, numbered in (row, tile) order
    nz = (H.reshape(N, nt, T) & 0x7FFF).astype(bool).sum(axis=2)
    over = nz > C
    assert t["n_fb"] == int(over.sum())
    assert np.array_equal(t["counts"] == DENSE, over)
    slots = t["values"][:, :, 0].astype(np.int64) | (t["idx"][:, :, 0].astype(np.int64) << 16)
    assert np.array_equal(slots[over], np.arange(int(over.sum())))
    for (n, k) in zip(*np.nonzero(over)):
        assert np.array_equal(t["pool"][slots[n, k]], H[n, k * T:(k + 1) * T])
    # the rows the row-granular hybrid sends whole are those holding a dense tile
    assert np.array_equal(r["row_fb"] >= 0, over.any(axis=1))


def test_tiles_packed_product_equals_dense_bitwise():
    H = _random_h()
    N, f = H.shape
    rng = np.random.default_rng(3)
    W = synth.f32_to_bf16_bits(rng.standard_normal((f, 48)).astype(np.float32))
    t = oracle.pack_tiles(H, 64, 4, pool_cap=N * (f // 64))
    assert t["n_fb"] > 0
    assert np.array_equal(oracle.down_packed(t, W).view(np.uint32), oracle.down_dense(H, W).view(np.uint32))


def test_tiles_special_cases():
    H = _random_h()
    N, f = H.shape
    z = oracle.pack_tiles(np.zeros_like(H), 64, 4, pool_cap=8)
    assert z["n_fb"] == 0 and not z["counts"].any()
    full = oracle.pack_tiles(H, 64, 64, pool_cap=8)        # C = T: nothing can overflow
    assert full["n_fb"] == 0
    assert np.array_equal(oracle.unpack(full, f), H)


def test_tiles_format_checker_catches_violations():
    H = _random_h()
    N, f = H.shape
    t = oracle.pack_tiles(H, 64, 4, pool_cap=N * (f // 64))
    assert oracle.check_format(t, f) == 0
    dense = np.argwhere(t["counts"] == DENSE)
    assert len(dense) >= 2

    def broken(mut):
        u = {k: (v.copy() if isinstance(v, np.ndarray) else v) for k, v in t.items()}
        mut(u)
        return oracle.check_format(u, f)

    (n0, k0), (n1, k1) = dense[0], dense[1]

    def swap_slots(u):
        u["values"][n0, k0, 0], u["values"][n1, k1, 0] = u["values"][n1, k1, 0], u["values"][n0, k0, 0]

    def row_routed(u):
        u["row_fb"][n0] = 0

    def thin_pool_tile(u):
        u["pool"][0][:] = 0

    def miscount(u):
        u["n_fb"] += 1

    def dirty_padding(u):
        u["idx"][n0, k0, 1] = 5

    assert broken(swap_slots) == 10
    assert broken(row_routed) == 7
    assert broken(thin_pool_tile) == 12
    assert broken(miscount) == 11
    assert broken(dirty_padding) == 6
