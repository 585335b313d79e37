"""Randomised pins of the oracle's packers and format checkers: on random
shapes, capacities, fallback capacities and activities (negative values and
-0.0 included), the packed layout satisfies invariants computed here with
numpy, independently of the oracle: per-tile counts, which rows (or tiles)
leave TwELL, their numbering, and the round trip back to H (bit for bit in
the dense parts, with -0.0 read as zero in the cells)."""
import numpy as np
import pytest

import oracle
import synth

hypothesis = pytest.importorskip("hypothesis")
from hypothesis import given, settings, strategies as st  # noqa: E402


def _random_h(N, f, seed, act, dense_frac):
    rng = np.random.default_rng(seed)
    dense_rows = np.flatnonzero(rng.random(N) < dense_frac)
    H = synth.make_dense_h(N, f, seed, activity=act, dense_rows=dense_rows, dense_activity=0.5)
    flip = rng.random((N, f)) < 0.1
    H = np.where(flip, H | np.uint16(0x8000), H)          # negatives, and -0.0 where H was +0
    return H.astype(np.uint16)


def _nonzero(H):
    return (H & 0x7FFF) != 0


SHAPES = dict(N=st.integers(0, 24), nt=st.integers(1, 4), T=st.sampled_from([32, 64]), C=st.integers(1, 8),
              cap=st.integers(0, 6), act=st.floats(0.0, 0.3), dense=st.floats(0.0, 0.5),
              seed=st.integers(0, 2 ** 31 - 1))


@settings(max_examples=80, deadline=None)
@given(**SHAPES)
def test_row_hybrid_invariants(N, nt, T, C, cap, act, dense, seed):
    f = nt * T
    H = _random_h(N, f, seed, act, dense)
    p = oracle.pack(H, T, C, cap)
    assert oracle.check_format(p, f) == 0
    nz = _nonzero(H).reshape(N, nt, T)
    per_tile = nz.sum(2)
    over = (per_tile > C).any(1)
    # a row leaves TwELL exactly when one of its tiles holds more than C non-zeros
    assert np.array_equal(p["row_fb"] >= 0, over)
    assert p["n_fb"] == int(over.sum())
    # its slot is its rank among those rows, also past the capacity
    assert np.array_equal(p["row_fb"][over], np.arange(int(over.sum())))
    assert np.array_equal(p["counts"][~over], per_tile[~over])
    assert not p["counts"][over].any()
    if p["n_fb"] <= cap:
        # TwELL cells keep only non-zeros (-0.0 comes back as +0.0); a
        # fallback row is kept verbatim in fb_dense
        canon = np.where(_nonzero(H) | over[:, None], H, np.uint16(0))
        assert np.array_equal(oracle.unpack(p, f), canon)


@settings(max_examples=80, deadline=None)
@given(**SHAPES)
def test_tile_hybrid_invariants(N, nt, T, C, cap, act, dense, seed):
    f = nt * T
    H = _random_h(N, f, seed, act, dense)
    pool_cap = cap * nt
    p = oracle.pack_tiles(H, T, C, pool_cap)
    assert oracle.check_format(p, f) == 0
    per_tile = _nonzero(H).reshape(N, nt, T).sum(2)
    dense_tiles = per_tile > C
    assert p["n_fb"] == int(dense_tiles.sum())
    stored = p["counts"] == 255
    # dense tiles take the pool's slots in (row, tile) order until it is full
    order = np.flatnonzero(dense_tiles.reshape(-1))
    assert np.array_equal(np.flatnonzero(stored.reshape(-1)), order[:pool_cap])
    sparse = ~dense_tiles
    assert np.array_equal(p["counts"][sparse], per_tile[sparse])
    if p["n_fb"] <= pool_cap:
        # a dense tile is kept verbatim in the pool, sparse tiles only their non-zeros
        whole = np.repeat(dense_tiles, T, axis=1)
        canon = np.where(_nonzero(H) | whole, H, np.uint16(0))
        assert np.array_equal(oracle.unpack(p, f), canon)
