"""Pins for the CPU oracle: each test ties it to something other than itself.

Sources of truth used here: a hand-worked example of the format (golden
fixture), the IEEE-754 definition of round-to-nearest-even and a library
conversion, brute force over every sparsity pattern of a small tile, exact
integer arithmetic (numpy int64), closed forms of the backward, and torch
autograd on the dense float64 definition of the layer.
"""
import json
import math
import os

import numpy as np
import pytest

import oracle
import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
bf = synth.bf16_bits_to_f32
to_bf = synth.f32_to_bf16_bits


# ---------------------------------------------------------------- bf16 rounding
def test_bf16_rounding_hand_cases():
    # IEEE-754 round to nearest, ties to even, on the top 16 bits.
    one = 1.0
    cases = [
        (1.0, 0x3F80),
        (one + 2.0 ** -8, 0x3F80),          # exact tie, 0x3F80 is even -> stays
        (one + 3 * 2.0 ** -8, 0x3F82),      # exact tie, 0x3F81 odd -> up to 0x3F82
        (one + 2.0 ** -8 + 2.0 ** -20, 0x3F81),  # just above the tie -> up
        (-2.0, 0xC000),
        (0.0, 0x0000),
        (-0.0, 0x8000),
        (3.0, 0x4040),
        (2.0 ** -130, None),                # subnormal, checked against torch below
    ]
    for x, want in cases:
        if want is not None:
            assert oracle.bf16_round(x) == want, (x, hex(oracle.bf16_round(x)))


def test_bf16_rounding_matches_library():
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(7)
    x = np.concatenate([
        rng.standard_normal(100000).astype(np.float32),
        (rng.standard_normal(1000) * 1e-39).astype(np.float32),   # subnormals
        # exact ties between two bf16 neighbours
        (bf(rng.integers(0, 0x7F00, 2000).astype(np.uint16)).view(np.uint32) | 0x8000).view(np.float32),
    ])
    want = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(oracle.round_bf16(x), want)


# ---------------------------------------------------------------- packing
def _golden():
    with open(os.path.join(GOLDEN, "twell_hand_example.json")) as fh:
        return json.load(fh)


def test_pack_hand_example():
    g = _golden()
    H = to_bf(np.array(g["H"], dtype=np.float32))
    p = oracle.pack(H, g["T"], g["C"], g["fb_cap"])
    e = g["expected"]
    assert p["n_fb"] == e["n_fb"]
    assert p["counts"].tolist() == e["counts"]
    assert bf(p["values"]).tolist() == e["values"]
    assert p["idx"].tolist() == e["idx"]
    assert p["row_fb"].tolist() == e["row_fb"]
    assert p["fb_rows"].tolist() == e["fb_rows"]
    assert np.array_equal(p["fb_dense"], H[[1, 3]])
    # padding is +0.0 bit-for-bit (never -0.0)
    assert np.all(p["values"][p["idx"] == 0][bf(p["values"][p["idx"] == 0]) == 0] == 0)
    assert oracle.check_format(p, H.shape[1]) == 0
    assert np.array_equal(oracle.unpack(p, H.shape[1]), H)


@pytest.mark.parametrize("C", list(range(0, 9)))
def test_pack_brute_force_all_patterns(C):
    # every 8-column pattern of one tile (T = 8): 256 rows
    T = 8
    pats = np.array([[(m >> i) & 1 for i in range(T)] for m in range(256)], dtype=np.float32)
    vals = (np.arange(256 * T, dtype=np.float32).reshape(256, T) % 7 + 1.0) * 0.5
    H = to_bf(pats * vals)
    p = oracle.pack(H, T, C, fb_cap=256)
    pop = pats.sum(1).astype(int)
    over = pop > C
    assert p["n_fb"] == int(over.sum())
    assert np.array_equal(p["row_fb"] >= 0, over)
    assert np.array_equal(p["fb_rows"][:p["n_fb"]], np.nonzero(over)[0])
    for r in range(256):
        if over[r]:
            assert p["counts"][r, 0] == 0
            assert np.array_equal(p["fb_dense"][p["row_fb"][r]], H[r])
            continue
        nz = np.nonzero(pats[r])[0]
        assert p["counts"][r, 0] == len(nz)
        assert p["idx"][r, 0, :len(nz)].tolist() == nz.tolist()
        assert np.array_equal(p["values"][r, 0, :len(nz)], H[r, nz])
        assert np.all(p["values"][r, 0, len(nz):] == 0) and np.all(p["idx"][r, 0, len(nz):] == 0)
    assert oracle.check_format(p, T) == 0
    assert np.array_equal(oracle.unpack(p, T), H)


def test_pack_special_cases():
    N, f, T, C = 64, 512, 64, 8
    # H = 0: nothing stored, no fallback
    p = oracle.pack(np.zeros((N, f), np.uint16), T, C, 16)
    assert p["n_fb"] == 0 and not p["counts"].any() and not p["values"].any()
    # C = T: no row can overflow, even a fully dense one
    H = to_bf(np.abs(np.random.default_rng(0).standard_normal((N, f))).astype(np.float32) + 1)
    p = oracle.pack(H, T, T, 16)
    assert p["n_fb"] == 0 and np.all(p["counts"] == T)
    # T = f is plain ELLPACK: one tile per row, idx = column
    H = synth.make_dense_h(N, 128, seed=3, activity=0.03)
    p = oracle.pack(H, 128, 16, 16)
    assert p["n_fb"] == 0
    for r in range(N):
        nz = np.nonzero(bf(H[r]))[0]
        assert p["counts"][r, 0] == len(nz) and p["idx"][r, 0, :len(nz)].tolist() == nz.tolist()
    # exactly C fits, C + 1 overflows
    H = np.zeros((2, 64), np.float32)
    H[0, :8] = 1.0
    H[1, :9] = 1.0
    p = oracle.pack(to_bf(H), 64, 8, 4)
    assert p["row_fb"].tolist() == [-1, 0] and p["counts"][0, 0] == 8


def test_pack_negative_zero_is_zero():
    H = np.zeros((1, 8), np.uint16)
    H[0, 2] = 0x8000          # -0.0 is not a non-zero
    H[0, 5] = to_bf(np.array([2.0], np.float32))[0]
    p = oracle.pack(H, 8, 2, 1)
    assert p["counts"][0, 0] == 1 and p["idx"][0, 0, 0] == 5


def test_pack_roundtrip_and_counts_random():
    N, f, T, C = 300, 1024, 64, 8
    H = synth.make_dense_h(N, f, seed=11, activity=0.02, dense_rows=np.arange(0, N, 37))
    p = oracle.pack(H, T, C, 64)
    assert oracle.check_format(p, f) == 0
    assert np.array_equal(oracle.unpack(p, f), H)
    nnz = int((bf(H) != 0).sum())
    fb = p["row_fb"] >= 0
    assert int(p["counts"].sum()) + int((bf(H[fb]) != 0).sum()) == nnz
    # a row is in the fallback iff one of its tiles holds more than C non-zeros
    tile_nnz = (bf(H) != 0).reshape(N, f // T, T).sum(2)
    assert np.array_equal(fb, (tile_nnz > C).any(1))


def test_format_checker_catches_each_violation():
    N, f, T, C = 40, 256, 64, 4
    H = synth.make_dense_h(N, f, seed=2, activity=0.02, dense_rows=[3, 17])
    good = oracle.pack(H, T, C, 8)
    assert oracle.check_format(good, f) == 0

    def mutated(fn):
        p = {k: (v.copy() if isinstance(v, np.ndarray) else v) for k, v in good.items()}
        fn(p)
        return oracle.check_format(p, f)

    r, t = next((r, t) for r in range(N) for t in range(f // T) if good["counts"][r, t] >= 2)
    assert mutated(lambda p: p["counts"].__setitem__((r, t), C + 1)) == 1
    assert mutated(lambda p: p["counts"].__setitem__((3, 0), 1)) == 2
    assert mutated(lambda p: p["idx"].__setitem__((r, t, 0), T)) == 3
    assert mutated(lambda p: p["idx"].__setitem__((r, t, 1), p["idx"][r, t, 0])) == 4
    assert mutated(lambda p: p["values"].__setitem__((r, t, 0), 0)) == 5
    r0, t0 = next((r, t) for r in range(N) for t in range(f // T)
                  if good["counts"][r, t] < C and good["row_fb"][r] < 0)
    assert mutated(lambda p: p["idx"].__setitem__((r0, t0, C - 1), 1)) == 6
    assert mutated(lambda p: p["row_fb"].__setitem__(0, 1)) == 7
    assert mutated(lambda p: p["fb_rows"].__setitem__(slice(0, 2), p["fb_rows"][1::-1].copy())) in (7, 8)
    assert mutated(lambda p: p.__setitem__("n_fb", 1)) == 9
    # slots must be the rows' ranks: an inverse pair (last fallback row <-> a
    # free slot) is not enough
    fbr = [int(r) for r in np.flatnonzero(good["row_fb"] >= 0)]
    assert len(fbr) >= 2 and {3, 17} <= set(fbr) and good["n_fb"] == len(fbr) < 7

    def renumber(p):
        p["row_fb"][fbr[-1]] = 7
        p["fb_rows"][7] = fbr[-1]
    assert mutated(renumber) == 8

    def swap_slots(p):
        p["row_fb"][fbr[0]], p["row_fb"][fbr[1]] = 1, 0
        p["fb_rows"][:2] = [fbr[1], fbr[0]]
    assert mutated(swap_slots) == 8
    # an overflowed fallback (rows past fb_cap keep their numbers, unstored) is well formed
    over = oracle.pack(H, T, C, 1)
    assert over["n_fb"] == len(fbr) and list(over["row_fb"][fbr]) == list(range(len(fbr)))
    assert oracle.check_format(over, f) == 0
    over["fb_rows"][0] = fbr[1]
    assert oracle.check_format(over, f) == 7


# ---------------------------------------------------------------- forward arithmetic
def _exact_int_forward(inp):
    X = bf(inp["X"]).astype(np.int64)
    W = bf(inp["W_inT"]).astype(np.int64)
    b = bf(inp["b"]).astype(np.int64)
    Wd = bf(inp["W_down"]).astype(np.int64)
    z = X @ W.T + b
    h = np.where(z > 0, z, 0)
    return z, h, h @ Wd


def test_hidden_and_down_exact_on_integers():
    inp = synth.make_integer_inputs(256, 256, 1024, seed=5, sparsity=0.97)
    z, h, y = _exact_int_forward(inp)
    assert np.abs(z).max() < 2 ** 24 and np.abs(y).max() < 2 ** 24
    Z, H = oracle.hidden(inp["X"], inp["W_inT"], inp["b"])
    assert np.array_equal(Z.astype(np.int64), z)
    # h = bf16(z) for z > 0: compare with the library rounding of the exact integer
    assert np.array_equal(H, to_bf(h.astype(np.float32)))
    Hf = bf(H).astype(np.int64)
    y_exact = Hf @ bf(inp["W_down"]).astype(np.int64)
    Y = oracle.down_dense(H, inp["W_down"])
    assert np.array_equal(Y.astype(np.int64), y_exact)
    p = oracle.pack(H, 64, 8, 256)
    assert np.array_equal(oracle.down_packed(p, inp["W_down"]), Y)
    assert 0.005 < (h > 0).mean() < 0.1


def test_hidden_row_selection_and_relu_sign():
    inp = synth.make_integer_inputs(128, 64, 256, seed=9, sparsity=0.9)
    z, h, _ = _exact_int_forward(inp)
    rows = np.array([127, 0, 64, 5], np.int32)
    Z, H = oracle.hidden(inp["X"], inp["W_inT"], inp["b"], rows=rows)
    assert np.array_equal(Z.astype(np.int64), z[rows])
    assert np.all(bf(H)[z[rows] <= 0] == 0) and np.all(H[z[rows] <= 0] == 0)   # +0, never -0
    assert np.all(bf(H)[z[rows] > 0] > 0)


def test_down_packed_equals_dense_bitwise():
    # Adding exact zero products never changes an fp32 sum, so the packed
    # product (j ascending over stored entries) equals the dense one bit for bit.
    inp = synth.make_ffn_inputs(synth.CONFIGS["pr1"])
    out = oracle.forward(inp["X"], inp["W_inT"], inp["b"], inp["W_down"], 64, 8, 64)
    Yd = oracle.down_dense(out["H"], inp["W_down"])
    assert np.array_equal(out["Y"].view(np.uint32), Yd.view(np.uint32))
    # and both agree with a float64 library matmul within the fp32 summation bound
    Hf = bf(out["H"]).astype(np.float64)
    Wf = bf(inp["W_down"]).astype(np.float64)
    ref = Hf @ Wf
    bound = 1024 * 2.0 ** -24 * (np.abs(Hf) @ np.abs(Wf)) + 1e-30
    assert np.all(np.abs(Yd - ref) <= bound)


def test_hidden_matches_float64_library():
    inp = synth.make_ffn_inputs(synth.CONFIGS["pr1"])
    Z, H = oracle.hidden(inp["X"], inp["W_inT"], inp["b"])
    X = bf(inp["X"]).astype(np.float64)
    W = bf(inp["W_inT"]).astype(np.float64)
    b = bf(inp["b"]).astype(np.float64)
    ref = X @ W.T + b
    bound = 256 * 2.0 ** -24 * (np.abs(X) @ np.abs(W).T + np.abs(b)) + 1e-30
    assert np.all(np.abs(Z - ref) <= bound)
    act = (bf(H) != 0).mean()
    assert 0.005 < act < 0.02            # the bias calibration gives ~99% sparsity


# ---------------------------------------------------------------- backward
def test_backward_closed_form_zero_upstream():
    # dY = 0: dZ = lambda exactly on the pattern, db[j] = lambda * #active(j),
    # dX = lambda * sum of the active rows of W_in^T, dW_down = 0.
    inp = synth.make_integer_inputs(96, 64, 256, seed=4, sparsity=0.9)
    lam = 0.25
    _, H = oracle.hidden(inp["X"], inp["W_inT"], inp["b"])
    dY = np.zeros((96, 64), np.uint16)
    dH, dZ = oracle.grad_hidden(dY, inp["W_down"], H, lam)
    act = bf(H) > 0
    assert np.array_equal(dZ, np.where(act, np.float32(lam), np.float32(0)))
    dX = oracle.grad_input(dZ, inp["W_inT"])
    assert np.array_equal(dX, (lam * (act.astype(np.float64) @ bf(inp["W_inT"]).astype(np.float64))).astype(np.float32))
    dWin, dWdown, db = oracle.grad_weights(inp["X"], inp["W_down"], H, dY, lam)
    assert not dWdown.any()
    assert np.array_equal(db, (lam * act.sum(0)).astype(np.float32))
    assert np.array_equal(dWin, (lam * (act.T.astype(np.float64) @ bf(inp["X"]).astype(np.float64))).astype(np.float32))


def test_backward_single_active_unit_rank_one():
    # one active unit j* per row, lambda = 0: dW_down[j*] = sum_n h[n,j*] dY[n],
    # every other row of dW_down is 0, dX[n] = (dY[n].W_down[j*]) W_in^T[j*].
    rng = np.random.default_rng(1)
    N, d, f, js = 16, 32, 64, 5
    H = np.zeros((N, f), np.float32)
    H[:, js] = rng.integers(1, 5, N)
    Hb = to_bf(H)
    dY = to_bf(rng.integers(-3, 4, (N, d)).astype(np.float32))
    Wd = to_bf(rng.integers(-2, 3, (f, d)).astype(np.float32))
    Wi = to_bf(rng.integers(-2, 3, (f, d)).astype(np.float32))
    X = to_bf(rng.integers(-2, 3, (N, d)).astype(np.float32))
    _, dZ = oracle.grad_hidden(dY, Wd, Hb, 0.0)
    g = bf(dY).astype(np.int64) @ bf(Wd[js]).astype(np.int64)
    assert np.array_equal(dZ[:, js].astype(np.int64), g) and not np.delete(dZ, js, 1).any()
    dX = oracle.grad_input(dZ, Wi)
    assert np.array_equal(dX.astype(np.int64), np.outer(g, bf(Wi[js]).astype(np.int64)))
    dWin, dWdown, db = oracle.grad_weights(X, Wd, Hb, dY, 0.0)
    assert np.array_equal(dWdown[js].astype(np.int64), H[:, js].astype(np.int64) @ bf(dY).astype(np.int64))
    assert not np.delete(dWdown, js, 0).any()
    assert db[js] == g.sum() and not np.delete(db, js).any()


def test_backward_matches_autograd():
    torch = pytest.importorskip("torch")
    N, d, f = 48, 64, 256
    cfg = synth.FFNConfig("t", N, d, f, 64, 8, seed=21, sparsity=0.9)
    inp = synth.make_ffn_inputs(cfg)
    dYb = synth.make_grad_output(N, d, 99)
    lam = 0.01
    _, H = oracle.hidden(inp["X"], inp["W_inT"], inp["b"])
    # autograd of L = sum(Y * dY) + lam * sum|h| through the float64 dense layer,
    # with h's bf16 rounding treated as the identity (straight-through)
    X = torch.tensor(bf(inp["X"]), dtype=torch.float64, requires_grad=True)
    Wi = torch.tensor(bf(inp["W_inT"]), dtype=torch.float64, requires_grad=True)
    b = torch.tensor(bf(inp["b"]), dtype=torch.float64, requires_grad=True)
    Wd = torch.tensor(bf(inp["W_down"]), dtype=torch.float64, requires_grad=True)
    Hq = torch.tensor(bf(H), dtype=torch.float64)
    z = X @ Wi.T + b
    h = torch.relu(z)
    h = h + (Hq - h).detach()
    Y = h @ Wd
    loss = (Y * torch.tensor(bf(dYb), dtype=torch.float64)).sum() + lam * h.abs().sum()
    loss.backward()
    dH, dZ = oracle.grad_hidden(dYb, inp["W_down"], H, lam)
    dX = oracle.grad_input(dZ, inp["W_inT"])
    dWin, dWdown, db = oracle.grad_weights(inp["X"], inp["W_down"], H, dYb, lam)

    def close(a, ref):
        ref = ref.detach().numpy()
        return np.abs(a - ref).max() <= 1e-5 * max(1.0, np.abs(ref).max())

    assert close(dX, X.grad) and close(dWin, Wi.grad) and close(db, b.grad) and close(dWdown, Wd.grad)


def test_weight_grad_column_selection():
    cfg = synth.FFNConfig("t", 40, 32, 128, 32, 4, seed=8, sparsity=0.9)
    inp = synth.make_ffn_inputs(cfg)
    dY = synth.make_grad_output(40, 32, 1)
    _, H = oracle.hidden(inp["X"], inp["W_inT"], inp["b"])
    full = oracle.grad_weights(inp["X"], inp["W_down"], H, dY, 0.1)
    cols = np.array([100, 3, 64], np.int32)
    sel = oracle.grad_weights(inp["X"], inp["W_down"], H, dY, 0.1, cols=cols)
    for a, b in zip(full, sel):
        assert np.array_equal(a[cols], b)


def test_generator_statistics_1b_shape():
    # the throughput workload's recipe: ~1% mean activity on ordinary rows,
    # 2% of rows forced to 20% (all of which overflow C = 8 at T = 128)
    cfg = synth.FFNConfig("1b_small", 512, 256, 2048, 128, 8, seed=1, row_spread="lognormal",
                          forced_frac_rows=0.02)
    inp = synth.make_ffn_inputs(cfg)
    _, H = oracle.hidden(inp["X"], inp["W_inT"], inp["b"])
    act = (bf(H) != 0).mean(1)
    forced = inp["forced_rows"]
    assert len(forced) == round(0.02 * 512)
    assert np.all(np.abs(act[forced] - 0.2) < 0.02)
    rest = np.delete(act, forced)
    assert 0.007 < rest.mean() < 0.013
    p = oracle.pack(H, 128, 8, 128)
    assert set(forced.tolist()) <= set(np.nonzero(p["row_fb"] >= 0)[0].tolist())


def test_gated_hidden_exact_on_integers():
    # gated (Llama-style) variant: h = bf16(zg * zu) where zg > 0, else +0
    inp = synth.make_integer_inputs(128, 64, 256, seed=12, sparsity=0.9)
    rng = np.random.default_rng(13)
    Wu = to_bf(rng.integers(-2, 3, (256, 64)).astype(np.float32))
    X = bf(inp["X"]).astype(np.int64)
    zg = X @ bf(inp["W_inT"]).astype(np.int64).T + bf(inp["b"]).astype(np.int64)
    zu = X @ bf(Wu).astype(np.int64).T
    want = np.where(zg > 0, zg * zu, 0)
    assert np.abs(want).max() < 2 ** 24
    Zg, H = oracle.hidden_gated(inp["X"], inp["W_inT"], Wu, inp["b"])
    assert np.array_equal(Zg.astype(np.int64), zg)
    got = bf(H)
    assert np.array_equal(got, bf(to_bf(want.astype(np.float32))))
    assert np.all(H[zg <= 0] == 0)


def test_overflowed_layout_unpacks_rows_past_capacity_as_zeros():
    """Reading 15: a fallback row past fb_cap is stored nowhere and its cells
    are emptied, so unpacking the layout gives a zero row for it, and the packed
    product gives it a zero output row; the stored rows come back exactly."""
    H = synth.make_dense_h(40, 256, seed=21, activity=0.01, dense_rows=np.arange(0, 40, 5))
    p = oracle.pack(H, 64, 8, 3)
    assert p["n_fb"] >= 6
    over = np.nonzero(p["row_fb"] >= 3)[0]
    assert len(over) == p["n_fb"] - 3 and (p["counts"][over] == 0).all()
    want = H.copy()
    want[over] = 0
    assert np.array_equal(oracle.unpack(p, 256), want)
    W = synth.f32_to_bf16_bits(np.random.default_rng(3).standard_normal((256, 64), dtype=np.float32))
    Y = oracle.down_packed(p, W)
    assert not Y[over].any()
    assert np.array_equal(Y, oracle.down_dense(want, W))
