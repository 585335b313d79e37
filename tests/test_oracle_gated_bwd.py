"""Pins of the oracle's backward of the gated layer (H = bf16(g * u) where
g = X.W_g + b > 0, u = X.W_u; L = sum(Y * dY) + lambda * sum|h|), each tied to
something other than the oracle: float64 autograd of the dense layer with h's
rounding passed straight through, the closed form with no upstream gradient
(h negative as well as positive), and the swap of the gate and up roles."""
import numpy as np
import pytest

import oracle
import synth

bf = synth.bf16_bits_to_f32


def _layer(N, d, f, seed, sparsity=0.7):
    cfg = synth.FFNConfig("g", N, d, f, 64, 8, seed=seed, sparsity=sparsity, gated=True)
    inp = synth.make_ffn_inputs(cfg)
    _, H = oracle.hidden_gated(inp["X"], inp["W_inT"], inp["W_uT"], inp["b"])
    return inp, H


def _oracle_all(inp, H, dY, lam):
    dG, dU = oracle.grad_hidden_gated(inp["X"], inp["W_inT"], inp["W_uT"], inp["b"], dY, inp["W_down"], H, lam)
    dX = oracle.grad_input_gated(dG, dU, inp["W_inT"], inp["W_uT"])
    dWg, dWu, dWd, db = oracle.grad_weights_gated(inp["X"], inp["W_inT"], inp["W_uT"], inp["b"], inp["W_down"], H,
                                                  dY, lam)
    return dG, dU, dX, dWg, dWu, dWd, db


def test_gated_backward_matches_autograd():
    torch = pytest.importorskip("torch")
    N, d, f = 40, 64, 192
    inp, H = _layer(N, d, f, seed=31)
    assert (bf(H) < 0).any() and (bf(H) > 0).any()
    dYb = synth.make_grad_output(N, d, 7)
    lam = 0.02
    X = torch.tensor(bf(inp["X"]), dtype=torch.float64, requires_grad=True)
    Wg = torch.tensor(bf(inp["W_inT"]), dtype=torch.float64, requires_grad=True)
    Wu = torch.tensor(bf(inp["W_uT"]), dtype=torch.float64, requires_grad=True)
    b = torch.tensor(bf(inp["b"]), dtype=torch.float64, requires_grad=True)
    Wd = torch.tensor(bf(inp["W_down"]), dtype=torch.float64, requires_grad=True)
    Hq = torch.tensor(bf(H), dtype=torch.float64)
    mask = torch.tensor(H != 0)          # the stored pattern: h != 0
    g = X @ Wg.T + b
    u = X @ Wu.T
    h = torch.where(mask, g * u, torch.zeros_like(g))
    h = h + (Hq - h).detach()            # straight through the bf16 rounding
    loss = (h @ Wd * torch.tensor(bf(dYb), dtype=torch.float64)).sum() + lam * h.abs().sum()
    loss.backward()
    _, _, dX, dWg, dWu, dWd, db = _oracle_all(inp, H, dYb, lam)

    def close(a, ref):
        ref = ref.detach().numpy()
        return np.abs(a - ref).max() <= 1e-5 * max(1.0, np.abs(ref).max())

    assert close(dX, X.grad), "dX"
    assert close(dWg, Wg.grad), "dW_g"
    assert close(dWu, Wu.grad), "dW_u"
    assert close(db, b.grad), "db"
    assert close(dWd, Wd.grad), "dW_down"


def test_gated_backward_zero_upstream_closed_form():
    """dY = 0: dh is lambda * sign(h) at the pattern, so dG = lambda sign(h) u
    and dU = lambda sign(h) g there (g, u from float64 dot products of the bf16
    inputs), zero elsewhere; dW_down is 0."""
    N, d, f = 24, 32, 128
    inp, H = _layer(N, d, f, seed=5)
    dY = np.zeros((N, d), np.uint16)
    lam = 0.5
    dG, dU, dX, dWg, dWu, dWd, db = _oracle_all(inp, H, dY, lam)
    X, Wg, Wu, b = (bf(inp[k]).astype(np.float64) for k in ("X", "W_inT", "W_uT", "b"))
    g = X @ Wg.T + b
    u = X @ Wu.T
    hs = np.sign(bf(H))
    assert (hs < 0).any() and (hs > 0).any()
    assert np.allclose(dG, lam * hs * u, rtol=1e-5, atol=1e-6)
    assert np.allclose(dU, lam * hs * g, rtol=1e-5, atol=1e-6)
    assert not dWd.any()
    assert np.allclose(db, (lam * hs * u).sum(axis=0), rtol=1e-4, atol=1e-5)
    assert np.allclose(dX, (lam * hs * u) @ Wg + (lam * hs * g) @ Wu, rtol=1e-4, atol=1e-4)


def test_gated_backward_role_swap():
    """Exchanging the gate and up matrices where both are positive exchanges
    dG and dU: with X >= 0 and W_g, W_u >= 0, zero bias, every g, u > 0, so
    h = bf16(g * u) is symmetric in the two roles."""
    rng = np.random.default_rng(3)
    N, d, f = 16, 32, 64
    X = synth.f32_to_bf16_bits(np.abs(rng.standard_normal((N, d))).astype(np.float32))
    Wa = synth.f32_to_bf16_bits(np.abs(rng.standard_normal((f, d))).astype(np.float32) / 8)
    Wb = synth.f32_to_bf16_bits(np.abs(rng.standard_normal((f, d))).astype(np.float32) / 8)
    Wd = synth.f32_to_bf16_bits(rng.standard_normal((f, d)).astype(np.float32) / 8)
    b0 = np.zeros(f, np.uint16)
    dY = synth.make_grad_output(N, d, 2)
    _, H1 = oracle.hidden_gated(X, Wa, Wb, b0)
    _, H2 = oracle.hidden_gated(X, Wb, Wa, b0)
    assert np.array_equal(H1, H2) and (H1 != 0).all()
    dG1, dU1 = oracle.grad_hidden_gated(X, Wa, Wb, b0, dY, Wd, H1, 0.1)
    dG2, dU2 = oracle.grad_hidden_gated(X, Wb, Wa, b0, dY, Wd, H2, 0.1)
    assert np.array_equal(dG1, dU2) and np.array_equal(dU1, dG2)


def test_gated_weight_grad_column_selection():
    inp, H = _layer(30, 32, 128, seed=9)
    dY = synth.make_grad_output(30, 32, 4)
    full = oracle.grad_weights_gated(inp["X"], inp["W_inT"], inp["W_uT"], inp["b"], inp["W_down"], H, dY, 0.1)
    cols = np.array([100, 3, 64], np.int32)
    sel = oracle.grad_weights_gated(inp["X"], inp["W_inT"], inp["W_uT"], inp["b"], inp["W_down"], H, dY, 0.1,
                                    cols=cols)
    for a, s in zip(full, sel):
        assert np.array_equal(a[cols], s)
