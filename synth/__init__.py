"""Seeded synthetic inputs for the TwELL activation-sparse FFN layer.

This module is shared by the CPU oracle's tests and by the CUDA path's tests and
bench. It holds no part of the layer's own arithmetic (no ReLU, no packing, no
projection): only random draws, bf16 rounding of the drawn inputs, and the
calibration that places the per-column bias so that the layer's activations come
out about 99% sparse, as the pages' trained models are.

Workloads follow "Sparser, Faster, Lighter Transformer Language Models": the
pages measure ~1B-parameter sparse LMs whose feed-forward layers are more than
99% inactive after L1 training (bayesiansapien note, TL;DR and "What it claims").
No checkpoint or dataset is available, so every tensor is drawn here instead.

Recipe (one config = one seed, numpy PCG64):
  * X0 ~ N(0, 1) [N, d]; W_in^T ~ N(0, 1/sqrt(d)) [f, d]; W_down ~ N(0, 1/sqrt(f)) [f, d];
    each drawn in float32 and rounded to bf16 (round to nearest, ties to even).
  * u = X0 . W_in (float32 numpy matmul, calibration only).  b_j = -bf16(q_j) with
    q_j the order statistic at 0-based index ceil(s*N)-1 of column j of u, s the
    target inactive fraction (0.99 by default), so a unit fires on ~1% of tokens.
  * "lognormal" configs: per-row active fraction p_n ~ exp(N(mu, sigma^2)) with
    sigma = 0.5 and mu = ln(mean) - sigma^2/2, clipped to [0.001, 0.1]; a seeded
    subset of rows is forced to p = 0.2 (the dense-fallback rows).  Row n is
    scaled by s_n so that exactly round(p_n * f) units of s_n*u_n + b are > 0,
    then X_n = bf16(s_n * X0_n).
  * dY ~ N(0, 1) in bf16 for training configs.
  * gated configs add W_u^T ~ N(0, 1/sqrt(d)); the bias places the gate's quantile.
  * decode configs take the bias from a separate calibration batch (seed + 500)
    of calib_rows tokens, since a quantile over 16 tokens says little.
  * another batch for the same layer (batch_seed, e.g. a data-parallel rank's):
    X0 drawn from batch_seed, row activities from batch_seed + 1, row scales
    against the layer's bias.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional

import numpy as np

__all__ = [
    "FFNConfig", "CONFIGS", "f32_to_bf16_bits", "bf16_bits_to_f32", "make_ffn_inputs",
    "make_integer_inputs", "make_dense_h", "make_grad_output",
]


@dataclasses.dataclass(frozen=True)
class FFNConfig:
    name: str
    n_rows: int          # N tokens
    d_model: int         # d
    d_ff: int            # f
    tile: int            # T
    cap: int             # C
    seed: int
    sparsity: float = 0.99            # inactive fraction the column bias targets
    row_spread: str = "uniform"       # "uniform" or "lognormal"
    forced_frac_rows: float = 0.0     # fraction of rows forced to forced_activity
    forced_activity: float = 0.2
    l1_lambda: float = 0.0
    fb_cap: Optional[int] = None      # dense-fallback capacity; default below
    gated: bool = False               # Llama-style: H = ReLU(X.W_g + b) * (X.W_u)
    calib_rows: Optional[int] = None  # bias from a separate calibration batch of this many tokens

    @property
    def n_tiles(self) -> int:
        return self.d_ff // self.tile

    @property
    def fallback_capacity(self) -> int:
        if self.fb_cap is not None:
            return self.fb_cap
        return max(16, self.n_rows // 8)


CONFIGS = {
    # small correctness layer (uniform 99% sparsity, bias at the 99th percentile)
    "pr1": FFNConfig("pr1", 256, 256, 1024, 64, 8, seed=0),
    # ~1B-parameter-model FFN shape: the throughput workload
    "1b": FFNConfig("1b", 4096, 2048, 8192, 128, 8, seed=1, row_spread="lognormal",
                    forced_frac_rows=0.02),
    # training step shape (forward + backward, L1 on H)
    "train": FFNConfig("train", 8192, 2048, 8192, 128, 8, seed=4, row_spread="lognormal",
                       forced_frac_rows=0.01, l1_lambda=1e-4),
    # gated (Llama-style) layer, bias at the gate's 99th percentile
    "gated": FFNConfig("gated", 4096, 4096, 14336, 128, 16, seed=2, gated=True),
    # gated layer's training shape: lognormal row activity, 1% forced-dense rows, L1 on H
    "gated_train": FFNConfig("gated_train", 4096, 4096, 14336, 128, 16, seed=5, gated=True, row_spread="lognormal",
                             forced_frac_rows=0.01, l1_lambda=1e-4),
    # decode-shaped step: 16 tokens, bias calibrated on 4096 other tokens
    "decode": FFNConfig("decode", 16, 4096, 14336, 128, 16, seed=3, sparsity=0.995, calib_rows=4096),
}


def decode_sweep():
    """The decode shape at the sweep's sparsity levels."""
    return [dataclasses.replace(CONFIGS["decode"], name=f"decode_{int(round(s * 1000))}", sparsity=s)
            for s in (0.90, 0.95, 0.99, 0.995)]


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 to bf16 (nearest, ties to even); inputs must be finite."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    lsb = (u >> np.uint64(16)) & np.uint64(1)
    r = (u + np.uint64(0x7FFF) + lsb) >> np.uint64(16)
    return r.astype(np.uint16)


def bf16_bits_to_f32(h: np.ndarray) -> np.ndarray:
    return (np.ascontiguousarray(h, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def _column_bias(u: np.ndarray, sparsity: float) -> np.ndarray:
    n = u.shape[0]
    k = max(0, min(n - 1, int(math.ceil(sparsity * n)) - 1))
    q = np.partition(u, k, axis=0)[k]
    return f32_to_bf16_bits(-q.astype(np.float32))


def _row_scales(u: np.ndarray, b: np.ndarray, active: np.ndarray) -> np.ndarray:
    """Per-row scale s_n > 0 with exactly active[n] entries of s_n*u_n + b above 0.

    With b_j < 0 an entry fires once s exceeds theta = -b_j/u_nj (u_nj > 0), so
    the scale is taken between the k-th and (k+1)-th smallest thresholds.
    """
    bf = bf16_bits_to_f32(b).astype(np.float64)
    n, f = u.shape
    scales = np.empty(n, dtype=np.float64)
    for r0 in range(0, n, 512):
        uu = u[r0:r0 + 512].astype(np.float64)
        with np.errstate(divide="ignore", invalid="ignore"):
            theta = np.where(uu > 0, -bf[None, :] / uu, np.inf)
        theta = np.where((uu > 0) & (bf[None, :] >= 0), 0.0, theta)
        theta.sort(axis=1)
        for i in range(theta.shape[0]):
            k = int(active[r0 + i])
            lo = theta[i, k - 1] if k > 0 else 0.0
            hi = theta[i, k] if k < f else lo * 2 + 1
            if not np.isfinite(hi):
                hi = lo * 2 + 1
            if not np.isfinite(lo):
                lo = 0.0
            scales[r0 + i] = 0.5 * (lo + hi) if k > 0 else 0.5 * hi
    return scales


def make_ffn_inputs(cfg: FFNConfig, rows: Optional[int] = None, batch_seed: Optional[int] = None) -> dict:
    """Draw one layer's inputs: bf16 bit patterns (uint16) plus calibration facts.

    With batch_seed, the layer (weights and bias, calibrated on the config's own
    batch) is the config's, and the returned batch X is drawn afresh from
    batch_seed by the same recipe: another batch for the same layer, as the
    ranks of a data-parallel job each hold one."""
    n = cfg.n_rows if rows is None else rows
    d, f = cfg.d_model, cfg.d_ff
    if batch_seed is not None:
        layer = make_ffn_inputs(cfg, rows=rows)
        x0 = f32_to_bf16_bits(np.random.default_rng(batch_seed).standard_normal((n, d), dtype=np.float32))
        # the batch's activity recipe against the shared layer's bias
        x = _batch_for_layer(cfg, x0, layer["W_inT"], layer["b"], np.random.default_rng(batch_seed + 1))
        out = dict(layer)
        out.update(X=x["X"], X0=x0, target_activity=x["target"], forced_rows=x["forced"])
        if "dY" in layer:
            out["dY"] = make_grad_output(n, d, batch_seed + 1000)
        return out
    rng = np.random.default_rng(cfg.seed)
    x0 = f32_to_bf16_bits(rng.standard_normal((n, d), dtype=np.float32))
    w_in_t = f32_to_bf16_bits(rng.standard_normal((f, d), dtype=np.float32) / np.float32(math.sqrt(d)))
    w_down = f32_to_bf16_bits(rng.standard_normal((f, d), dtype=np.float32) / np.float32(math.sqrt(f)))
    w_u_t = None
    if cfg.gated:
        w_u_t = f32_to_bf16_bits(rng.standard_normal((f, d), dtype=np.float32) / np.float32(math.sqrt(d)))
    if cfg.calib_rows:
        crng = np.random.default_rng(cfg.seed + 500)
        xc = f32_to_bf16_bits(crng.standard_normal((cfg.calib_rows, d), dtype=np.float32))
        u = bf16_bits_to_f32(xc) @ bf16_bits_to_f32(w_in_t).T
    else:
        u = bf16_bits_to_f32(x0) @ bf16_bits_to_f32(w_in_t).T
    b = _column_bias(u, cfg.sparsity)
    target = np.full(n, 1.0 - cfg.sparsity)
    forced = np.zeros(0, dtype=np.int64)
    if cfg.row_spread == "lognormal":
        sigma = 0.5
        mu = math.log(1.0 - cfg.sparsity) - sigma * sigma / 2
        target = np.clip(np.exp(rng.normal(mu, sigma, size=n)), 0.001, 0.1)
        n_forced = int(round(cfg.forced_frac_rows * n))
        if n_forced:
            forced = np.sort(rng.choice(n, size=n_forced, replace=False))
            target[forced] = cfg.forced_activity
        active = np.maximum(1, np.rint(target * f)).astype(np.int64)
        # the scales act on this batch's own pre-activations (not the calibration batch's)
        u_rows = u if not cfg.calib_rows else bf16_bits_to_f32(x0) @ bf16_bits_to_f32(w_in_t).T
        s = _row_scales(u_rows, b, active)
        x = f32_to_bf16_bits((bf16_bits_to_f32(x0) * s[:, None]).astype(np.float32))
    else:
        x = x0
    out = {"X": x, "X0": x0, "W_inT": w_in_t, "b": b, "W_down": w_down, "target_activity": target,
           "forced_rows": forced}
    if w_u_t is not None:
        out["W_uT"] = w_u_t
    if cfg.l1_lambda or cfg.name == "train":
        out["dY"] = make_grad_output(n, d, cfg.seed + 1000)
    return out


def _batch_for_layer(cfg: FFNConfig, x0: np.ndarray, w_in_t: np.ndarray, b: np.ndarray, rng) -> dict:
    """A batch for an existing layer: rows of x0 scaled so that row n fires
    round(p_n * f) units of the layer (lognormal p_n and forced rows as in
    make_ffn_inputs), or x0 itself for a uniform-activity config."""
    n, f = x0.shape[0], w_in_t.shape[0]
    target = np.full(n, 1.0 - cfg.sparsity)
    forced = np.zeros(0, dtype=np.int64)
    if cfg.row_spread != "lognormal":
        return {"X": x0, "target": target, "forced": forced}
    sigma = 0.5
    mu = math.log(1.0 - cfg.sparsity) - sigma * sigma / 2
    target = np.clip(np.exp(rng.normal(mu, sigma, size=n)), 0.001, 0.1)
    n_forced = int(round(cfg.forced_frac_rows * n))
    if n_forced:
        forced = np.sort(rng.choice(n, size=n_forced, replace=False))
        target[forced] = cfg.forced_activity
    active = np.maximum(1, np.rint(target * f)).astype(np.int64)
    u = bf16_bits_to_f32(x0) @ bf16_bits_to_f32(w_in_t).T
    s = _row_scales(u, b, active)
    x = f32_to_bf16_bits((bf16_bits_to_f32(x0) * s[:, None]).astype(np.float32))
    return {"X": x, "target": target, "forced": forced}


def make_grad_output(n: int, d: int, seed: int) -> np.ndarray:
    rng = np.random.default_rng(seed)
    return f32_to_bf16_bits(rng.standard_normal((n, d), dtype=np.float32))


def make_integer_inputs(n: int, d: int, f: int, seed: int, lo: int = -2, hi: int = 2,
                        sparsity: float = 0.99, gated: bool = False) -> dict:
    """Small-integer layer inputs.  Every product and partial sum is an exact
    float32 integer, so any summation order gives the same bits (the exact
    parity case).  The bias is the negated integer column quantile, so about
    (1 - sparsity) of the units fire."""
    rng = np.random.default_rng(seed)
    x = rng.integers(lo, hi + 1, size=(n, d)).astype(np.float32)
    w_in_t = rng.integers(lo, hi + 1, size=(f, d)).astype(np.float32)
    w_down = rng.integers(lo, hi + 1, size=(f, d)).astype(np.float32)
    b = _column_bias(x @ w_in_t.T, sparsity)
    out = {"X": f32_to_bf16_bits(x), "W_inT": f32_to_bf16_bits(w_in_t), "b": b,
           "W_down": f32_to_bf16_bits(w_down)}
    if gated:
        out["W_uT"] = f32_to_bf16_bits(rng.integers(lo, hi + 1, size=(f, d)).astype(np.float32))
    return out


def make_dense_h(n: int, f: int, seed: int, activity: float = 0.01,
                 dense_rows: Optional[np.ndarray] = None, dense_activity: float = 0.2) -> np.ndarray:
    """A non-negative bf16 activation matrix with a given fraction of non-zeros
    per row (input for the standalone pack / unpack calls)."""
    rng = np.random.default_rng(seed)
    p = np.full((n, 1), activity)
    if dense_rows is not None and len(dense_rows):
        p[np.asarray(dense_rows)] = dense_activity
    mask = rng.random((n, f)) < p
    vals = np.abs(rng.standard_normal((n, f), dtype=np.float32)) + np.float32(1e-3)
    h = np.where(mask, vals, np.float32(0.0)).astype(np.float32)
    return f32_to_bf16_bits(h)
