"""CPU oracle for the TwELL activation-sparse FFN (test infrastructure only).

Only tests/, the smoke check and the bench's CPU-baseline leg may import this
package.  It wraps `liboracle.so`, compiled from `twell_oracle.c` (plain C,
fp32 loops, summation index ascending), with numpy arrays; bf16 tensors travel
as uint16 bit patterns.  It shares no code with the CUDA library.

Every function states the passage of "Sparser, Faster, Lighter Transformer
Language Models" (as the pages describe it) that it restates; see the C source.
"""
from __future__ import annotations

import contextlib
import ctypes
import os
import subprocess
from typing import Optional

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "twell_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle (gcc, OpenMP, no fused multiply-add)."""
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-fopenmp", "-ffp-contract=off", "-fno-fast-math",
                               "-fPIC", "-shared", "-o", tmp, _SRC])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _configure(lib):
    P = ctypes.c_void_p
    I = ctypes.c_int32
    lib.oracle_bf16_round.restype = ctypes.c_uint16
    lib.oracle_bf16_round.argtypes = [ctypes.c_float]
    lib.oracle_hidden.argtypes = [P, P, P, I, I, P, I, P, P]
    lib.oracle_hidden_gated.argtypes = [P, P, P, P, I, I, P, I, P, P]
    lib.oracle_pack.restype = I
    lib.oracle_pack.argtypes = [P, I, I, I, I, I, P, P, P, P, P, P]
    lib.oracle_unpack.argtypes = [P, P, P, P, P, I, I, I, I, I, P]
    lib.oracle_down_dense.argtypes = [P, P, I, I, I, P]
    lib.oracle_down_packed.argtypes = [P, P, P, P, P, P, I, I, I, I, I, I, P]
    lib.oracle_round_bf16.argtypes = [P, ctypes.c_int64, P]
    lib.oracle_grad_hidden.argtypes = [P, P, P, ctypes.c_float, P, I, I, I, P, P]
    lib.oracle_grad_input.argtypes = [P, P, I, I, I, P]
    lib.oracle_grad_weights.argtypes = [P, P, P, P, ctypes.c_float, I, I, I, P, I, P, P, P]
    lib.oracle_grad_hidden_gated.argtypes = [P, P, P, P, P, P, P, ctypes.c_float, P, I, I, I, P, P]
    lib.oracle_grad_input_gated.argtypes = [P, P, P, P, I, I, I, P]
    lib.oracle_grad_weights_gated.argtypes = [P, P, P, P, P, P, P, ctypes.c_float, I, I, I, P, I, P, P, P, P]
    lib.oracle_check_format.restype = I
    lib.oracle_check_format.argtypes = [P, P, P, P, P, I, I, I, I, I, I]
    lib.oracle_pack_tiles.restype = I
    lib.oracle_pack_tiles.argtypes = [P, I, I, I, I, I, P, P, P, P, P]
    lib.oracle_unpack_tiles.argtypes = [P, P, P, P, I, I, I, I, P]
    lib.oracle_down_packed_tiles.argtypes = [P, P, P, P, P, I, I, I, I, I, P]
    lib.oracle_check_format_tiles.restype = I
    lib.oracle_check_format_tiles.argtypes = [P, P, P, P, P, I, I, I, I, I, I]
    return lib


def _load():
    global _lib
    if _lib is None:
        _lib = _configure(ctypes.CDLL(build()))
    return _lib


@contextlib.contextmanager
def use_library(path: str):
    """Run the wrappers against another build of the oracle source (used by the
    tests that plant a mistake in a copy of the oracle and expect a pin to fail)."""
    global _lib
    saved = _load()
    _lib = _configure(ctypes.CDLL(path))
    try:
        yield
    finally:
        _lib = saved


def _p(a: Optional[np.ndarray]):
    return None if a is None else a.ctypes.data


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def bf16_round(x: float) -> int:
    return int(_load().oracle_bf16_round(float(x)))


def round_bf16(x: np.ndarray) -> np.ndarray:
    x = _c(x, np.float32)
    out = np.empty(x.shape, dtype=np.uint16)
    _load().oracle_round_bf16(_p(x), x.size, _p(out))
    return out


def _rows(rows, n):
    if rows is None:
        return np.arange(n, dtype=np.int32)
    return _c(rows, np.int32)


def hidden(X, W_inT, b, rows=None):
    """Pre-activation z (fp32) and h = bf16(z) where z > 0 else +0 for the selected rows."""
    X, W_inT, b = _c(X, np.uint16), _c(W_inT, np.uint16), _c(b, np.uint16)
    f, d = W_inT.shape
    r = _rows(rows, X.shape[0])
    Z = np.empty((len(r), f), dtype=np.float32)
    H = np.empty((len(r), f), dtype=np.uint16)
    _load().oracle_hidden(_p(X), _p(W_inT), _p(b), d, f, _p(r), len(r), _p(Z), _p(H))
    return Z, H


def hidden_gated(X, W_gT, W_uT, b, rows=None):
    X, W_gT, W_uT, b = (_c(a, np.uint16) for a in (X, W_gT, W_uT, b))
    f, d = W_gT.shape
    r = _rows(rows, X.shape[0])
    Z = np.empty((len(r), f), dtype=np.float32)
    H = np.empty((len(r), f), dtype=np.uint16)
    _load().oracle_hidden_gated(_p(X), _p(W_gT), _p(W_uT), _p(b), d, f, _p(r), len(r), _p(Z), _p(H))
    return Z, H


def pack(H, T: int, C: int, fb_cap: int) -> dict:
    """Scalar-loop TwELL packer (hybrid, row-granular fallback)."""
    H = _c(H, np.uint16)
    N, f = H.shape
    nt = f // T
    out = {
        "values": np.empty((N, nt, C), dtype=np.uint16),
        "idx": np.empty((N, nt, C), dtype=np.uint8),
        "counts": np.empty((N, nt), dtype=np.uint8),
        "row_fb": np.empty((N,), dtype=np.int32),
        "fb_rows": np.full((fb_cap,), -1, dtype=np.int32),
        "fb_dense": np.zeros((fb_cap, f), dtype=np.uint16),
    }
    n_fb = _load().oracle_pack(_p(H), N, f, T, C, fb_cap, _p(out["values"]), _p(out["idx"]),
                               _p(out["counts"]), _p(out["row_fb"]), _p(out["fb_rows"]),
                               _p(out["fb_dense"]))
    out["n_fb"] = int(n_fb)
    out["T"], out["C"], out["fb_cap"] = T, C, fb_cap
    return out


def pack_tiles(H, T: int, C: int, pool_cap: int) -> dict:
    """Scalar-loop packer of the tile-granular hybrid: tiles with more than C
    non-zeros are kept densely in a pool (slots in (row, tile) order)."""
    H = _c(H, np.uint16)
    N, f = H.shape
    nt = f // T
    out = {
        "values": np.empty((N, nt, C), dtype=np.uint16),
        "idx": np.empty((N, nt, C), dtype=np.uint8),
        "counts": np.empty((N, nt), dtype=np.uint8),
        "row_fb": np.empty((N,), dtype=np.int32),
        "pool": np.zeros((pool_cap, T), dtype=np.uint16),
    }
    n = _load().oracle_pack_tiles(_p(H), N, f, T, C, pool_cap, _p(out["values"]), _p(out["idx"]),
                                  _p(out["counts"]), _p(out["row_fb"]), _p(out["pool"]))
    out["n_fb"] = int(n)
    out["T"], out["C"], out["pool_cap"], out["hybrid"] = T, C, pool_cap, "tiles"
    return out


def unpack(packed: dict, f: int) -> np.ndarray:
    v, i, c = packed["values"], packed["idx"], packed["counts"]
    N = c.shape[0]
    H = np.empty((N, f), dtype=np.uint16)
    if packed.get("hybrid") == "tiles":
        _load().oracle_unpack_tiles(_p(_c(v, np.uint16)), _p(_c(i, np.uint8)), _p(_c(c, np.uint8)),
                                    _p(_c(packed["pool"], np.uint16)), N, f, packed["T"], packed["C"], _p(H))
        return H
    fbd = _c(packed["fb_dense"], np.uint16)
    _load().oracle_unpack(_p(_c(v, np.uint16)), _p(_c(i, np.uint8)), _p(_c(c, np.uint8)),
                          _p(_c(packed["row_fb"], np.int32)), _p(fbd),
                          N, f, packed["T"], packed["C"], packed.get("fb_cap", fbd.shape[0]), _p(H))
    return H


def down_dense(H, W_down) -> np.ndarray:
    H, W_down = _c(H, np.uint16), _c(W_down, np.uint16)
    n, f = H.shape
    d = W_down.shape[1]
    Y = np.empty((n, d), dtype=np.float32)
    _load().oracle_down_dense(_p(H), _p(W_down), n, f, d, _p(Y))
    return Y


def down_packed(packed: dict, W_down) -> np.ndarray:
    W_down = _c(W_down, np.uint16)
    f, d = W_down.shape
    N = packed["counts"].shape[0]
    Y = np.empty((N, d), dtype=np.float32)
    if packed.get("hybrid") == "tiles":
        _load().oracle_down_packed_tiles(_p(_c(packed["values"], np.uint16)), _p(_c(packed["idx"], np.uint8)),
                                         _p(_c(packed["counts"], np.uint8)), _p(_c(packed["pool"], np.uint16)),
                                         _p(W_down), N, f, d, packed["T"], packed["C"], _p(Y))
        return Y
    _load().oracle_down_packed(_p(_c(packed["values"], np.uint16)), _p(_c(packed["idx"], np.uint8)),
                               _p(_c(packed["counts"], np.uint8)), _p(_c(packed["row_fb"], np.int32)),
                               _p(_c(packed["fb_dense"], np.uint16)), _p(W_down), N, f, d,
                               packed["T"], packed["C"], packed.get("fb_cap", packed["fb_dense"].shape[0]), _p(Y))
    return Y


def grad_hidden(dY, W_down, H_sel, lam: float, rows=None):
    """(dH, dZ) for the selected rows; H_sel holds those rows of H."""
    dY, W_down, H_sel = _c(dY, np.uint16), _c(W_down, np.uint16), _c(H_sel, np.uint16)
    f, d = W_down.shape
    r = _rows(rows, dY.shape[0])
    dH = np.empty((len(r), f), dtype=np.float32)
    dZ = np.empty((len(r), f), dtype=np.float32)
    _load().oracle_grad_hidden(_p(dY), _p(W_down), _p(H_sel), float(lam), _p(r), len(r), d, f,
                               _p(dH), _p(dZ))
    return dH, dZ


def grad_input(dZ, W_inT) -> np.ndarray:
    dZ, W_inT = _c(dZ, np.float32), _c(W_inT, np.uint16)
    f, d = W_inT.shape
    n = dZ.shape[0]
    dX = np.empty((n, d), dtype=np.float32)
    _load().oracle_grad_input(_p(dZ), _p(W_inT), n, d, f, _p(dX))
    return dX


def grad_weights(X, W_down, H, dY, lam: float, cols=None):
    """(dW_inT, dW_down, db) restricted to the hidden units `cols` (all by default)."""
    X, W_down, H, dY = (_c(a, np.uint16) for a in (X, W_down, H, dY))
    N, d = X.shape
    f = W_down.shape[0]
    c = _rows(cols, f)
    dWin = np.empty((len(c), d), dtype=np.float32)
    dWdown = np.empty((len(c), d), dtype=np.float32)
    db = np.empty((len(c),), dtype=np.float32)
    _load().oracle_grad_weights(_p(X), _p(W_down), _p(H), _p(dY), float(lam), N, d, f, _p(c), len(c),
                                _p(dWin), _p(dWdown), _p(db))
    return dWin, dWdown, db


def grad_hidden_gated(X, W_gT, W_uT, b, dY, W_down, H, lam: float, rows=None):
    """(dG, dU) of the gated layer for the selected rows; H is the full [N][f]."""
    X, W_gT, W_uT, b, dY, W_down, H = (_c(a, np.uint16) for a in (X, W_gT, W_uT, b, dY, W_down, H))
    f, d = W_gT.shape
    r = _rows(rows, X.shape[0])
    dG = np.empty((len(r), f), dtype=np.float32)
    dU = np.empty((len(r), f), dtype=np.float32)
    _load().oracle_grad_hidden_gated(_p(X), _p(W_gT), _p(W_uT), _p(b), _p(dY), _p(W_down), _p(H), float(lam),
                                     _p(r), len(r), d, f, _p(dG), _p(dU))
    return dG, dU


def grad_input_gated(dG, dU, W_gT, W_uT) -> np.ndarray:
    dG, dU = _c(dG, np.float32), _c(dU, np.float32)
    W_gT, W_uT = _c(W_gT, np.uint16), _c(W_uT, np.uint16)
    f, d = W_gT.shape
    n = dG.shape[0]
    dX = np.empty((n, d), dtype=np.float32)
    _load().oracle_grad_input_gated(_p(dG), _p(dU), _p(W_gT), _p(W_uT), n, d, f, _p(dX))
    return dX


def grad_weights_gated(X, W_gT, W_uT, b, W_down, H, dY, lam: float, cols=None):
    """(dW_gT, dW_uT, dW_down, db) of the gated layer for the hidden units `cols`."""
    X, W_gT, W_uT, b, W_down, H, dY = (_c(a, np.uint16) for a in (X, W_gT, W_uT, b, W_down, H, dY))
    N, d = X.shape
    f = W_gT.shape[0]
    c = _rows(cols, f)
    out = [np.empty((len(c), d), dtype=np.float32) for _ in range(3)]
    db = np.empty((len(c),), dtype=np.float32)
    _load().oracle_grad_weights_gated(_p(X), _p(W_gT), _p(W_uT), _p(b), _p(W_down), _p(H), _p(dY), float(lam),
                                      N, d, f, _p(c), len(c), _p(out[0]), _p(out[1]), _p(out[2]), _p(db))
    return out[0], out[1], out[2], db


def check_format(packed: dict, f: int) -> int:
    """0 when the packed layer satisfies the TwELL format invariants, else a rule code."""
    N = packed["counts"].shape[0]
    if packed.get("hybrid") == "tiles":
        return int(_load().oracle_check_format_tiles(
            _p(_c(packed["values"], np.uint16)), _p(_c(packed["idx"], np.uint8)),
            _p(_c(packed["counts"], np.uint8)), _p(_c(packed["row_fb"], np.int32)),
            _p(_c(packed["pool"], np.uint16)), int(packed["n_fb"]), N, f, packed["T"], packed["C"],
            packed["pool_cap"]))
    return int(_load().oracle_check_format(
        _p(_c(packed["values"], np.uint16)), _p(_c(packed["idx"], np.uint8)), _p(_c(packed["counts"], np.uint8)),
        _p(_c(packed["row_fb"], np.int32)), _p(_c(packed["fb_rows"], np.int32)), int(packed["n_fb"]),
        N, f, packed["T"], packed["C"], packed["fb_cap"]))


def forward(X, W_inT, b, W_down, T: int, C: int, fb_cap: int, rows=None, hybrid: str = "rows") -> dict:
    """Whole forward for the selected rows: z, h, packed h, Y (fp32) and bf16(Y).
    hybrid="tiles" packs with the tile-granular hybrid, a pool of
    fb_cap * (d_ff / T) dense tiles."""
    Z, H = hidden(X, W_inT, b, rows)
    if hybrid == "tiles":
        packed = pack_tiles(H, T, C, fb_cap * (H.shape[1] // T))
    else:
        packed = pack(H, T, C, fb_cap)
    Y = down_packed(packed, W_down)
    return {"Z": Z, "H": H, "packed": packed, "Y": Y, "Y_bf16": round_bf16(Y)}
