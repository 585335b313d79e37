"""Python binding of libtwell.so, the TwELL activation-sparse FFN for GB300.

Argument marshalling only: every step of the layer runs in the library's CUDA
kernels (include/twell.h documents each call).  torch supplies device memory
and the current stream; bf16 tensors are passed by pointer.  If the library
has not been built, every call raises -- there is no CPU or eager fallback.

One training step of a layer (X [N, d] bf16; W_inT, W_down [f, d] bf16; b [f]
bf16; T the tile width, C the per-tile capacity, fb_cap the dense fallback
rows):

    import activation_sparse_transformer_gb300 as tw
    H = tw.alloc_packed(N, f, T, C, fb_cap, "cuda")      # the packed activations
    ws = torch.empty(max(tw.fwd_workspace_bytes(N, d, f, T, C, fb_cap),
                         tw.bwd_workspace_bytes(N, d, f, T, C, fb_cap)),
                     dtype=torch.uint8, device="cuda")      # one scratch for both calls
    tw.twell_ffn_fwd(X, W_inT, b, W_down, H, Y, ws)          # Y [N, d] bf16
    tw.twell_ffn_bwd(X, W_inT, W_down, H, dY, l1_lambda,     # dX bf16; dW_inT, dW_down,
                     dX, dW_inT, dW_down, db, ws)           # db fp32
    assert tw.twell_read_status(H) == 0                      # e.g. fallback overflow

The calls are asynchronous on the current stream and can be captured in a CUDA
graph; twell_pack / twell_unpack convert between dense bf16 H and the packed form.
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass
from typing import Optional

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libtwell.so")

TWELL_OK = 0
KERNELS = {
    "up_pack": 0, "route": 1, "fb_assemble": 2, "spmm": 4, "fb_down": 5, "pack": 6,
    "check_format": 3, "unpack": 7, "sddmm": 8, "dx": 9, "dw": 10, "dense_gemm": 11, "aux": 12,
    "dw_fallback": 13, "dx_fallback": 14,
}
EXPORTED = [
    "twell_pack", "twell_unpack", "twell_ffn_fwd", "twell_fwd_workspace_bytes", "twell_ffn_bwd",
    "twell_bwd_workspace_bytes", "twell_dense_ffn_fwd", "twell_read_status", "twell_status_string",
    "twell_launch_count", "twell_profile_enable", "twell_profile_reset", "twell_profile_read",
    "twell_profile_timeline",
    "twell_ffn_fwd_noalloc", "twell_ffn_fwd_noalloc_max_scratch", "twell_gated_ffn_fwd",
    "twell_selftest_wait_timeout", "twell_check_format", "twell_dense_ffn_bwd", "twell_dense_bwd_workspace_bytes",
    "twell_bwd_tiles_workspace_bytes", "twell_gated_ffn_fwd_train", "twell_gated_ffn_bwd",
    "twell_gated_bwd_workspace_bytes", "twell_gated_bwd_tiles_workspace_bytes",
]


class TwellError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__(f"{where}: {status_string(code)} ({code})")


class twell_t(ctypes.Structure):
    _fields_ = [
        ("n_rows", ctypes.c_int32), ("d_ff", ctypes.c_int32), ("tile", ctypes.c_int32),
        ("cap", ctypes.c_int32), ("fb_cap", ctypes.c_int32), ("hybrid", ctypes.c_int32),
        ("values", ctypes.c_void_p), ("idx", ctypes.c_void_p), ("counts", ctypes.c_void_p),
        ("row_fb", ctypes.c_void_p), ("fb_rows", ctypes.c_void_p), ("fb_dense", ctypes.c_void_p),
        ("n_fb", ctypes.c_void_p), ("status", ctypes.c_void_p),
    ]


_lib_handle = None


def load_library() -> ctypes.CDLL:
    """Loads libtwell.so; raises if it is missing (build it with __graft_entry__.build())."""
    global _lib_handle
    if _lib_handle is not None:
        return _lib_handle
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"{LIB_PATH} is not built; run `python -c 'import __graft_entry__ as g; g.build()'`")
    lib = ctypes.CDLL(LIB_PATH)
    P, I32, I64, SZ = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t
    L = ctypes.POINTER(twell_t)
    sig = {
        "twell_pack": (ctypes.c_int, [P, I64, L, P]),
        "twell_unpack": (ctypes.c_int, [L, P, I64, P]),
        "twell_ffn_fwd": (ctypes.c_int, [P, P, P, P, I32, I32, I32, L, P, P, SZ, P]),
        "twell_fwd_workspace_bytes": (SZ, [I32, I32, I32, I32, I32, I32]),
        "twell_ffn_bwd": (ctypes.c_int, [P, P, P, L, I32, P, ctypes.c_float, P, P, P, P, P, SZ, P]),
        "twell_bwd_workspace_bytes": (SZ, [I32, I32, I32, I32, I32, I32]),
        "twell_bwd_tiles_workspace_bytes": (SZ, [I32, I32, I32, I32, I32, I32]),
        "twell_dense_ffn_fwd": (ctypes.c_int, [P, P, P, P, I32, I32, I32, P, P, P]),
        "twell_read_status": (ctypes.c_int, [L, P]),
        "twell_status_string": (ctypes.c_char_p, [ctypes.c_int]),
        "twell_launch_count": (I64, []),
        "twell_profile_enable": (ctypes.c_int, [ctypes.c_int]),
        "twell_profile_reset": (ctypes.c_int, []),
        "twell_profile_read": (ctypes.c_int, [ctypes.c_int, ctypes.POINTER(I64), ctypes.POINTER(ctypes.c_double)]),
        "twell_profile_timeline": (ctypes.c_int, [ctypes.c_int, ctypes.POINTER(ctypes.c_int32),
                                                  ctypes.POINTER(ctypes.c_uint64), ctypes.POINTER(ctypes.c_double),
                                                  ctypes.POINTER(ctypes.c_double)]),
        "twell_ffn_fwd_noalloc": (ctypes.c_int, [P, P, P, P, I32, I32, I32, L, P, P]),
        "twell_ffn_fwd_noalloc_max_scratch": (SZ, []),
        "twell_gated_ffn_fwd": (ctypes.c_int, [P, P, P, P, P, I32, I32, I32, L, P, P, SZ, P]),
        "twell_gated_ffn_fwd_train": (ctypes.c_int, [P, P, P, P, P, I32, I32, I32, L, P, P, P, SZ, P]),
        "twell_gated_ffn_bwd": (ctypes.c_int, [P, P, P, P, P, L, P, I32, P, ctypes.c_float, P, P, P, P, P, P, SZ,
                                               P]),
        "twell_gated_bwd_workspace_bytes": (SZ, [I32, I32, I32, I32, I32, I32]),
        "twell_gated_bwd_tiles_workspace_bytes": (SZ, [I32, I32, I32, I32, I32, I32]),
        "twell_selftest_wait_timeout": (ctypes.c_int, [P, ctypes.c_uint64, P]),
        "twell_check_format": (ctypes.c_int, [L, P, P]),
        "twell_dense_ffn_bwd": (ctypes.c_int, [P, P, P, P, I32, I32, I32, P, ctypes.c_float, P, P, P, P, P, SZ, P]),
        "twell_dense_bwd_workspace_bytes": (SZ, [I32, I32, I32]),
    }
    for name, (res, args) in sig.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib_handle = lib
    return lib


def status_string(code: int) -> str:
    return load_library().twell_status_string(int(code)).decode()


def _check(code: int, where: str) -> None:
    if code != TWELL_OK:
        raise TwellError(code, where)


def _stream(stream=None) -> int:
    import torch
    s = stream if stream is not None else torch.cuda.current_stream()
    return int(s.cuda_stream)


def _need(t, nbytes: int, name: str) -> None:
    """Rejects a buffer smaller than the bytes the call reads or writes through
    it (the C ABI receives only the pointer)."""
    have = 0 if t is None else t.numel() * t.element_size()
    if have < nbytes:
        raise ValueError(f"{name}: {have} bytes, the call needs {nbytes}")


def _need_dense(t, rows: int, row_elems: int, ld: int, elem_bytes: int, name: str) -> None:
    """A [rows][ld] buffer of which the first row_elems of every row are used."""
    _need(t, ((rows - 1) * ld + row_elems) * elem_bytes if rows > 0 else 0, name)


def _ptr(t) -> Optional[int]:
    if t is None:
        return None
    if not (t.is_cuda and t.is_contiguous()):
        raise ValueError("tensors passed to libtwell must be contiguous CUDA tensors")
    return t.data_ptr()


@dataclass
class Packed:
    """Device buffers of one TwELL hybrid layout and the twell_t that names them."""
    values: "object"
    idx: "object"
    counts: "object"
    row_fb: "object"
    fb_rows: "object"
    fb_dense: "object"
    n_fb: "object"
    status: "object"
    n_rows: int
    d_ff: int
    tile: int
    cap: int
    fb_cap: int
    hybrid: int = 0   # HYBRID_ROWS or HYBRID_TILES

    def struct(self) -> twell_t:
        N, nt = self.n_rows, self.d_ff // self.tile
        cells = N * nt
        _need(self.values, cells * self.cap * 2, "values")
        _need(self.idx, cells * self.cap, "idx")
        _need(self.counts, cells, "counts")
        _need(self.row_fb, N * 4, "row_fb")
        _need(self.fb_rows, self.fb_cap * 4, "fb_rows")
        _need(self.fb_dense, self.fb_cap * self.d_ff * 2, "fb_dense")
        _need(self.n_fb, 4, "n_fb")
        _need(self.status, 4, "status")
        p = lambda t: t.data_ptr() if t is not None and t.numel() else None
        return twell_t(self.n_rows, self.d_ff, self.tile, self.cap, self.fb_cap, self.hybrid,
                       p(self.values), p(self.idx), p(self.counts), p(self.row_fb), p(self.fb_rows),
                       p(self.fb_dense), p(self.n_fb), p(self.status))


HYBRID_ROWS, HYBRID_TILES, DENSE_TILE = 0, 1, 255


def alloc_packed(n_rows: int, d_ff: int, tile: int, cap: int, fb_cap: int, device="cuda",
                 hybrid: int = HYBRID_ROWS) -> Packed:
    """Buffers of a packed layer.  With hybrid=HYBRID_TILES, fb_dense is the pool
    of fb_cap * d_ff / tile dense tiles."""
    import torch
    nt = d_ff // tile
    kw = dict(device=device)
    return Packed(
        values=torch.empty((n_rows, nt, cap), dtype=torch.bfloat16, **kw),
        idx=torch.empty((n_rows, nt, cap), dtype=torch.uint8, **kw),
        counts=torch.empty((n_rows, nt), dtype=torch.uint8, **kw),
        row_fb=torch.empty((max(n_rows, 1),), dtype=torch.int32, **kw),
        fb_rows=torch.empty((max(fb_cap, 1),), dtype=torch.int32, **kw),
        fb_dense=torch.empty((max(fb_cap, 1), d_ff), dtype=torch.bfloat16, **kw),
        n_fb=torch.zeros((4,), dtype=torch.int32, **kw),
        status=torch.zeros((4,), dtype=torch.int32, **kw),
        n_rows=n_rows, d_ff=d_ff, tile=tile, cap=cap, fb_cap=fb_cap, hybrid=hybrid,
    )


def twell_pack(H, packed: Packed, stream=None) -> None:
    """Dense bf16 H [n_rows, >= d_ff] -> TwELL hybrid (asynchronous)."""
    _need_dense(H, packed.n_rows, packed.d_ff, H.stride(0), 2, "H")
    st = packed.struct()
    _check(load_library().twell_pack(_ptr(H), H.stride(0), ctypes.byref(st), _stream(stream)), "twell_pack")


def twell_unpack(packed: Packed, H, stream=None) -> None:
    _need_dense(H, packed.n_rows, packed.d_ff, H.stride(0), 2, "H")
    st = packed.struct()
    _check(load_library().twell_unpack(ctypes.byref(st), _ptr(H), H.stride(0), _stream(stream)), "twell_unpack")


def fwd_workspace_bytes(n_rows, d_model, d_ff, tile, cap, fb_cap) -> int:
    return int(load_library().twell_fwd_workspace_bytes(n_rows, d_model, d_ff, tile, cap, fb_cap))


def bwd_workspace_bytes(n_rows, d_model, d_ff, tile, cap, fb_cap, hybrid=None) -> int:
    """Workspace of twell_ffn_bwd; hybrid=HYBRID_TILES for a tile-granular layout."""
    lib = load_library()
    fn = lib.twell_bwd_tiles_workspace_bytes if hybrid == HYBRID_TILES else lib.twell_bwd_workspace_bytes
    return int(fn(n_rows, d_model, d_ff, tile, cap, fb_cap))


def _need_layer(n, d, f, W_inT, b, W_down, Y) -> None:
    _need(W_inT, f * d * 2, "W_inT")
    _need(b, f * 2, "b")
    _need(W_down, f * d * 2, "W_down")
    _need(Y, n * d * 2, "Y")


def twell_ffn_fwd(X, W_inT, b, W_down, packed: Packed, Y, workspace, stream=None) -> None:
    n, d = X.shape
    f = W_inT.shape[0]
    _need_layer(n, d, f, W_inT, b, W_down, Y)
    st = packed.struct()
    _check(load_library().twell_ffn_fwd(_ptr(X), _ptr(W_inT), _ptr(b), _ptr(W_down), n, d, f, ctypes.byref(st),
                                        _ptr(Y), _ptr(workspace), workspace.numel() * workspace.element_size(),
                                        _stream(stream)), "twell_ffn_fwd")


def twell_gated_ffn_fwd(X, W_gT, W_uT, b, W_down, packed: Packed, Y, workspace, stream=None) -> None:
    """Gated ReLU layer: H = ReLU(X.W_g + b) * (X.W_u) packed in TwELL, Y = H.W_down."""
    n, d = X.shape
    f = W_gT.shape[0]
    _need_layer(n, d, f, W_gT, b, W_down, Y)
    _need(W_uT, f * d * 2, "W_uT")
    st = packed.struct()
    _check(load_library().twell_gated_ffn_fwd(_ptr(X), _ptr(W_gT), _ptr(W_uT), _ptr(b), _ptr(W_down), n, d, f,
                                              ctypes.byref(st), _ptr(Y), _ptr(workspace),
                                              workspace.numel() * workspace.element_size(), _stream(stream)),
           "twell_gated_ffn_fwd")


def twell_gated_ffn_fwd_train(X, W_gT, W_uT, b, W_down, packed: Packed, Y, gu, workspace, stream=None) -> None:
    """twell_gated_ffn_fwd that also keeps (g, u) fp32 at every stored slot in gu
    ([n_rows][d_ff / tile][cap][2] float32), for twell_gated_ffn_bwd."""
    n, d = X.shape
    f = W_gT.shape[0]
    _need_layer(n, d, f, W_gT, b, W_down, Y)
    _need(W_uT, f * d * 2, "W_uT")
    _need(gu, n * (f // packed.tile) * packed.cap * 8, "gu")
    st = packed.struct()
    _check(load_library().twell_gated_ffn_fwd_train(_ptr(X), _ptr(W_gT), _ptr(W_uT), _ptr(b), _ptr(W_down), n, d,
                                                    f, ctypes.byref(st), _ptr(Y), _ptr(gu), _ptr(workspace),
                                                    workspace.numel() * workspace.element_size(), _stream(stream)),
           "twell_gated_ffn_fwd_train")


def twell_ffn_fwd_noalloc(X, W_inT, b, W_down, packed: Packed, Y, stream=None) -> None:
    """twell_ffn_fwd without a workspace argument: the library's fixed scratch
    array is used (for callers that cannot allocate device memory)."""
    n, d = X.shape
    f = W_inT.shape[0]
    _need_layer(n, d, f, W_inT, b, W_down, Y)
    st = packed.struct()
    _check(load_library().twell_ffn_fwd_noalloc(_ptr(X), _ptr(W_inT), _ptr(b), _ptr(W_down), n, d, f,
                                                ctypes.byref(st), _ptr(Y), _stream(stream)),
           "twell_ffn_fwd_noalloc")


def twell_ffn_bwd(X, W_inT, W_down, packed: Packed, dY, l1_lambda: float, dX, dW_inT, dW_down, db, workspace,
                  stream=None) -> None:
    d = X.shape[1]
    n, f = packed.n_rows, packed.d_ff
    for t, nbytes, name in ((X, n * d * 2, "X"), (W_inT, f * d * 2, "W_inT"), (W_down, f * d * 2, "W_down"),
                            (dY, n * d * 2, "dY"), (dX, n * d * 2, "dX"), (dW_inT, f * d * 4, "dW_inT"),
                            (dW_down, f * d * 4, "dW_down"), (db, f * 4, "db")):
        _need(t, nbytes, name)
    st = packed.struct()
    _check(load_library().twell_ffn_bwd(_ptr(X), _ptr(W_inT), _ptr(W_down), ctypes.byref(st), d, _ptr(dY),
                                        float(l1_lambda), _ptr(dX), _ptr(dW_inT), _ptr(dW_down), _ptr(db),
                                        _ptr(workspace), workspace.numel() * workspace.element_size(),
                                        _stream(stream)), "twell_ffn_bwd")


def gated_bwd_workspace_bytes(n_rows, d_model, d_ff, tile, cap, fb_cap, hybrid=None) -> int:
    """Workspace of twell_gated_ffn_bwd; hybrid=HYBRID_TILES for a tile-granular layout."""
    lib = load_library()
    fn = lib.twell_gated_bwd_tiles_workspace_bytes if hybrid == HYBRID_TILES else lib.twell_gated_bwd_workspace_bytes
    return int(fn(n_rows, d_model, d_ff, tile, cap, fb_cap))


def twell_gated_ffn_bwd(X, W_gT, W_uT, b, W_down, packed: Packed, gu, dY, l1_lambda: float, dX, dW_gT, dW_uT,
                        dW_down, db, workspace, stream=None) -> None:
    """Backward of the gated layer; gu is what twell_gated_ffn_fwd_train kept."""
    d = X.shape[1]
    n, f = packed.n_rows, packed.d_ff
    for t, nbytes, name in ((X, n * d * 2, "X"), (W_gT, f * d * 2, "W_gT"), (W_uT, f * d * 2, "W_uT"),
                            (b, f * 2, "b"), (W_down, f * d * 2, "W_down"),
                            (gu, n * (f // packed.tile) * packed.cap * 8, "gu"), (dY, n * d * 2, "dY"),
                            (dX, n * d * 2, "dX"), (dW_gT, f * d * 4, "dW_gT"), (dW_uT, f * d * 4, "dW_uT"),
                            (dW_down, f * d * 4, "dW_down"), (db, f * 4, "db")):
        _need(t, nbytes, name)
    st = packed.struct()
    _check(load_library().twell_gated_ffn_bwd(_ptr(X), _ptr(W_gT), _ptr(W_uT), _ptr(b), _ptr(W_down),
                                              ctypes.byref(st), _ptr(gu), d, _ptr(dY), float(l1_lambda), _ptr(dX),
                                              _ptr(dW_gT), _ptr(dW_uT), _ptr(dW_down), _ptr(db), _ptr(workspace),
                                              workspace.numel() * workspace.element_size(), _stream(stream)),
           "twell_gated_ffn_bwd")


def twell_dense_ffn_fwd(X, W_inT, b, W_down, Hbuf, Y, stream=None) -> None:
    """Dense comparator: Y = ReLU(X.W_in + b).W_down on the same tensor-core GEMM."""
    n, d = X.shape
    f = W_inT.shape[0]
    _need_layer(n, d, f, W_inT, b, W_down, Y)
    _need(Hbuf, n * f * 2, "Hbuf")
    _check(load_library().twell_dense_ffn_fwd(_ptr(X), _ptr(W_inT), _ptr(b), _ptr(W_down), n, d, f, _ptr(Hbuf),
                                              _ptr(Y), _stream(stream)), "twell_dense_ffn_fwd")


def dense_bwd_workspace_bytes(n_rows, d_model, d_ff) -> int:
    return int(load_library().twell_dense_bwd_workspace_bytes(n_rows, d_model, d_ff))


def twell_dense_ffn_bwd(X, W_inT, W_down, Hbuf, dY, l1_lambda: float, dX, dW_inT, dW_down, db, workspace,
                        stream=None) -> None:
    """Dense comparator's backward: the gradients of twell_ffn_bwd for the layer
    run densely (Hbuf = the dense forward's H), with no sparsity used."""
    n, d = X.shape
    f = W_inT.shape[0]
    for t, nbytes, name in ((X, n * d * 2, "X"), (W_inT, f * d * 2, "W_inT"), (W_down, f * d * 2, "W_down"),
                            (Hbuf, n * f * 2, "Hbuf"), (dY, n * d * 2, "dY"), (dX, n * d * 2, "dX"),
                            (dW_inT, f * d * 4, "dW_inT"), (dW_down, f * d * 4, "dW_down"), (db, f * 4, "db"),
                            (workspace, dense_bwd_workspace_bytes(n, d, f), "workspace")):
        _need(t, nbytes, name)
    _check(load_library().twell_dense_ffn_bwd(_ptr(X), _ptr(W_inT), _ptr(W_down), _ptr(Hbuf), n, d, f, _ptr(dY),
                                              float(l1_lambda), _ptr(dX), _ptr(dW_inT), _ptr(dW_down), _ptr(db),
                                              _ptr(workspace), workspace.numel() * workspace.element_size(),
                                              _stream(stream)), "twell_dense_ffn_bwd")


def twell_check_format(packed: Packed, violations, stream=None) -> None:
    """Check the layout's format rules on the device (asynchronous): bit k of
    the device int32 tensor `violations` is set when rule k is broken."""
    _need(violations, 4, "violations")
    st = packed.struct()
    _check(load_library().twell_check_format(ctypes.byref(st), _ptr(violations), _stream(stream)),
           "twell_check_format")


def twell_read_status(packed: Packed, stream=None) -> int:
    st = packed.struct()
    return int(load_library().twell_read_status(ctypes.byref(st), _stream(stream)))


def twell_selftest_wait_timeout(status, limit_ns: int, stream=None) -> None:
    """Run the pipelines' bounded wait on a barrier nothing arrives on; status
    (a device int32 tensor) becomes TWELL_ERR_WAIT_TIMEOUT once limit_ns pass."""
    _check(load_library().twell_selftest_wait_timeout(_ptr(status), int(limit_ns), _stream(stream)),
           "twell_selftest_wait_timeout")


def twell_launch_count() -> int:
    return int(load_library().twell_launch_count())


def twell_profile_enable(on: bool) -> None:
    _check(load_library().twell_profile_enable(1 if on else 0), "twell_profile_enable")


def twell_profile_reset() -> None:
    _check(load_library().twell_profile_reset(), "twell_profile_reset")


def twell_profile_timeline(max_entries: int = 4096) -> list:
    """Recorded launches in order: dicts with kernel (name), stream, start_ms,
    end_ms (device times relative to the first recorded launch)."""
    k = (ctypes.c_int32 * max_entries)()
    st = (ctypes.c_uint64 * max_entries)()
    a = (ctypes.c_double * max_entries)()
    b = (ctypes.c_double * max_entries)()
    n = load_library().twell_profile_timeline(max_entries, k, st, a, b)
    _check(min(n, 0), "twell_profile_timeline")
    names = {v: name for name, v in KERNELS.items()}
    return [{"kernel": names.get(k[i], str(k[i])), "stream": int(st[i]), "start_ms": a[i], "end_ms": b[i]}
            for i in range(n)]


def twell_profile_read(kernel) -> tuple:
    """(launches, total_ms) of one kernel id or name since the last reset."""
    k = KERNELS[kernel] if isinstance(kernel, str) else int(kernel)
    n = ctypes.c_int64(0)
    ms = ctypes.c_double(0.0)
    _check(load_library().twell_profile_read(k, ctypes.byref(n), ctypes.byref(ms)), "twell_profile_read")
    return int(n.value), float(ms.value)
