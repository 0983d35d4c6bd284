"""CPU oracle for the N:4 2bit-CSR INT4 SparseGemv (test infrastructure).

Only the test suite, ``__graft_entry__.smoke()`` and the benchmark's CPU
baseline leg may import this package.  The product library never does, and
this package imports nothing from the product.

The arithmetic lives in ``sgemv_oracle.c`` (plain C, fp64 dequantisation and
naive matvec); this module only builds it with gcc and marshals numpy arrays.
The method follows Dong et al., "Efficient LLM ad generation via model
compression and parallel verification" (arXiv 2605.11582), sections 1 and
3.2; the readings of what those sections leave open are documented in the C
source.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "sgemv_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

ORC_OK = 0
ORC_ERR_ARG = -1
ORC_ERR_NONFINITE = -6
ORC_ERR_RANGE = -7


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (no fast-math, no FMA contraction)."""
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= max(
                os.path.getmtime(_SRC),
                os.path.getmtime(os.path.join(_HERE, "sgemv_oracle.h")))):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-std=c11", "-O2", "-ffp-contract=off", "-fno-fast-math",
           "-fPIC", "-shared", "-Wall", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        build()
        lib = ctypes.CDLL(_LIB_PATH)
        P = ctypes.c_void_p
        I64 = ctypes.c_int64
        I = ctypes.c_int
        lib.orc_f64_to_f16.argtypes = [ctypes.c_double]
        lib.orc_f64_to_f16.restype = ctypes.c_uint16
        lib.orc_f32_to_f16.argtypes = [ctypes.c_float]
        lib.orc_f32_to_f16.restype = ctypes.c_uint16
        lib.orc_f16_to_f64.argtypes = [ctypes.c_uint16]
        lib.orc_f16_to_f64.restype = ctypes.c_double
        lib.orc_vals_row_bytes.argtypes = [I64, I]
        lib.orc_vals_row_bytes.restype = I64
        lib.orc_idx_row_bytes.argtypes = [I64, I]
        lib.orc_idx_row_bytes.restype = I64
        lib.orc_prune.argtypes = [P, I64, I64, I, P]
        lib.orc_prune.restype = I
        lib.orc_quantize.argtypes = [P, P, I64, I64, I, I, P, P, P]
        lib.orc_quantize.restype = I
        lib.orc_encode.argtypes = [P, P, I64, I64, I, P, P]
        lib.orc_encode.restype = None
        lib.orc_decode.argtypes = [P, P, I64, I64, I, P, P]
        lib.orc_decode.restype = None
        lib.orc_pack.argtypes = [P, I64, I64, I, I, P, P, P, P]
        lib.orc_pack.restype = I
        lib.orc_prune_scored.argtypes = [P, P, P, I64, I64, I, P]
        lib.orc_prune_scored.restype = I
        lib.orc_pack_scored.argtypes = [P, P, P, I64, I64, I, I, P, P, P, P]
        lib.orc_pack_scored.restype = I
        lib.orc_quantize_rowg.argtypes = [P, P, I64, I64, I, P, P, P, P]
        lib.orc_quantize_rowg.restype = I
        lib.orc_pack_rowg.argtypes = [P, I64, I64, I, P, P, P, P, P]
        lib.orc_pack_rowg.restype = I
        lib.orc_dequant_rows_rowg.argtypes = [P, P, P, P, I64, I, P, I64, I64, P]
        lib.orc_dequant_rows_rowg.restype = None
        lib.orc_matvec_rowg.argtypes = [P, P, P, P, I64, I64, I, P, P, I, P, I64, P]
        lib.orc_matvec_rowg.restype = None
        lib.orc_dequant_rows.argtypes = [P, P, P, P, I64, I, I, I64, I64, P]
        lib.orc_dequant_rows.restype = None
        lib.orc_matvec.argtypes = [P, P, P, P, I64, I, I, P, I, P, I64, P]
        lib.orc_matvec.restype = None
        _lib = lib
        return lib


class OracleError(RuntimeError):
    def __init__(self, code: int, what: str):
        super().__init__(f"oracle {what} failed with code {code}")
        self.code = code


def _ptr(a: np.ndarray) -> int:
    return a.ctypes.data


def _c(a, dtype) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=dtype)


def f64_to_f16_bits(v: float) -> int:
    return int(_load().orc_f64_to_f16(float(v)))


def f32_to_f16_bits(v: float) -> int:
    return int(_load().orc_f32_to_f16(float(v)))


def f16_bits_to_f64(h: int) -> float:
    return float(_load().orc_f16_to_f64(int(h) & 0xFFFF))


def f64_to_f16_array(a: np.ndarray) -> np.ndarray:
    """Element-wise binary16 rounding of a float64 array (bit patterns)."""
    lib = _load()
    flat = np.asarray(a, dtype=np.float64).ravel()
    out = np.fromiter((lib.orc_f64_to_f16(float(v)) for v in flat),
                      dtype=np.uint16, count=flat.size)
    return out.reshape(np.shape(a))


def row_bytes(cols: int, n_keep: int) -> tuple[int, int]:
    lib = _load()
    return int(lib.orc_vals_row_bytes(cols, n_keep)), int(
        lib.orc_idx_row_bytes(cols, n_keep))


def prune(W: np.ndarray, n_keep: int) -> np.ndarray:
    W = _c(W, np.float32)
    rows, cols = W.shape
    pos = np.zeros((rows, cols // 4, n_keep), dtype=np.uint8)
    rc = _load().orc_prune(_ptr(W), rows, cols, n_keep, _ptr(pos))
    if rc:
        raise OracleError(rc, "prune")
    return pos


def prune_scored(W: np.ndarray, xnorm: np.ndarray, grad, n_keep: int) -> np.ndarray:
    """Eq. 3 pruning: keep per quad the N largest |w|*xnorm + |w|*|grad|."""
    W = _c(W, np.float32)
    rows, cols = W.shape
    xn = _c(xnorm, np.float32)
    g = None if grad is None else _c(grad, np.float32)
    pos = np.zeros((rows, cols // 4, n_keep), dtype=np.uint8)
    rc = _load().orc_prune_scored(_ptr(W), _ptr(xn), None if g is None else _ptr(g),
                                  rows, cols, n_keep, _ptr(pos))
    if rc:
        raise OracleError(rc, "prune_scored")
    return pos


def quantize(W: np.ndarray, pos: np.ndarray, n_keep: int, group: int):
    W = _c(W, np.float32)
    pos = _c(pos, np.uint8)
    rows, cols = W.shape
    P = cols // 4 * n_keep
    q = np.zeros((rows, P), dtype=np.uint8)
    ng = cols // group if group else 0
    scale = np.zeros((rows, ng), dtype=np.uint16)
    zero = np.zeros((rows, ng), dtype=np.uint16)
    rc = _load().orc_quantize(_ptr(W), _ptr(pos), rows, cols, n_keep, group,
                              _ptr(q), _ptr(scale), _ptr(zero))
    if rc:
        raise OracleError(rc, "quantize")
    return q, scale, zero


def encode(pos: np.ndarray, q: np.ndarray, rows: int, cols: int, n_keep: int):
    pos = _c(pos, np.uint8)
    q = _c(q, np.uint8)
    vb, ib = row_bytes(cols, n_keep)
    vals = np.zeros((rows, vb), dtype=np.uint8)
    idx = np.zeros((rows, ib), dtype=np.uint8)
    _load().orc_encode(_ptr(pos), _ptr(q), rows, cols, n_keep, _ptr(vals),
                       _ptr(idx))
    return vals, idx


def decode(vals: np.ndarray, idx: np.ndarray, rows: int, cols: int,
           n_keep: int):
    vals = _c(vals, np.uint8)
    idx = _c(idx, np.uint8)
    P = cols // 4 * n_keep
    pos = np.zeros((rows, P), dtype=np.uint8)
    q = np.zeros((rows, P), dtype=np.uint8)
    _load().orc_decode(_ptr(vals), _ptr(idx), rows, cols, n_keep, _ptr(pos),
                       _ptr(q))
    return pos, q


class Packed:
    """Canonical 2bit-CSR arrays of one weight matrix.  With per-row group
    sizes, `row_group` holds them (int32, one per row), `group` is None and
    scale/zero are flat: each row's cols/row_group[r] entries in row order."""

    def __init__(self, rows, cols, n_keep, group, vals, idx, scale, zero, row_group=None):
        self.rows, self.cols, self.n_keep, self.group = rows, cols, n_keep, group
        self.vals, self.idx, self.scale, self.zero = vals, idx, scale, zero
        self.row_group = row_group


def pack(W: np.ndarray, n_keep: int, group: int) -> Packed:
    W = _c(W, np.float32)
    rows, cols = W.shape
    vb, ib = row_bytes(cols, n_keep)
    ng = cols // group if group else 0
    vals = np.zeros((rows, vb), dtype=np.uint8)
    idx = np.zeros((rows, ib), dtype=np.uint8)
    scale = np.zeros((rows, ng), dtype=np.uint16)
    zero = np.zeros((rows, ng), dtype=np.uint16)
    rc = _load().orc_pack(_ptr(W), rows, cols, n_keep, group, _ptr(vals),
                          _ptr(idx), _ptr(scale), _ptr(zero))
    if rc:
        raise OracleError(rc, "pack")
    return Packed(rows, cols, n_keep, group, vals, idx, scale, zero)


def dequant(p: Packed, row0: int = 0, nrows: int | None = None) -> np.ndarray:
    if nrows is None:
        nrows = p.rows - row0
    out = np.zeros((nrows, p.cols), dtype=np.float64)
    if p.row_group is not None:
        _load().orc_dequant_rows_rowg(_ptr(p.vals), _ptr(p.idx), _ptr(p.scale),
                                      _ptr(p.zero), p.cols, p.n_keep,
                                      _ptr(p.row_group), row0, nrows, _ptr(out))
        return out
    _load().orc_dequant_rows(_ptr(p.vals), _ptr(p.idx), _ptr(p.scale),
                             _ptr(p.zero), p.cols, p.n_keep, p.group, row0,
                             nrows, _ptr(out))
    return out


def matvec(p: Packed, x_f16: np.ndarray, rows=None) -> np.ndarray:
    """fp64 y (m x len(rows)) for binary16 x (m x cols)."""
    x = np.ascontiguousarray(x_f16)
    if x.dtype == np.float16:
        x = x.view(np.uint16)
    x = _c(x, np.uint16)
    if x.ndim == 1:
        x = x.reshape(1, -1)
    m = x.shape[0]
    if rows is None:
        rows = np.arange(p.rows, dtype=np.int64)
    rows = _c(rows, np.int64)
    y = np.zeros((rows.size, m), dtype=np.float64)
    if p.row_group is not None:
        _load().orc_matvec_rowg(_ptr(p.vals), _ptr(p.idx), _ptr(p.scale), _ptr(p.zero),
                                p.rows, p.cols, p.n_keep, _ptr(p.row_group), _ptr(x), m,
                                _ptr(rows), rows.size, _ptr(y))
        return np.ascontiguousarray(y.T)
    _load().orc_matvec(_ptr(p.vals), _ptr(p.idx), _ptr(p.scale), _ptr(p.zero),
                       p.cols, p.n_keep, p.group, _ptr(x), m, _ptr(rows),
                       rows.size, _ptr(y))
    return np.ascontiguousarray(y.T)


def pack_scored(W: np.ndarray, xnorm: np.ndarray, grad, n_keep: int,
                group: int) -> Packed:
    """Eq. 3 pruning, then the same quantisation and encoding as pack()."""
    W = _c(W, np.float32)
    rows, cols = W.shape
    xn = _c(xnorm, np.float32)
    g = None if grad is None else _c(grad, np.float32)
    vb, ib = row_bytes(cols, n_keep)
    ng = cols // group if group else 0
    vals = np.zeros((rows, vb), dtype=np.uint8)
    idx = np.zeros((rows, ib), dtype=np.uint8)
    scale = np.zeros((rows, ng), dtype=np.uint16)
    zero = np.zeros((rows, ng), dtype=np.uint16)
    rc = _load().orc_pack_scored(_ptr(W), _ptr(xn), None if g is None else _ptr(g),
                                 rows, cols, n_keep, group, _ptr(vals), _ptr(idx),
                                 _ptr(scale), _ptr(zero))
    if rc:
        raise OracleError(rc, "pack_scored")
    return Packed(rows, cols, n_keep, group, vals, idx, scale, zero)


def pack_rowg(W: np.ndarray, n_keep: int, row_group) -> Packed:
    """Magnitude pruning and quantisation with a group size per row."""
    W = _c(W, np.float32)
    rows, cols = W.shape
    rg = _c(row_group, np.int32)
    if rg.shape != (rows,):
        raise ValueError("one group size per row")
    vb, ib = row_bytes(cols, n_keep)
    ng = int(sum(cols // int(g) for g in rg)) if rows else 0
    vals = np.zeros((rows, vb), dtype=np.uint8)
    idx = np.zeros((rows, ib), dtype=np.uint8)
    scale = np.zeros(ng, dtype=np.uint16)
    zero = np.zeros(ng, dtype=np.uint16)
    rc = _load().orc_pack_rowg(_ptr(W), rows, cols, n_keep, _ptr(rg), _ptr(vals),
                               _ptr(idx), _ptr(scale), _ptr(zero))
    if rc:
        raise OracleError(rc, "pack_rowg")
    return Packed(rows, cols, n_keep, None, vals, idx, scale, zero, row_group=rg)


def quantize_rowg(W: np.ndarray, pos: np.ndarray, n_keep: int, row_group):
    W = _c(W, np.float32)
    pos = _c(pos, np.uint8)
    rows, cols = W.shape
    rg = _c(row_group, np.int32)
    P = cols // 4 * n_keep
    ng = int(sum(cols // int(g) for g in rg)) if rows else 0
    q = np.zeros((rows, P), dtype=np.uint8)
    scale = np.zeros(ng, dtype=np.uint16)
    zero = np.zeros(ng, dtype=np.uint16)
    rc = _load().orc_quantize_rowg(_ptr(W), _ptr(pos), rows, cols, n_keep, _ptr(rg),
                                   _ptr(q), _ptr(scale), _ptr(zero))
    if rc:
        raise OracleError(rc, "quantize_rowg")
    return q, scale, zero
