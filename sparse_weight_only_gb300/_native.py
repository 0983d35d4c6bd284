"""ctypes binding of libsgemv (include/sgemv.h).

Argument marshalling only: every step of pack and run executes in the CUDA
kernels of the shared library.  PyTorch supplies device memory and streams.
There is no CPU fallback: if the library is not built, loading fails.
"""
from __future__ import annotations

import ctypes
import os
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libsgemv.so")

SGEMV_OK = 0
SGEMV_ERR_ARG = -1
SGEMV_ERR_UNSUPPORTED = -2
SGEMV_ERR_CUDA = -3
SGEMV_ERR_STATE = -4
SGEMV_ERR_TIMEOUT = -5
SGEMV_ERR_NONFINITE = -6
SGEMV_ERR_RANGE = -7
SGEMV_MAX_M = 64

# Every symbol include/sgemv.h declares, with (restype, argtypes).
_P = ctypes.c_void_p
_I = ctypes.c_int
_SZ = ctypes.c_size_t
_PSZ = ctypes.POINTER(ctypes.c_size_t)
SIGNATURES = {
    "sgemv_create": (_I, [ctypes.POINTER(_P), _I, _I, _I, _I, _I, _I]),
    "sgemv_create_rowgroups": (_I, [ctypes.POINTER(_P), _I, _I, _I, _P, _I, _I]),
    "sgemv_pack": (_I, [_P, _P]),
    "sgemv_pack_device": (_I, [_P, _P, _P]),
    "sgemv_pack_scored": (_I, [_P, _P, _P, _P]),
    "sgemv_import": (_I, [_P, _P, _P, _P, _P]),
    "sgemv_export": (_I, [_P, _P, _P, _P, _P]),
    "sgemv_run": (_I, [_P, _P, _P, _I, _P]),
    "sgemv_run_host": (_I, [_P, _P, _P, _I, _P]),
    "sgemv_run_group": (_I, [_P, _I, _P, _P, _I, _P]),
    "sgemv_run_group_host": (_I, [_P, _I, _P, _P, _I, _P]),
    "sgemv_run_noalloc": (_I, [_P, _P, _P, _I, _P]),
    "sgemv_status": (_I, [_P]),
    "sgemv_debug_withhold": (_I, [_P, _I]),
    "sgemv_sizes": (_I, [_P, _PSZ, _PSZ, _PSZ, _PSZ]),
    "sgemv_packed_bytes": (_SZ, [_P]),
    "sgemv_last_error": (ctypes.c_char_p, []),
    "sgemv_destroy": (_I, [_P]),
}

_lock = threading.Lock()
_lib = None


def load(path: str | None = None):
    """Load the in-tree libsgemv.so (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        p = path or LIB_PATH
        if not os.path.exists(p):
            raise RuntimeError(
                f"{p} is missing: the CUDA extension is not built "
                "(run `python -c 'import __graft_entry__ as g; g.build()'`)")
        lib = ctypes.CDLL(p)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
        return lib


class SgemvError(RuntimeError):
    def __init__(self, code: int, what: str, msg: str):
        super().__init__(f"{what} failed ({code}): {msg}")
        self.code = code


def _check(rc: int, what: str) -> None:
    if rc != SGEMV_OK:
        msg = load().sgemv_last_error().decode(errors="replace")
        raise SgemvError(rc, what, msg)


def _stream_ptr(stream) -> int | None:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


class SparseGemv:
    """A packed N:4 2bit-CSR INT4 weight on one GPU.

    rows x cols is out features x in features; n_keep is N (1 or 2); group
    is the quantisation group in dense columns (64, 128 or 256).  With
    row_group (one size per row) group is None and each row has its own.
    """

    def __init__(self, rows: int, cols: int, n_keep: int, group, max_m: int = 1,
                 device: int = 0, row_group=None):
        lib = load()
        h = ctypes.c_void_p()
        self.row_group = None
        if row_group is not None:
            rg = np.ascontiguousarray(row_group, dtype=np.int32)
            if rg.shape != (rows,):
                raise ValueError(f"row_group shape {rg.shape} != {(rows,)}")
            _check(lib.sgemv_create_rowgroups(ctypes.byref(h), rows, cols, n_keep,
                                              rg.ctypes.data, max_m, device),
                   "sgemv_create_rowgroups")
            self.row_group = rg
            group = None
        else:
            _check(lib.sgemv_create(ctypes.byref(h), rows, cols, n_keep, group,
                                    max_m, device), "sgemv_create")
        self._h = h
        self.rows, self.cols, self.n_keep, self.group = rows, cols, n_keep, group
        self.max_m, self.device = max_m, device

    # -- lifetime ---------------------------------------------------------
    def close(self) -> None:
        if getattr(self, "_h", None) is not None and self._h.value:
            load().sgemv_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()

    @property
    def handle(self) -> int:
        return self._h.value

    # -- format -----------------------------------------------------------
    def sizes(self) -> dict:
        v, i, g, d = (ctypes.c_size_t() for _ in range(4))
        _check(load().sgemv_sizes(self._h, ctypes.byref(v), ctypes.byref(i),
                                  ctypes.byref(g), ctypes.byref(d)),
               "sgemv_sizes")
        return {"vals": v.value, "idx": i.value, "groups": g.value,
                "device": d.value}

    def packed_bytes(self) -> int:
        return int(load().sgemv_packed_bytes(self._h))

    def pack(self, w: np.ndarray) -> None:
        w = np.ascontiguousarray(w, dtype=np.float32)
        if w.shape != (self.rows, self.cols):
            raise ValueError(f"weight shape {w.shape} != {(self.rows, self.cols)}")
        _check(load().sgemv_pack(self._h, w.ctypes.data), "sgemv_pack")

    def pack_scored(self, w: np.ndarray, xnorm: np.ndarray, grad=None) -> None:
        """Eq. 3 importance pruning: |w| * xnorm[col] + |w| * |grad| per
        weight (grad None: zero gradient), then the usual quantisation."""
        w = np.ascontiguousarray(w, dtype=np.float32)
        if w.shape != (self.rows, self.cols):
            raise ValueError(f"weight shape {w.shape} != {(self.rows, self.cols)}")
        xn = np.ascontiguousarray(xnorm, dtype=np.float32)
        if xn.shape != (self.cols,):
            raise ValueError(f"xnorm shape {xn.shape} != {(self.cols,)}")
        g = None
        if grad is not None:
            g = np.ascontiguousarray(grad, dtype=np.float32)
            if g.shape != w.shape:
                raise ValueError(f"grad shape {g.shape} != {w.shape}")
        _check(load().sgemv_pack_scored(self._h, w.ctypes.data, xn.ctypes.data,
                                        None if g is None else g.ctypes.data),
               "sgemv_pack_scored")

    def pack_device(self, w, stream=None) -> None:
        """w: a torch float32 CUDA tensor of shape (rows, cols)."""
        if tuple(w.shape) != (self.rows, self.cols) or not w.is_contiguous():
            raise ValueError("w must be a contiguous (rows, cols) tensor")
        _check(load().sgemv_pack_device(self._h, w.data_ptr(),
                                        _stream_ptr(stream)),
               "sgemv_pack_device")

    def import_canonical(self, vals, idx, scale, zero) -> None:
        s = self.sizes()
        arrs = []
        for a, dt, n in ((vals, np.uint8, s["vals"]), (idx, np.uint8, s["idx"]),
                         (scale, np.uint16, s["groups"]),
                         (zero, np.uint16, s["groups"])):
            a = np.ascontiguousarray(a, dtype=dt)
            if a.size != n:
                raise ValueError(f"canonical array of {a.size} elements, want {n}")
            arrs.append(a)
        _check(load().sgemv_import(self._h, *(a.ctypes.data for a in arrs)),
               "sgemv_import")

    def export_canonical(self):
        s = self.sizes()
        vb = s["vals"] // max(self.rows, 1) if self.rows else 0
        ib = s["idx"] // max(self.rows, 1) if self.rows else 0
        vals = np.zeros((self.rows, vb), np.uint8)
        idx = np.zeros((self.rows, ib), np.uint8)
        if self.row_group is None:
            ng = self.cols // self.group
            scale = np.zeros((self.rows, ng), np.uint16)
            zero = np.zeros((self.rows, ng), np.uint16)
        else:   # flat: each row's entries after those of the rows before it
            scale = np.zeros(s["groups"], np.uint16)
            zero = np.zeros(s["groups"], np.uint16)
        _check(load().sgemv_export(self._h, vals.ctypes.data, idx.ctypes.data,
                                   scale.ctypes.data, zero.ctypes.data),
               "sgemv_export")
        return vals, idx, scale, zero

    # -- product ----------------------------------------------------------
    def run(self, x, y, stream=None) -> None:
        """y (m x rows, fp16, CUDA) = W_hat . x (m x cols, fp16, CUDA)."""
        m = x.shape[0] if x.dim() == 2 else 1
        _check(load().sgemv_run(self._h, x.data_ptr(), y.data_ptr(), m,
                                _stream_ptr(stream)), "sgemv_run")

    def run_noalloc(self, x, y, stream=None) -> None:
        """As run(), for 2 <= m <= min(64, max_m), with the split-K workspace
        in the library's fixed device array instead of the handle's: the call
        allocates nothing.  Calls of this kind must not overlap on the GPU."""
        m = x.shape[0] if x.dim() == 2 else 1
        _check(load().sgemv_run_noalloc(self._h, x.data_ptr(), y.data_ptr(), m,
                                        _stream_ptr(stream)), "sgemv_run_noalloc")

    def __call__(self, x, stream=None):
        import torch
        x2 = x if x.dim() == 2 else x.reshape(1, -1)
        y = torch.empty((x2.shape[0], self.rows), dtype=torch.float16,
                        device=x.device)
        self.run(x2, y, stream)
        return y if x.dim() == 2 else y.reshape(-1)

    def run_host(self, x: np.ndarray, y: np.ndarray, stream=None) -> None:
        """Host-buffer variant: x (m x cols) and y (m x rows) are float16
        numpy arrays (ideally page-locked).  Asynchronous on `stream`."""
        m = x.shape[0] if x.ndim == 2 else 1
        _check(load().sgemv_run_host(self._h, x.ctypes.data, y.ctypes.data, m,
                                     _stream_ptr(stream)), "sgemv_run_host")

    def status(self) -> int:
        return int(load().sgemv_status(self._h))

    def debug_withhold(self, runs: int) -> None:
        """Failure-detection test hook: the next `runs` batch products with
        2 <= m <= 8 or m >= 33 make their bounded wait run out (sgemv_status
        then reports SGEMV_ERR_TIMEOUT)."""
        _check(load().sgemv_debug_withhold(self._h, runs), "sgemv_debug_withhold")


def run_group(mats, x, ys, stream=None) -> None:
    """y_i = W_hat_i . x for matrices that share x (one launch per N at
    m = 1).  mats: SparseGemv list; x: (m, cols) fp16 CUDA tensor; ys: list
    of (m, rows_i) fp16 CUDA tensors."""
    n = len(mats)
    if len(ys) != n:
        raise ValueError("one output per matrix")
    hs = (ctypes.c_void_p * max(n, 1))(*[h.handle for h in mats])
    yp = (ctypes.c_void_p * max(n, 1))(*[y.data_ptr() for y in ys])
    m = x.shape[0] if x.dim() == 2 else 1
    _check(load().sgemv_run_group(hs, n, x.data_ptr(), yp, m, _stream_ptr(stream)),
           "sgemv_run_group")


def run_group_host(mats, x, ys, stream=None) -> None:
    """run_group with host buffers: x (m x cols) and each ys[i] (m x rows_i)
    are float16 numpy arrays or CPU tensors (ideally page-locked).
    Asynchronous on `stream`: synchronise it before reading ys."""
    n = len(mats)
    if len(ys) != n:
        raise ValueError("one output per matrix")

    def ptr(a):
        return a.data_ptr() if hasattr(a, "data_ptr") else a.ctypes.data
    hs = (ctypes.c_void_p * max(n, 1))(*[h.handle for h in mats])
    yp = (ctypes.c_void_p * max(n, 1))(*[ptr(y) for y in ys])
    m = x.shape[0] if len(x.shape) == 2 else 1
    _check(load().sgemv_run_group_host(hs, n, ptr(x), yp, m, _stream_ptr(stream)),
           "sgemv_run_group_host")
