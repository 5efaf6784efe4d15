"""Thin ctypes binding over libsnk: the C-ABI entry points under the same names.

Argument marshalling only: every step of the layer runs in the library's CUDA
kernels.  Tensors are passed by device pointer, streams by handle.  PyTorch
serves as the device-memory allocator and stream provider.  If the library
has not been built, loading fails loudly; there is no fallback.
"""
from __future__ import annotations

import ctypes
import os
import re
import threading

_PKG = os.path.dirname(os.path.abspath(__file__))
# the in-tree library that build.py writes; nothing selects another one
LIB_PATH = os.path.join(_PKG, "libsnk.so")
HEADER = os.path.join(os.path.dirname(_PKG), "include", "snk.h")

SNK_OK, SNK_ERR_ARG, SNK_ERR_DUP, SNK_ERR_RANGE = 0, 1, 2, 3
SNK_ERR_CUDA, SNK_ERR_OOM, SNK_ERR_NOSPACE, SNK_ERR_LIMIT = 4, 5, 6, 7

_lock = threading.Lock()
_lib = None


class SnkError(RuntimeError):
    def __init__(self, status: int, call: str):
        super().__init__(f"{call} failed: {snk_status_string(status)} (status {status})")
        self.status = status


def lib():
    """Load libsnk.so (built by ``sparse_linear_layer_gb300.build``)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"libsnk.so is not built ({LIB_PATH}); run "
                               "sparse_linear_layer_gb300.build.build() first")
        L = ctypes.CDLL(LIB_PATH)
        i64, u64, f32, P, I = (ctypes.c_int64, ctypes.c_uint64, ctypes.c_float,
                               ctypes.c_void_p, ctypes.c_int)
        L.snk_create.argtypes = [ctypes.POINTER(P), i64, i64, i64, P, P, P, P]
        L.snk_forward.argtypes = [P, P, i64, P, P, P]
        L.snk_backward_input.argtypes = [P, P, i64, P, P]
        L.snk_backward_weight.argtypes = [P, P, P, i64, P, P, P]
        L.snk_prune_regrow.argtypes = [P, f32, u64, P]
        L.snk_prune_regrow_gradient.argtypes = [P, f32, P, P, i64, P]
        L.snk_destroy.argtypes = [P]
        L.snk_status_string.argtypes = [I]
        L.snk_status_string.restype = ctypes.c_char_p
        L.snk_get_shape.argtypes = [P, ctypes.POINTER(i64), ctypes.POINTER(i64),
                                    ctypes.POINTER(i64), ctypes.POINTER(i64)]
        L.snk_copy_topology.argtypes = [P, P, P, P, P, P]
        L.snk_check.argtypes = [P, P]
        L.snk_forward_csr_noalloc.argtypes = [i64, i64, i64, P, P, P, P, i64, P, P, P]
        L.snk_pcsr_build.argtypes = [P, I, P]
        L.snk_pcsr_info.argtypes = [P, ctypes.POINTER(i64), ctypes.POINTER(i64),
                                    ctypes.POINTER(i64), P]
        L.snk_pcsr_copy.argtypes = [P, P, P, P, P, P, P]
        L.snk_pcsr_insert.argtypes = [P, i64, P, P, P, P]
        L.snk_pcsr_delete.argtypes = [P, i64, P, P, P]
        L.snk_pcsr_compact.argtypes = [P, P]
        L.snk_pcsr_export.argtypes = [P, P, P, P, i64, ctypes.POINTER(i64), P]
        for name in ("snk_create", "snk_forward", "snk_backward_input", "snk_backward_weight",
                     "snk_prune_regrow", "snk_prune_regrow_gradient", "snk_destroy",
                     "snk_get_shape", "snk_copy_topology", "snk_check", "snk_forward_csr_noalloc",
                     "snk_pcsr_build", "snk_pcsr_info", "snk_pcsr_copy", "snk_pcsr_insert",
                     "snk_pcsr_delete", "snk_pcsr_compact", "snk_pcsr_export"):
            getattr(L, name).restype = I
        _lib = L
        return L


def declared_symbols():
    """Function names declared in include/snk.h."""
    with open(HEADER) as f:
        text = f.read()
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\*?\s+\*?(snk_\w+)\s*\(", text, re.M)))


def _check(status: int, call: str):
    if status != SNK_OK:
        raise SnkError(status, call)


def _ptr(t):
    if t is None:
        return None
    if isinstance(t, int):
        return t
    if not t.is_contiguous():
        raise ValueError("tensor must be contiguous")
    return t.data_ptr()


def _stream(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def snk_status_string(status: int) -> str:
    return lib().snk_status_string(status).decode()


def snk_create(out_features: int, in_features: int, values, rows, cols, stream=None) -> int:
    """Bind a layer to (values, rows, cols); sorts them in place.  Returns the handle."""
    h = ctypes.c_void_p()
    nnz = values.numel() if hasattr(values, "numel") else int(values)
    _check(lib().snk_create(ctypes.byref(h), out_features, in_features, nnz, _ptr(values),
                            _ptr(rows), _ptr(cols), _stream(stream)), "snk_create")
    return h.value


def snk_forward(handle: int, X, bias, Y, stream=None, batch: int | None = None):
    b = X.shape[0] if batch is None else batch
    _check(lib().snk_forward(handle, _ptr(X), b, _ptr(bias), _ptr(Y), _stream(stream)),
           "snk_forward")


def snk_backward_input(handle: int, dY, dX, stream=None, batch: int | None = None):
    b = dY.shape[0] if batch is None else batch
    _check(lib().snk_backward_input(handle, _ptr(dY), b, _ptr(dX), _stream(stream)),
           "snk_backward_input")


def snk_backward_weight(handle: int, X, dY, dW, db=None, stream=None, batch: int | None = None):
    b = X.shape[0] if batch is None else batch
    _check(lib().snk_backward_weight(handle, _ptr(X), _ptr(dY), b, _ptr(dW), _ptr(db),
                                     _stream(stream)), "snk_backward_weight")


def snk_prune_regrow(handle: int, zeta: float, seed: int, stream=None):
    _check(lib().snk_prune_regrow(handle, float(zeta), seed & (2**64 - 1), _stream(stream)),
           "snk_prune_regrow")


def snk_prune_regrow_gradient(handle: int, zeta: float, X, dY, stream=None,
                              batch: int | None = None):
    b = X.shape[0] if batch is None else batch
    _check(lib().snk_prune_regrow_gradient(handle, float(zeta), _ptr(X), _ptr(dY), b,
                                           _stream(stream)), "snk_prune_regrow_gradient")


def snk_destroy(handle: int):
    _check(lib().snk_destroy(handle), "snk_destroy")


def snk_check(handle: int, stream=None):
    """Synchronise the stream and raise SnkError(SNK_ERR_LIMIT) if a
    tensor-core kernel of this handle stopped on a wait limit since the last
    check (its outputs were written as NaN)."""
    _check(lib().snk_check(handle, _stream(stream)), "snk_check")


def snk_get_shape(handle: int):
    o, i, n, v = (ctypes.c_int64() for _ in range(4))
    _check(lib().snk_get_shape(handle, ctypes.byref(o), ctypes.byref(i), ctypes.byref(n),
                               ctypes.byref(v)), "snk_get_shape")
    return o.value, i.value, n.value, v.value


def snk_copy_topology(handle: int, row_ptr=None, col_ptr=None, rows_c=None, perm=None,
                      stream=None):
    _check(lib().snk_copy_topology(handle, _ptr(row_ptr), _ptr(col_ptr), _ptr(rows_c),
                                   _ptr(perm), _stream(stream)), "snk_copy_topology")


def snk_forward_csr_noalloc(out_features: int, in_features: int, row_ptr, cols, values, X, bias,
                            Y, stream=None, batch: int | None = None):
    """Forward product on a caller's CSR without any device allocation (the
    library's fixed scratch array is used instead)."""
    b = X.shape[0] if batch is None else batch
    nnz = values.numel() if hasattr(values, "numel") else 0
    _check(lib().snk_forward_csr_noalloc(out_features, in_features, nnz, _ptr(row_ptr), _ptr(cols),
                                         _ptr(values), _ptr(X), b, _ptr(bias), _ptr(Y),
                                         _stream(stream)), "snk_forward_csr_noalloc")


def snk_pcsr_build(handle: int, padding_pct: int = 20, stream=None):
    _check(lib().snk_pcsr_build(handle, int(padding_pct), _stream(stream)), "snk_pcsr_build")


def snk_pcsr_info(handle: int, stream=None):
    """(used_slots, n_live, version)"""
    u, n, v = ctypes.c_int64(), ctypes.c_int64(), ctypes.c_int64()
    _check(lib().snk_pcsr_info(handle, ctypes.byref(u), ctypes.byref(n), ctypes.byref(v),
                               _stream(stream)), "snk_pcsr_info")
    return u.value, n.value, v.value


def snk_pcsr_copy(handle: int, slot_values=None, slot_cols=None, row_start=None, row_nnz=None,
                  row_capacity=None, stream=None):
    _check(lib().snk_pcsr_copy(handle, _ptr(slot_values), _ptr(slot_cols), _ptr(row_start),
                               _ptr(row_nnz), _ptr(row_capacity), _stream(stream)),
           "snk_pcsr_copy")


def snk_pcsr_insert(handle: int, rows, cols, values, stream=None):
    _check(lib().snk_pcsr_insert(handle, rows.numel(), _ptr(rows), _ptr(cols), _ptr(values),
                                 _stream(stream)), "snk_pcsr_insert")


def snk_pcsr_delete(handle: int, rows, cols, stream=None):
    _check(lib().snk_pcsr_delete(handle, rows.numel(), _ptr(rows), _ptr(cols), _stream(stream)),
           "snk_pcsr_delete")


def snk_pcsr_compact(handle: int, stream=None):
    _check(lib().snk_pcsr_compact(handle, _stream(stream)), "snk_pcsr_compact")


def snk_pcsr_export(handle: int, values, rows, cols, stream=None) -> int:
    """Canonical live triple into the given tensors; returns nnz."""
    n = ctypes.c_int64()
    _check(lib().snk_pcsr_export(handle, _ptr(values), _ptr(rows), _ptr(cols), values.numel(),
                                 ctypes.byref(n), _stream(stream)), "snk_pcsr_export")
    return n.value


class SparseLinear:
    """Convenience owner of one layer: keeps the caller-side tensors alive for
    the handle's lifetime and allocates outputs with torch."""

    def __init__(self, out_features: int, in_features: int, values, rows, cols, stream=None):
        self.out_features, self.in_features = out_features, in_features
        self.values, self.rows, self.cols = values, rows, cols
        self.handle = snk_create(out_features, in_features, values, rows, cols, stream)

    @property
    def nnz(self) -> int:
        return self.values.numel()

    @property
    def topology_version(self) -> int:
        return snk_get_shape(self.handle)[3]

    def forward(self, X, bias=None, out=None, stream=None):
        import torch
        Y = out if out is not None else torch.empty((X.shape[0], self.out_features),
                                                    dtype=torch.float32, device=X.device)
        snk_forward(self.handle, X, bias, Y, stream)
        return Y

    def backward_input(self, dY, out=None, stream=None):
        import torch
        dX = out if out is not None else torch.empty((dY.shape[0], self.in_features),
                                                     dtype=torch.float32, device=dY.device)
        snk_backward_input(self.handle, dY, dX, stream)
        return dX

    def backward_weight(self, X, dY, with_bias: bool = False, out=None, stream=None):
        import torch
        dW = out if out is not None else torch.empty_like(self.values)
        db = torch.empty(self.out_features, dtype=torch.float32, device=dY.device) if with_bias else None
        snk_backward_weight(self.handle, X, dY, dW, db, stream)
        return (dW, db) if with_bias else dW

    def prune_regrow(self, zeta: float, seed: int, stream=None):
        snk_prune_regrow(self.handle, zeta, seed, stream)

    def prune_regrow_gradient(self, zeta: float, X, dY, stream=None):
        snk_prune_regrow_gradient(self.handle, zeta, X, dY, stream)

    def pcsr(self):
        """The Padded-CSR view as host-readable torch tensors (slot arrays cut
        to the used slots)."""
        import torch
        dev = self.values.device
        used, live, version = snk_pcsr_info(self.handle)
        out = dict(slot_values=torch.empty(used, dtype=torch.float32, device=dev),
                   slot_cols=torch.empty(used, dtype=torch.int32, device=dev),
                   row_start=torch.empty(self.out_features, dtype=torch.int32, device=dev),
                   row_nnz=torch.empty(self.out_features, dtype=torch.int32, device=dev),
                   row_capacity=torch.empty(self.out_features, dtype=torch.int32, device=dev))
        snk_pcsr_copy(self.handle, out["slot_values"], out["slot_cols"], out["row_start"],
                      out["row_nnz"], out["row_capacity"])
        out["n_live"], out["version"] = live, version
        return out

    def topology(self):
        import torch
        dev = self.values.device
        out = dict(row_ptr=torch.empty(self.out_features + 1, dtype=torch.int32, device=dev),
                   col_ptr=torch.empty(self.in_features + 1, dtype=torch.int32, device=dev),
                   rows_c=torch.empty(self.nnz, dtype=torch.int32, device=dev),
                   perm=torch.empty(self.nnz, dtype=torch.int32, device=dev))
        snk_copy_topology(self.handle, out["row_ptr"], out["col_ptr"], out["rows_c"], out["perm"])
        return out

    def close(self):
        if getattr(self, "handle", None):
            snk_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
