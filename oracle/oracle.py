"""ctypes wrapper around ``snk_oracle.c`` (plain C, fp64 accumulation).

Test infrastructure only.  Nothing in the CUDA library imports this module.

Page titles cited below:
  [SNACK] "Beyond Masked Sparsity: SNACK Enables Truly Sparse Neural Networks on GPU"
  [PCSR]  "Padded-CSR: A sparse storage format for dynamic sparse training on CPU"
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

__all__ = [
    "OracleError", "build", "canonicalize", "forward", "backward_input",
    "backward_weight", "prune_count", "prune", "regrow", "prune_regrow",
    "grad_at", "grad_key", "grad_keys", "grow_gradient", "grad_count_below",
    "prune_regrow_gradient",
    "splitmix64_nth", "mulhi64", "candidate", "regrow_limit", "openmp_available", "threads",
    "ORC_OK", "ORC_ERR_ARG", "ORC_ERR_DUP", "ORC_ERR_RANGE", "ORC_ERR_OOM",
    "ORC_ERR_NOSPACE", "ORC_ERR_LIMIT",
]

ORC_OK, ORC_ERR_ARG, ORC_ERR_DUP, ORC_ERR_RANGE = 0, 1, 2, 3
ORC_ERR_OOM, ORC_ERR_NOSPACE, ORC_ERR_LIMIT = 5, 6, 7

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "snk_oracle.c")
_OUT_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_OUT_DIR, "libsnk_oracle.so")
# the same source built with OpenMP: the products split their outputs among
# the host's cores (same terms in the same order per output, same bits); used
# for the benchmark's all-core CPU baseline
_OMP_PATH = os.path.join(_OUT_DIR, "libsnk_oracle_omp.so")
_lock = threading.Lock()
_lib = None
_omp_lib = None


class OracleError(RuntimeError):
    def __init__(self, status: int, what: str):
        super().__init__(f"oracle {what}: status {status}")
        self.status = status


def _compile(path: str, extra, force: bool) -> str:
    os.makedirs(_OUT_DIR, exist_ok=True)
    stale = (not os.path.exists(path) or os.path.getmtime(path) < os.path.getmtime(_SRC))
    if force or stale:
        tmp = path + f".tmp{os.getpid()}"
        subprocess.run(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", *extra, "-o", tmp,
                        _SRC, "-lm"], check=True)
        os.replace(tmp, path)
    return path


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (portable C, no target-specific flags),
    single-threaded, and the same source with OpenMP when the compiler has
    it (the all-core CPU baseline; tests use the single-threaded build)."""
    path = _compile(_LIB_PATH, [], force)
    try:
        _compile(_OMP_PATH, ["-fopenmp"], force)
    except (subprocess.CalledProcessError, OSError):
        pass
    return path


def openmp_available() -> bool:
    build()
    return os.path.exists(_OMP_PATH)


def _load(omp: bool = False):
    global _lib, _omp_lib
    if omp and not openmp_available():
        raise OracleError(-1, "OpenMP build not available")
    with _lock:
        if (_omp_lib if omp else _lib) is not None:
            return _omp_lib if omp else _lib
        lib = ctypes.CDLL(_OMP_PATH if omp else build())
        i64, u64, f32 = ctypes.c_int64, ctypes.c_uint64, ctypes.c_float
        P = ctypes.c_void_p
        lib.orc_canonicalize.argtypes = [i64, i64, i64, P, P, P, P, P, P, P]
        lib.orc_canonicalize.restype = ctypes.c_int
        lib.orc_forward.argtypes = [i64, i64, i64, P, P, P, P, i64, P, P, P]
        lib.orc_forward.restype = None
        lib.orc_backward_input.argtypes = [i64, i64, i64, P, P, P, P, i64, P, P]
        lib.orc_backward_input.restype = None
        lib.orc_backward_weight.argtypes = [i64, i64, i64, P, P, P, P, i64, P, P, P, P]
        lib.orc_backward_weight.restype = None
        lib.orc_prune_count.argtypes = [f32, i64]
        lib.orc_prune_count.restype = i64
        lib.orc_prune.argtypes = [i64, i64, i64, P, P, P, f32, P, P]
        lib.orc_prune.restype = ctypes.c_int
        lib.orc_regrow.argtypes = [i64, i64, i64, P, P, i64, u64, P, P]
        lib.orc_regrow.restype = ctypes.c_int
        lib.orc_prune_regrow.argtypes = [i64, i64, i64, P, P, P, f32, u64]
        lib.orc_prune_regrow.restype = ctypes.c_int
        lib.orc_grad_at.argtypes = [i64, i64, P, P, i64, i64, i64]
        lib.orc_grad_at.restype = ctypes.c_float
        lib.orc_grad_key.argtypes = [ctypes.c_float, u64]
        lib.orc_grad_key.restype = u64
        lib.orc_grad_keys.argtypes = [i64, i64, P, P, i64, P, i64, P]
        lib.orc_grad_keys.restype = None
        lib.orc_grow_gradient.argtypes = [i64, i64, i64, P, P, P, P, i64, i64, P]
        lib.orc_grow_gradient.restype = ctypes.c_int
        lib.orc_grad_count_below.argtypes = [i64, i64, i64, P, P, P, P, i64, u64]
        lib.orc_grad_count_below.restype = i64
        lib.orc_prune_regrow_gradient.argtypes = [i64, i64, i64, P, P, P, f32, P, P, i64]
        lib.orc_prune_regrow_gradient.restype = ctypes.c_int
        lib.orc_splitmix64_nth.argtypes = [u64, u64]
        lib.orc_splitmix64_nth.restype = u64
        lib.orc_mulhi64.argtypes = [u64, u64]
        lib.orc_mulhi64.restype = u64
        lib.orc_candidate.argtypes = [u64, u64, u64]
        lib.orc_candidate.restype = u64
        lib.orc_threads.argtypes = []
        lib.orc_threads.restype = ctypes.c_int
        if omp:
            _omp_lib = lib
        else:
            _lib = lib
        return lib


def threads(omp: bool = False) -> int:
    """Threads the products of a build use (1 without OpenMP)."""
    return int(_load(omp).orc_threads())


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _f32(a):
    return np.ascontiguousarray(a, dtype=np.float32)


def _i32(a):
    return np.ascontiguousarray(a, dtype=np.int32)


def canonicalize(out_f: int, in_f: int, v, r, c):
    """Canonical (row, col) order plus CSR and CSC ([PCSR] sec. 3.2, 4.1, 7.2;
    [SNACK] Table 7).  Returns a dict of numpy arrays; inputs are not modified."""
    lib = _load()
    v, r, c = _f32(v).copy(), _i32(r).copy(), _i32(c).copy()
    nnz = v.shape[0]
    row_ptr = np.zeros(out_f + 1, np.int32)
    col_ptr = np.zeros(in_f + 1, np.int32)
    rows_c = np.zeros(max(nnz, 1), np.int32)[:nnz]
    perm = np.zeros(max(nnz, 1), np.int32)[:nnz]
    st = lib.orc_canonicalize(out_f, in_f, nnz, _ptr(v), _ptr(r), _ptr(c),
                              _ptr(row_ptr), _ptr(col_ptr), _ptr(rows_c), _ptr(perm))
    if st != ORC_OK:
        raise OracleError(st, "canonicalize")
    return dict(values=v, rows=r, cols=c, row_ptr=row_ptr, col_ptr=col_ptr,
                rows_c=rows_c, perm=perm)


def forward(out_f: int, in_f: int, v, r, c, X, bias=None, omp: bool = False):
    """Y = X (W.M)^T + bias in fp64, and the magnitude sum A ([PCSR] sec. 6.1).
    omp: run the OpenMP build (same bits)."""
    lib = _load(omp)
    v, r, c, X = _f32(v), _i32(r), _i32(c), _f32(X)
    b = X.shape[0]
    assert X.shape == (b, in_f)
    bias = None if bias is None else _f32(bias)
    Y = np.empty((b, out_f), np.float64)
    A = np.empty((b, out_f), np.float64)
    lib.orc_forward(out_f, in_f, v.shape[0], _ptr(v), _ptr(r), _ptr(c), _ptr(X), b,
                    _ptr(bias), _ptr(Y), _ptr(A))
    return Y, A


def backward_input(out_f: int, in_f: int, v, r, c, dY, omp: bool = False):
    """dX = dY (W.M) in fp64, and its magnitude sum ([PCSR] sec. 7.1)."""
    lib = _load(omp)
    v, r, c, dY = _f32(v), _i32(r), _i32(c), _f32(dY)
    b = dY.shape[0]
    assert dY.shape == (b, out_f)
    dX = np.empty((b, in_f), np.float64)
    A = np.empty((b, in_f), np.float64)
    lib.orc_backward_input(out_f, in_f, v.shape[0], _ptr(v), _ptr(r), _ptr(c), _ptr(dY),
                           b, _ptr(dX), _ptr(A))
    return dX, A


def backward_weight(out_f: int, in_f: int, r, c, X, dY, omp: bool = False):
    """dW on the support and db, each with its magnitude sum ([PCSR] sec. 7.1)."""
    lib = _load(omp)
    r, c, X, dY = _i32(r), _i32(c), _f32(X), _f32(dY)
    b = X.shape[0]
    assert X.shape == (b, in_f) and dY.shape == (b, out_f)
    nnz = r.shape[0]
    dW = np.empty(nnz, np.float64)
    A = np.empty(nnz, np.float64)
    db = np.empty(out_f, np.float64)
    Adb = np.empty(out_f, np.float64)
    lib.orc_backward_weight(out_f, in_f, nnz, _ptr(r), _ptr(c), _ptr(X), _ptr(dY), b,
                            _ptr(dW), _ptr(A), _ptr(db), _ptr(Adb))
    return dW, A, db, Adb


def prune_count(zeta: float, nnz: int) -> int:
    return int(_load().orc_prune_count(float(np.float32(zeta)), nnz))


def prune(out_f: int, in_f: int, v, r, c, zeta: float):
    """Boolean mask of the floor(zeta*nnz) entries with the smallest (|v|, lin)."""
    lib = _load()
    v, r, c = _f32(v), _i32(r), _i32(c)
    nnz = v.shape[0]
    removed = np.zeros(max(nnz, 1), np.uint8)[:nnz]
    k = ctypes.c_int64(0)
    st = lib.orc_prune(out_f, in_f, nnz, _ptr(v), _ptr(r), _ptr(c), float(np.float32(zeta)),
                       _ptr(removed), ctypes.byref(k))
    if st != ORC_OK:
        raise OracleError(st, "prune")
    return removed.astype(bool), int(k.value)


def regrow(out_f: int, in_f: int, r_kept, c_kept, k: int, seed: int):
    """The k positions drawn by the seeded sequential regrow, in draw order."""
    lib = _load()
    r_kept, c_kept = _i32(r_kept), _i32(c_kept)
    new_lin = np.zeros(max(k, 1), np.int64)[:k]
    draws = ctypes.c_int64(0)
    st = lib.orc_regrow(out_f, in_f, r_kept.shape[0], _ptr(r_kept), _ptr(c_kept), k,
                        ctypes.c_uint64(seed & (2**64 - 1)), _ptr(new_lin), ctypes.byref(draws))
    if st != ORC_OK:
        raise OracleError(st, "regrow")
    return new_lin, int(draws.value)


def prune_regrow(out_f: int, in_f: int, v, r, c, zeta: float, seed: int):
    """Prune + regrow + canonical re-emission; returns new (v, r, c)."""
    lib = _load()
    v, r, c = _f32(v).copy(), _i32(r).copy(), _i32(c).copy()
    st = lib.orc_prune_regrow(out_f, in_f, v.shape[0], _ptr(v), _ptr(r), _ptr(c),
                              float(np.float32(zeta)), ctypes.c_uint64(seed & (2**64 - 1)))
    if st != ORC_OK:
        raise OracleError(st, "prune_regrow")
    return v, r, c


def grad_at(out_f: int, in_f: int, X, dY, row: int, col: int) -> float:
    """The fp32 gradient of position (row, col) as the fmaf chain over the batch."""
    X, dY = _f32(X), _f32(dY)
    return float(_load().orc_grad_at(out_f, in_f, _ptr(X), _ptr(dY), X.shape[0], row, col))


def grad_key(g: float, lin: int) -> int:
    return int(_load().orc_grad_key(ctypes.c_float(g), ctypes.c_uint64(lin)))


def grad_keys(out_f: int, in_f: int, X, dY, lin) -> np.ndarray:
    """Ranking keys (complement of bits(|g|) << 32 | position) of positions."""
    X, dY = _f32(X), _f32(dY)
    lin = np.ascontiguousarray(lin, np.int64)
    keys = np.zeros(len(lin), np.uint64)
    _load().orc_grad_keys(out_f, in_f, _ptr(X), _ptr(dY), X.shape[0], _ptr(lin), len(lin),
                          _ptr(keys))
    return keys


def grow_gradient(out_f: int, in_f: int, r_kept, c_kept, X, dY, k: int):
    """The k candidate positions with the largest |gradient| (ties: smaller
    position), ascending."""
    lib = _load()
    r_kept, c_kept, X, dY = _i32(r_kept), _i32(c_kept), _f32(X), _f32(dY)
    new_lin = np.zeros(max(k, 1), np.int64)[:k]
    st = lib.orc_grow_gradient(out_f, in_f, r_kept.shape[0], _ptr(r_kept), _ptr(c_kept),
                               _ptr(X), _ptr(dY), X.shape[0], k, _ptr(new_lin))
    if st != ORC_OK:
        raise OracleError(st, "grow_gradient")
    return new_lin


def grad_count_below(out_f: int, in_f: int, r_kept, c_kept, X, dY, theta: int) -> int:
    lib = _load()
    r_kept, c_kept, X, dY = _i32(r_kept), _i32(c_kept), _f32(X), _f32(dY)
    n = lib.orc_grad_count_below(out_f, in_f, r_kept.shape[0], _ptr(r_kept), _ptr(c_kept),
                                 _ptr(X), _ptr(dY), X.shape[0], ctypes.c_uint64(theta))
    if n < 0:
        raise OracleError(ORC_ERR_OOM, "grad_count_below")
    return int(n)


def prune_regrow_gradient(out_f: int, in_f: int, v, r, c, zeta: float, X, dY):
    """Prune + gradient grow + canonical re-emission; returns new (v, r, c)."""
    lib = _load()
    v, r, c = _f32(v).copy(), _i32(r).copy(), _i32(c).copy()
    X, dY = _f32(X), _f32(dY)
    st = lib.orc_prune_regrow_gradient(out_f, in_f, v.shape[0], _ptr(v), _ptr(r), _ptr(c),
                                       ctypes.c_float(zeta), _ptr(X), _ptr(dY), X.shape[0])
    if st != ORC_OK:
        raise OracleError(st, "prune_regrow_gradient")
    return v, r, c


def splitmix64_nth(state: int, n: int) -> int:
    return int(_load().orc_splitmix64_nth(ctypes.c_uint64(state & (2**64 - 1)), n))


def mulhi64(a: int, b: int) -> int:
    return int(_load().orc_mulhi64(ctypes.c_uint64(a), ctypes.c_uint64(b)))


def candidate(seed: int, t: int, n_positions: int) -> int:
    return int(_load().orc_candidate(ctypes.c_uint64(seed & (2**64 - 1)), t, n_positions))


def regrow_limit(k: int) -> int:
    """Number of draws after which the regrow gives up (64 k + 1024)."""
    return 64 * k + 1024
