"""Plain CPU oracle for the SNACK truly-sparse linear layer.

TEST INFRASTRUCTURE ONLY.  The product library never imports, links or runs
anything in this package; only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` do.  The arithmetic lives in
``snack_oracle.c`` (plain C, fp64 accumulation) and is written from the paper
"Beyond Masked Sparsity: SNACK Enables Truly Sparse Neural Networks on GPU":

* ``canonicalize``        Appendix B, Table 7 (COO / CSR / CSC)
* ``forward``             §3.1 Algorithm 1
* ``backward_input``      §3.4, Appendix F (W^T by swapping index arrays)
* ``backward_weight``     §3.4, Appendix F (sparse outer product, mini-batch)
* ``weight_gradient64``   the same gradient left in float64
* ``sgd_update``          §3.4 / §4.1 SGD on the stored entries (textbook rule)
* ``adam_update``         Appendix G Adam on the stored entries (Kingma & Ba)
* ``uniform_init``        §3.3 Algorithm 2 (getrand = counter SplitMix64)
* ``prune_regrow``        Appendix G (magnitude prune, Algorithm 2 regrow)

``snack_oracle_omp.c`` holds an all-cores copy of the three product loops
(``forward_omp``, ``backward_input_omp``, ``backward_weight_omp``) for the
benchmark's CPU baseline: the same terms summed in the same order per output
element, split over threads by whole rows / columns / entries, so its
results are bit-identical to the single-threaded routines.

Every function is pinned by ``tests/test_oracle_pins.py`` against something
other than itself (Table 7, dense matmul, scipy.sparse, closed forms,
published generator outputs, brute force on tiny inputs).

This module is a thin ctypes loader: arrays are passed as contiguous numpy
buffers and results come back as numpy arrays.
"""

from __future__ import annotations

import ctypes
import os
import platform
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "snack_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liboracle.so")
_lock = threading.Lock()
_lib = None

OK, ERR_RANGE, ERR_DUPLICATE, ERR_ALLOC, ERR_ARG = 0, 1, 2, 3, 4


def build(force: bool = False) -> str:
    """Compile snack_oracle.c into oracle/_build/liboracle.so (plain gcc)."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    stamp = os.path.join(_BUILD_DIR, "machine.txt")
    try:
        with open(stamp) as f:
            same_machine = f.read().strip() == platform.machine()
    except OSError:
        same_machine = False
    if (not force and same_machine and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared",
                           "-fno-fast-math", "-ffp-contract=off",
                           _SRC, "-o", tmp, "-lm"])
    os.replace(tmp, _LIB_PATH)
    with open(stamp, "w") as f:
        f.write(platform.machine())
    return _LIB_PATH


_OMP_SRC = os.path.join(_HERE, "snack_oracle_omp.c")
_OMP_LIB_PATH = os.path.join(_BUILD_DIR, "liboracle_omp.so")
_omp_lib = None


def build_omp(force: bool = False) -> str:
    """Compile snack_oracle_omp.c (gcc -fopenmp) into oracle/_build/."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    stamp = os.path.join(_BUILD_DIR, "machine_omp.txt")
    try:
        with open(stamp) as f:
            same_machine = f.read().strip() == platform.machine()
    except OSError:
        same_machine = False
    if (not force and same_machine and os.path.exists(_OMP_LIB_PATH)
            and os.path.getmtime(_OMP_LIB_PATH) >= os.path.getmtime(_OMP_SRC)):
        return _OMP_LIB_PATH
    tmp = _OMP_LIB_PATH + f".tmp{os.getpid()}"
    subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp",
                           "-fno-fast-math", "-ffp-contract=off",
                           _OMP_SRC, "-o", tmp, "-lm"])
    os.replace(tmp, _OMP_LIB_PATH)
    with open(stamp, "w") as f:
        f.write(platform.machine())
    return _OMP_LIB_PATH


def _load_omp():
    global _omp_lib
    with _lock:
        if _omp_lib is not None:
            return _omp_lib
        lib = ctypes.CDLL(build_omp())
        i64, p, ci = ctypes.c_int64, ctypes.c_void_p, ctypes.c_int
        lib.oracle_omp_threads.restype = ci
        lib.oracle_omp_forward.argtypes = [i64, i64, p, p, p, i64, p, p, p, ci]
        lib.oracle_omp_backward_input.argtypes = [i64, i64, p, p, p, p, i64, p, p, p, ci]
        lib.oracle_omp_backward_weight.argtypes = [i64, i64, i64, p, p, i64, p, p, p, p, ci]
        for fn in (lib.oracle_omp_forward, lib.oracle_omp_backward_input,
                   lib.oracle_omp_backward_weight):
            fn.restype = ci
        _omp_lib = lib
        return lib


def host_cores() -> int:
    """CPU cores this process may run on (its affinity mask)."""
    try:
        return len(os.sched_getaffinity(0))
    except (AttributeError, OSError):
        return os.cpu_count() or 1


def forward_omp(out: int, inp: int, ref: dict, X, threads: int | None = None):
    """Y = X W^T on all cores; ``ref`` is a canonicalize() result.  Returns (Y, S),
    bit-identical to forward() on ref's canonical arrays."""
    lib = _load_omp()
    X = _c(X, np.float32)
    B = X.shape[0]
    assert X.shape == (B, inp)
    Y = np.empty((B, out), np.float32)
    S = np.empty((B, out), np.float64)
    lib.oracle_omp_forward(out, inp, _ptr(_c(ref["row_ptr"], np.int32)),
                           _ptr(_c(ref["col"], np.int32)), _ptr(_c(ref["val"], np.float32)), B,
                           _ptr(X), _ptr(Y), _ptr(S), threads or host_cores())
    return Y, S


def backward_input_omp(out: int, inp: int, ref: dict, dY, threads: int | None = None):
    """dX = dY W on all cores (column-partitioned).  Returns (dX, S)."""
    lib = _load_omp()
    dY = _c(dY, np.float32)
    B = dY.shape[0]
    assert dY.shape == (B, out)
    dX = np.empty((B, inp), np.float32)
    S = np.empty((B, inp), np.float64)
    lib.oracle_omp_backward_input(out, inp, _ptr(_c(ref["col_ptr"], np.int32)),
                                  _ptr(_c(ref["csc_perm"], np.int32)),
                                  _ptr(_c(ref["row"], np.int32)), _ptr(_c(ref["val"], np.float32)),
                                  B, _ptr(dY), _ptr(dX), _ptr(S), threads or host_cores())
    return dX, S


def backward_weight_omp(out: int, inp: int, ref: dict, X, dY, threads: int | None = None):
    """dW at the stored entries on all cores.  Returns (dW, S)."""
    lib = _load_omp()
    X, dY = _c(X, np.float32), _c(dY, np.float32)
    B = X.shape[0]
    assert X.shape == (B, inp) and dY.shape == (B, out)
    n = ref["row"].size
    dW = np.empty(n, np.float32)
    S = np.empty(n, np.float64)
    lib.oracle_omp_backward_weight(out, inp, n, _ptr(_c(ref["row"], np.int32)),
                                   _ptr(_c(ref["col"], np.int32)), B, _ptr(X), _ptr(dY),
                                   _ptr(dW), _ptr(S), threads or host_cores())
    return dW, S


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        i64, u64, p = ctypes.c_int64, ctypes.c_uint64, ctypes.c_void_p
        lib.oracle_canonicalize.argtypes = [i64, i64, i64, p, p, p, p, p, p, p,
                                            p, p, p, p, p]
        lib.oracle_canonicalize.restype = ctypes.c_int
        for name in ("oracle_forward", "oracle_backward_input"):
            fn = getattr(lib, name)
            fn.argtypes = [i64, i64, i64, p, p, p, i64, p, p, p]
            fn.restype = ctypes.c_int
        lib.oracle_backward_weight.argtypes = [i64, i64, i64, p, p, i64, p, p, p, p]
        lib.oracle_weight_gradient64.argtypes = [i64, i64, i64, p, p, i64, p, p, p, p]
        lib.oracle_weight_gradient64.restype = ctypes.c_int
        d = ctypes.c_double
        lib.oracle_sgd_update.argtypes = [i64, p, p, p, d, d, d, p, p]
        lib.oracle_sgd_update.restype = ctypes.c_int
        lib.oracle_adam_update.argtypes = [i64, p, p, p, p, d, d, d, d, d, i64, p, p, p]
        lib.oracle_adam_update.restype = ctypes.c_int
        lib.oracle_backward_weight.restype = ctypes.c_int
        lib.oracle_splitmix64.argtypes = [u64, u64]
        lib.oracle_splitmix64.restype = u64
        lib.oracle_cell_index.argtypes = [u64, u64]
        lib.oracle_cell_index.restype = u64
        lib.oracle_uniform_init.argtypes = [i64, i64, i64, u64, p, p, p]
        lib.oracle_uniform_init.restype = ctypes.c_int
        lib.oracle_prune_count.argtypes = [ctypes.c_float, i64]
        lib.oracle_prune_count.restype = i64
        lib.oracle_prune_regrow.argtypes = [i64, i64, i64, p, p, p, ctypes.c_float,
                                            u64, p, p, p, p, p]
        lib.oracle_prune_regrow.restype = ctypes.c_int
        _lib = lib
        return lib


def _ptr(a: np.ndarray | None):
    return None if a is None else ctypes.c_void_p(a.ctypes.data)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


class OracleError(RuntimeError):
    def __init__(self, code: int, bad: int = -1):
        names = {ERR_RANGE: "index out of range", ERR_DUPLICATE: "duplicate (row, col)",
                 ERR_ALLOC: "allocation failed", ERR_ARG: "invalid argument"}
        super().__init__(f"oracle: {names.get(code, code)} (entry {bad})")
        self.code = code
        self.bad = bad


def canonicalize(out: int, inp: int, row, col, val=None) -> dict:
    """Canonical COO + CSR + CSC of a user COO triple (Table 7 construction)."""
    lib = _load()
    row = _c(row, np.int32)
    col = _c(col, np.int32)
    nnz = row.size
    val = None if val is None else _c(val, np.float32)
    res = dict(row=np.empty(nnz, np.int32), col=np.empty(nnz, np.int32),
               val=np.empty(nnz, np.float32), src=np.empty(nnz, np.int64),
               row_ptr=np.empty(out + 1, np.int32), col_ptr=np.empty(inp + 1, np.int32),
               csc_row=np.empty(nnz, np.int32), csc_perm=np.empty(nnz, np.int32))
    bad = ctypes.c_int64(-1)
    rc = lib.oracle_canonicalize(out, inp, nnz, _ptr(row), _ptr(col), _ptr(val),
                                 _ptr(res["row"]), _ptr(res["col"]), _ptr(res["val"]),
                                 _ptr(res["src"]), _ptr(res["row_ptr"]),
                                 _ptr(res["col_ptr"]), _ptr(res["csc_row"]),
                                 _ptr(res["csc_perm"]), ctypes.byref(bad))
    if rc != OK:
        raise OracleError(rc, bad.value)
    return res


def forward(out: int, inp: int, row, col, val, X):
    """Y = X W^T (Algorithm 1).  Returns (Y fp32 [B][out], S fp64 [B][out])."""
    lib = _load()
    row, col, val = _c(row, np.int32), _c(col, np.int32), _c(val, np.float32)
    X = _c(X, np.float32)
    B = X.shape[0]
    assert X.shape == (B, inp)
    Y = np.empty((B, out), np.float32)
    S = np.empty((B, out), np.float64)
    rc = lib.oracle_forward(out, inp, row.size, _ptr(row), _ptr(col), _ptr(val), B,
                            _ptr(X), _ptr(Y), _ptr(S))
    if rc != OK:
        raise OracleError(rc)
    return Y, S


def backward_input(out: int, inp: int, row, col, val, dY):
    """dX = dY W (W^T by swapped index arrays).  Returns (dX [B][in], S)."""
    lib = _load()
    row, col, val = _c(row, np.int32), _c(col, np.int32), _c(val, np.float32)
    dY = _c(dY, np.float32)
    B = dY.shape[0]
    assert dY.shape == (B, out)
    dX = np.empty((B, inp), np.float32)
    S = np.empty((B, inp), np.float64)
    rc = lib.oracle_backward_input(out, inp, row.size, _ptr(row), _ptr(col), _ptr(val),
                                   B, _ptr(dY), _ptr(dX), _ptr(S))
    if rc != OK:
        raise OracleError(rc)
    return dX, S


def backward_weight(out: int, inp: int, row, col, X, dY):
    """dW[k] = sum_b dY[b,row_k] X[b,col_k] at stored entries.  Returns (dW, S)."""
    lib = _load()
    row, col = _c(row, np.int32), _c(col, np.int32)
    X, dY = _c(X, np.float32), _c(dY, np.float32)
    B = X.shape[0]
    assert X.shape == (B, inp) and dY.shape == (B, out)
    dW = np.empty(row.size, np.float32)
    S = np.empty(row.size, np.float64)
    rc = lib.oracle_backward_weight(out, inp, row.size, _ptr(row), _ptr(col), B,
                                    _ptr(X), _ptr(dY), _ptr(dW), _ptr(S))
    if rc != OK:
        raise OracleError(rc)
    return dW, S


def weight_gradient64(out: int, inp: int, row, col, X, dY):
    """The weight gradient at stored entries in float64 (not rounded).
    Returns (g, S)."""
    lib = _load()
    row, col = _c(row, np.int32), _c(col, np.int32)
    X, dY = _c(X, np.float32), _c(dY, np.float32)
    B = X.shape[0]
    assert X.shape == (B, inp) and dY.shape == (B, out)
    g = np.empty(row.size, np.float64)
    S = np.empty(row.size, np.float64)
    rc = lib.oracle_weight_gradient64(out, inp, row.size, _ptr(row), _ptr(col), B,
                                      _ptr(X), _ptr(dY), _ptr(g), _ptr(S))
    if rc != OK:
        raise OracleError(rc)
    return g, S


def sgd_update(val, g, buf, lr: float, momentum: float = 0.0, weight_decay: float = 0.0):
    """One SGD step on stored values (float32 val / buf in, float64 out).
    Returns (val_new, buf_new); buf may be None when momentum == 0."""
    lib = _load()
    val = _c(val, np.float32)
    g = _c(g, np.float64)
    n = val.size
    out = np.empty(n, np.float64)
    if momentum != 0.0:
        buf = _c(buf, np.float32)
        bout = np.empty(n, np.float64)
        bp, bo = _ptr(buf), _ptr(bout)
    else:
        bout, bp, bo = None, None, None
    rc = lib.oracle_sgd_update(n, _ptr(val), _ptr(g), bp, lr, momentum, weight_decay,
                               _ptr(out), bo)
    if rc != OK:
        raise OracleError(rc)
    return out, bout


def adam_update(val, g, m, v, lr: float, beta1: float, beta2: float, eps: float,
                weight_decay: float, step: int):
    """One Adam step on stored values (float32 val / m / v in, float64 out).
    Returns (val_new, m_new, v_new)."""
    lib = _load()
    val = _c(val, np.float32)
    g = _c(g, np.float64)
    m, v = _c(m, np.float32), _c(v, np.float32)
    n = val.size
    out, mo, vo = (np.empty(n, np.float64) for _ in range(3))
    rc = lib.oracle_adam_update(n, _ptr(val), _ptr(g), _ptr(m), _ptr(v), lr, beta1, beta2, eps,
                                weight_decay, step, _ptr(out), _ptr(mo), _ptr(vo))
    if rc != OK:
        raise OracleError(rc)
    return out, mo, vo


def splitmix64(seed: int, t: int) -> int:
    """Draw t of the counter-based SplitMix64 stream started at `seed`."""
    return int(_load().oracle_splitmix64(seed & (2**64 - 1), t & (2**64 - 1)))


def cell_index(x: int, n: int) -> int:
    """floor(x * n / 2^64)."""
    return int(_load().oracle_cell_index(x & (2**64 - 1), n))


def uniform_init(out: int, inp: int, count: int, seed: int):
    """Algorithm 2: `count` distinct cells.  Returns (row, col, trials)."""
    lib = _load()
    row = np.empty(count, np.int32)
    col = np.empty(count, np.int32)
    trials = ctypes.c_int64(0)
    rc = lib.oracle_uniform_init(out, inp, count, seed & (2**64 - 1), _ptr(row),
                                 _ptr(col), ctypes.byref(trials))
    if rc != OK:
        raise OracleError(rc)
    return row, col, int(trials.value)


def prune_count(frac: float, nnz: int) -> int:
    return int(_load().oracle_prune_count(ctypes.c_float(frac), nnz))


def prune_regrow(out: int, inp: int, row, col, val, frac: float, seed: int):
    """One magnitude-prune / uniform-regrow step on a canonical layer.

    Returns dict(row, col, val, pruned, trials) in canonical order."""
    lib = _load()
    row, col, val = _c(row, np.int32), _c(col, np.int32), _c(val, np.float32)
    nnz = row.size
    n_row = np.empty(nnz, np.int32)
    n_col = np.empty(nnz, np.int32)
    n_val = np.empty(nnz, np.float32)
    pruned = ctypes.c_int64(0)
    trials = ctypes.c_int64(0)
    rc = lib.oracle_prune_regrow(out, inp, nnz, _ptr(row), _ptr(col), _ptr(val),
                                 ctypes.c_float(frac), seed & (2**64 - 1), _ptr(n_row),
                                 _ptr(n_col), _ptr(n_val), ctypes.byref(pruned),
                                 ctypes.byref(trials))
    if rc != OK:
        raise OracleError(rc)
    return dict(row=n_row, col=n_col, val=n_val, pruned=int(pruned.value),
                trials=int(trials.value))
