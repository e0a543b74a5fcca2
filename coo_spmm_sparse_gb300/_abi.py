"""ctypes declarations of the C ABI in include/snack.h.

The library is the in-tree coo_spmm_sparse_gb300/_build/libsnack.so.  There
is no fallback: if it is missing, or cannot be loaded, importing the binding
fails with an error that says how to build it.
"""

from __future__ import annotations

import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_build", "libsnack.so")

i32, i64, u64, f32 = ctypes.c_int32, ctypes.c_int64, ctypes.c_uint64, ctypes.c_float
vp, sz = ctypes.c_void_p, ctypes.c_size_t
P = ctypes.POINTER

# name -> (restype, argtypes), mirroring include/snack.h
SIGNATURES = {
    "snack_create": (ctypes.c_int, [i64, i64, i64, vp, vp, vp, ctypes.c_int, vp, P(vp)]),
    "snack_create_random": (ctypes.c_int, [i64, i64, i64, u64, vp, P(vp), P(i64)]),
    "snack_forward": (ctypes.c_int, [vp, vp, vp, i64, vp]),
    "snack_backward_input": (ctypes.c_int, [vp, vp, vp, i64, vp]),
    "snack_backward_weight": (ctypes.c_int, [vp, vp, vp, vp, i64, vp]),
    "snack_backward": (ctypes.c_int, [vp, vp, vp, vp, vp, i64, vp]),
    "snack_sgd_step": (ctypes.c_int, [vp, vp, vp, i64, f32, f32, f32, vp]),
    "snack_adam_step": (ctypes.c_int, [vp, vp, vp, i64, f32, f32, f32, f32, f32, i64, vp]),
    "snack_optimizer_state": (ctypes.c_int, [vp, ctypes.c_int, P(vp)]),
    "snack_prune_regrow": (ctypes.c_int, [vp, f32, u64, vp, P(i64), P(i64)]),
    "snack_values": (ctypes.c_int, [vp, P(vp)]),
    "snack_values_changed": (ctypes.c_int, [vp, vp]),
    "snack_export": (ctypes.c_int, [vp, vp, vp, vp, ctypes.c_int, vp]),
    "snack_export_segments": (ctypes.c_int, [vp, vp, vp, vp, vp, vp]),
    "snack_plan": (ctypes.c_int, [vp, ctypes.c_int, i64, P(i32), P(i32), P(i64), P(i32)]),
    "snack_forward_csr_static": (ctypes.c_int, [i64, i64, i64, vp, vp, vp, vp, vp, i64, vp]),
    "snack_launch_count": (u64, []),
    "snack_debug_fail_alloc": (None, [i64]),
    "snack_device_error": (ctypes.c_int, [vp, P(ctypes.c_int), vp]),
    "snack_selftest_wait": (ctypes.c_int, [vp, P(ctypes.c_int)]),
    "snack_nnz": (i64, [vp]),
    "snack_out_features": (i64, [vp]),
    "snack_in_features": (i64, [vp]),
    "snack_device_bytes": (sz, [vp]),
    "snack_last_error": (ctypes.c_char_p, [vp]),
    "snack_status_string": (ctypes.c_char_p, [ctypes.c_int]),
    "snack_destroy": (None, [vp]),
}

STATUS = {0: "SNACK_OK", 1: "SNACK_ERR_INVALID_ARG", 2: "SNACK_ERR_OUT_OF_RANGE",
          3: "SNACK_ERR_DUPLICATE", 4: "SNACK_ERR_ALLOC", 5: "SNACK_ERR_CUDA",
          6: "SNACK_ERR_UNSUPPORTED", 7: "SNACK_ERR_TIMEOUT"}

_lib = None


def load(path: str = LIB_PATH):
    """Load libsnack.so and declare every entry point (no fallback)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise ImportError(
            f"libsnack.so not found at {path}; build it with "
            "`python -c 'import __graft_entry__ as g; g.build()'` or "
            "`python coo_spmm_sparse_gb300/build.py` (needs nvcc)")
    lib = ctypes.CDLL(path)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib
