"""CPU-only checks of the C ABI boundary: the library builds, loads, exports
every entry point declared in include/snack.h, and is independent of the
oracle.  No compute call is made (there may be no GPU)."""

import importlib.util
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "snack.h")
PKG = os.path.join(ROOT, "coo_spmm_sparse_gb300")


def _builder():
    spec = importlib.util.spec_from_file_location("_snack_build_t",
                                                  os.path.join(PKG, "build.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


@pytest.fixture(scope="module")
def libpath():
    return _builder().build()


def declared_symbols():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(snack_[a-z_]+)\s*\(", text)))


def test_header_declares_the_five_operations():
    names = declared_symbols()
    for need in ("snack_create", "snack_forward", "snack_backward_input",
                 "snack_backward_weight", "snack_prune_regrow"):
        assert need in names


def test_library_exports_every_declared_symbol(libpath):
    out = subprocess.run(["nm", "-D", "--defined-only", libpath], capture_output=True,
                         text=True, check=True).stdout
    exported = set(re.findall(r"\bT (snack_[a-z_]+)\b", out))
    missing = [n for n in declared_symbols() if n not in exported]
    assert not missing, f"declared but not exported: {missing}"


def test_binding_declares_every_symbol_and_loads(libpath):
    import ctypes
    from coo_spmm_sparse_gb300 import _abi
    assert sorted(_abi.SIGNATURES) == declared_symbols()
    lib = ctypes.CDLL(libpath)
    for n in declared_symbols():
        assert hasattr(lib, n)
    # pure host calls that need no device
    lib.snack_status_string.restype = ctypes.c_char_p
    assert lib.snack_status_string(0) == b"ok"
    lib.snack_nnz.restype = ctypes.c_int64
    lib.snack_nnz.argtypes = [ctypes.c_void_p]
    assert lib.snack_nnz(None) == -1


def test_library_does_not_contain_or_load_the_oracle(libpath):
    out = subprocess.run(["nm", "-D", libpath], capture_output=True, text=True).stdout
    assert "oracle_" not in out
    deps = subprocess.run(["ldd", libpath], capture_output=True, text=True).stdout
    assert "oracle" not in deps
    for dirpath, _, files in os.walk(PKG):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h")):
                src = open(os.path.join(dirpath, f)).read()
                assert "import oracle" not in src and "from oracle" not in src, f


def test_missing_library_fails_loudly(tmp_path):
    from coo_spmm_sparse_gb300 import _abi
    saved = _abi._lib
    try:
        _abi._lib = None
        with pytest.raises(ImportError):
            _abi.load(str(tmp_path / "nope.so"))
    finally:
        _abi._lib = saved
