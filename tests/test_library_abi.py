"""CPU checks of the C-ABI library: it builds, loads without a GPU, exports
every symbol include/*.h declares, and rejects bad arguments on the host
before touching a device."""
import ctypes
import glob
import os
import re

import pytest

from decode_attention_paged_gb300 import _build, _lib

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    _build.build()
    return _lib.load()


def declared_symbols():
    names = []
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        txt = open(h).read()
        names += re.findall(r"MLA_API\s+[\w\s\*]*?\b(mla_\w+)\s*\(", txt)
    return sorted(set(names))


def test_header_declares_the_boundary():
    names = declared_symbols()
    for required in ("mla_get_metadata", "mla_decode_fwd", "mla_metadata_size",
                     "mla_workspace_size", "mla_strerror", "mla_last_device_error"):
        assert required in names


def test_every_declared_symbol_is_exported(lib):
    for name in declared_symbols():
        assert hasattr(lib, name), f"{name} declared in include/ but not exported"
        assert name in _lib.SIGNATURES, f"{name} missing from the Python binding"


def test_nothing_else_is_exported():
    import subprocess

    out = subprocess.run(["nm", "-D", "--defined-only", _lib.SO_PATH], capture_output=True,
                         text=True, check=True).stdout
    exported = sorted(l.split()[-1] for l in out.splitlines() if " T " in l)
    assert set(exported) <= set(declared_symbols()), exported


def test_strerror_and_version(lib):
    assert lib.mla_strerror(0) == b"ok"
    assert b"timed out" in lib.mla_strerror(_lib.MLA_ERR_DEVICE_TIMEOUT)
    assert lib.mla_strerror(12345) == b"unknown error"
    assert lib.mla_version() >= 100


def test_host_side_argument_checks(lib):
    mb, sb = ctypes.c_size_t(), ctypes.c_size_t()
    assert lib.mla_metadata_size(0, 16, 1, 1, ctypes.byref(mb), ctypes.byref(sb)) == _lib.MLA_ERR_INVALID_ARGUMENT
    assert lib.mla_metadata_size(1, 0, 1, 1, ctypes.byref(mb), ctypes.byref(sb)) == _lib.MLA_ERR_INVALID_ARGUMENT
    assert lib.mla_metadata_size(1, 16, 1, 2, ctypes.byref(mb), ctypes.byref(sb)) == _lib.MLA_ERR_UNSUPPORTED
    ws = ctypes.c_size_t()
    assert lib.mla_workspace_size(1, 16, 1, 1, None) == _lib.MLA_ERR_INVALID_ARGUMENT
    assert lib.mla_workspace_size(1, 16, 0, 1, ctypes.byref(ws)) == _lib.MLA_ERR_INVALID_ARGUMENT
    # page size other than 64 is refused before any device work
    st = lib.mla_decode_fwd(None, 0, None, 0, 0, 1, 32, None, 0, 1, None, 1, 1, 16, 1, 1.0, 0,
                            None, None, None, 0, None, 0, 0, 0, None, None)
    assert st == _lib.MLA_ERR_UNSUPPORTED
    st = lib.mla_decode_fwd(None, 0, None, 0, 0, 1, 64, None, 0, 1, None, 1, 1, 16, 1, 1.0, 0,
                            None, None, None, 0, None, 0, 0, 0, None, None)
    assert st == _lib.MLA_ERR_INVALID_ARGUMENT


def test_without_gpu_calls_report_no_device(lib):
    import torch

    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    mb, sb = ctypes.c_size_t(), ctypes.c_size_t()
    assert lib.mla_metadata_size(4, 16, 1, 1, ctypes.byref(mb), ctypes.byref(sb)) == _lib.MLA_ERR_NO_DEVICE
