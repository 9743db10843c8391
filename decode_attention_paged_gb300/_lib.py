"""ctypes loader for libmla.so (the C ABI in include/mla_decode.h).

There is no fallback: if the library is missing or fails to load, importing
the binding raises.  Build it with ``__graft_entry__.build()`` or
``python -m decode_attention_paged_gb300._build``.
"""
from __future__ import annotations

import ctypes
import os

HERE = os.path.dirname(os.path.abspath(__file__))
SO_PATH = os.path.join(HERE, "libmla.so")

# Status codes (mirror of include/mla_decode.h).
MLA_OK = 0
MLA_ERR_INVALID_ARGUMENT = -1
MLA_ERR_UNSUPPORTED = -2
MLA_ERR_WORKSPACE_TOO_SMALL = -3
MLA_ERR_CUDA = -4
MLA_ERR_DEVICE_TIMEOUT = -5
MLA_ERR_METADATA_MISMATCH = -6
MLA_ERR_NO_DEVICE = -7
MLA_ERR_SEQ_TOO_LONG = -8
MLA_ERR_BAD_ALIGNMENT = -9
MLA_ERR_BAD_INDEX = -10

# Every symbol include/mla_decode.h declares, with its ctypes signature.
_P = ctypes.c_void_p
_I = ctypes.c_int
_I64 = ctypes.c_int64
_SZ = ctypes.c_size_t
_F = ctypes.c_float
SIGNATURES = {
    "mla_strerror": (ctypes.c_char_p, [_I]),
    "mla_version": (_I, []),
    "mla_metadata_size": (_I, [_I, _I, _I, _I, ctypes.POINTER(_SZ), ctypes.POINTER(_SZ)]),
    "mla_get_metadata": (_I, [_P, _I, _I, _I, _I, _P, _P, _P]),
    "mla_workspace_size": (_I, [_I, _I, _I, _I, ctypes.POINTER(_SZ)]),
    "mla_decode_fwd": (_I, [_P, _I64, _P, _I64, _I64, _I, _I, _P, _I64, _I, _P, _I, _I, _I, _I, _F,
                            _I, _P, _P, _P, _SZ, _P, _I64, _I64, _I64, _P, _P]),
    "mla_decode_fwd_dims": (_I, [_P, _I64, _P, _I64, _I64, _I, _I, _P, _I64, _I, _P, _I, _I, _I,
                                 _I, _I, _I, _F, _I, _P, _P, _P, _SZ, _P, _I64, _I64, _I64, _P,
                                 _P]),
    "mla_decode_splitkv": (_I, [_P, _I64, _P, _I64, _I64, _I, _I, _P, _I64, _I, _P, _I, _I, _I, _I,
                                _F, _I, _P, _P, _P, _SZ, _P, _I64, _I64, _I64, _P, _P]),
    "mla_decode_combine": (_I, [_P, _P, _P, _SZ, _I, _I, _I, _I, _P, _I64, _I64, _I64, _P, _P]),
    "mla_decode_fwd_noalloc": (_I, [_P, _I64, _P, _I64, _I64, _I, _I, _P, _I64, _I, _P, _I, _I,
                                    _I, _I, _F, _I, _P, _P, _P, _I64, _I64, _I64, _P, _P]),
    "mla_decode_fp8_fwd": (_I, [_P, _I64, _P, _I64, _I, _I, _P, _I64, _I, _P, _I, _I, _I, _I, _F,
                                _I, _P, _P, _P, _SZ, _P, _I64, _I64, _I64, _P, _P]),
    "mla_metadata_size_sparse": (_I, [_I, _I, _I, _I, ctypes.POINTER(_SZ), ctypes.POINTER(_SZ)]),
    "mla_get_metadata_sparse": (_I, [_I, _I, _I, _I, _I, _P, _P, _P]),
    "mla_workspace_size_sparse": (_I, [_I, _I, _I, _I, ctypes.POINTER(_SZ)]),
    "mla_decode_sparse_fwd": (_I, [_P, _I64, _P, _I64, _I64, _I, _I, _P, _I, _I, _I, _I, _I, _F,
                                   _P, _P, _P, _SZ, _P, _I64, _I64, _I64, _P, _P]),
    "mla_last_device_error": (_I, [_P, ctypes.POINTER(_I)]),
    "mla_set_wait_budget_ns": (_I, [ctypes.c_uint64]),
    "mla_set_fixed_overhead": (_I, [_I]),
    "mla_set_decode_kernel": (_I, [_I]),
    "mla_get_decode_kernel": (_I, []),
}

_lib = None


def load() -> ctypes.CDLL:
    global _lib
    if _lib is None:
        if not os.path.exists(SO_PATH):
            raise ImportError(f"libmla.so not built ({SO_PATH}); run __graft_entry__.build()")
        lib = ctypes.CDLL(SO_PATH)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
    return _lib


class MLAError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        msg = load().mla_strerror(code).decode()
        super().__init__(f"{where}: {msg} (code {code})")


def check(code: int, where: str) -> None:
    if code != MLA_OK:
        raise MLAError(code, where)
