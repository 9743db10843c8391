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
    # cache heads: h_q must split into equal groups; a query tile takes whole
    # groups of 64/g tokens or a 64-head slice, so g divides 64 or 64 divides g
    assert lib.mla_metadata_size(1, 16, 1, 3, ctypes.byref(mb), ctypes.byref(sb)) == _lib.MLA_ERR_INVALID_ARGUMENT
    assert lib.mla_metadata_size(1, 96, 1, 2, ctypes.byref(mb), ctypes.byref(sb)) == _lib.MLA_ERR_UNSUPPORTED
    assert lib.mla_metadata_size(1, 16, 1, 0, ctypes.byref(mb), ctypes.byref(sb)) == _lib.MLA_ERR_INVALID_ARGUMENT
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
    # a valid cache-head split passes the host checks
    assert lib.mla_metadata_size(4, 16, 2, 2, ctypes.byref(mb), ctypes.byref(sb)) == _lib.MLA_ERR_NO_DEVICE
    assert lib.mla_metadata_size(4, 256, 1, 2, ctypes.byref(mb), ctypes.byref(sb)) == _lib.MLA_ERR_NO_DEVICE


def test_sparse_host_side_argument_checks(lib):
    E = _lib
    mb, sb = ctypes.c_size_t(), ctypes.c_size_t()
    assert lib.mla_metadata_size_sparse(0, 16, 1, 1, ctypes.byref(mb), ctypes.byref(sb)) == E.MLA_ERR_INVALID_ARGUMENT
    assert lib.mla_metadata_size_sparse(1, 16, 1, 2, ctypes.byref(mb), ctypes.byref(sb)) == E.MLA_ERR_UNSUPPORTED
    # batch * s_q is the scheduler's request count: at most 16384
    assert lib.mla_metadata_size_sparse(16384, 16, 2, 1, ctypes.byref(mb), ctypes.byref(sb)) == E.MLA_ERR_UNSUPPORTED
    assert lib.mla_get_metadata_sparse(-1, 1, 16, 1, 1, None, None, None) == E.MLA_ERR_INVALID_ARGUMENT
    assert lib.mla_get_metadata_sparse(64, 1, 16, 1, 1, None, None, None) == E.MLA_ERR_INVALID_ARGUMENT
    ws = ctypes.c_size_t()
    assert lib.mla_workspace_size_sparse(1, 16, 1, 1, None) == E.MLA_ERR_INVALID_ARGUMENT

    # Fake, never dereferenced, 256-byte aligned addresses: every check below
    # happens on the host before the device is queried.
    P = 1 << 20
    D, DV = 576, 512

    def call(**kw):
        a = dict(q=P, qsb=16 * D, kc=P, kps=64 * D, kts=D, pages=4, page=64, idx=P, topk=64,
                 b=1, s_q=1, h_q=16, h_kv=1, scale=1.0, meta=P, ns=P, ws=P, wsb=1 << 30, out=P,
                 osb=16 * DV, oss=16 * DV, osh=DV, lse=P)
        a.update(kw)
        return lib.mla_decode_sparse_fwd(a["q"], a["qsb"], a["kc"], a["kps"], a["kts"], a["pages"],
                                         a["page"], a["idx"], a["topk"], a["b"], a["s_q"], a["h_q"],
                                         a["h_kv"], a["scale"], a["meta"], a["ns"], a["ws"],
                                         a["wsb"], a["out"], a["osb"], a["oss"], a["osh"],
                                         a["lse"], None)

    assert call(page=32) == E.MLA_ERR_UNSUPPORTED
    assert call(idx=None) == E.MLA_ERR_INVALID_ARGUMENT
    assert call(topk=-1) == E.MLA_ERR_INVALID_ARGUMENT
    assert call(kps=65 * D) == E.MLA_ERR_UNSUPPORTED          # pages not packed
    assert call(b=2, s_q=2, qsb=2 * 16 * D + 8, oss=16 * DV, osb=2 * 16 * DV) == E.MLA_ERR_UNSUPPORTED
    assert call(idx=P + 2) == E.MLA_ERR_BAD_ALIGNMENT
    assert call(q=P + 8) == E.MLA_ERR_BAD_ALIGNMENT
    assert call(scale=float("nan")) == E.MLA_ERR_INVALID_ARGUMENT
    import torch

    if not torch.cuda.is_available():
        assert call() == E.MLA_ERR_NO_DEVICE


def _noalloc_args(**override):
    """CPU tensors shaped like a valid no-allocation call (b=2, s_q=1, h_q=16)."""
    import torch

    b, s_q, h_q = 2, 1, 16
    a = dict(
        q=torch.zeros(b, s_q, h_q, 576, dtype=torch.bfloat16),
        k_cache=torch.zeros(4, 64, 1, 576, dtype=torch.bfloat16),
        block_table=torch.zeros(b, 2, dtype=torch.int32),
        cache_seqlens=torch.full((b,), 64, dtype=torch.int32),
        softmax_scale=576 ** -0.5, causal=False,
        meta=torch.zeros(8 + 8 * 256, dtype=torch.int32),
        num_splits=torch.zeros(b + 1, dtype=torch.int32),
        out=torch.zeros(b, s_q, h_q, 512, dtype=torch.bfloat16),
        lse=torch.zeros(b, h_q, s_q, dtype=torch.float32))
    a.update(override)
    return a


@pytest.mark.parametrize("bad", [
    dict(block_table="int64"), dict(cache_seqlens="int64"), dict(out="float32"),
    dict(out="short"), dict(lse="transposed")])
def test_noalloc_wrapper_rejects_wrong_dtypes_and_shapes(bad):
    """The Python wrapper checks what the C ABI cannot see (dtypes and shapes)
    before it passes raw pointers: an int64 block table would otherwise be read
    as pairs of int32 words, an undersized out written past its end."""
    import torch

    from decode_attention_paged_gb300 import api

    a = _noalloc_args()
    key, kind = next(iter(bad.items()))
    if kind == "int64":
        a[key] = a[key].to(torch.int64)
    elif kind == "float32":
        a[key] = a[key].float()
    elif kind == "short":
        a[key] = a[key][:, :, :, :256]
    elif kind == "transposed":
        a[key] = torch.zeros(2, 1, 16, dtype=torch.float32)
    with pytest.raises(AssertionError):
        api.mla_decode_fwd_noalloc(**a)


def test_decode_wrappers_refuse_metadata_below_the_floor():
    """A decode CTA may read its part record before it has checked the plan
    header, which is in bounds because every metadata buffer holds room for
    256 records.  The Python wrappers refuse a smaller buffer before any
    device call."""
    import torch

    from decode_attention_paged_gb300 import api

    small = torch.zeros(8 + 8 * 152, dtype=torch.int32)
    a = _noalloc_args(meta=small)
    with pytest.raises(AssertionError):
        api.mla_decode_fwd_noalloc(**a)
    with pytest.raises(AssertionError):
        api.DecodeCall(a["q"], a["k_cache"], a["block_table"], a["cache_seqlens"],
                       a["softmax_scale"], False, small, a["num_splits"])
    with pytest.raises(AssertionError):
        api.mla_decode_fwd_dims(a["q"], a["k_cache"], a["block_table"], a["cache_seqlens"],
                                a["softmax_scale"], False, small, a["num_splits"], 512)
    idx = torch.zeros(2, 1, 64, dtype=torch.int32)
    with pytest.raises(AssertionError):
        api.SparseDecodeCall(a["q"], a["k_cache"], idx, a["softmax_scale"], small,
                             a["num_splits"])
    assert api.META_MIN_INTS == 8 + 8 * 256
