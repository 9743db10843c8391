"""fp64 CPU oracle for paged MLA decode -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product (the CUDA library and its
Python binding) never imports, links or calls it, and shares no code with it.

The C sources (``mla_oracle.c``, ``sparse_oracle.c``, ``plan_oracle.c``, ``fp8_oracle.c``) hold the arithmetic and
cite the pages they follow; this module only compiles them with gcc and
marshals numpy arrays through ctypes.

Inputs are raw bf16 bit patterns (``uint16`` arrays); the C code widens them to
fp64 exactly.  Outputs are fp64.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SO = os.path.join(_HERE, "liboracle.so")
_SRCS = [os.path.join(_HERE, "mla_oracle.c"), os.path.join(_HERE, "sparse_oracle.c"),
         os.path.join(_HERE, "plan_oracle.c"), os.path.join(_HERE, "fp8_oracle.c")]
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle into ``oracle/liboracle.so`` (plain C, fp64, no FMA
    contraction so x86 and Arm give the same bits)."""
    newest = max(os.path.getmtime(s) for s in _SRCS)
    if not force and os.path.exists(_SO) and os.path.getmtime(_SO) >= newest:
        return _SO
    tmp = _SO + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared",
           "-pthread", "-o", tmp] + _SRCS + ["-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _SO)
    return _SO


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_SO)
            P = ctypes.c_void_p
            I = ctypes.c_int
            D = ctypes.c_double
            I64 = ctypes.c_int64
            lib.oracle_mla_decode.argtypes = [P, P, P, P, I, I, I, I, I, I, I, I, D, I, P, P, I]
            lib.oracle_mla_decode.restype = I
            lib.oracle_mla_decode_rows.argtypes = [P, P, P, P, I, I, I, I, I, I, I, I, D, I, P,
                                                   I64, P, P, I]
            lib.oracle_mla_decode_rows.restype = I
            lib.oracle_mla_partial.argtypes = [P, P, P, P, I, I, I, I, I, I, I, I, D, I, I, I, I,
                                               I, P, P]
            lib.oracle_mla_partial.restype = I
            lib.oracle_merge_pair.argtypes = [P, P, P, D, D, P, I]
            lib.oracle_merge_pair.restype = None
            lib.oracle_lse_combine.argtypes = [I, P, P, I, P, P]
            lib.oracle_lse_combine.restype = None
            lib.oracle_mla_sparse.argtypes = [P, P, P, I, I, I, I, I, I, I64, D, P, P, I]
            lib.oracle_mla_sparse.restype = I
            lib.oracle_mla_sparse_rows.argtypes = [P, P, P, I, I, I, I, I, I, I64, D, P, I64, P,
                                                   P, I]
            lib.oracle_mla_sparse_rows.restype = I
            lib.oracle_plan.argtypes = [P, I, I, I, I, P, P]
            lib.oracle_plan.restype = I
            lib.oracle_e4m3_value.argtypes = [ctypes.c_uint8]
            lib.oracle_e4m3_value.restype = D
            lib.oracle_bf16_round.argtypes = [D]
            lib.oracle_bf16_round.restype = ctypes.c_uint16
            lib.oracle_fp8_dequant.argtypes = [P, I64, I64, P]
            lib.oracle_fp8_dequant.restype = I
            _lib = lib
    return _lib


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def bf16_bits(t) -> np.ndarray:
    """uint16 bit patterns of a torch bf16 tensor (CPU), C-contiguous."""
    import torch

    assert t.dtype == torch.bfloat16
    return np.ascontiguousarray(t.detach().cpu().contiguous().view(torch.int16).numpy()).view(np.uint16)


class Problem:
    """One decode problem in the oracle's layout.

    q      : uint16 [b, s_q, h_q, d]        (bf16 bits)
    kv     : uint16 [num_pages, page, d]    (bf16 bits, the single KV head)
    block_table : int32 [b, max_blocks]
    seqlens     : int32 [b]
    """

    def __init__(self, q, kv, block_table, seqlens, scale, causal):
        self.q = np.ascontiguousarray(q, dtype=np.uint16)
        kv = np.asarray(kv, dtype=np.uint16)
        if kv.ndim == 4:  # [pages, page, h_kv=1, d]
            assert kv.shape[2] == 1
            kv = kv.reshape(kv.shape[0], kv.shape[1], kv.shape[3])
        self.kv = np.ascontiguousarray(kv)
        self.block_table = np.ascontiguousarray(block_table, dtype=np.int32)
        self.seqlens = np.ascontiguousarray(seqlens, dtype=np.int32)
        self.b, self.s_q, self.h_q, self.d = self.q.shape
        self.num_pages, self.page, d2 = self.kv.shape
        assert d2 == self.d
        self.max_blocks = self.block_table.shape[1] if self.block_table.ndim == 2 else 0
        self.scale = float(scale)
        self.causal = int(bool(causal))

    def _args(self, dv):
        return (_ptr(self.q), _ptr(self.kv), _ptr(self.block_table), _ptr(self.seqlens), self.b,
                self.s_q, self.h_q, self.d, dv, self.page, self.max_blocks, self.num_pages,
                self.scale, self.causal)


def mla_decode(p: Problem, dv: int = 512, nthreads: int = 1):
    """Full decode: returns (out [b, s_q, h_q, dv] fp64, lse [b, h_q, s_q] fp64)."""
    lib = _load()
    out = np.zeros((p.b, p.s_q, p.h_q, dv), dtype=np.float64)
    lse = np.zeros((p.b, p.h_q, p.s_q), dtype=np.float64)
    st = lib.oracle_mla_decode(*p._args(dv), _ptr(out), _ptr(lse), int(nthreads))
    if st != 0:
        raise RuntimeError(f"oracle_mla_decode failed: {st}")
    return out, lse


def mla_decode_rows(p: Problem, units, dv: int = 512, nthreads: int = 1):
    """Selected rows only.  units: int array [n, 2] of (request, row = s*h_q + h).
    Returns (out [n, dv], lse [n]) in fp64."""
    lib = _load()
    units = np.ascontiguousarray(np.asarray(units, dtype=np.int32).reshape(-1, 2))
    n = units.shape[0]
    out = np.zeros((n, dv), dtype=np.float64)
    lse = np.zeros((n,), dtype=np.float64)
    st = lib.oracle_mla_decode_rows(*p._args(dv), _ptr(units), n, _ptr(out), _ptr(lse),
                                    int(nthreads))
    if st != 0:
        raise RuntimeError(f"oracle_mla_decode_rows failed: {st}")
    return out, lse


def mla_partial(p: Problem, i: int, rho: int, t_begin: int, t_end: int, dv: int = 512):
    """Partial (normalised o[dv], lse) of row rho of request i over keys [t_begin, t_end)."""
    lib = _load()
    o = np.zeros((dv,), dtype=np.float64)
    lse = np.zeros((1,), dtype=np.float64)
    st = lib.oracle_mla_partial(*p._args(dv), int(i), int(rho), int(t_begin), int(t_end), _ptr(o),
                                _ptr(lse))
    if st != 0:
        raise RuntimeError(f"oracle_mla_partial failed: {st}")
    return o, float(lse[0])


def merge_pair(state1, state2):
    """Two-way merge of unnormalised states (m, l, o~).  Returns a new state."""
    lib = _load()
    m1, l1, o1 = state1
    m2, l2, o2 = state2
    m = np.array([m1], dtype=np.float64)
    l = np.array([l1], dtype=np.float64)
    o = np.array(o1, dtype=np.float64, copy=True)
    o2 = np.ascontiguousarray(o2, dtype=np.float64)
    lib.oracle_merge_pair(_ptr(m), _ptr(l), _ptr(o), float(m2), float(l2), _ptr(o2), o.shape[0])
    return float(m[0]), float(l[0]), o


def lse_combine(lse_parts, o_parts):
    """n-way combine of normalised partials.  lse_parts [n], o_parts [n, dv]."""
    lib = _load()
    lse_parts = np.ascontiguousarray(lse_parts, dtype=np.float64).reshape(-1)
    o_parts = np.ascontiguousarray(o_parts, dtype=np.float64).reshape(lse_parts.shape[0], -1)
    dv = o_parts.shape[1]
    o = np.zeros((dv,), dtype=np.float64)
    lse = np.zeros((1,), dtype=np.float64)
    lib.oracle_lse_combine(lse_parts.shape[0], _ptr(lse_parts), _ptr(o_parts), dv, _ptr(o),
                           _ptr(lse))
    return o, float(lse[0])


PLAN_FIELDS = ("begin_req", "end_req", "begin_block", "end_block", "begin_split_idx",
               "is_first_req_splitted", "is_last_req_splitted", "pad")


def plan(seqlens, num_parts: int, fixed_overhead: int, page: int = 64):
    """Tile-scheduler plan: returns (parts int32 [num_parts, 8], num_splits int32 [b+1])."""
    lib = _load()
    seqlens = np.ascontiguousarray(seqlens, dtype=np.int32).reshape(-1)
    b = seqlens.shape[0]
    parts = np.zeros((num_parts, 8), dtype=np.int32)
    ns = np.zeros((b + 1,), dtype=np.int32)
    st = lib.oracle_plan(_ptr(seqlens), b, int(page), int(num_parts), int(fixed_overhead),
                         _ptr(parts), _ptr(ns))
    if st != 0:
        raise RuntimeError(f"oracle_plan failed: {st}")
    return parts, ns


class SparseProblem:
    """One sparse decode problem in the oracle's layout.

    q       : uint16 [b, s_q, h_q, d]           (bf16 bits)
    kv      : uint16 [num_pages, page, d] or [num_pages, page, 1, d]
    indices : int32 [b, s_q, topk]  physical token = page_id * page + offset,
              < 0 for padding
    """

    def __init__(self, q, kv, indices, scale):
        self.q = np.ascontiguousarray(q, dtype=np.uint16)
        kv = np.asarray(kv, dtype=np.uint16)
        if kv.ndim == 4:
            assert kv.shape[2] == 1
            kv = kv.reshape(kv.shape[0], kv.shape[1], kv.shape[3])
        self.kv = np.ascontiguousarray(kv)
        self.indices = np.ascontiguousarray(indices, dtype=np.int32)
        self.b, self.s_q, self.h_q, self.d = self.q.shape
        assert self.indices.shape[:2] == (self.b, self.s_q)
        self.topk = self.indices.shape[2]
        self.num_tokens = self.kv.shape[0] * self.kv.shape[1]
        self.scale = float(scale)

    def _args(self, dv):
        return (_ptr(self.q), _ptr(self.kv), _ptr(self.indices), self.b, self.s_q, self.h_q,
                self.topk, self.d, dv, self.num_tokens, self.scale)


def mla_sparse(p: SparseProblem, dv: int = 512, nthreads: int = 1, allow_bad_index=False):
    """Sparse decode: (out [b, s_q, h_q, dv], lse [b, h_q, s_q]) in fp64."""
    lib = _load()
    out = np.zeros((p.b, p.s_q, p.h_q, dv), dtype=np.float64)
    lse = np.zeros((p.b, p.h_q, p.s_q), dtype=np.float64)
    st = lib.oracle_mla_sparse(*p._args(dv), _ptr(out), _ptr(lse), int(nthreads))
    if st != 0 and not (st == -5 and allow_bad_index):
        raise RuntimeError(f"oracle_mla_sparse failed: {st}")
    return out, lse


def mla_sparse_rows(p: SparseProblem, units, dv: int = 512, nthreads: int = 1):
    """Selected rows (request, row = s*h_q + h) of a sparse decode, fp64."""
    lib = _load()
    units = np.ascontiguousarray(np.asarray(units, dtype=np.int32).reshape(-1, 2))
    n = units.shape[0]
    out = np.zeros((n, dv), dtype=np.float64)
    lse = np.zeros((n,), dtype=np.float64)
    st = lib.oracle_mla_sparse_rows(*p._args(dv), _ptr(units), n, _ptr(out), _ptr(lse),
                                    int(nthreads))
    if st != 0:
        raise RuntimeError(f"oracle_mla_sparse_rows failed: {st}")
    return out, lse


# ------------------------------------------------------------ FP8 KV cache
FP8_ROW_BYTES = 656  # 512 e4m3 + 4 fp32 scales + 64 bf16 ("[DeepSeek-3] FlashMLA", sec. 12)


def e4m3_value(code: int) -> float:
    """Value of one float8_e4m3 code (fp8_oracle.c)."""
    return float(_load().oracle_e4m3_value(int(code)))


def bf16_round(x: float) -> int:
    """bf16 bit pattern of x rounded to nearest even (fp8_oracle.c)."""
    return int(_load().oracle_bf16_round(float(x)))


def fp8_dequant(cache_bytes) -> np.ndarray:
    """FP8 cache [pages, 64, 1, 656] uint8 (numpy or torch) -> bf16 bit patterns
    [pages, 64, 1, 576] of the dequantised rows."""
    a = cache_bytes.cpu().numpy() if hasattr(cache_bytes, "cpu") else np.asarray(cache_bytes)
    a = np.ascontiguousarray(a, dtype=np.uint8)
    assert a.shape[-1] == FP8_ROW_BYTES
    n = a.size // FP8_ROW_BYTES
    out = np.empty(a.shape[:-1] + (576,), dtype=np.uint16)
    st = _load().oracle_fp8_dequant(_ptr(a), n, FP8_ROW_BYTES, _ptr(out))
    if st != 0:
        raise RuntimeError(f"oracle_fp8_dequant failed: {st}")
    return out


def mla_decode_fp8(q_bits, cache_bytes, block_table, cache_seqlens, scale, causal,
                   dv: int = 512, nthreads: int = 1):
    """Dense decode over an FP8 cache: the dense oracle on the dequantised rows."""
    p = Problem(q_bits, fp8_dequant(cache_bytes), block_table, cache_seqlens, scale, causal)
    return mla_decode(p, dv, nthreads)


# ------------------------------------------------------------ h_kv > 1
def mla_decode_gqa(q_bits, kv_bits, block_table, cache_seqlens, scale, causal, dv: int = 512,
                   nthreads: int = 1):
    """Decode with h_kv cache heads ("[DeepSeek-3] FlashMLA", sec. 4: k_cache is
    [blocks, 64, h_kv, 576]; the dense tests cover MQA and GQA).  Reading: the
    h_q query heads form h_kv groups of g = h_q / h_kv consecutive heads, and
    group j attends to cache head j only -- so each group is one dense decode
    (mla_oracle.c) over that head's rows.
    q_bits [b, s_q, h_q, 576], kv_bits [pages, 64, h_kv, 576] (bf16 bits).
    Returns out [b, s_q, h_q, dv], lse [b, h_q, s_q] in fp64."""
    q_bits = np.asarray(q_bits, dtype=np.uint16)
    kv_bits = np.asarray(kv_bits, dtype=np.uint16)
    b, s_q, h_q, d = q_bits.shape
    h_kv = kv_bits.shape[2]
    assert h_q % h_kv == 0
    g = h_q // h_kv
    out = np.zeros((b, s_q, h_q, dv), dtype=np.float64)
    lse = np.zeros((b, h_q, s_q), dtype=np.float64)
    for j in range(h_kv):
        p = Problem(q_bits[:, :, j * g:(j + 1) * g, :], kv_bits[:, :, j, :], block_table,
                    cache_seqlens, scale, causal)
        o, l = mla_decode(p, dv, nthreads)
        out[:, :, j * g:(j + 1) * g] = o
        lse[:, j * g:(j + 1) * g] = l
    return out, lse
