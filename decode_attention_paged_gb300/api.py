"""Python binding of libmla.so: argument marshalling only.

Every step of the decode path (tile scheduling, paged TMA gathers, tcgen05
QK^T / PV, online softmax, split combine) runs in the library's CUDA kernels.
PyTorch only provides device memory (torch.empty) and the current stream.
The functions carry the C ABI's names; see include/mla_decode.h for the exact
contract of each.
"""
from __future__ import annotations

import ctypes
from typing import Optional, Tuple

import torch

from . import _lib

D_QK = 576
D_V = 512
# Smallest metadata buffer a decode call accepts: the header and room for 256
# part records (mla_metadata_size never returns less).
META_MIN_INTS = 8 + 8 * 256


def _check_plan(meta: torch.Tensor, num_splits: torch.Tensor) -> None:
    assert meta.dtype == torch.int32 and num_splits.dtype == torch.int32
    assert meta.is_contiguous() and meta.numel() >= META_MIN_INTS, \
        "meta must be a buffer of mla_metadata_size() bytes"


PAGE = 64


def _stream_ptr(stream: Optional[torch.cuda.Stream]) -> ctypes.c_void_p:
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _ptr(t: torch.Tensor) -> ctypes.c_void_p:
    return ctypes.c_void_p(t.data_ptr())


def metadata_size(batch: int, h_q: int, s_q: int, h_kv: int = 1) -> Tuple[int, int]:
    mb, sb = ctypes.c_size_t(), ctypes.c_size_t()
    _lib.check(_lib.load().mla_metadata_size(batch, h_q, s_q, h_kv, ctypes.byref(mb),
                                             ctypes.byref(sb)), "mla_metadata_size")
    return mb.value, sb.value


def workspace_size(batch: int, h_q: int, s_q: int, h_kv: int = 1) -> int:
    b = ctypes.c_size_t()
    _lib.check(_lib.load().mla_workspace_size(batch, h_q, s_q, h_kv, ctypes.byref(b)),
               "mla_workspace_size")
    return b.value


def mla_get_metadata(cache_seqlens: torch.Tensor, h_q: int, s_q: int, h_kv: int = 1,
                     stream: Optional[torch.cuda.Stream] = None,
                     meta: Optional[torch.Tensor] = None,
                     num_splits: Optional[torch.Tensor] = None):
    """Tile-scheduler plan for one decode step.  Returns (meta int32 [header + parts*8],
    num_splits int32 [batch + 1]), both on cache_seqlens' device; pass meta /
    num_splits to fill existing buffers (e.g. inside a CUDA graph)."""
    assert cache_seqlens.is_cuda and cache_seqlens.dtype == torch.int32
    cache_seqlens = cache_seqlens.contiguous()
    batch = cache_seqlens.shape[0]
    with torch.cuda.device(cache_seqlens.device):
        mb, sb = metadata_size(batch, h_q, s_q, h_kv)
        if meta is None:
            meta = torch.empty(mb // 4, dtype=torch.int32, device=cache_seqlens.device)
        if num_splits is None:
            num_splits = torch.empty(sb // 4, dtype=torch.int32, device=cache_seqlens.device)
        assert meta.dtype == torch.int32 and meta.numel() * 4 >= mb and meta.is_contiguous()
        assert num_splits.dtype == torch.int32 and num_splits.numel() * 4 >= sb
        _lib.check(_lib.load().mla_get_metadata(_ptr(cache_seqlens), batch, h_q, s_q, h_kv,
                                                _ptr(meta), _ptr(num_splits), _stream_ptr(stream)),
                   "mla_get_metadata")
    return meta, num_splits


class DecodeCall:
    """Marshalled arguments of one decode call (validated shapes, allocated
    outputs and workspace), reusable for the fused call or its two halves."""

    def __init__(self, q, k_cache, block_table, cache_seqlens, softmax_scale, causal, meta,
                 num_splits, workspace=None, out=None, lse=None, stream=None):
        assert q.dtype == torch.bfloat16 and k_cache.dtype == torch.bfloat16
        assert block_table.dtype == torch.int32 and cache_seqlens.dtype == torch.int32
        _check_plan(meta, num_splits)
        b, s_q, h_q, d = q.shape
        assert d == D_QK and q.stride(3) == 1 and q.stride(2) == D_QK and \
            q.stride(1) == h_q * D_QK, \
            "q rows must be packed: [b][s_q][h_q][576] with the (s_q, h_q) rows contiguous"
        num_pages, page, h_kv, dk = k_cache.shape
        assert dk == D_QK and k_cache.stride(3) == 1
        assert block_table.stride(1) == 1
        dev = q.device
        with torch.cuda.device(dev):
            if out is None:
                out = torch.empty(b, s_q, h_q, D_V, dtype=torch.bfloat16, device=dev)
            if lse is None:
                lse = torch.empty(b, h_q, s_q, dtype=torch.float32, device=dev)
            assert out.stride(3) == 1 and lse.is_contiguous()
            if workspace is None:
                workspace = torch.empty(workspace_size(b, h_q, s_q, h_kv), dtype=torch.uint8,
                                        device=dev)
        cache_seqlens = cache_seqlens.contiguous()
        self.device = dev
        self.out, self.lse, self.workspace = out, lse, workspace
        self._keep = (q, k_cache, block_table, cache_seqlens, meta, num_splits)
        self.stream = stream
        ws_bytes = workspace.numel() * workspace.element_size()
        self.full_args = (
            _ptr(q), q.stride(0), _ptr(k_cache), k_cache.stride(0), k_cache.stride(1), num_pages,
            page, _ptr(block_table), block_table.stride(0), block_table.shape[1],
            _ptr(cache_seqlens), b, s_q, h_q, h_kv, float(softmax_scale), int(bool(causal)),
            _ptr(meta), _ptr(num_splits), _ptr(workspace), ws_bytes, _ptr(out), out.stride(0),
            out.stride(1), out.stride(2), _ptr(lse))
        self.combine_args = (_ptr(meta), _ptr(num_splits), _ptr(workspace), ws_bytes, b, s_q, h_q,
                             h_kv, _ptr(out), out.stride(0), out.stride(1), out.stride(2),
                             _ptr(lse))

    def fwd(self):
        with torch.cuda.device(self.device):
            _lib.check(_lib.load().mla_decode_fwd(*self.full_args, _stream_ptr(self.stream)),
                       "mla_decode_fwd")
        return self.out, self.lse

    def splitkv(self):
        with torch.cuda.device(self.device):
            _lib.check(_lib.load().mla_decode_splitkv(*self.full_args, _stream_ptr(self.stream)),
                       "mla_decode_splitkv")

    def combine(self):
        with torch.cuda.device(self.device):
            _lib.check(_lib.load().mla_decode_combine(*self.combine_args, _stream_ptr(self.stream)),
                       "mla_decode_combine")
        return self.out, self.lse


def mla_decode_fwd(q: torch.Tensor, k_cache: torch.Tensor, block_table: torch.Tensor,
                   cache_seqlens: torch.Tensor, softmax_scale: float, causal: bool,
                   meta: torch.Tensor, num_splits: torch.Tensor,
                   workspace: Optional[torch.Tensor] = None, out: Optional[torch.Tensor] = None,
                   lse: Optional[torch.Tensor] = None,
                   stream: Optional[torch.cuda.Stream] = None):
    """out [b, s_q, h_q, 512] bf16 and lse [b, h_q, s_q] fp32 for absorbed queries
    q [b, s_q, h_q, 576] over the paged cache k_cache [pages, 64, 1, 576]."""
    return DecodeCall(q, k_cache, block_table, cache_seqlens, softmax_scale, causal, meta,
                      num_splits, workspace, out, lse, stream).fwd()


def mla_decode_fwd_dims(q: torch.Tensor, k_cache: torch.Tensor, block_table: torch.Tensor,
                        cache_seqlens: torch.Tensor, softmax_scale: float, causal: bool,
                        meta: torch.Tensor, num_splits: torch.Tensor, head_dim_v: int,
                        workspace: Optional[torch.Tensor] = None,
                        stream: Optional[torch.cuda.Stream] = None):
    """Other head sizes: q [b, s_q, h_q, d] over k_cache [pages, 64, 1, d],
    V the first head_dim_v dims of each cache row; returns out
    [b, s_q, h_q, head_dim_v] bf16 and lse [b, h_q, s_q] fp32
    (mla_decode_fwd_dims in include/mla_decode.h: d and head_dim_v multiples
    of 64, head_dim_v <= min(d, 512), d <= 576)."""
    assert q.dtype == torch.bfloat16 and k_cache.dtype == torch.bfloat16
    assert block_table.dtype == torch.int32 and cache_seqlens.dtype == torch.int32
    _check_plan(meta, num_splits)
    b, s_q, h_q, d = q.shape
    assert q.stride(3) == 1 and q.stride(2) == d and q.stride(1) == h_q * d, \
        "q rows must be packed: [b][s_q][h_q][d] with the (s_q, h_q) rows contiguous"
    num_pages, page, h_kv, dk = k_cache.shape
    assert dk == d and k_cache.stride(3) == 1 and block_table.stride(1) == 1
    assert block_table.dim() == 2 and block_table.shape[0] == b
    for t in (k_cache, block_table, cache_seqlens, meta, num_splits):
        assert t.device == q.device, "every tensor must be on q's device"
    dev = q.device
    cache_seqlens = cache_seqlens.contiguous()
    with torch.cuda.device(dev):
        out = torch.empty(b, s_q, h_q, head_dim_v, dtype=torch.bfloat16, device=dev)
        lse = torch.empty(b, h_q, s_q, dtype=torch.float32, device=dev)
        if workspace is None:
            workspace = torch.empty(workspace_size(b, h_q, s_q, h_kv), dtype=torch.uint8,
                                    device=dev)
        st = _lib.load().mla_decode_fwd_dims(
            _ptr(q), q.stride(0), _ptr(k_cache), k_cache.stride(0), k_cache.stride(1), num_pages,
            page, _ptr(block_table), block_table.stride(0), block_table.shape[1],
            _ptr(cache_seqlens), b, s_q, h_q, h_kv, d, int(head_dim_v), float(softmax_scale),
            int(bool(causal)), _ptr(meta), _ptr(num_splits), _ptr(workspace),
            workspace.numel() * workspace.element_size(), _ptr(out), out.stride(0),
            out.stride(1), out.stride(2), _ptr(lse), _stream_ptr(stream))
        _lib.check(st, "mla_decode_fwd_dims")
    return out, lse


def mla_decode_fwd_noalloc(q: torch.Tensor, k_cache: torch.Tensor, block_table: torch.Tensor,
                           cache_seqlens: torch.Tensor, softmax_scale: float, causal: bool,
                           meta: torch.Tensor, num_splits: torch.Tensor, out: torch.Tensor,
                           lse: torch.Tensor, stream: Optional[torch.cuda.Stream] = None):
    """mla_decode_fwd for callers that cannot allocate device memory: the
    library supplies the split-KV scratch from a fixed 32 MiB device array
    (see include/mla_decode.h).  The caller passes out and lse; nothing here
    allocates."""
    assert q.dtype == torch.bfloat16 and k_cache.dtype == torch.bfloat16
    assert block_table.dtype == torch.int32 and cache_seqlens.dtype == torch.int32
    _check_plan(meta, num_splits)
    b, s_q, h_q, d = q.shape
    assert d == D_QK and q.stride(3) == 1 and q.stride(2) == D_QK and q.stride(1) == h_q * D_QK
    num_pages, page, h_kv, dk = k_cache.shape
    assert dk == D_QK and k_cache.stride(3) == 1 and block_table.stride(1) == 1
    assert block_table.dim() == 2 and block_table.shape[0] == b
    assert cache_seqlens.shape == (b,) and cache_seqlens.is_contiguous()
    assert out.dtype == torch.bfloat16 and tuple(out.shape) == (b, s_q, h_q, D_V)
    assert out.stride(3) == 1
    assert lse.dtype == torch.float32 and tuple(lse.shape) == (b, h_q, s_q)
    assert lse.is_contiguous()
    for t in (k_cache, block_table, cache_seqlens, meta, num_splits, out, lse):
        assert t.device == q.device, "every tensor must be on q's device"
    with torch.cuda.device(q.device):
        st = _lib.load().mla_decode_fwd_noalloc(
            _ptr(q), q.stride(0), _ptr(k_cache), k_cache.stride(0), k_cache.stride(1), num_pages,
            page, _ptr(block_table), block_table.stride(0), block_table.shape[1],
            _ptr(cache_seqlens), b, s_q, h_q, h_kv, float(softmax_scale), int(bool(causal)),
            _ptr(meta), _ptr(num_splits), _ptr(out), out.stride(0), out.stride(1), out.stride(2),
            _ptr(lse), _stream_ptr(stream))
        _lib.check(st, "mla_decode_fwd_noalloc")
    return out, lse


class Fp8DecodeCall:
    """Marshalled arguments of one decode over an FP8-layout cache
    (include/mla_decode.h, mla_decode_fp8_fwd): k_cache uint8
    [pages, 64, 1, 656] with packed rows."""

    def __init__(self, q, k_cache, block_table, cache_seqlens, softmax_scale, causal, meta,
                 num_splits, workspace=None, out=None, lse=None, stream=None):
        assert q.dtype == torch.bfloat16 and k_cache.dtype == torch.uint8
        assert block_table.dtype == torch.int32 and cache_seqlens.dtype == torch.int32
        _check_plan(meta, num_splits)
        b, s_q, h_q, d = q.shape
        assert d == D_QK and q.stride(3) == 1 and q.stride(2) == D_QK and \
            q.stride(1) == h_q * D_QK
        num_pages, page, h_kv, row = k_cache.shape
        assert row == 656 and k_cache.stride(3) == 1 and k_cache.stride(1) == 656 * h_kv
        assert block_table.stride(1) == 1
        dev = q.device
        with torch.cuda.device(dev):
            if out is None:
                out = torch.empty(b, s_q, h_q, D_V, dtype=torch.bfloat16, device=dev)
            if lse is None:
                lse = torch.empty(b, h_q, s_q, dtype=torch.float32, device=dev)
            assert out.stride(3) == 1 and lse.is_contiguous()
            if workspace is None:
                workspace = torch.empty(workspace_size(b, h_q, s_q, h_kv), dtype=torch.uint8,
                                        device=dev)
        cache_seqlens = cache_seqlens.contiguous()
        self.device = dev
        self.out, self.lse, self.workspace = out, lse, workspace
        self._keep = (q, k_cache, block_table, cache_seqlens, meta, num_splits)
        self.stream = stream
        self.args = (
            _ptr(q), q.stride(0), _ptr(k_cache), k_cache.stride(0), num_pages, page,
            _ptr(block_table), block_table.stride(0), block_table.shape[1], _ptr(cache_seqlens), b,
            s_q, h_q, h_kv, float(softmax_scale), int(bool(causal)), _ptr(meta), _ptr(num_splits),
            _ptr(workspace), workspace.numel() * workspace.element_size(), _ptr(out),
            out.stride(0), out.stride(1), out.stride(2), _ptr(lse))

    def fwd(self):
        with torch.cuda.device(self.device):
            _lib.check(_lib.load().mla_decode_fp8_fwd(*self.args, _stream_ptr(self.stream)),
                       "mla_decode_fp8_fwd")
        return self.out, self.lse


def mla_decode_fp8_fwd(q, k_cache, block_table, cache_seqlens, softmax_scale, causal, meta,
                       num_splits, workspace=None, out=None, lse=None, stream=None):
    """Decode over an FP8-layout cache (656-byte rows: e4m3 latent, fp32
    scales, bf16 RoPE); the metadata is mla_get_metadata's."""
    return Fp8DecodeCall(q, k_cache, block_table, cache_seqlens, softmax_scale, causal, meta,
                         num_splits, workspace, out, lse, stream).fwd()


def metadata_size_sparse(batch: int, h_q: int, s_q: int, h_kv: int = 1) -> Tuple[int, int]:
    mb, sb = ctypes.c_size_t(), ctypes.c_size_t()
    _lib.check(_lib.load().mla_metadata_size_sparse(batch, h_q, s_q, h_kv, ctypes.byref(mb),
                                                    ctypes.byref(sb)), "mla_metadata_size_sparse")
    return mb.value, sb.value


def workspace_size_sparse(batch: int, h_q: int, s_q: int, h_kv: int = 1) -> int:
    b = ctypes.c_size_t()
    _lib.check(_lib.load().mla_workspace_size_sparse(batch, h_q, s_q, h_kv, ctypes.byref(b)),
               "mla_workspace_size_sparse")
    return b.value


def mla_get_metadata_sparse(topk: int, batch: int, h_q: int, s_q: int, h_kv: int = 1,
                            device=None, stream: Optional[torch.cuda.Stream] = None,
                            meta: Optional[torch.Tensor] = None,
                            num_splits: Optional[torch.Tensor] = None):
    """Split plan for sparse decode: every (request, query token) pair attends
    to a list of `topk` selected positions.  Returns (meta, num_splits
    int32 [batch * s_q + 1])."""
    dev = torch.device(device) if device is not None else torch.device("cuda",
                                                                      torch.cuda.current_device())
    with torch.cuda.device(dev):
        mb, sb = metadata_size_sparse(batch, h_q, s_q, h_kv)
        if meta is None:
            meta = torch.empty(mb // 4, dtype=torch.int32, device=dev)
        if num_splits is None:
            num_splits = torch.empty(sb // 4, dtype=torch.int32, device=dev)
        assert meta.dtype == torch.int32 and meta.numel() * 4 >= mb and meta.is_contiguous()
        assert num_splits.dtype == torch.int32 and num_splits.numel() * 4 >= sb
        _lib.check(_lib.load().mla_get_metadata_sparse(int(topk), batch, h_q, s_q, h_kv,
                                                       _ptr(meta), _ptr(num_splits),
                                                       _stream_ptr(stream)),
                   "mla_get_metadata_sparse")
    return meta, num_splits


class SparseDecodeCall:
    """Marshalled arguments of one sparse decode call (see include/mla_decode.h,
    mla_decode_sparse_fwd): q [b, s_q, h_q, 576], k_cache [pages, 64, 1, 576]
    with packed pages, indices int32 [b, s_q, topk] of positions page * 64 +
    offset (< 0: padding)."""

    def __init__(self, q, k_cache, indices, softmax_scale, meta, num_splits, workspace=None,
                 out=None, lse=None, stream=None):
        assert q.dtype == torch.bfloat16 and k_cache.dtype == torch.bfloat16
        assert indices.dtype == torch.int32 and indices.is_contiguous()
        _check_plan(meta, num_splits)
        b, s_q, h_q, d = q.shape
        assert d == D_QK and q.stride(3) == 1 and q.stride(2) == D_QK and \
            q.stride(1) == h_q * D_QK
        num_pages, page, h_kv, dk = k_cache.shape
        assert dk == D_QK and k_cache.stride(3) == 1
        assert tuple(indices.shape[:2]) == (b, s_q)
        topk = indices.shape[2]
        dev = q.device
        with torch.cuda.device(dev):
            if out is None:
                out = torch.empty(b, s_q, h_q, D_V, dtype=torch.bfloat16, device=dev)
            if lse is None:
                lse = torch.empty(b, h_q, s_q, dtype=torch.float32, device=dev)
            assert out.stride(3) == 1 and lse.is_contiguous()
            if workspace is None:
                workspace = torch.empty(workspace_size_sparse(b, h_q, s_q, h_kv),
                                        dtype=torch.uint8, device=dev)
        self.device = dev
        self.out, self.lse, self.workspace = out, lse, workspace
        self._keep = (q, k_cache, indices, meta, num_splits)
        self.stream = stream
        self.args = (
            _ptr(q), q.stride(0), _ptr(k_cache), k_cache.stride(0), k_cache.stride(1), num_pages,
            page, _ptr(indices), topk, b, s_q, h_q, h_kv, float(softmax_scale), _ptr(meta),
            _ptr(num_splits), _ptr(workspace), workspace.numel() * workspace.element_size(),
            _ptr(out), out.stride(0), out.stride(1), out.stride(2), _ptr(lse))

    def fwd(self):
        with torch.cuda.device(self.device):
            _lib.check(_lib.load().mla_decode_sparse_fwd(*self.args, _stream_ptr(self.stream)),
                       "mla_decode_sparse_fwd")
        return self.out, self.lse


def mla_decode_sparse_fwd(q: torch.Tensor, k_cache: torch.Tensor, indices: torch.Tensor,
                          softmax_scale: float, meta: torch.Tensor, num_splits: torch.Tensor,
                          workspace: Optional[torch.Tensor] = None,
                          out: Optional[torch.Tensor] = None, lse: Optional[torch.Tensor] = None,
                          stream: Optional[torch.cuda.Stream] = None):
    """Sparse decode: out [b, s_q, h_q, 512] bf16 and lse [b, h_q, s_q] fp32 over
    the positions listed in indices [b, s_q, topk]."""
    return SparseDecodeCall(q, k_cache, indices, softmax_scale, meta, num_splits, workspace, out,
                            lse, stream).fwd()


def mla_last_device_error(stream: Optional[torch.cuda.Stream] = None) -> int:
    """Synchronise the stream and read/clear the device error word."""
    code = ctypes.c_int()
    _lib.check(_lib.load().mla_last_device_error(_stream_ptr(stream), ctypes.byref(code)),
               "mla_last_device_error")
    return code.value


def set_wait_budget_ns(ns: int) -> None:
    _lib.check(_lib.load().mla_set_wait_budget_ns(int(ns)), "mla_set_wait_budget_ns")


def set_fixed_overhead(blocks: int) -> None:
    _lib.check(_lib.load().mla_set_fixed_overhead(int(blocks)), "mla_set_fixed_overhead")


KERNEL_SINGLE = 1  # one CTA per SM holding all 576 dims
KERNEL_TQ = 2      # one CTA per SM, most of Q in tensor memory, three KV stages
KERNEL_AUTO = 3    # default: TQ for s_q * h_q <= 32, DUO for >= 128 (one cache head), else SINGLE
KERNEL_DUO = 4     # a 2-CTA cluster per SM pair, 128-row tiles, pages split by head dims


def set_decode_kernel(kind: int) -> None:
    """Select the decode kernel (process-wide); rebuild metadata afterwards."""
    _lib.check(_lib.load().mla_set_decode_kernel(int(kind)), "mla_set_decode_kernel")


def get_decode_kernel() -> int:
    return int(_lib.load().mla_get_decode_kernel())


def flash_mla_with_kvcache(q, k_cache, block_table, cache_seqlens, head_dim_v, meta, num_splits,
                           softmax_scale=None, causal=False):
    """The pages' call shape (flash_mla_with_kvcache) mapped onto mla_decode_fwd
    (or mla_decode_fwd_dims for head sizes other than 576 / 512)."""
    if softmax_scale is None:
        softmax_scale = q.shape[-1] ** -0.5
    if q.shape[-1] != D_QK or head_dim_v != D_V:
        return mla_decode_fwd_dims(q, k_cache, block_table, cache_seqlens, softmax_scale, causal,
                                   meta, num_splits, head_dim_v)
    return mla_decode_fwd(q, k_cache, block_table, cache_seqlens, softmax_scale, causal, meta,
                          num_splits)
