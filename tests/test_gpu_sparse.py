"""Sparse decode ("[DeepSeek-3] FlashMLA", sec. 11: attention over per-query
selected cache positions, index = page * 64 + offset) on the GPU against the
fp64 sparse oracle, element by element, on the automatic kernel choice (the
CTA pair for lists of 128 or more query rows) and on the single-CTA kernel.
Tolerances: |out - ref| <= 1e-2 + 1e-2 |ref|, |lse - ref| <= 1e-3."""
import numpy as np
import pytest
import torch

import oracle
from decode_attention_paged_gb300 import _lib
from decode_attention_paged_gb300 import workloads as W
from tests._helpers import (NTHREADS, assert_close, problem, run_gpu, run_gpu_sparse,
                            sparse_problem)

pytestmark = pytest.mark.gpu

CASES = [
    # (b, s_q, h_q, topk, context, pad_frac): one page, a ragged last page,
    # padding, two query tiles with splits, many small lists per SM part,
    # topk larger than the context (trailing padding)
    (2, 1, 16, 64, 100, 0.0),
    (3, 2, 64, 200, 300, 0.2),
    (1, 1, 128, 2048, 5000, 0.0),
    (2, 2, 128, 130, 1000, 0.5),
    (64, 1, 16, 512, 700, 0.0),
    (4, 3, 32, 100, 40, 0.0),
    (1, 1, 1, 77, 77, 0.0),
]


@pytest.fixture
def kernel_kind(request):
    from decode_attention_paged_gb300 import api

    default = api.get_decode_kernel()
    api.set_decode_kernel(request.param)
    yield request.param
    api.set_decode_kernel(default)


SPARSE_EXTRA = [
    # lists of 128 and 256 rows on the CTA pair: ragged pages, heavy padding,
    # splits over many parts, two tiles, several query tokens
    (3, 2, 128, 700, 900, 0.3),
    (2, 1, 256, 300, 400, 0.1),
    (40, 1, 128, 1000, 1200, 0.0),
]


@pytest.mark.parametrize("kernel_kind", [3, 1], indirect=True, ids=["auto", "single"])
@pytest.mark.parametrize("case", CASES + SPARSE_EXTRA,
                         ids=[str(i) for i in range(len(CASES) + len(SPARSE_EXTRA))])
def test_sparse_parity(kernel_kind, case):
    b, s_q, h_q, topk, ctx, pad = case
    w = W.random_sparse_case(500 + (CASES + SPARSE_EXTRA).index(case), b, s_q, h_q, topk, ctx, pad)
    out, lse = run_gpu_sparse(w)
    ref_out, ref_lse = oracle.mla_sparse(sparse_problem(w), nthreads=NTHREADS)
    assert_close(out, lse, ref_out, ref_lse, f"sparse {case} kernel {kernel_kind}")


def test_sparse_empty_lists():
    """topk = 0, and lists that are all padding: out = 0, lse = -inf."""
    w = W.random_sparse_case(520, 3, 2, 16, 0, 64)
    out, lse = run_gpu_sparse(w)
    assert torch.all(out == 0) and torch.all(torch.isneginf(lse))
    w = W.random_sparse_case(521, 3, 2, 16, 70, 200)
    w.indices[1] = -1
    w.indices[2, 1] = -1
    out, lse = run_gpu_sparse(w)
    ref_out, ref_lse = oracle.mla_sparse(sparse_problem(w), nthreads=NTHREADS)
    assert_close(out, lse, ref_out, ref_lse, "padding-only lists")
    assert torch.all(out[1] == 0) and torch.all(out[2, 1] == 0)


def test_sparse_duplicates_count_twice():
    w = W.random_sparse_case(522, 2, 1, 16, 96, 200)
    w.indices[:, :, 48:] = w.indices[:, :, :48]
    out, lse = run_gpu_sparse(w)
    ref_out, ref_lse = oracle.mla_sparse(sparse_problem(w), nthreads=NTHREADS)
    assert_close(out, lse, ref_out, ref_lse, "duplicates")


def test_sparse_index_past_the_cache_is_masked_and_reported():
    w = W.random_sparse_case(523, 2, 2, 64, 150, 300)
    n = w.num_tokens
    w.indices[0, 0, 3] = n
    w.indices[1, 1, 140] = n + 1000
    w.indices[1, 0, 0] = 2 ** 31 - 1
    out, lse = run_gpu_sparse(w, expect_code=_lib.MLA_ERR_BAD_INDEX)
    ref_out, ref_lse = oracle.mla_sparse(sparse_problem(w), nthreads=NTHREADS,
                                         allow_bad_index=True)
    assert_close(out, lse, ref_out, ref_lse, "bad indices")


def test_sparse_equals_dense_when_lists_are_the_prefix():
    """Lists naming every token of a request's prefix in page order give the
    dense decode result (both against the dense oracle)."""
    b, h_q, seqlens = 3, 64, [700, 64, 1500]
    w = W.random_case(524, b, 1, h_q, seqlens, False)
    topk = max(seqlens)
    idx = torch.full((b, 1, topk), -1, dtype=torch.int32)
    for i, L in enumerate(seqlens):
        t = torch.arange(L)
        idx[i, 0, :L] = w.block_table[i, t // W.PAGE] * W.PAGE + t % W.PAGE
    sw = W.SparseWorkload("prefix", w.q, w.k_cache, idx, w.softmax_scale)
    s_out, s_lse = run_gpu_sparse(sw)
    d_out, d_lse, _, _ = run_gpu(w)
    ref_out, ref_lse = oracle.mla_decode(problem(w), nthreads=NTHREADS)
    assert_close(s_out, s_lse, ref_out, ref_lse, "sparse prefix")
    assert_close(d_out, d_lse, ref_out, ref_lse, "dense")


def test_sparse_rejects_unpacked_pages():
    from decode_attention_paged_gb300 import api

    w = W.random_sparse_case(525, 1, 1, 16, 64, 64).to("cuda")
    big = torch.zeros(w.k_cache.shape[0], W.PAGE + 1, 1, W.D_QK, dtype=torch.bfloat16,
                      device="cuda")
    big[:, : W.PAGE] = w.k_cache
    kc = big[:, : W.PAGE]  # page stride 65 rows
    meta, ns = api.mla_get_metadata_sparse(w.topk, w.b, w.h_q, w.s_q)
    with pytest.raises(_lib.MLAError) as e:
        api.mla_decode_sparse_fwd(w.q, kc, w.indices, w.softmax_scale, meta, ns)
    assert e.value.code == _lib.MLA_ERR_UNSUPPORTED


def test_sparse_workload_full_size():
    """The sparse benchmark workload (batch 128, s_q 2, h_q 128, topk 2048) at
    full size, in the launch configuration the benchmark times; every element
    against the oracle."""
    w = W.sparse()
    out, lse = run_gpu_sparse(w)
    ro, rl = oracle.mla_sparse(sparse_problem(w), nthreads=NTHREADS)
    assert_close(out, lse, ro, rl, "sparse full size")
