"""GPU parity: the CUDA path (through the C ABI) against the fp64 oracle, element
by element, on seeded inputs.

- small cases (several 64-row tiles, ragged tails, causal and not, splits):
  every output element;
- the five benchmark workloads at full size, in the launch configuration the
  benchmark times: every output element against the oracle;
- edge cases: empty sequences, one token, causal rows that see nothing,
  NaN-poisoned tails and unreferenced pages, strided tensors, metadata reuse.
Tolerances: |out - ref| <= 1e-2 + 1e-2 |ref|, |lse - ref| <= 1e-3.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from decode_attention_paged_gb300 import workloads as W
from tests._helpers import NTHREADS, assert_close, problem, run_gpu

pytestmark = pytest.mark.gpu


def full_check(w, what, k_cache_gpu=None):
    out, lse, meta, ns = run_gpu(w, k_cache_gpu)
    ref_out, ref_lse = oracle.mla_decode(problem(w), nthreads=NTHREADS)
    errs = assert_close(out, lse, ref_out, ref_lse, what)
    return errs, ns


def test_tiny_config_full():
    errs, _ = full_check(W.tiny(), "tiny")
    print("tiny max errs", errs)


SMALL = [
    # (b, s_q, h_q, seqlens, causal)
    (1, 1, 16, [256], False),
    (2, 1, 16, [1, 64], False),
    (3, 1, 64, [65, 127, 130], False),
    (2, 1, 128, [300, 1000], False),
    (2, 2, 128, [200, 77], True),
    (3, 3, 20, [5, 64, 190], True),
    (1, 1, 96, [777], False),
    (4, 2, 1, [1, 2, 3, 129], True),
    (2, 1, 200, [64, 640], False),
    (5, 4, 16, [0, 1, 3, 65, 300], True),
]


@pytest.mark.parametrize("case", SMALL, ids=[str(i) for i in range(len(SMALL))])
def test_small_cases_full(case):
    b, s_q, h_q, seqlens, causal = case
    w = W.random_case(100 + SMALL.index(case), b, s_q, h_q, seqlens, causal)
    full_check(w, f"small {case}")


@pytest.mark.parametrize("L,h_q", [(20000, 16), (5000, 128), (70000, 1)])
def test_long_single_sequence_is_split_and_combined(L, h_q):
    """One long sequence spread over many SM parts: exercises the split
    partials and the combine kernel."""
    w = W.random_case(7, 1, 1, h_q, [L], False)
    _, ns = full_check(w, f"split L={L} h_q={h_q}")
    assert int(ns[1]) > 1, "the plan was expected to split this sequence"


def test_ragged_batch_with_splits_causal_mtp():
    w = W.random_case(8, 6, 2, 64, [1, 2, 4000, 64, 9000, 130], True)
    _, ns = full_check(w, "ragged mtp")
    counts = np.diff(ns.cpu().numpy())
    assert counts.max() > 1


def test_empty_and_degenerate_rows():
    """L = 0 requests, L = 1, and causal rows with L < s_q (nothing visible):
    out = 0 and lse = -inf there."""
    w = W.random_case(9, 4, 3, 16, [0, 1, 2, 0], True)
    out, lse, _, _ = run_gpu(w)
    ref_out, ref_lse = oracle.mla_decode(problem(w))
    assert_close(out, lse, ref_out, ref_lse, "degenerate")
    assert torch.all(out[0] == 0) and torch.all(torch.isneginf(lse[0]))
    assert torch.all(out[1, :2] == 0) and torch.all(torch.isneginf(lse[1, :, :2]))


def test_nan_poisoned_tails_and_unreferenced_pages():
    """Cache slots past each sequence's length and pages nobody references hold
    NaN: they must not reach any output."""
    w = W.random_case(10, 3, 2, 32, [100, 64, 1], True, extra_pages=5)
    kc = w.k_cache.clone()
    used = set()
    for i in range(w.b):
        L = int(w.cache_seqlens[i])
        nb = -(-L // 64)
        for j in range(nb):
            used.add(int(w.block_table[i, j]))
        if L % 64:
            kc[int(w.block_table[i, nb - 1]), L % 64:] = float("nan")
    for pg in range(kc.shape[0]):
        if pg not in used:
            kc[pg] = float("nan")
    w.k_cache = kc
    full_check(w, "nan poison")


def test_strided_tensors():
    """q with a padded batch stride, k_cache as a slice of a wider page pool,
    out with padded strides."""
    from decode_attention_paged_gb300 import api

    w = W.random_case(11, 3, 2, 16, [90, 300, 64], False)
    g = w.to("cuda")
    b, s_q, h_q, _ = w.q.shape
    qbig = torch.zeros(b, s_q * h_q * 576 + 64, dtype=torch.bfloat16, device="cuda")
    qbig[:, : s_q * h_q * 576] = g.q.reshape(b, -1)
    q = qbig[:, : s_q * h_q * 576].view(b, s_q, h_q, 576)
    assert q.stride(0) != s_q * h_q * 576
    kbig = torch.zeros(w.k_cache.shape[0], 64 * 2, 1, 576, dtype=torch.bfloat16, device="cuda")
    kbig[:, ::2] = g.k_cache
    kc = kbig[:, ::2]  # token stride 2*576, page stride 128*576
    out_big = torch.full((b, s_q, h_q + 3, 512 + 8), 7.0, dtype=torch.bfloat16, device="cuda")
    out = out_big[:, :, :h_q, :512]
    meta, ns = api.mla_get_metadata(g.cache_seqlens, h_q, s_q)
    api.mla_decode_fwd(q, kc, g.block_table, g.cache_seqlens, w.softmax_scale, False, meta, ns,
                       out=out)
    lse = torch.empty(b, h_q, s_q, device="cuda")
    _, lse = api.mla_decode_fwd(q, kc, g.block_table, g.cache_seqlens, w.softmax_scale, False,
                                meta, ns, out=out, lse=lse)
    assert api.mla_last_device_error() == 0
    ref_out, ref_lse = oracle.mla_decode(problem(w))
    assert_close(out, lse, ref_out, ref_lse, "strided")
    assert torch.all(out_big[:, :, h_q:] == 7.0) and torch.all(out_big[..., 512:] == 7.0)


def test_metadata_reused_across_layers_and_deterministic():
    """One plan serves several layers (different q and caches, same lengths);
    repeated calls give bit-identical results."""
    from decode_attention_paged_gb300 import api

    w1 = W.random_case(12, 4, 1, 128, [3000, 10, 600, 1500], False)
    w2 = W.random_case(13, 4, 1, 128, [3000, 10, 600, 1500], False)
    g1, g2 = w1.to("cuda"), w2.to("cuda")
    meta, ns = api.mla_get_metadata(g1.cache_seqlens, 128, 1)
    o1, l1 = api.mla_decode_fwd(g1.q, g1.k_cache, g1.block_table, g1.cache_seqlens,
                                w1.softmax_scale, False, meta, ns)
    o2, l2 = api.mla_decode_fwd(g2.q, g2.k_cache, g2.block_table, g2.cache_seqlens,
                                w2.softmax_scale, False, meta, ns)
    o1b, l1b = api.mla_decode_fwd(g1.q, g1.k_cache, g1.block_table, g1.cache_seqlens,
                                  w1.softmax_scale, False, meta, ns)
    assert api.mla_last_device_error() == 0
    assert torch.equal(o1, o1b) and torch.equal(l1, l1b)
    for w, o, l in ((w1, o1, l1), (w2, o2, l2)):
        ro, rl = oracle.mla_decode(problem(w), nthreads=NTHREADS)
        assert_close(o, l, ro, rl, "reuse")


@pytest.mark.parametrize("name", ["memory_bound", "compute_bound", "mtp", "long_ragged"])
def test_benchmark_workloads_full_size(name):
    """Full-size workloads in the benchmark's launch configuration: every
    element of out and lse against the oracle (all rows, all 512 dims)."""
    w = W.CONFIGS[name]()
    out, lse, meta, ns = run_gpu(w)
    ref_o, ref_l = oracle.mla_decode(problem(w), nthreads=NTHREADS)
    errs = assert_close(out, lse, ref_o, ref_l, name)
    print(name, "max errs", errs, "pieces", int(ns[-1].item()))
