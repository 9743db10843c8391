"""Pins for the sparse-decode oracle ("[DeepSeek-3] FlashMLA", sec. 11: attention
over per-query selected tokens, index = page_id * page + offset).  CPU only.

The pins tie it to the dense oracle (itself pinned in test_oracle_pins.py) and
to closed forms:
- indices listing a request's visible tokens in page order reproduce dense
  decode exactly (same keys, same order, same arithmetic), also with a
  different list per query token (the causal triangle);
- a key listed twice adds ln 2 to lse and leaves out unchanged;
- padding (-1) anywhere changes nothing; an all-padding list gives out = 0,
  lse = -inf;
- an index past the cache is left out and reported.
"""
import math

import numpy as np
import pytest
import torch

import oracle

D, DV, PAGE = 576, 512, 64


def rand_problem(seed, b, s_q, h_q, seqlens, extra_pages=2):
    g = torch.Generator().manual_seed(seed)
    nb = [max(1, -(-L // PAGE)) for L in seqlens]
    max_blocks = max(nb)
    num_pages = b * max_blocks + extra_pages
    q = torch.randn(b, s_q, h_q, D, generator=g).to(torch.bfloat16)
    kv = torch.randn(num_pages, PAGE, 1, D, generator=g).to(torch.bfloat16)
    bt = torch.randperm(num_pages, generator=g)[: b * max_blocks].view(b, max_blocks).to(torch.int32)
    return q, kv, bt


def indices_from_pages(bt, seqlens, s_q, causal, topk=None):
    """indices[i][s][k] = physical position of logical token k of request i,
    for the tokens row s may see; -1 after them."""
    b = len(seqlens)
    topk = topk or max(1, max(seqlens))
    idx = np.full((b, s_q, topk), -1, dtype=np.int32)
    for i, L in enumerate(seqlens):
        for s in range(s_q):
            lim = L if not causal else max(0, min(L, L - s_q + s + 1))
            for k in range(lim):
                idx[i, s, k] = int(bt[i, k // PAGE]) * PAGE + k % PAGE
    return idx


@pytest.mark.parametrize("causal", [False, True])
def test_equals_dense_oracle_when_indices_list_the_pages(causal):
    b, s_q, h_q, seqlens = 3, 2, 4, [70, 1, 130]
    q, kv, bt = rand_problem(11, b, s_q, h_q, seqlens)
    scale = D ** -0.5
    dense = oracle.Problem(oracle.bf16_bits(q), oracle.bf16_bits(kv), bt.numpy(),
                           np.array(seqlens, np.int32), scale, causal)
    ref_out, ref_lse = oracle.mla_decode(dense, nthreads=4)
    sp = oracle.SparseProblem(oracle.bf16_bits(q), oracle.bf16_bits(kv),
                              indices_from_pages(bt.numpy(), seqlens, s_q, causal), scale)
    out, lse = oracle.mla_sparse(sp, nthreads=4)
    # same keys, same order, same fp64 arithmetic: identical bits
    assert np.array_equal(out, ref_out)
    assert np.array_equal(lse, ref_lse)


def test_padding_anywhere_changes_nothing():
    b, s_q, h_q, seqlens = 2, 1, 3, [90, 40]
    q, kv, bt = rand_problem(12, b, s_q, h_q, seqlens)
    idx = indices_from_pages(bt.numpy(), seqlens, s_q, False)
    base = oracle.mla_sparse(oracle.SparseProblem(oracle.bf16_bits(q), oracle.bf16_bits(kv), idx,
                                                  0.05))
    # interleave -1 slots, keeping the order of the real keys
    rng = np.random.default_rng(0)
    wide = np.full((b, s_q, idx.shape[2] * 2), -1, dtype=np.int32)
    for i in range(b):
        pos = np.sort(rng.choice(wide.shape[2], idx.shape[2], replace=False))
        wide[i, 0, pos] = idx[i, 0]
    got = oracle.mla_sparse(oracle.SparseProblem(oracle.bf16_bits(q), oracle.bf16_bits(kv), wide,
                                                 0.05))
    assert np.array_equal(got[0], base[0]) and np.array_equal(got[1], base[1])


def test_duplicate_key_adds_ln2_to_lse():
    b, s_q, h_q, seqlens = 1, 1, 2, [64]
    q, kv, bt = rand_problem(13, b, s_q, h_q, seqlens)
    idx = indices_from_pages(bt.numpy(), seqlens, s_q, False)
    once = oracle.mla_sparse(oracle.SparseProblem(oracle.bf16_bits(q), oracle.bf16_bits(kv), idx,
                                                  0.04))
    twice = oracle.mla_sparse(oracle.SparseProblem(oracle.bf16_bits(q), oracle.bf16_bits(kv),
                                                   np.concatenate([idx, idx], axis=2), 0.04))
    np.testing.assert_allclose(twice[0], once[0], rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(twice[1], once[1] + math.log(2.0), rtol=0, atol=1e-12)


def test_single_key_returns_its_value_row():
    """One selected token: softmax weight 1, out = V row exactly, lse = its score."""
    q, kv, bt = rand_problem(14, 1, 1, 2, [64])
    t = 37
    idx = np.array([[[int(bt[0, 0]) * PAGE + t, -1, -1]]], dtype=np.int32)
    out, lse = oracle.mla_sparse(oracle.SparseProblem(oracle.bf16_bits(q), oracle.bf16_bits(kv),
                                                      idx, 0.1))
    row = kv[int(bt[0, 0]), t, 0].double().numpy()
    for h in range(2):
        np.testing.assert_array_equal(out[0, 0, h], row[:DV])
        qs = q[0, 0, h].double().numpy()
        np.testing.assert_allclose(lse[0, h, 0], 0.1 * float(qs @ row), rtol=1e-12, atol=1e-12)


def test_all_padding_gives_empty_row():
    q, kv, bt = rand_problem(15, 2, 1, 2, [64, 64])
    idx = np.full((2, 1, 8), -1, dtype=np.int32)
    out, lse = oracle.mla_sparse(oracle.SparseProblem(oracle.bf16_bits(q), oracle.bf16_bits(kv),
                                                      idx, 0.1))
    assert np.all(out == 0.0) and np.all(np.isneginf(lse))


def test_index_past_the_cache_is_left_out_and_reported():
    q, kv, bt = rand_problem(16, 1, 1, 2, [64])
    good = indices_from_pages(bt.numpy(), [64], 1, False)
    num_tokens = kv.shape[0] * PAGE
    bad = np.concatenate([good, np.array([[[num_tokens, num_tokens + 5]]], np.int32)], axis=2)
    sp_bad = oracle.SparseProblem(oracle.bf16_bits(q), oracle.bf16_bits(kv), bad, 0.07)
    with pytest.raises(RuntimeError):
        oracle.mla_sparse(sp_bad)
    got = oracle.mla_sparse(sp_bad, allow_bad_index=True)
    ref = oracle.mla_sparse(oracle.SparseProblem(oracle.bf16_bits(q), oracle.bf16_bits(kv), good,
                                                 0.07))
    assert np.array_equal(got[0], ref[0]) and np.array_equal(got[1], ref[1])


def test_rows_entry_matches_full():
    b, s_q, h_q = 2, 2, 3
    q, kv, bt = rand_problem(17, b, s_q, h_q, [100, 30])
    rng = np.random.default_rng(3)
    idx = rng.integers(-1, kv.shape[0] * PAGE, size=(b, s_q, 50)).astype(np.int32)
    sp = oracle.SparseProblem(oracle.bf16_bits(q), oracle.bf16_bits(kv), idx, 0.05)
    out, lse = oracle.mla_sparse(sp, nthreads=3)
    units = np.array([[1, 4], [0, 0], [1, 2]], np.int32)
    ro, rl = oracle.mla_sparse_rows(sp, units)
    for n, (i, row) in enumerate(units):
        s, h = row // h_q, row % h_q
        assert np.array_equal(ro[n], out[i, s, h]) and rl[n] == lse[i, h, s]
