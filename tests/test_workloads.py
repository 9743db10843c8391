"""The synthetic input recipe (seeded draws shared by the CUDA path and the
oracle): every configuration has the shapes, lengths, page pool and scale its
description states, the draws are reproducible from their seeds, and block
tables are permutations (no page is shared between or within requests)."""
import math

import numpy as np
import pytest
import torch

from decode_attention_paged_gb300 import workloads as W

# (config, b, s_q, h_q, seqlens or None for the seeded uniform draw, pool pages,
#  blocks per row, causal)
SPECS = [
    ("tiny", 1, 1, 16, [256], 4, 4, False),
    ("memory_bound", 64, 1, 16, [4096] * 64, 4096, 64, False),
    ("compute_bound", 64, 1, 128, None, 64 * 128, 128, False),
    ("mtp", 128, 2, 128, [4096] * 128, 8192, 64, True),
    ("long_ragged", 8, 1, 64, [1, 64, 1000, 8191, 16384, 32768, 49152, 65536], 8192, 1024, False),
]


@pytest.mark.parametrize("spec", SPECS, ids=[s[0] for s in SPECS])
def test_config_shapes_and_tables(spec):
    name, b, s_q, h_q, seqlens, pages, max_blocks, causal = spec
    w = W.CONFIGS[name]()
    assert w.q.shape == (b, s_q, h_q, W.D_QK) and w.q.dtype == torch.bfloat16
    assert w.k_cache.shape == (pages, W.PAGE, 1, W.D_QK) and w.k_cache.dtype == torch.bfloat16
    assert w.block_table.shape == (b, max_blocks) and w.block_table.dtype == torch.int32
    assert w.cache_seqlens.dtype == torch.int32 and w.cache_seqlens.shape == (b,)
    if seqlens is not None:
        assert w.cache_seqlens.tolist() == seqlens
    else:  # compute-bound: L ~ U[1, 8192]
        L = w.cache_seqlens.numpy()
        assert L.min() >= 1 and L.max() <= 8192 and len(set(L.tolist())) > 32
    assert w.causal == causal
    assert math.isclose(w.softmax_scale, 576 ** -0.5, rel_tol=1e-12)
    bt = w.block_table.numpy()
    assert bt.min() >= 0 and bt.max() < pages
    assert len(np.unique(bt)) == bt.size, "a page appears twice in the block table"
    if name == "tiny":
        assert bt.tolist() == [[0, 1, 2, 3]]  # identity table
    # every block a sequence uses is inside its row
    need = (w.cache_seqlens.numpy() + W.PAGE - 1) // W.PAGE
    assert (need <= max_blocks).all()


def test_draws_are_seeded_and_distinct():
    a, b = W.tiny(), W.tiny()
    assert torch.equal(a.q, b.q) and torch.equal(a.k_cache, b.k_cache)
    c = W.tiny(seed_offset=1)
    assert not torch.equal(a.q, c.q) and not torch.equal(a.k_cache, c.k_cache)
    # q and the cache come from different seeds
    assert not torch.equal(a.q[0, 0, :4].float(), a.k_cache[0, :4, 0].float())
    m1, m2 = W.compute_bound(), W.compute_bound()
    assert torch.equal(m1.cache_seqlens, m2.cache_seqlens)
    assert torch.equal(m1.block_table, m2.block_table)


def test_values_are_standard_normal_in_bf16():
    w = W.memory_bound()
    x = w.k_cache.view(-1)[: 1 << 22].float()
    assert abs(x.mean().item()) < 5e-3 and abs(x.std().item() - 1.0) < 5e-3
    # bf16: the low 16 bits of the fp32 pattern are zero after the cast back
    assert (x.view(torch.int32) & 0xFFFF).eq(0).all()


def test_sparse_lists_are_distinct_tokens_of_their_context():
    w = W.make_sparse("t", 3, 2, 16, 96, 300, pad_frac=0.1, seed_offset=7)
    idx = w.indices.numpy()
    assert idx.shape == (3, 2, 96)
    num_tokens = w.k_cache.shape[0] * W.PAGE
    pages_of = []
    for i in range(3):
        own = set()
        for s in range(2):
            row = idx[i, s]
            valid = row[row >= 0]
            assert len(set(valid.tolist())) == len(valid), "a key listed twice"
            assert valid.max() < num_tokens
            own |= set((valid // W.PAGE).tolist())
        pages_of.append(own)
    # requests own disjoint pages (a permutation of the pool)
    assert not (pages_of[0] & pages_of[1]) and not (pages_of[1] & pages_of[2])
    assert (idx < 0).mean() > 0.05  # padding slots drawn


def test_fp8_layout_round_trip():
    w = W.tiny()
    c8 = W.fp8_cache(w.k_cache)
    assert c8.shape == (4, W.PAGE, 1, 656) and c8.dtype == torch.uint8
    rope = c8[..., 528:].contiguous().view(torch.bfloat16)
    assert torch.equal(rope, w.k_cache[..., 512:])
    lat = c8[..., :512].contiguous().view(torch.float8_e4m3fn).float()
    sc = c8[..., 512:528].contiguous().view(torch.float32).repeat_interleave(128, -1)
    deq = lat * sc
    ref = w.k_cache[..., :512].float()
    # e4m3 keeps 3 mantissa bits: relative error of a quantised value <= 2^-4
    # of the tile's largest magnitude (scale = amax / 448)
    tol = sc * 448 * 2.0 ** -4
    assert ((deq - ref).abs() <= tol).all()
