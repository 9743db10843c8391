"""Pins for decode with several cache heads (h_kv > 1; "[DeepSeek-3] FlashMLA",
sec. 4: k_cache [blocks, 64, h_kv, 576], dense tests over MQA and GQA).  CPU
only.  Reading: query heads j*g .. j*g+g-1 (g = h_q / h_kv) attend to cache
head j.

Pinned against a brute force written out in plain Python/numpy on a tiny
paged problem (scores, softmax, weighted V sum, natural-log lse, bottom-right
causal rule), and against the special cases h_kv = 1 (the dense oracle) and
h_kv = h_q (multi-head attention: every head its own cache head)."""
import math

import numpy as np
import pytest
import torch

import oracle

D, DV, PAGE = 576, 512, 64


def tiny(seed, b, s_q, h_q, h_kv, seqlens):
    g = torch.Generator().manual_seed(seed)
    nb = max(1, max(-(-L // PAGE) for L in seqlens))
    pages = b * nb + 1
    q = torch.randn(b, s_q, h_q, D, generator=g).to(torch.bfloat16)
    kv = torch.randn(pages, PAGE, h_kv, D, generator=g).to(torch.bfloat16)
    bt = torch.randperm(pages, generator=g)[: b * nb].view(b, nb).to(torch.int32)
    return q, kv, bt


def brute(q, kv, bt, seqlens, scale, causal):
    b, s_q, h_q, _ = q.shape
    h_kv = kv.shape[2]
    g = h_q // h_kv
    qd, kd = q.double().numpy(), kv.double().numpy()
    out = np.zeros((b, s_q, h_q, DV))
    lse = np.zeros((b, h_q, s_q))
    for i in range(b):
        L = seqlens[i]
        for s in range(s_q):
            vis = L if not causal else max(0, min(L, L - s_q + s + 1))
            for h in range(h_q):
                j = h // g
                rows = [kd[bt[i, t // PAGE], t % PAGE, j] for t in range(vis)]
                if not rows:
                    lse[i, h, s] = -math.inf
                    continue
                x = np.array([scale * float(np.dot(qd[i, s, h], r)) for r in rows])
                m = x.max()
                l = m + math.log(np.exp(x - m).sum())
                w = np.exp(x - l)
                out[i, s, h] = (w[:, None] * np.array(rows)[:, :DV]).sum(0)
                lse[i, h, s] = l
    return out, lse


@pytest.mark.parametrize("h_kv,causal", [(2, False), (4, True), (8, False)])
def test_gqa_matches_brute_force(h_kv, causal):
    b, s_q, h_q, seqlens = 2, 2, 8, [70, 3]
    q, kv, bt = tiny(40 + h_kv, b, s_q, h_q, h_kv, seqlens)
    scale = 0.05
    got = oracle.mla_decode_gqa(oracle.bf16_bits(q), oracle.bf16_bits(kv), bt.numpy(),
                                np.array(seqlens, np.int32), scale, causal)
    ref = brute(q, kv, bt.numpy(), seqlens, scale, causal)
    np.testing.assert_allclose(got[0], ref[0], rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(got[1], ref[1], rtol=1e-12, atol=1e-10)


def test_one_cache_head_is_the_dense_oracle():
    q, kv, bt = tiny(50, 2, 1, 4, 1, [100, 64])
    args = (bt.numpy(), np.array([100, 64], np.int32), 0.04, False)
    got = oracle.mla_decode_gqa(oracle.bf16_bits(q), oracle.bf16_bits(kv), *args)
    ref = oracle.mla_decode(oracle.Problem(oracle.bf16_bits(q), oracle.bf16_bits(kv), *args))
    assert np.array_equal(got[0], ref[0]) and np.array_equal(got[1], ref[1])


def test_a_head_attends_only_to_its_own_cache_head():
    """Changing cache head j changes exactly the query heads of group j."""
    b, s_q, h_q, h_kv, seqlens = 1, 1, 6, 3, [90]
    q, kv, bt = tiny(51, b, s_q, h_q, h_kv, seqlens)
    args = (bt.numpy(), np.array(seqlens, np.int32), 0.05, False)
    base = oracle.mla_decode_gqa(oracle.bf16_bits(q), oracle.bf16_bits(kv), *args)
    kv2 = kv.clone()
    kv2[:, :, 1] = torch.randn(kv.shape[0], PAGE, D).to(torch.bfloat16)
    alt = oracle.mla_decode_gqa(oracle.bf16_bits(q), oracle.bf16_bits(kv2), *args)
    changed = [not np.array_equal(base[0][0, 0, h], alt[0][0, 0, h]) for h in range(h_q)]
    assert changed == [False, False, True, True, False, False]
