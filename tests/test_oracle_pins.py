"""Pins for the fp64 oracle: each test checks it against something other than
itself -- closed forms, a library routine (torch SDPA in fp64), pure-Python
brute force, and invariants the pages fix.  CPU only."""
import math

import numpy as np
import pytest
import torch

import oracle
from decode_attention_paged_gb300 import workloads as W


def _bits(t):
    return oracle.bf16_bits(t)


def _problem(w: W.Workload):
    return oracle.Problem(_bits(w.q), _bits(w.k_cache), w.block_table.numpy(),
                          w.cache_seqlens.numpy(), w.softmax_scale, w.causal)


def _bf(x):
    """float array -> bf16 tensor (exactly representable test values)."""
    return torch.tensor(np.asarray(x, dtype=np.float32)).to(torch.bfloat16)


def _gather(w: W.Workload, i: int):
    """K/V of request i as contiguous fp64 [L, 576] (CPU, torch indexing only)."""
    L = int(w.cache_seqlens[i])
    nb = (L + W.PAGE - 1) // W.PAGE
    pages = w.block_table[i, :nb].long()
    kv = w.k_cache[pages].reshape(nb * W.PAGE, -1)[:L]
    return kv.double()


# ---------------------------------------------------------------- library pin
@pytest.mark.parametrize("causal,s_q,h_q", [(False, 1, 16), (True, 2, 8), (True, 3, 4)])
def test_matches_torch_sdpa_fp64(causal, s_q, h_q):
    """The definition reduces to scaled_dot_product_attention with K = kv[:, :576]
    and V = kv[:, :512] per request ("[DeepSeek-3] FlashMLA", sec. 3)."""
    w = W.random_case(7, 3, s_q, h_q, [130, 64, 5], causal)
    out, lse = oracle.mla_decode(_problem(w), nthreads=2)
    for i in range(w.b):
        kv = _gather(w, i)
        L = kv.shape[0]
        q = w.q[i].double().reshape(s_q * h_q, -1)  # rows rho = s*h_q + h
        s_idx = torch.arange(s_q * h_q) // h_q
        t = torch.arange(L)
        if causal:
            mask = t[None, :] <= (L - s_q + s_idx)[:, None]
        else:
            mask = torch.ones(s_q * h_q, L, dtype=torch.bool)
        ref = torch.nn.functional.scaled_dot_product_attention(
            q[None], kv[None], kv[None, :, :512], attn_mask=mask[None], scale=w.softmax_scale)[0]
        scores = (q @ kv.T) * w.softmax_scale
        scores = scores.masked_fill(~mask, float("-inf"))
        ref_lse = torch.logsumexp(scores, dim=-1)
        got = torch.from_numpy(out[i].reshape(s_q * h_q, 512))
        got_lse = torch.from_numpy(lse[i].T.reshape(-1))  # [h, s] -> rows s*h_q + h
        assert torch.allclose(got, ref, atol=1e-12, rtol=1e-10)
        assert torch.allclose(got_lse, ref_lse, atol=1e-10, rtol=0)


# ----------------------------------------------------------- brute force pin
def test_pure_python_bruteforce_tiny():
    """Pure-Python loops with math.exp on a tiny problem (d=6, dv=4, page 4),
    causal, two pages plus a partial one."""
    rng = np.random.default_rng(3)
    b, s_q, h_q, d, dv, page = 2, 2, 2, 6, 4, 4
    seqlens = [9, 3]
    num_pages = 7
    q = _bf(rng.standard_normal((b, s_q, h_q, d)))
    kv = _bf(rng.standard_normal((num_pages, page, d)))
    bt = np.array([[5, 0, 3], [2, 6, 1]], dtype=np.int32)
    scale = 0.37
    p = oracle.Problem(_bits(q), _bits(kv), bt, np.array(seqlens, np.int32), scale, True)
    out, lse = oracle.mla_decode(p, dv=dv)
    qf, kf = q.double().numpy(), kv.double().numpy()
    for i in range(b):
        L = seqlens[i]
        for s in range(s_q):
            for h in range(h_q):
                vis = [t for t in range(L) if t <= L - s_q + s]
                xs = []
                for t in vis:
                    row = kf[bt[i][t // page]][t % page]
                    xs.append(scale * sum(qf[i, s, h, c] * row[c] for c in range(d)))
                if not vis:
                    assert lse[i, h, s] == -math.inf
                    assert np.all(out[i, s, h] == 0)
                    continue
                m = max(xs)
                tot = sum(math.exp(x - m) for x in xs)
                ref_lse = m + math.log(tot)
                ref = [0.0] * dv
                for x, t in zip(xs, vis):
                    row = kf[bt[i][t // page]][t % page]
                    for c in range(dv):
                        ref[c] += math.exp(x - ref_lse) * row[c]
                assert abs(lse[i, h, s] - ref_lse) < 1e-12
                assert np.allclose(out[i, s, h], ref, atol=1e-13, rtol=1e-12)


# ------------------------------------------------------------ closed forms
def test_one_token_returns_v_exactly():
    """L = 1: the softmax weight is 1, so out is the token's first 512 dims and
    lse is its single scaled score."""
    w = W.random_case(1, 2, 1, 16, [1, 1], False)
    out, lse = oracle.mla_decode(_problem(w))
    for i in range(w.b):
        kv0 = w.k_cache[int(w.block_table[i, 0]), 0, 0].double()
        for h in range(16):
            assert np.array_equal(out[i, 0, h], kv0[:512].numpy())
            x0 = float(np.dot(w.q[i, 0, h].double().numpy(), kv0.numpy())) * w.softmax_scale
            assert abs(lse[i, h, 0] - x0) < 1e-12


def test_softmax_rows_sum_to_one():
    """With V = 1 in every dim the output is the sum of the softmax weights."""
    w = W.random_case(2, 3, 2, 4, [200, 64, 7], True)
    kc = w.k_cache.clone()
    kc[..., :512] = 1.0
    w.k_cache = kc
    out, _ = oracle.mla_decode(_problem(w))
    assert np.allclose(out, 1.0, atol=1e-12, rtol=0)


def test_constant_keys():
    """All cached tokens equal: out = that token, lse = x + ln L."""
    L = 150
    w = W.random_case(3, 1, 1, 4, [L], False)
    kc = w.k_cache.clone()
    kc[:] = kc[0, 0]
    w.k_cache = kc
    out, lse = oracle.mla_decode(_problem(w))
    kv0 = kc[0, 0, 0].double().numpy()
    for h in range(4):
        x = float(np.dot(w.q[0, 0, h].double().numpy(), kv0)) * w.softmax_scale
        assert np.allclose(out[0, 0, h], kv0[:512], atol=1e-12, rtol=1e-12)
        assert abs(lse[0, h, 0] - (x + math.log(L))) < 1e-10


def test_zero_query_gives_mean_of_v():
    """q = 0: every score is 0, weights are uniform, lse = ln |visible|."""
    w = W.random_case(4, 2, 2, 2, [77, 130], True)
    w.q = torch.zeros_like(w.q)
    out, lse = oracle.mla_decode(_problem(w))
    for i in range(w.b):
        kv = _gather(w, i)
        L = kv.shape[0]
        for s in range(2):
            vis = L - 2 + s + 1
            mean = kv[:vis, :512].mean(0).numpy()
            for h in range(2):
                assert np.allclose(out[i, s, h], mean, atol=1e-13)
                assert abs(lse[i, h, s] - math.log(vis)) < 1e-13


def test_causal_visible_set_is_bottom_right_tril():
    """One-hot V exposes the visible set: with q = 0, out * |visible| is its
    indicator.  It must equal numpy's tril(ones(s_q, L), k = L - s_q) ("3.4
    Attention kernel", 代码: the causal mask of naive_attention)."""
    s_q, L, page = 4, 11, 4
    d = dv = 16
    nb = (L + page - 1) // page
    kv = np.zeros((nb, page, d), np.float32)
    for t in range(L):
        kv[t // page, t % page, t] = 1.0
    q = np.zeros((1, s_q, 1, d), np.float32)
    p = oracle.Problem(_bits(_bf(q)), _bits(_bf(kv)), np.arange(nb, dtype=np.int32)[None],
                       np.array([L], np.int32), 1.0, True)
    out, lse = oracle.mla_decode(p, dv=dv)
    tril = np.tril(np.ones((s_q, L)), k=L - s_q)
    for s in range(s_q):
        ind = out[0, s, 0, :L] * tril[s].sum()
        assert np.allclose(ind, tril[s], atol=1e-12)
        assert np.allclose(out[0, s, 0, L:], 0)


def test_empty_visible_set():
    """L = 0, and causal rows that see nothing (L < s_q): out = 0, lse = -inf."""
    w = W.random_case(5, 2, 3, 2, [0, 2], True)
    out, lse = oracle.mla_decode(_problem(w))
    assert np.all(out[0] == 0) and np.all(np.isneginf(lse[0]))
    # request 1 has L = 2, s_q = 3: token s sees t <= s - 1 -> s = 0 sees nothing
    assert np.all(out[1, 0] == 0) and np.all(np.isneginf(lse[1, :, 0]))
    assert np.all(np.isfinite(lse[1, :, 1:]))


def test_block_table_permutation_invariance():
    """Moving pages around in the pool, with the block table updated to match,
    leaves every result bit-identical."""
    w = W.random_case(6, 2, 1, 8, [300, 129], False)
    out, lse = oracle.mla_decode(_problem(w))
    g = torch.Generator().manual_seed(99)
    perm = torch.randperm(w.k_cache.shape[0], generator=g)
    inv = torch.empty_like(perm)
    inv[perm] = torch.arange(perm.numel())
    w2 = W.Workload(w.name, w.q, w.k_cache[perm].contiguous(), inv[w.block_table.long()].int(),
                    w.cache_seqlens, w.softmax_scale, w.causal)
    out2, lse2 = oracle.mla_decode(_problem(w2))
    assert np.array_equal(out, out2) and np.array_equal(lse, lse2)


def test_scale_multiplies_the_score():
    """score *= softmax_scale: doubling q equals doubling the scale."""
    w = W.random_case(8, 1, 1, 4, [70], False)
    o1, l1 = oracle.mla_decode(_problem(w))
    w2 = W.Workload(w.name, w.q, w.k_cache, w.block_table, w.cache_seqlens, 2 * w.softmax_scale,
                    False)
    w3 = W.Workload(w.name, (w.q.float() * 2).bfloat16(), w.k_cache, w.block_table,
                    w.cache_seqlens, w.softmax_scale, False)
    o2, l2 = oracle.mla_decode(_problem(w2))
    o3, l3 = oracle.mla_decode(_problem(w3))
    assert np.allclose(o2, o3, atol=1e-12) and np.allclose(l2, l3, atol=1e-12)
    assert not np.allclose(o1, o2)


# ------------------------------------------------------- split invariance
@pytest.mark.parametrize("causal", [False, True])
def test_split_then_combine_equals_unsplit(causal):
    """Split-KV is exact ("3.4 Attention kernel", 解码 attention 与
    Flash-Decoding; FlashMLA overview sec. 7): any cut of the key range into
    pieces -- empty pieces included -- merged by the LSE combine, or by the
    pairwise (m, l, o~) merge, gives the unsplit row."""
    rng = np.random.default_rng(11)
    w = W.random_case(9, 2, 2, 4, [333, 90], causal)
    p = _problem(w)
    out, lse = oracle.mla_decode(p)
    for i in range(w.b):
        L = int(w.cache_seqlens[i])
        for rho in range(w.s_q * w.h_q):
            s, h = divmod(rho, w.h_q)
            for n_split in (1, 2, 5, 17, 64):
                cuts = np.sort(rng.integers(0, L + 1, size=n_split - 1))
                bounds = [0] + cuts.tolist() + [L]
                parts = [oracle.mla_partial(p, i, rho, a, b_) for a, b_ in zip(bounds, bounds[1:])]
                lse_k = np.array([pl for _, pl in parts])
                o_k = np.stack([po for po, _ in parts])
                o, l = oracle.lse_combine(lse_k, o_k)
                assert np.allclose(o, out[i, s, h], atol=1e-12, rtol=1e-12)
                assert abs(l - lse[i, h, s]) < 1e-12
                # pairwise merge of unnormalised states: m = lse, l = 1, o~ = o
                st = (-math.inf, 0.0, np.zeros(512))
                for po, pl in parts:
                    if pl == -math.inf:
                        st = oracle.merge_pair(st, (pl, 0.0, po))
                    else:
                        st = oracle.merge_pair(st, (pl, 1.0, po))
                m, lsum, ot = st
                assert np.allclose(ot / lsum, out[i, s, h], atol=1e-12, rtol=1e-12)
                assert abs(m + math.log(lsum) - lse[i, h, s]) < 1e-12


def test_combine_edge_cases():
    o = np.arange(4.0)
    got, l = oracle.lse_combine([0.5], o[None])
    assert np.array_equal(got, o) and l == 0.5  # one piece: identity
    got, l = oracle.lse_combine([-math.inf, -math.inf], np.ones((2, 4)))
    assert np.all(got == 0) and l == -math.inf  # all empty: zeros, -inf
    got, l = oracle.lse_combine([-math.inf, 1.0], np.stack([np.full(4, np.nan), o]))
    assert np.array_equal(got, o) and l == 1.0  # an empty piece is skipped entirely


def test_full_problem_row_subset_matches():
    """The row-subset entry point gives the same bits as the full decode."""
    w = W.random_case(10, 3, 2, 4, [100, 1, 64], True)
    p = _problem(w)
    out, lse = oracle.mla_decode(p, nthreads=3)
    units = np.array([[0, 0], [2, 7], [1, 3], [0, 5]], np.int32)
    o, l = oracle.mla_decode_rows(p, units)
    for k, (i, rho) in enumerate(units):
        s, h = divmod(int(rho), 4)
        assert np.array_equal(o[k], out[i, s, h]) and l[k] == lse[i, h, s]


@pytest.mark.parametrize("d,dv", [(192, 128), (64, 64), (320, 192), (576, 448)])
def test_other_head_sizes_match_torch_sdpa(d, dv):
    """Head sizes other than 576 / 512 (V = the first dv dims of each cache
    row): the definition again reduces to fp64 scaled_dot_product_attention
    per request, causal rows included."""
    w = W.random_case(11, 3, 2, 8, [130, 64, 5], True, d=d)
    out, lse = oracle.mla_decode(_problem(w), dv=dv, nthreads=2)
    for i in range(w.b):
        kv = _gather(w, i)
        L = kv.shape[0]
        q = w.q[i].double().reshape(2 * 8, -1)
        s_idx = torch.arange(2 * 8) // 8
        mask = torch.arange(L)[None, :] <= (L - 2 + s_idx)[:, None]
        ref = torch.nn.functional.scaled_dot_product_attention(
            q[None], kv[None], kv[None, :, :dv], attn_mask=mask[None], scale=w.softmax_scale)[0]
        scores = ((q @ kv.T) * w.softmax_scale).masked_fill(~mask, float("-inf"))
        got = torch.from_numpy(out[i].reshape(2 * 8, dv))
        assert torch.allclose(got, ref, atol=1e-12, rtol=1e-10)
        assert torch.allclose(torch.from_numpy(lse[i].T.reshape(-1)), torch.logsumexp(scores, -1),
                              atol=1e-10, rtol=0)
