"""Decode with several cache heads (h_kv > 1; "[DeepSeek-3] FlashMLA", sec. 4:
k_cache [blocks, 64, h_kv, 576], query heads j*g..j*g+g-1 attend to cache head
j) on the GPU against the fp64 oracle, element by element.
Tolerances: |out - ref| <= 1e-2 + 1e-2 |ref|, |lse - ref| <= 1e-3."""
import pytest
import torch

import oracle
from decode_attention_paged_gb300 import _lib
from decode_attention_paged_gb300 import workloads as W
from tests._helpers import NTHREADS, assert_close

pytestmark = pytest.mark.gpu

CASES = [
    # (b, s_q, h_q, h_kv, seqlens, causal): the query tile layouts -- whole head
    # groups of one or several tokens (g = 8, 4), two tiles of two tokens each
    # (g = 32), 64-head slices of one token (g = 128), one head per group (MHA)
    (2, 1, 16, 2, [300, 4100], False),
    (3, 2, 32, 4, [0, 130, 2000], True),
    (2, 4, 64, 2, [700, 64], True),
    (1, 1, 256, 2, [5000], False),
    (4, 1, 8, 8, [63, 64, 65, 1], False),
    (2, 3, 16, 4, [100, 9], True),
]


def gqa_case(seed, b, s_q, h_q, h_kv, seqlens):
    g = torch.Generator().manual_seed(seed)
    nb = max(1, max(-(-L // W.PAGE) for L in seqlens))
    pages = b * nb + 3
    q = torch.randn(b, s_q, h_q, W.D_QK, generator=g).to(torch.bfloat16)
    kv = torch.randn(pages, W.PAGE, h_kv, W.D_QK, generator=g).to(torch.bfloat16)
    bt = torch.randperm(pages, generator=g)[: b * nb].view(b, nb).to(torch.int32)
    return q, kv, bt, torch.tensor(seqlens, dtype=torch.int32)


@pytest.mark.parametrize("case", CASES, ids=[str(i) for i in range(len(CASES))])
def test_gqa_parity(case):
    from decode_attention_paged_gb300 import api

    b, s_q, h_q, h_kv, seqlens, causal = case
    q, kv, bt, sl = gqa_case(900 + CASES.index(case), b, s_q, h_q, h_kv, seqlens)
    scale = W.SCALE
    qd, kvd, btd, sld = q.cuda(), kv.cuda(), bt.cuda(), sl.cuda()
    meta, ns = api.mla_get_metadata(sld, h_q, s_q, h_kv)
    out, lse = api.mla_decode_fwd(qd, kvd, btd, sld, scale, causal, meta, ns)
    assert api.mla_last_device_error() == 0
    ref_out, ref_lse = oracle.mla_decode_gqa(oracle.bf16_bits(q), oracle.bf16_bits(kv), bt.numpy(),
                                             sl.numpy(), scale, causal, nthreads=NTHREADS)
    assert_close(out, lse, ref_out, ref_lse, f"gqa {case}")


def test_gqa_unsupported_group_size_is_refused():
    from decode_attention_paged_gb300 import api

    with pytest.raises(_lib.MLAError) as e:
        api.mla_get_metadata(torch.zeros(2, dtype=torch.int32, device="cuda"), 96, 1, 2)
    assert e.value.code == _lib.MLA_ERR_UNSUPPORTED


def test_gqa_full_size():
    """The GQA workload the benchmark times (b 32, h_q 64, h_kv 4, L 4096) at
    full size through the same call; every element against the oracle (group
    j = query heads 16j..16j+15 over cache head j)."""
    from decode_attention_paged_gb300 import api

    w = W.gqa()
    g = w.to("cuda")
    meta, ns = api.mla_get_metadata(g.cache_seqlens, w.h_q, w.s_q, w.h_kv)
    out, lse = api.mla_decode_fwd(g.q, g.k_cache, g.block_table, g.cache_seqlens,
                                  w.softmax_scale, w.causal, meta, ns)
    assert api.mla_last_device_error() == 0
    ro, rl = oracle.mla_decode_gqa(oracle.bf16_bits(w.q), oracle.bf16_bits(w.k_cache),
                                   w.block_table.numpy(), w.cache_seqlens.numpy(),
                                   w.softmax_scale, w.causal, nthreads=NTHREADS)
    assert_close(out, lse, ro, rl, "gqa full size")
