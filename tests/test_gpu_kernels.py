"""Every dense decode kernel (the single-CTA one, the one that keeps most of the
query tile in tensor memory, and the CTA-pair one for 128-row tiles) against
the fp64 oracle on the same seeded cases, and against each other.
Tolerances: |out - ref| <= 1e-2 + 1e-2 |ref|, |lse - ref| <= 1e-3."""
import numpy as np
import pytest
import torch

import oracle
from decode_attention_paged_gb300 import _lib
from decode_attention_paged_gb300 import workloads as W
from tests._helpers import NTHREADS, assert_close, problem, run_gpu

pytestmark = pytest.mark.gpu

CASES = [
    # (b, s_q, h_q, seqlens, causal): tails, splits, causal rows that see
    # nothing, several query tiles, an empty request
    (2, 1, 16, [1, 6000], False),
    (3, 2, 64, [0, 130, 4097], True),
    (1, 1, 128, [20000], False),
    (4, 1, 16, [63, 64, 65, 1], False),
    # many short pieces per SM part (several requests in one part): the
    # softmax may run ahead of PV by two pages on the per-stage-P path
    (8, 1, 16, [4096] * 8, False),
    (128, 1, 16, [512] * 128, False),
    (24, 2, 16, [700] * 24, True),
    # 128-row tiles (the CTA-pair kernel's shape): one and two tiles per
    # request, a partial second tile, splits, empty requests, causal MTP
    (3, 1, 128, [0, 5000, 77], False),
    (4, 2, 128, [64, 1, 4097, 300], True),
    (2, 1, 200, [64, 6500], False),
    (40, 1, 128, [1000] * 40, False),
]


@pytest.fixture
def kernel_kind(request):
    from decode_attention_paged_gb300 import api

    default = api.get_decode_kernel()
    api.set_decode_kernel(request.param)
    yield request.param
    api.set_decode_kernel(default)


@pytest.mark.parametrize("kernel_kind", [1, 2, 4], indirect=True, ids=["single", "tq", "duo"])
@pytest.mark.parametrize("case", CASES, ids=[str(i) for i in range(len(CASES))])
def test_kernel_parity(kernel_kind, case):
    b, s_q, h_q, seqlens, causal = case
    w = W.random_case(300 + CASES.index(case), b, s_q, h_q, seqlens, causal)
    out, lse, _, _ = run_gpu(w)
    ref_out, ref_lse = oracle.mla_decode(problem(w), nthreads=NTHREADS)
    assert_close(out, lse, ref_out, ref_lse, f"kernel {kernel_kind} {case}")


def test_kernels_agree():
    from decode_attention_paged_gb300 import api

    w = W.random_case(333, 3, 1, 16, [5000, 70, 900], False)
    g = w.to("cuda")
    default = api.get_decode_kernel()
    try:
        api.set_decode_kernel(api.KERNEL_SINGLE)
        meta_one, ns_one = api.mla_get_metadata(g.cache_seqlens, w.h_q, w.s_q)
        o_one, l_one = api.mla_decode_fwd(g.q, g.k_cache, g.block_table, g.cache_seqlens,
                                          w.softmax_scale, w.causal, meta_one, ns_one)
        assert api.mla_last_device_error() == 0
        api.set_decode_kernel(api.KERNEL_TQ)
        meta_r, ns_r = api.mla_get_metadata(g.cache_seqlens, w.h_q, w.s_q)
        o_r, l_r = api.mla_decode_fwd(g.q, g.k_cache, g.block_table, g.cache_seqlens,
                                      w.softmax_scale, w.causal, meta_r, ns_r)
        assert api.mla_last_device_error() == 0
        # same function, same plan, different summation orders
        assert (o_r.float() - o_one.float()).abs().max().item() <= 2e-2
        assert (l_r - l_one).abs().max().item() <= 1e-3
        w2 = W.random_case(334, 3, 2, 128, [5000, 70, 900], True)
        g2 = w2.to("cuda")
        outs = []
        for kind in (api.KERNEL_SINGLE, api.KERNEL_DUO):
            api.set_decode_kernel(kind)
            m2, n2 = api.mla_get_metadata(g2.cache_seqlens, w2.h_q, w2.s_q)
            outs.append(api.mla_decode_fwd(g2.q, g2.k_cache, g2.block_table, g2.cache_seqlens,
                                           w2.softmax_scale, w2.causal, m2, n2))
            assert api.mla_last_device_error() == 0
        assert (outs[0][0].float() - outs[1][0].float()).abs().max().item() <= 2e-2
        assert (outs[0][1] - outs[1][1]).abs().max().item() <= 1e-3
    finally:
        api.set_decode_kernel(default)
    assert api.get_decode_kernel() == default
