"""Head sizes other than 576 / 512 (mla_decode_fwd_dims: q and cache rows of
d dims, V the first dv dims of each cache row, one cache head) against the
fp64 oracle, element by element.  Tolerances: |out - ref| <= 1e-2 +
1e-2 |ref|, |lse - ref| <= 1e-3."""
import pytest
import torch

import oracle
from decode_attention_paged_gb300 import _lib
from decode_attention_paged_gb300 import workloads as W
from tests._helpers import NTHREADS, assert_close, problem

pytestmark = pytest.mark.gpu

SIZES = [
    (192, 128),   # the 128 + 64 head of a model without weight absorption
    (128, 128),
    (64, 64),
    (320, 192),   # V in two PV groups (128 + 64 dims)
    (576, 448),   # three PV groups (256 + 128 + 64)
    (448, 384),
    (576, 512),   # the MLA sizes through the general entry point
]

CASES = [
    # (b, s_q, h_q, seqlens, causal): tails, splits, an empty request, causal
    # rows that see nothing, two query tiles
    (3, 1, 16, [0, 130, 4097], False),
    (2, 2, 64, [700, 1], True),
    (2, 1, 128, [5000, 77], False),
]


def run_dims(w, dv):
    from decode_attention_paged_gb300 import api

    g = w.to("cuda")
    meta, ns = api.mla_get_metadata(g.cache_seqlens, w.h_q, w.s_q)
    out, lse = api.mla_decode_fwd_dims(g.q, g.k_cache, g.block_table, g.cache_seqlens,
                                       w.softmax_scale, w.causal, meta, ns, dv)
    assert api.mla_last_device_error() == 0
    return out, lse


@pytest.mark.parametrize("case", CASES, ids=[str(i) for i in range(len(CASES))])
@pytest.mark.parametrize("d,dv", SIZES, ids=[f"{d}-{dv}" for d, dv in SIZES])
def test_dims_parity(d, dv, case):
    b, s_q, h_q, seqlens, causal = case
    w = W.random_case(500 + CASES.index(case), b, s_q, h_q, seqlens, causal, d=d)
    out, lse = run_dims(w, dv)
    assert tuple(out.shape) == (b, s_q, h_q, dv)
    ref_out, ref_lse = oracle.mla_decode(problem(w), dv=dv, nthreads=NTHREADS)
    assert_close(out, lse, ref_out, ref_lse, f"d {d} dv {dv} {case}")


def test_dims_576_512_equals_mla_decode_fwd():
    """The general entry point at 576 / 512 gives what mla_decode_fwd gives."""
    from decode_attention_paged_gb300 import api

    w = W.random_case(520, 3, 1, 16, [300, 4097, 64], False)
    g = w.to("cuda")
    meta, ns = api.mla_get_metadata(g.cache_seqlens, w.h_q, w.s_q)
    o1, l1 = api.mla_decode_fwd_dims(g.q, g.k_cache, g.block_table, g.cache_seqlens,
                                     w.softmax_scale, False, meta, ns, 512)
    o2, l2 = api.mla_decode_fwd(g.q, g.k_cache, g.block_table, g.cache_seqlens, w.softmax_scale,
                                False, meta, ns)
    assert (o1.float() - o2.float()).abs().max().item() <= 2e-2
    assert (l1 - l2).abs().max().item() <= 1e-3


@pytest.mark.parametrize("d,dv,h_kv", [(100, 64, 1), (192, 256, 1), (640, 512, 1),
                                        (576, 576, 1), (192, 0, 1), (192, 128, 2)])
def test_unsupported_sizes_refused(d, dv, h_kv):
    """Sizes that are not multiples of 64, V wider than K or than 512, K wider
    than 576, and other head sizes with several cache heads are refused
    before anything is enqueued."""
    from decode_attention_paged_gb300 import api

    w = W.random_case(521, 1, 1, 16, [64], False, d=d)
    g = w.to("cuda")
    meta, ns = api.mla_get_metadata(g.cache_seqlens, w.h_q, w.s_q)
    kc = g.k_cache if h_kv == 1 else torch.cat([g.k_cache] * h_kv, dim=2).contiguous()
    with pytest.raises(_lib.MLAError) as e:
        api.mla_decode_fwd_dims(g.q, kc, g.block_table, g.cache_seqlens, w.softmax_scale, False,
                                meta, ns, dv)
    assert e.value.code == _lib.MLA_ERR_UNSUPPORTED
