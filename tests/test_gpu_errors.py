"""Device-side error reporting, exercised without faulting the GPU: metadata
built for another shape, and pipeline waits that run out of their (tiny)
budget.  In both cases the kernels return cleanly, the error word says why, and
the next correct call still works."""
import pytest
import torch

import oracle
from decode_attention_paged_gb300 import _lib
from decode_attention_paged_gb300 import workloads as W
from tests._helpers import assert_close, problem

pytestmark = pytest.mark.gpu


def _call(g, w, meta, ns):
    from decode_attention_paged_gb300 import api

    return api.mla_decode_fwd(g.q, g.k_cache, g.block_table, g.cache_seqlens, w.softmax_scale,
                              w.causal, meta, ns)


def test_metadata_for_another_batch_is_detected():
    from decode_attention_paged_gb300 import api

    w = W.random_case(20, 3, 1, 16, [100, 200, 300], False)
    g = w.to("cuda")
    assert api.mla_last_device_error() == 0
    meta2, ns2 = api.mla_get_metadata(g.cache_seqlens[:2].contiguous(), 16, 1)
    _call(g, w, meta2, ns2)
    assert api.mla_last_device_error() == _lib.MLA_ERR_METADATA_MISMATCH
    meta, ns = api.mla_get_metadata(g.cache_seqlens, 16, 1)
    out, lse = _call(g, w, meta, ns)
    assert api.mla_last_device_error() == 0
    ro, rl = oracle.mla_decode(problem(w))
    assert_close(out, lse, ro, rl, "after mismatch")


def test_sequence_longer_than_block_table_is_reported():
    from decode_attention_paged_gb300 import api

    w = W.random_case(21, 2, 1, 16, [64, 100], False)
    g = w.to("cuda")
    bad = g.cache_seqlens.clone()
    bad[1] = 64 * w.block_table.shape[1] + 1
    meta, ns = api.mla_get_metadata(bad, 16, 1)
    api.mla_decode_fwd(g.q, g.k_cache, g.block_table, bad, w.softmax_scale, False, meta, ns)
    assert api.mla_last_device_error() == _lib.MLA_ERR_SEQ_TOO_LONG


def test_wait_budget_exhaustion_returns_cleanly():
    """A 1 ns wait budget makes the first pipeline wait that is not already
    satisfied give up: the CTA records a timeout, drains its own copies and
    MMAs, frees tensor memory and exits.  The context stays usable."""
    from decode_attention_paged_gb300 import api

    w = W.random_case(22, 2, 1, 64, [5000, 3000], False)
    g = w.to("cuda")
    meta, ns = api.mla_get_metadata(g.cache_seqlens, 64, 1)
    assert api.mla_last_device_error() == 0
    api.set_wait_budget_ns(1)
    try:
        _call(g, w, meta, ns)
        code = api.mla_last_device_error()
    finally:
        api.set_wait_budget_ns(0)
    assert code in (_lib.MLA_ERR_DEVICE_TIMEOUT, 0)
    assert code == _lib.MLA_ERR_DEVICE_TIMEOUT, "expected the tiny budget to run out"
    out, lse = _call(g, w, meta, ns)
    assert api.mla_last_device_error() == 0
    ro, rl = oracle.mla_decode(problem(w))
    assert_close(out, lse, ro, rl, "after timeout")


def test_host_rejects_bad_arguments_without_launching():
    from decode_attention_paged_gb300 import api

    w = W.random_case(23, 1, 1, 16, [64], False)
    g = w.to("cuda")
    meta, ns = api.mla_get_metadata(g.cache_seqlens, 16, 1)
    small_ws = torch.empty(16, dtype=torch.uint8, device="cuda")
    with pytest.raises(_lib.MLAError) as e:
        api.mla_decode_fwd(g.q, g.k_cache, g.block_table, g.cache_seqlens, w.softmax_scale, False,
                           meta, ns, workspace=small_ws)
    assert e.value.code == _lib.MLA_ERR_WORKSPACE_TOO_SMALL
    assert api.mla_last_device_error() == 0
