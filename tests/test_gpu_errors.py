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


def _timeout_then_recover(run, check):
    """Run once with a 1 ns wait budget (expect a recorded timeout and a clean
    return), then with the default budget (expect the oracle's result)."""
    from decode_attention_paged_gb300 import api

    assert api.mla_last_device_error() == 0
    api.set_wait_budget_ns(1)
    try:
        run()
        code = api.mla_last_device_error()
    finally:
        api.set_wait_budget_ns(0)
    assert code == _lib.MLA_ERR_DEVICE_TIMEOUT, f"expected a timeout, got {code}"
    out, lse = run()
    assert api.mla_last_device_error() == 0
    check(out, lse)


@pytest.mark.parametrize("kind,h_q", [(2, 16), (1, 64), (1, 128), (4, 128), (4, 256)],
                         ids=["tq", "single-stageP", "single-Pbuffer", "duo", "duo-2tiles"])
def test_every_dense_kernel_unwinds_on_timeout(kind, h_q):
    from decode_attention_paged_gb300 import api

    w = W.random_case(24, 2, 1, h_q, [3000, 700], False)
    g = w.to("cuda")
    default = api.get_decode_kernel()
    try:
        api.set_decode_kernel(kind)
        meta, ns = api.mla_get_metadata(g.cache_seqlens, h_q, 1)
        ro, rl = oracle.mla_decode(problem(w))
        _timeout_then_recover(lambda: _call(g, w, meta, ns),
                              lambda o, l: assert_close(o, l, ro, rl, f"kernel {kind}"))
    finally:
        api.set_decode_kernel(default)


@pytest.mark.parametrize("h_q", [64, 128])
def test_sparse_gather_warps_unwind_on_timeout(h_q):
    from decode_attention_paged_gb300 import api
    from tests._helpers import sparse_problem

    w = W.random_sparse_case(25, 2, 2, h_q, 700, 1500, 0.1)
    g = w.to("cuda")
    meta, ns = api.mla_get_metadata_sparse(w.topk, w.b, w.h_q, w.s_q)
    ro, rl = oracle.mla_sparse(sparse_problem(w))

    def run():
        return api.mla_decode_sparse_fwd(g.q, g.k_cache, g.indices, w.softmax_scale, meta, ns)

    _timeout_then_recover(run, lambda o, l: assert_close(o, l, ro, rl, "sparse"))


@pytest.mark.parametrize("h_q", [16, 128])
def test_fp8_dequant_warps_unwind_on_timeout(h_q):
    from decode_attention_paged_gb300 import api

    w = W.as_fp8(W.random_case(26, 2, 1, h_q, [3000, 700], False))
    g = w.to("cuda")
    meta, ns = api.mla_get_metadata(g.cache_seqlens, h_q, 1)
    ro, rl = oracle.mla_decode_fp8(oracle.bf16_bits(w.q), w.k_cache, w.block_table.numpy(),
                                   w.cache_seqlens.numpy(), w.softmax_scale, False)

    def run():
        return api.mla_decode_fp8_fwd(g.q, g.k_cache, g.block_table, g.cache_seqlens,
                                      w.softmax_scale, False, meta, ns)

    _timeout_then_recover(run, lambda o, l: assert_close(o, l, ro, rl, "fp8"))


def test_cache_head_kernel_unwinds_on_timeout():
    from decode_attention_paged_gb300 import api

    g_ = torch.Generator().manual_seed(27)
    b, s_q, h_q, h_kv, seqlens = 2, 2, 32, 4, [2000, 300]
    pages = b * 32 + 2
    q = torch.randn(b, s_q, h_q, 576, generator=g_).to(torch.bfloat16)
    kv = torch.randn(pages, 64, h_kv, 576, generator=g_).to(torch.bfloat16)
    bt = torch.randperm(pages, generator=g_)[: b * 32].view(b, 32).to(torch.int32)
    sl = torch.tensor(seqlens, dtype=torch.int32)
    qd, kvd, btd, sld = q.cuda(), kv.cuda(), bt.cuda(), sl.cuda()
    meta, ns = api.mla_get_metadata(sld, h_q, s_q, h_kv)
    ro, rl = oracle.mla_decode_gqa(oracle.bf16_bits(q), oracle.bf16_bits(kv), bt.numpy(),
                                   sl.numpy(), W.SCALE, True)

    def run():
        return api.mla_decode_fwd(qd, kvd, btd, sld, W.SCALE, True, meta, ns)

    _timeout_then_recover(run, lambda o, l: assert_close(o, l, ro, rl, "heads"))
