"""CUDA-graph capture of the decode step (Overview sec. 5: one plan per decode
step, reused by every layer; the calls allocate nothing and never
synchronise, so they can be captured).  A captured step is replayed after the
inputs were rewritten in place, and compared with the fp64 oracle on the new
inputs.  Tolerances: |out - ref| <= 1e-2 + 1e-2 |ref|, |lse - ref| <= 1e-3."""
import pytest
import torch

import oracle
from decode_attention_paged_gb300 import workloads as W
from tests._helpers import NTHREADS, assert_close, problem, sparse_problem

pytestmark = pytest.mark.gpu


def _capture(fn):
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        fn()  # warm-up outside the capture (library state, allocator)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fn()
    torch.cuda.synchronize()
    return g


def test_graph_replays_plan_and_decode_on_new_inputs():
    """Plan and decode both inside the graph: new seqlens, q and cache
    contents written in place between replays change the result accordingly."""
    from decode_attention_paged_gb300 import api

    b, s_q, h_q = 4, 2, 32
    w0 = W.random_case(700, b, s_q, h_q, [300, 1, 4000, 64], True)
    w1 = W.random_case(701, b, s_q, h_q, [3000, 70, 5, 4100], True)
    pages = max(w0.k_cache.shape[0], w1.k_cache.shape[0])
    mb = max(w0.block_table.shape[1], w1.block_table.shape[1])

    def pad(w):
        kc = torch.zeros(pages, 64, 1, 576, dtype=torch.bfloat16)
        kc[: w.k_cache.shape[0]] = w.k_cache
        bt = torch.zeros(b, mb, dtype=torch.int32)
        bt[:, : w.block_table.shape[1]] = w.block_table
        return W.Workload(w.name, w.q, kc, bt, w.cache_seqlens, w.softmax_scale, w.causal)

    w0, w1 = pad(w0), pad(w1)
    g = w0.to("cuda")
    meta, ns = api.mla_get_metadata(g.cache_seqlens, h_q, s_q)
    call = api.DecodeCall(g.q, g.k_cache, g.block_table, g.cache_seqlens, w0.softmax_scale,
                          True, meta, ns)

    def step():
        api.mla_get_metadata(g.cache_seqlens, h_q, s_q, meta=meta, num_splits=ns)
        call.fwd()

    graph = _capture(step)
    for w in (w0, w1, w0):
        g.q.copy_(w.q)
        g.k_cache.copy_(w.k_cache)
        g.block_table.copy_(w.block_table)
        g.cache_seqlens.copy_(w.cache_seqlens)
        graph.replay()
        torch.cuda.synchronize()
        assert api.mla_last_device_error() == 0
        ref_out, ref_lse = oracle.mla_decode(problem(w), nthreads=NTHREADS)
        assert_close(call.out, call.lse, ref_out, ref_lse, f"graph replay {w.name}")


def test_graph_reuses_one_plan_across_layers():
    """Several decode calls (layers) in one graph share one plan built in the
    same graph, as the plan is meant to be used."""
    from decode_attention_paged_gb300 import api

    b, s_q, h_q, layers = 3, 1, 64, 3
    ws = [W.random_case(710 + k, b, s_q, h_q, [900, 2500, 40], False) for k in range(layers)]
    gs = [w.to("cuda") for w in ws]
    meta, ns = api.mla_get_metadata(gs[0].cache_seqlens, h_q, s_q)
    calls = [api.DecodeCall(g.q, g.k_cache, gs[0].block_table, gs[0].cache_seqlens,
                            ws[0].softmax_scale, False, meta, ns) for g in gs]

    def step():
        api.mla_get_metadata(gs[0].cache_seqlens, h_q, s_q, meta=meta, num_splits=ns)
        for c in calls:
            c.fwd()

    graph = _capture(step)
    graph.replay()
    torch.cuda.synchronize()
    assert api.mla_last_device_error() == 0
    for k, w in enumerate(ws):
        wl = W.Workload(w.name, w.q, w.k_cache, ws[0].block_table, ws[0].cache_seqlens,
                        w.softmax_scale, False)
        ref_out, ref_lse = oracle.mla_decode(problem(wl), nthreads=NTHREADS)
        assert_close(calls[k].out, calls[k].lse, ref_out, ref_lse, f"layer {k}")


def test_graph_sparse_decode_on_new_indices():
    from decode_attention_paged_gb300 import api

    w0 = W.random_sparse_case(720, 2, 2, 64, 300, 500, 0.1)
    w1 = W.random_sparse_case(721, 2, 2, 64, 300, 500, 0.3)
    g = w0.to("cuda")
    meta, ns = api.mla_get_metadata_sparse(w0.topk, w0.b, w0.h_q, w0.s_q)
    call = api.SparseDecodeCall(g.q, g.k_cache, g.indices, w0.softmax_scale, meta, ns)
    graph = _capture(call.fwd)
    for w in (w1, w0):
        g.q.copy_(w.q)
        g.k_cache.copy_(w.k_cache)
        g.indices.copy_(w.indices)
        graph.replay()
        torch.cuda.synchronize()
        assert api.mla_last_device_error() == 0
        ref_out, ref_lse = oracle.mla_sparse(sparse_problem(w), nthreads=NTHREADS)
        assert_close(call.out, call.lse, ref_out, ref_lse, f"sparse graph {w.name}")
