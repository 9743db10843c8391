"""mla_decode_fwd_noalloc -- the decode entry point for callers that cannot
allocate device memory (a plugin whose host framework owns the whole memory
pool, a serving loop that forbids cudaMalloc because it can synchronise the
device, a process already at its memory limit).  It takes its split-KV scratch
from a fixed 32 MiB device array inside the library instead of a caller
workspace.

Checked here, through the C ABI: on two calls in a row (different inputs, so
the second call runs over scratch the first one left behind) its out / lse
match those of mla_decode_fwd within the parity tolerances, and both match the
fp64 oracle element by element; a problem whose scratch would exceed 32 MiB is
refused before anything runs.  This file is
collected last so a failure here never hides the other tests' results."""
import numpy as np
import pytest
import torch

import oracle
from decode_attention_paged_gb300 import _lib
from decode_attention_paged_gb300 import workloads as W
from tests._helpers import NTHREADS, assert_close, problem

pytestmark = pytest.mark.gpu


def test_noalloc_matches_fwd_on_two_calls_in_a_row():
    from decode_attention_paged_gb300 import api

    for seed in (31, 32):
        w = W.random_case(seed, 4, 2, 64, [3000, 10, 600, 1500], True)
        g = w.to("cuda")
        meta, ns = api.mla_get_metadata(g.cache_seqlens, w.h_q, w.s_q)
        ref_out, ref_lse = api.mla_decode_fwd(g.q, g.k_cache, g.block_table, g.cache_seqlens,
                                              w.softmax_scale, w.causal, meta, ns)
        out = torch.full_like(ref_out, float("nan"))
        lse = torch.full_like(ref_lse, float("nan"))
        api.mla_decode_fwd_noalloc(g.q, g.k_cache, g.block_table, g.cache_seqlens,
                                   w.softmax_scale, w.causal, meta, ns, out, lse)
        assert api.mla_last_device_error() == 0
        assert int(ns[-1]) > w.b, "the plan should split requests so the scratch is used"
        assert_close(out, lse, ref_out.double().cpu().numpy(), ref_lse.double().cpu().numpy(),
                     f"noalloc seed {seed} against mla_decode_fwd")
        o_out, o_lse = oracle.mla_decode(problem(w), nthreads=NTHREADS)
        assert_close(out, lse, o_out, o_lse, f"noalloc seed {seed} against the oracle")


def test_noalloc_refuses_problems_beyond_its_scratch():
    from decode_attention_paged_gb300 import api

    w = W.random_case(33, 300, 1, 128, [64] * 300, False)
    g = w.to("cuda")
    need = api.workspace_size(w.b, w.h_q, w.s_q)
    assert need > 32 * 1024 * 1024
    meta, ns = api.mla_get_metadata(g.cache_seqlens, w.h_q, w.s_q)
    out = torch.zeros(w.b, w.s_q, w.h_q, 512, dtype=torch.bfloat16, device="cuda")
    lse = torch.zeros(w.b, w.h_q, w.s_q, device="cuda")
    with pytest.raises(_lib.MLAError) as e:
        api.mla_decode_fwd_noalloc(g.q, g.k_cache, g.block_table, g.cache_seqlens,
                                   w.softmax_scale, False, meta, ns, out, lse)
    assert e.value.code == _lib.MLA_ERR_WORKSPACE_TOO_SMALL
    assert api.mla_last_device_error() == 0
    assert torch.all(out == 0) and torch.all(lse == 0)
