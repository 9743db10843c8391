"""Shared helpers for the GPU parity tests: run the CUDA path through the C ABI
binding, run the oracle, compare element by element within the stated
tolerances (out: 1e-2 absolute + 1e-2 relative; lse: 1e-3 absolute, -inf
exactly where the oracle has -inf)."""
import os

import numpy as np
import torch

import oracle
from decode_attention_paged_gb300 import workloads as W

OUT_ATOL = 1e-2
OUT_RTOL = 1e-2
LSE_ATOL = 1e-3
NTHREADS = max(1, min(16, os.cpu_count() or 1))


def problem(w: W.Workload) -> oracle.Problem:
    return oracle.Problem(oracle.bf16_bits(w.q), oracle.bf16_bits(w.k_cache),
                          w.block_table.numpy(), w.cache_seqlens.numpy(), w.softmax_scale,
                          w.causal)


def run_gpu(w: W.Workload, k_cache_gpu=None):
    from decode_attention_paged_gb300 import api

    g = w.to("cuda")
    kc = k_cache_gpu if k_cache_gpu is not None else g.k_cache
    meta, ns = api.mla_get_metadata(g.cache_seqlens, w.h_q, w.s_q)
    out, lse = api.mla_decode_fwd(g.q, kc, g.block_table, g.cache_seqlens, w.softmax_scale,
                                  w.causal, meta, ns)
    code = api.mla_last_device_error()
    assert code == 0, f"device error code {code}"
    return out, lse, meta, ns


def assert_close(got_out, got_lse, ref_out, ref_lse, what=""):
    """got_* are torch tensors (any device) or arrays; ref_* fp64 arrays of the same shape."""
    go = got_out.double().cpu().numpy() if torch.is_tensor(got_out) else np.asarray(got_out, np.float64)
    gl = got_lse.double().cpu().numpy() if torch.is_tensor(got_lse) else np.asarray(got_lse, np.float64)
    assert go.shape == ref_out.shape and gl.shape == ref_lse.shape
    assert np.all(np.isfinite(go)), f"{what}: non-finite out"
    excess = np.abs(go - ref_out) - (OUT_ATOL + OUT_RTOL * np.abs(ref_out))
    if excess.max() > 0:
        idx = np.unravel_index(np.argmax(excess), excess.shape)
        raise AssertionError(f"{what}: out mismatch at {idx}: got {go[idx]} ref {ref_out[idx]}")
    fin = np.isfinite(ref_lse)
    assert np.array_equal(fin, np.isfinite(gl)), f"{what}: lse finiteness differs"
    assert np.all(np.isneginf(gl[~fin])), f"{what}: empty rows must have lse = -inf"
    if fin.any():
        err = np.abs(gl[fin] - ref_lse[fin]).max()
        assert err <= LSE_ATOL, f"{what}: lse err {err}"
    return float(np.abs(go - ref_out).max()), float(np.abs(gl[fin] - ref_lse[fin]).max()) if fin.any() else 0.0


def sample_units(w: W.Workload, n: int, seed: int):
    """Sampled (request, row) units: random ones plus the first/last rows of the
    first/last/longest requests."""
    R = w.s_q * w.h_q
    rng = np.random.default_rng(seed)
    units = set()
    L = w.cache_seqlens.numpy()
    for i in {0, w.b - 1, int(np.argmax(L)), int(np.argmin(L))}:
        for rho in {0, R - 1, R // 2, min(R - 1, 63), min(R - 1, 64)}:
            units.add((i, rho))
    n = min(n, w.b * R)  # there are only b * R distinct units
    while len(units) < n:
        units.add((int(rng.integers(0, w.b)), int(rng.integers(0, R))))
    return np.array(sorted(units), dtype=np.int32)


def gather_units(out, lse, units, h_q):
    """Pick rows (request, rho = s*h_q + h) out of full GPU outputs."""
    o = out.double().cpu().numpy()
    l = lse.double().cpu().numpy()
    go = np.stack([o[i, rho // h_q, rho % h_q] for i, rho in units])
    gl = np.array([l[i, rho % h_q, rho // h_q] for i, rho in units])
    return go, gl


def sparse_problem(w) -> oracle.SparseProblem:
    return oracle.SparseProblem(oracle.bf16_bits(w.q), oracle.bf16_bits(w.k_cache),
                                w.indices.numpy(), w.softmax_scale)


def run_gpu_sparse(w, expect_code: int = 0):
    """Sparse decode of a SparseWorkload through the C ABI; checks the device
    error word against expect_code."""
    from decode_attention_paged_gb300 import api

    g = w.to("cuda")
    meta, ns = api.mla_get_metadata_sparse(w.topk, w.b, w.h_q, w.s_q)
    out, lse = api.mla_decode_sparse_fwd(g.q, g.k_cache, g.indices, w.softmax_scale, meta, ns)
    code = api.mla_last_device_error()
    assert code == expect_code, f"device error code {code}, expected {expect_code}"
    return out, lse
