"""Decode over an FP8-layout cache ("[DeepSeek-3] FlashMLA", sec. 12: 656-byte
rows of e4m3 latent values, fp32 scales and bf16 RoPE, dequantised to bf16) on
the GPU against the fp64 oracle (dense decode over the dequantised rows),
element by element, on both kernels that read it (the single-CTA one and the
one that keeps Q in tensor memory).  Tolerances: |out - ref| <= 1e-2 + 1e-2 |ref|,
|lse - ref| <= 1e-3."""
import numpy as np
import pytest
import torch

import oracle
from decode_attention_paged_gb300 import _lib
from decode_attention_paged_gb300 import workloads as W
from tests._helpers import NTHREADS, assert_close, gather_units, sample_units

pytestmark = pytest.mark.gpu

CASES = [
    # (b, s_q, h_q, seqlens, causal): one tile and P per page; several tiles
    # and the P buffer; ragged tails, splits, empty requests, causal rows
    (2, 1, 16, [1, 6000], False),
    (3, 2, 64, [0, 130, 4097], True),
    (1, 1, 128, [20000], False),
    (4, 1, 16, [63, 64, 65, 1], False),
    (128, 1, 16, [512] * 128, False),
    (2, 1, 1, [700, 64], False),
]


def run_fp8(w, expect_code=0):
    from decode_attention_paged_gb300 import api

    g = w.to("cuda")
    meta, ns = api.mla_get_metadata(g.cache_seqlens, w.h_q, w.s_q)
    out, lse = api.mla_decode_fp8_fwd(g.q, g.k_cache, g.block_table, g.cache_seqlens,
                                      w.softmax_scale, w.causal, meta, ns)
    code = api.mla_last_device_error()
    assert code == expect_code, f"device error {code}"
    return out, lse


def ref_fp8(w):
    return oracle.mla_decode_fp8(oracle.bf16_bits(w.q), w.k_cache, w.block_table.numpy(),
                                 w.cache_seqlens.numpy(), w.softmax_scale, w.causal,
                                 nthreads=NTHREADS)


@pytest.fixture
def kernel_kind(request):
    from decode_attention_paged_gb300 import api

    default = api.get_decode_kernel()
    api.set_decode_kernel(request.param)
    yield request.param
    api.set_decode_kernel(default)


@pytest.mark.parametrize("kernel_kind", [3, 1, 2], indirect=True, ids=["auto", "single", "tq"])
@pytest.mark.parametrize("case", CASES, ids=[str(i) for i in range(len(CASES))])
def test_fp8_parity(kernel_kind, case):
    b, s_q, h_q, seqlens, causal = case
    w = W.as_fp8(W.random_case(800 + CASES.index(case), b, s_q, h_q, seqlens, causal))
    out, lse = run_fp8(w)
    ref_out, ref_lse = ref_fp8(w)
    assert_close(out, lse, ref_out, ref_lse, f"fp8 {case}")


def test_fp8_tail_rows_never_reach_the_result():
    """Rows past a sequence's length in its last page hold NaN scales and
    NaN codes; unreferenced pages too."""
    w = W.as_fp8(W.random_case(820, 3, 1, 32, [70, 130, 5], False))
    kc = w.k_cache.clone()
    used = set()
    for i, L in enumerate(w.cache_seqlens.tolist()):
        nb = (L + 63) // 64
        for j in range(nb):
            used.add(int(w.block_table[i, j]))
        last = int(w.block_table[i, nb - 1])
        t0 = L - 64 * (nb - 1)
        kc[last, t0:, 0, :512] = 0x7F                        # e4m3 NaN
        kc[last, t0:, 0, 512:528] = torch.tensor([0xFF, 0xFF, 0xC0, 0x7F] * 4, dtype=torch.uint8)
    for pg in range(kc.shape[0]):
        if pg not in used:
            kc[pg] = 0xFF
    w2 = W.Fp8Workload(w.name, w.q, kc, w.block_table, w.cache_seqlens, w.softmax_scale, False)
    out, lse = run_fp8(w2)
    ref_out, ref_lse = ref_fp8(w)  # the clean cache: the tails must not matter
    assert_close(out, lse, ref_out, ref_lse, "fp8 NaN tails")


def test_fp8_matches_bf16_decode_of_the_dequantised_cache():
    """The FP8 kernel and the bf16 kernel fed the (torch-)dequantised cache agree."""
    from decode_attention_paged_gb300 import api

    w = W.as_fp8(W.random_case(821, 4, 2, 64, [300, 2000, 64, 1000], True))
    c8 = w.k_cache
    lat = c8[..., :512].contiguous().view(torch.float8_e4m3fn).double()
    sc = c8[..., 512:528].contiguous().view(torch.float32).double().repeat_interleave(128, -1)
    kc = torch.cat([(lat * sc).float().to(torch.bfloat16),
                    c8[..., 528:].contiguous().view(torch.bfloat16)], dim=-1)
    o8, l8 = run_fp8(w)
    g = w.to("cuda")
    meta, ns = api.mla_get_metadata(g.cache_seqlens, w.h_q, w.s_q)
    ob, lb = api.mla_decode_fwd(g.q, kc.cuda(), g.block_table, g.cache_seqlens, w.softmax_scale,
                                True, meta, ns)
    assert (o8.float() - ob.float()).abs().max().item() <= 2e-2
    assert (l8 - lb).abs().max().item() <= 1e-3


def test_fp8_memory_bound_full_size():
    """The memory-bound workload in the FP8 layout at full size, in the launch
    configuration the benchmark times; every element against the oracle."""
    w = W.memory_bound_fp8()
    out, lse = run_fp8(w)
    ro, rl = oracle.mla_decode_fp8(oracle.bf16_bits(w.q), w.k_cache, w.block_table.numpy(),
                                   w.cache_seqlens.numpy(), w.softmax_scale, False,
                                   nthreads=NTHREADS)
    assert_close(out, lse, ro, rl, "fp8 memory-bound")
