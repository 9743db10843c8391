"""Pins for the FP8 KV-cache oracle ("[DeepSeek-3] FlashMLA", sec. 12: 656-byte
rows of 512 e4m3 latent values, 4 fp32 scales and 64 bf16 RoPE values,
dequantised to bf16 before BF16 QK/PV).  CPU only.

The pins tie it to library routines and closed forms, not to itself:
- the e4m3 decoder equals torch's float8_e4m3fn conversion on all 256 codes;
- the bf16 rounding equals torch's float32 -> bfloat16 conversion (round to
  nearest even) on random, tie, subnormal and overflow inputs;
- the whole dequantisation equals a torch-only restatement (codes through
  torch's float8 type, the product in fp64, torch's bf16 rounding);
- power-of-two scales give products that bf16 holds exactly;
- FP8 decode equals the dense oracle over the torch-dequantised cache.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from decode_attention_paged_gb300 import workloads as W


def test_e4m3_decoder_matches_torch_on_every_code():
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).float().double().numpy()
    got = np.array([oracle.e4m3_value(c) for c in range(256)])
    nan = np.isnan(ref)
    assert np.array_equal(nan, np.isnan(got))
    assert nan.sum() == 2  # S.1111.111 only: the finite-only variant
    assert np.array_equal(got[~nan], ref[~nan])
    # closed forms: largest finite, smallest subnormal, one
    assert oracle.e4m3_value(0x7E) == 448.0
    assert oracle.e4m3_value(0x01) == 2.0 ** -9
    assert oracle.e4m3_value(0x38) == 1.0
    assert oracle.e4m3_value(0xB8) == -1.0


def _torch_bf16_bits(x32: np.ndarray) -> np.ndarray:
    t = torch.from_numpy(x32.astype(np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def test_bf16_rounding_matches_torch():
    rng = np.random.default_rng(0)
    # random finite fp32 bit patterns over the whole range
    bits = rng.integers(0, 2 ** 32, size=20000, dtype=np.uint64).astype(np.uint32)
    bits = bits[(bits & 0x7F800000) != 0x7F800000]
    # exact ties (low 16 bits = 0x8000), both parities, and subnormals
    ties = (rng.integers(0, 2 ** 16, size=2000, dtype=np.uint64).astype(np.uint32) << 16) | 0x8000
    ties = ties[(ties & 0x7F800000) != 0x7F800000]
    subn = rng.integers(1, 2 ** 23, size=2000, dtype=np.uint64).astype(np.uint32)
    allbits = np.concatenate([bits, ties, subn, subn | 0x80000000])
    x32 = allbits.view(np.float32)
    ref = _torch_bf16_bits(x32)
    got = np.array([oracle.bf16_round(float(v)) for v in x32], dtype=np.uint16)
    assert np.array_equal(got, ref)
    # overflow and signed zero
    assert oracle.bf16_round(3.5e38) == 0x7F80
    assert oracle.bf16_round(-3.5e38) == 0xFF80
    assert oracle.bf16_round(-0.0) == 0x8000
    assert oracle.bf16_round(1.0) == 0x3F80


def _random_fp8_rows(seed, n, general_scales):
    g = torch.Generator().manual_seed(seed)
    codes = torch.randint(0, 256, (n, 512), generator=g, dtype=torch.int32).to(torch.uint8)
    codes[(codes & 0x7F) == 0x7F] = 0x3F  # no NaN codes
    if general_scales:
        scales = (torch.rand(n, 4, generator=g) * 3 + 1e-3).to(torch.float32)
    else:
        scales = torch.ldexp(torch.ones(n, 4), torch.randint(-20, 20, (n, 4), generator=g))
    rope = torch.randn(n, 64, generator=g).to(torch.bfloat16)
    rows = torch.empty(n, 656, dtype=torch.uint8)
    rows[:, :512] = codes
    rows[:, 512:528] = scales.contiguous().view(torch.uint8)
    rows[:, 528:] = rope.contiguous().view(torch.uint8)
    return rows, codes, scales, rope


def test_power_of_two_scales_are_exact():
    rows, codes, scales, rope = _random_fp8_rows(1, 64, general_scales=False)
    got = oracle.fp8_dequant(rows.view(1, 64, 1, 656)).reshape(64, 576)
    vals = codes.view(torch.float8_e4m3fn).double() * scales.double().repeat_interleave(128, 1)
    ref = vals.float().to(torch.bfloat16)  # exact: 4 significant bits, no rounding
    assert torch.equal(ref.double(), vals)
    assert np.array_equal(got[:, :512], ref.view(torch.int16).numpy().view(np.uint16))
    assert np.array_equal(got[:, 512:], rope.view(torch.int16).numpy().view(np.uint16))


def test_dequant_matches_torch_restatement():
    """General scales: the product has up to 28 significant bits, exact in fp64;
    torch rounds it to fp32 first, so the two may differ by one bf16 step only
    at exact fp32 ties of the bf16 rounding."""
    rows, codes, scales, rope = _random_fp8_rows(2, 256, general_scales=True)
    got = oracle.fp8_dequant(rows.view(4, 64, 1, 656)).reshape(256, 576)
    prod = codes.view(torch.float8_e4m3fn).double() * scales.double().repeat_interleave(128, 1)
    ref = prod.float().to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    same = got[:, :512] == ref
    assert same.mean() > 0.999
    diff = np.abs(got[:, :512].astype(np.int32) - ref.astype(np.int32))
    assert diff.max() <= 1
    # the oracle is the exact rounding: check the differing ones against fp64
    for i, c in zip(*np.nonzero(~same)):
        x = float(prod[i, c])
        lo = torch.tensor([got[i, c]], dtype=torch.int16).view(torch.bfloat16).double().item()
        step = abs(lo - torch.tensor([ref[i, c]], dtype=torch.int16).view(torch.bfloat16).double().item())
        assert abs(x - lo) <= step / 2
    assert np.array_equal(got[:, 512:], rope.view(torch.int16).numpy().view(np.uint16))


@pytest.mark.parametrize("causal", [False, True])
def test_fp8_decode_is_dense_decode_over_the_dequantised_cache(causal):
    w = W.random_case(31, 3, 2, 16, [200, 64, 1], causal)
    c8 = W.fp8_cache(w.k_cache)
    # dequantised through torch only
    lat = c8[..., :512].contiguous().view(torch.float8_e4m3fn).double()
    sc = c8[..., 512:528].contiguous().view(torch.float32).double().repeat_interleave(128, -1)
    kc = torch.cat([(lat * sc).float().to(torch.bfloat16),
                    c8[..., 528:].contiguous().view(torch.bfloat16)], dim=-1)
    ref = oracle.mla_decode(oracle.Problem(oracle.bf16_bits(w.q), oracle.bf16_bits(kc),
                                           w.block_table.numpy(), w.cache_seqlens.numpy(),
                                           w.softmax_scale, causal), nthreads=4)
    got = oracle.mla_decode_fp8(oracle.bf16_bits(w.q), c8, w.block_table.numpy(),
                                w.cache_seqlens.numpy(), w.softmax_scale, causal, nthreads=4)
    # e4m3 codes times amax/448 scales: fp32 rounding of the product is the
    # only possible difference (one bf16 step, rarely); both lse within 1e-9
    np.testing.assert_allclose(got[1], ref[1], rtol=0, atol=1e-6)
    np.testing.assert_allclose(got[0], ref[0], rtol=1e-5, atol=1e-6)


def test_fp8_cache_rows_round_trip_the_rope_and_scale_layout():
    w = W.random_case(32, 1, 1, 16, [64], False)
    c8 = W.fp8_cache(w.k_cache)
    assert c8.shape[-1] == 656
    sc = c8[..., 512:528].contiguous().view(torch.float32)
    amax = w.k_cache[..., :512].float().reshape(*w.k_cache.shape[:-1], 4, 128).abs().amax(-1)
    assert torch.allclose(sc * 448.0, amax, rtol=1e-6)
    d = oracle.fp8_dequant(c8)
    assert np.array_equal(d[..., 512:], oracle.bf16_bits(w.k_cache)[..., 512:])
    # e4m3 keeps 4 significant bits: relative error <= 2^-4 of the tile's scale step
    x = torch.from_numpy(d[..., :512].astype(np.int16)).view(torch.bfloat16).float()
    err = (x - w.k_cache[..., :512].float()).abs()
    assert float(err.max()) <= float(amax.max()) / 448.0 * 16 + 1e-6
