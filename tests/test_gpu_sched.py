"""The device tile scheduler (mla_get_metadata) against the oracle's plan
(the page's greedy walk): integer for integer, plus the plan invariants and
the greedy-fill property."""
import numpy as np
import pytest
import torch

import oracle
from tests.test_plan_oracle import check_greedy_fill, check_plan_invariants

pytestmark = pytest.mark.gpu

HEADER = 8


def device_plan(seqlens, h_q, s_q):
    from decode_attention_paged_gb300 import api

    sl = torch.tensor(seqlens, dtype=torch.int32, device="cuda")
    meta, ns = api.mla_get_metadata(sl, h_q, s_q)
    torch.cuda.synchronize()
    meta = meta.cpu().numpy()
    num_parts = int(meta[3])  # the buffer has room for more records than the plan writes
    return meta[:HEADER], meta[HEADER:HEADER + 8 * num_parts].reshape(-1, 8), ns.cpu().numpy()


CASES = [
    ([256], 16, 1),
    ([4096] * 64, 16, 1),
    ([1, 64, 1000, 8191, 16384, 32768, 49152, 65536], 64, 1),
    ([4096] * 128, 128, 2),
    ([0, 0, 5, 0], 16, 1),
    (list(range(0, 3000, 37)), 20, 3),
    ([70000] * 3, 1, 1),
]


@pytest.mark.parametrize("seqlens,h_q,s_q", CASES)
def test_device_plan_equals_oracle(seqlens, h_q, s_q):
    hdr, parts, ns = device_plan(seqlens, h_q, s_q)
    R = s_q * h_q
    assert hdr[0] == 0x4D4C4131 and hdr[1] == len(seqlens) and hdr[2] == R
    num_parts, n_mtiles, fixed = int(hdr[3]), int(hdr[4]), int(hdr[5])
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    if R >= 128:
        # the default for 128-row tiles is the CTA-pair kernel: one part per
        # co-resident 2-CTA cluster and 128-row tile, at most one per SM pair
        assert n_mtiles == -(-R // 128)
        assert 1 <= num_parts <= max(1, (sms // 2) // n_mtiles)
        assert num_parts >= max(1, (sms // 2 - 8) // n_mtiles)
    else:
        # one CTA per SM: one SM part per SM and 64-row tile
        assert n_mtiles == -(-R // 64)
        assert num_parts == max(1, sms // n_mtiles)
    ref_parts, ref_ns = oracle.plan(seqlens, num_parts, fixed)
    assert np.array_equal(parts, ref_parts)
    assert np.array_equal(ns, ref_ns)
    assert hdr[7] == ns[-1]
    check_plan_invariants(seqlens, parts, ns, num_parts, fixed)
    check_greedy_fill(seqlens, parts, num_parts, fixed)


def test_random_seqlens_plans():
    rng = np.random.default_rng(5)
    for _ in range(20):
        b = int(rng.integers(1, 300))
        seqlens = rng.integers(0, 20000, size=b).tolist()
        h_q = int(rng.choice([1, 16, 64, 128]))
        s_q = int(rng.choice([1, 2]))
        hdr, parts, ns = device_plan(seqlens, h_q, s_q)
        ref_parts, ref_ns = oracle.plan(seqlens, int(hdr[3]), int(hdr[5]))
        assert np.array_equal(parts, ref_parts) and np.array_equal(ns, ref_ns)
        check_greedy_fill(seqlens, parts, int(hdr[3]), int(hdr[5]))


@pytest.mark.parametrize("fixed", [1, 3, 9, 64])
def test_fixed_overhead_and_many_requests(fixed):
    """Many short requests (more requests than parts, parts closing at
    boundaries and mid-request) under several overheads."""
    from decode_attention_paged_gb300 import api

    rng = np.random.default_rng(40 + fixed)
    seqlens = rng.integers(0, 700, size=2000).tolist()
    api.set_fixed_overhead(fixed)
    try:
        hdr, parts, ns = device_plan(seqlens, 16, 1)
    finally:
        api.set_fixed_overhead(-1)
    assert int(hdr[5]) == fixed
    ref_parts, ref_ns = oracle.plan(seqlens, int(hdr[3]), fixed)
    assert np.array_equal(parts, ref_parts) and np.array_equal(ns, ref_ns)
    check_plan_invariants(seqlens, parts, ns, int(hdr[3]), fixed)
    check_greedy_fill(seqlens, parts, int(hdr[3]), fixed)


def test_default_overhead_follows_the_kernel():
    """With no overhead set, the plan charges each kernel's measured boundary
    cost: 4 blocks for tiles the tensor-memory-Q kernel runs (s_q*h_q <= 32),
    5 for the CTA-pair kernel (>= 128 rows), 2 for the single-CTA kernel."""
    from decode_attention_paged_gb300 import api

    api.set_fixed_overhead(-1)
    assert int(device_plan([4096] * 4, 16, 1)[0][5]) == 4
    assert int(device_plan([4096] * 4, 64, 1)[0][5]) == 2
    default = api.get_decode_kernel()
    try:
        api.set_decode_kernel(api.KERNEL_SINGLE)
        assert int(device_plan([4096] * 4, 128, 1)[0][5]) == 2
    finally:
        api.set_decode_kernel(default)
    hdr = device_plan([4096] * 4, 128, 1)[0]
    # one 128-row tile: the CTA-pair kernel (two 64-row tiles if its clusters
    # cannot be resident and the single-CTA kernel runs instead)
    assert int(hdr[5]) == (5 if int(hdr[4]) == 1 else 2)


def test_metadata_has_room_for_256_records():
    """Decode CTAs read their part record beside the header: every metadata
    buffer the library sizes holds the header and at least 256 records."""
    from decode_attention_paged_gb300 import api

    for shape in ((1, 16, 1, 1), (64, 128, 1, 1), (32, 64, 1, 4), (128, 128, 2, 1)):
        mb, _ = api.metadata_size(*shape)
        assert mb >= 4 * (8 + 8 * 256)
        mbs, _ = api.metadata_size_sparse(shape[0], shape[1], shape[2])
        assert mbs >= 4 * (8 + 8 * 256)
