"""Pins for the oracle's restatement of the tile scheduler (FlashMLA deep
dive, section "Tile Scheduler"): hand-worked plans from the page's payload
formula, and the invariants any valid plan must keep.  CPU only."""
import numpy as np
import pytest

import oracle

BEGIN_REQ, END_REQ, BEGIN_BLOCK, END_BLOCK, BEGIN_SPLIT, FIRST_SPLIT, LAST_SPLIT, PAD = range(8)


def check_plan_invariants(seqlens, parts, num_splits, num_parts, c, page=64):
    """Every block of every request is covered exactly once, in order; the
    non-empty parts follow one another without gaps; no part exceeds the cap
    payload = ceil(total / parts) + c; num_splits is the prefix sum of pieces;
    split indices and flags line up."""
    seqlens = [max(0, int(x)) for x in seqlens]
    b = len(seqlens)
    n = [(L + page - 1) // page for L in seqlens]
    total = sum(x + c for x in n)
    payload = -(-total // num_parts) + c
    covered = [[] for _ in range(b)]
    piece_of = {}
    next_req, next_block = 0, 0
    for p in range(num_parts):
        r = parts[p]
        if r[BEGIN_REQ] >= b:
            assert r[END_REQ] == b - 1 and r[BEGIN_BLOCK] == 0 and r[END_BLOCK] == 0
            continue
        assert (r[BEGIN_REQ], r[BEGIN_BLOCK]) == (next_req, next_block)
        cost = 0
        for i in range(r[BEGIN_REQ], r[END_REQ] + 1):
            b0 = r[BEGIN_BLOCK] if i == r[BEGIN_REQ] else 0
            b1 = r[END_BLOCK] if i == r[END_REQ] else n[i]
            assert 0 <= b0 <= b1 <= n[i]
            covered[i].append((b0, b1))
            piece_of[(p, i)] = len(covered[i]) - 1
            cost += b1 - b0 + c
        assert cost <= payload
        if r[END_BLOCK] == n[r[END_REQ]]:
            next_req, next_block = r[END_REQ] + 1, 0
        else:
            next_req, next_block = r[END_REQ], r[END_BLOCK]
    assert next_req == b
    for i in range(b):
        pieces = covered[i]
        assert len(pieces) >= 1
        assert pieces[0][0] == 0 and pieces[-1][1] == n[i]
        for (a0, a1), (b0_, _) in zip(pieces, pieces[1:]):
            assert a1 == b0_
        if len(pieces) > 1:
            assert all(a1 > a0 for a0, a1 in pieces)  # a split never makes an empty piece
    assert num_splits[0] == 0
    for i in range(b):
        assert num_splits[i + 1] - num_splits[i] == len(covered[i])
    for p in range(num_parts):
        r = parts[p]
        if r[BEGIN_REQ] >= b:
            assert r[BEGIN_SPLIT] == num_splits[b]
            continue
        br, er = r[BEGIN_REQ], r[END_REQ]
        assert r[BEGIN_SPLIT] == num_splits[br] + piece_of[(p, br)]
        assert r[FIRST_SPLIT] == int(len(covered[br]) > 1)
        assert r[LAST_SPLIT] == int(len(covered[er]) > 1)
        assert r[PAD] == 0


def test_hand_worked_no_split():
    """seqlens [100, 200, 300, 0], 2 parts, c = 1: blocks [2, 4, 5, 0].
    Cost line: request 0 = units 0..2 (overhead 0, blocks 1..2), request 1 =
    3..7 (blocks 4..7), request 2 = 8..13 (blocks 9..13), request 3 = unit 14;
    total 15, q = ceil(15/2) = 8.  Part 0 = units [0, 8): all blocks of
    requests 0 and 1.  Part 1 = [8, 15): request 2 and the empty request 3."""
    parts, ns = oracle.plan([100, 200, 300, 0], 2, 1)
    assert parts.tolist() == [[0, 1, 0, 4, 0, 0, 0, 0], [2, 3, 0, 0, 2, 0, 0, 0]]
    assert ns.tolist() == [0, 1, 2, 3, 4]


def test_hand_worked_split():
    """seqlens [640, 64], 2 parts, c = 1: blocks [10, 1].  Request 0 = units
    0..10 (blocks at 1..10), request 1 = 11..12 (block at 12); total 13,
    q = 7.  Part 0 = [0, 7): blocks 0..5 of request 0.  Part 1 = [7, 13):
    blocks 6..9 of request 0 and block 0 of request 1.  Request 0 has two
    pieces (indices 0, 1); cost of part 0 = 6 + 1, of part 1 = 5 + 2, both
    <= payload = 7 + 1."""
    parts, ns = oracle.plan([640, 64], 2, 1)
    assert parts.tolist() == [[0, 0, 0, 6, 0, 1, 1, 0], [0, 1, 6, 1, 1, 1, 0, 0]]
    assert ns.tolist() == [0, 2, 3]


def test_more_parts_than_work():
    parts, ns = oracle.plan([64], 4, 5)
    check_plan_invariants([64], parts, ns, 4, 5)
    assert parts[1].tolist() == [1, 0, 0, 0, 1, 0, 0, 0]


@pytest.mark.parametrize("seed", range(12))
def test_random_plans_are_valid(seed):
    rng = np.random.default_rng(seed)
    b = int(rng.integers(1, 200))
    kind = seed % 3
    if kind == 0:
        seqlens = rng.integers(0, 9000, size=b)
    elif kind == 1:
        seqlens = np.full(b, int(rng.integers(1, 70000)))
    else:
        seqlens = (2.0 ** rng.uniform(0, 16.5, size=b)).astype(np.int64)
    num_parts = int(rng.choice([1, 2, 37, 38, 76, 152, 300]))
    c = int(rng.integers(1, 9))
    parts, ns = oracle.plan(seqlens, num_parts, c)
    check_plan_invariants(seqlens, parts, ns, num_parts, c)


def test_balance_on_uniform_lengths():
    """Equal requests over many parts: no part exceeds the cap."""
    seqlens = [4096] * 64
    parts, ns = oracle.plan(seqlens, 152, 2)
    check_plan_invariants(seqlens, parts, ns, 152, 2)
    costs = []
    for r in parts:
        if r[BEGIN_REQ] >= 64:
            costs.append(0)
            continue
        cost = 0
        for i in range(r[BEGIN_REQ], r[END_REQ] + 1):
            b0 = r[BEGIN_BLOCK] if i == r[BEGIN_REQ] else 0
            b1 = r[END_BLOCK] if i == r[END_REQ] else 64
            cost += b1 - b0 + 2
        costs.append(cost)
    payload = -(-(64 * 66) // 152) + 2
    assert max(costs) <= payload


def test_tiny_share_leaves_leading_parts_empty():
    """One block, many parts: q = 1, so the first parts cover only overhead
    units and stay empty; the block goes to the part holding its unit."""
    parts, ns = oracle.plan([64], 152, 2)
    check_plan_invariants([64], parts, ns, 152, 2)
    assert parts[2].tolist() == [0, 0, 0, 1, 0, 0, 0, 0]
    assert all(parts[p][0] == 1 for p in range(152) if p != 2)
