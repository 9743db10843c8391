"""Pins for the oracle's restatement of the tile scheduler (FlashMLA deep
dive, section "Tile Scheduler"): hand-worked plans from the page's payload
formula, and the invariants any valid plan must keep.  CPU only."""
import numpy as np
import pytest

import oracle

BEGIN_REQ, END_REQ, BEGIN_BLOCK, END_BLOCK, BEGIN_SPLIT, FIRST_SPLIT, LAST_SPLIT, PAD = range(8)


def check_plan_invariants(seqlens, parts, num_splits, num_parts, c, page=64):
    """Every block of every request is covered exactly once, in order; parts
    are contiguous; all but the last part stay within the payload cap;
    num_splits is the prefix sum of pieces; split indices line up."""
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
            assert next_req == b
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
        if p < num_parts - 1:
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
    """seqlens [100, 200, 300, 0], 2 parts, c = 1: blocks [2, 4, 5, 0];
    total = 3 + 5 + 6 + 1 = 15; payload = ceil(15/2) + 1 = 9.
    Part 0 takes request 0 (cost 3, 6 left) and request 1 (cost 5, 1 left);
    request 2 costs 6 > 1 and 1 <= c, so part 0 closes.  Part 1, the last,
    takes requests 2 and 3."""
    parts, ns = oracle.plan([100, 200, 300, 0], 2, 1)
    assert parts.tolist() == [[0, 1, 0, 4, 0, 0, 0, 0], [2, 3, 0, 0, 2, 0, 0, 0]]
    assert ns.tolist() == [0, 1, 2, 3, 4]


def test_hand_worked_split():
    """seqlens [640, 64], 2 parts, c = 1: blocks [10, 1]; total = 11 + 2 = 13;
    payload = ceil(13/2) + 1 = 8.  Request 0 costs 11 > 8, so part 0 takes
    8 - 1 = 7 of its blocks; part 1 takes blocks 7..10 of request 0 and all of
    request 1.  Request 0 has two pieces: indices 0 and 1."""
    parts, ns = oracle.plan([640, 64], 2, 1)
    assert parts.tolist() == [[0, 0, 0, 7, 0, 1, 1, 0], [0, 1, 7, 1, 1, 1, 0, 0]]
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
    c = int(rng.integers(0, 8))
    parts, ns = oracle.plan(seqlens, num_parts, c)
    check_plan_invariants(seqlens, parts, ns, num_parts, c)


def test_balance_on_uniform_lengths():
    """Equal requests over many parts: no part exceeds the cap, and the work
    is spread so that the busiest part carries at most payload units."""
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
    assert max(costs[:-1]) <= payload
