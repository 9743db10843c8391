"""Pins for the oracle's restatement of the tile scheduler (FlashMLA deep
dive, section "Tile Scheduler"): plans worked by hand from the page's payload
cap and greedy fill, the invariants any valid plan must keep, and the
property that makes a fill greedy (no closed part could have taken more).
CPU only."""
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


def check_greedy_fill(seqlens, parts, num_parts, c, page=64):
    """The page's fill is greedy, request by request, under the cap: a part
    is closed only when the next piece cannot go in.  So every non-empty part
    before the last one ends either mid-request with its cost exactly the
    payload (it took as many blocks as fit), or at a request boundary with
    less than c + 1 left (not one more block fits; a request without blocks,
    cost c, did not fit either); the non-empty parts come first."""
    seqlens = [max(0, int(x)) for x in seqlens]
    b = len(seqlens)
    n = [(L + page - 1) // page for L in seqlens]
    total = sum(x + c for x in n)
    payload = -(-total // num_parts) + c
    used = [p for p in range(num_parts) if parts[p][BEGIN_REQ] < b]
    assert used == list(range(len(used)))
    for p in used[:-1]:
        r = parts[p]
        cost = 0
        for i in range(r[BEGIN_REQ], r[END_REQ] + 1):
            b0 = r[BEGIN_BLOCK] if i == r[BEGIN_REQ] else 0
            b1 = r[END_BLOCK] if i == r[END_REQ] else n[i]
            cost += b1 - b0 + c
        left = payload - cost
        if r[END_BLOCK] < n[r[END_REQ]]:
            assert left == 0, (p, cost, payload)
        else:
            k = r[END_REQ] + 1
            assert k < b
            assert left <= c and n[k] + c > left, (p, left)


def test_hand_worked_no_split():
    """seqlens [100, 200, 300, 0], 2 parts, c = 1: blocks [2, 4, 5, 0], each
    request costing blocks + 1: total = 3 + 5 + 6 + 1 = 15, payload =
    ceil(15 / 2) + 1 = 9.  Part 0: request 0 (3) and request 1 (5) fit, 1
    left; request 2 (6) does not, and 1 - c = 0 blocks of it would, so the
    part closes.  Part 1: request 2 (6) and the empty request 3 (1)."""
    parts, ns = oracle.plan([100, 200, 300, 0], 2, 1)
    assert parts.tolist() == [[0, 1, 0, 4, 0, 0, 0, 0], [2, 3, 0, 0, 2, 0, 0, 0]]
    assert ns.tolist() == [0, 1, 2, 3, 4]


def test_hand_worked_split():
    """seqlens [640, 64], 2 parts, c = 1: blocks [10, 1]; total = 11 + 2 =
    13, payload = 7 + 1 = 8.  Part 0: request 0 (11) does not fit; it takes
    8 - 1 = 7 blocks (0..7).  Part 1: the rest of request 0 (3 blocks + the
    overhead paid again = 4) and request 1 (2).  Request 0 has two pieces."""
    parts, ns = oracle.plan([640, 64], 2, 1)
    assert parts.tolist() == [[0, 0, 0, 7, 0, 1, 1, 0], [0, 1, 7, 1, 1, 1, 0, 0]]
    assert ns.tolist() == [0, 2, 3]


def test_hand_worked_three_pieces():
    """seqlens [640], 3 parts, c = 2: 10 blocks; total 12, payload = 4 + 2 =
    6.  Every part pays the overhead again and takes 6 - 2 = 4 blocks until
    the rest (2 blocks + 2 = 4) fits: pieces 0..4, 4..8, 8..10."""
    parts, ns = oracle.plan([640], 3, 2)
    assert parts.tolist() == [[0, 0, 0, 4, 0, 1, 1, 0], [0, 0, 4, 8, 1, 1, 1, 0],
                              [0, 0, 8, 10, 2, 1, 1, 0]]
    assert ns.tolist() == [0, 3]


def test_hand_worked_split_then_whole():
    """seqlens [192, 192, 64], 2 parts, c = 2: blocks [3, 3, 1]; total =
    5 + 5 + 3 = 13, payload = 7 + 2 = 9.  Part 0: request 0 (5), 4 left;
    request 1 (5) does not fit, 4 - 2 = 2 blocks of it do: blocks 0..2.
    Part 1: the rest of request 1 (1 + 2 = 3) and request 2 (3)."""
    parts, ns = oracle.plan([192, 192, 64], 2, 2)
    assert parts.tolist() == [[0, 1, 0, 2, 0, 0, 1, 0], [1, 2, 2, 1, 2, 1, 0, 0]]
    assert ns.tolist() == [0, 1, 3, 4]


def test_hand_worked_waste_at_boundary():
    """seqlens [256, 64, 64], 3 parts, c = 2: blocks [4, 1, 1]; total =
    6 + 3 + 3 = 12, payload = 4 + 2 = 6.  Part 0: request 0 (6) fills it.
    Part 1: request 1 (3), 3 left; request 2 (3) fits: both.  Part 2 stays
    empty."""
    parts, ns = oracle.plan([256, 64, 64], 3, 2)
    assert parts.tolist() == [[0, 0, 0, 4, 0, 0, 0, 0], [1, 2, 0, 1, 1, 0, 0, 0],
                              [3, 2, 0, 0, 3, 0, 0, 0]]
    assert ns.tolist() == [0, 1, 2, 3]


def test_hand_worked_split_after_whole_request():
    """seqlens [128, 320], 2 parts, c = 3: blocks [2, 5]; total = 5 + 8 =
    13, payload = 7 + 3 = 10.  Part 0: request 0 (5), 5 left; request 1 (8)
    does not fit, 5 - 3 = 2 blocks do: blocks 0..2.  Part 1: the rest, 3 +
    3 = 6 (request 1's second piece, global index 2)."""
    parts, ns = oracle.plan([128, 320], 2, 3)
    assert parts.tolist() == [[0, 1, 0, 2, 0, 0, 1, 0], [1, 1, 2, 5, 2, 1, 1, 0]]
    assert ns.tolist() == [0, 1, 3]


def test_hand_worked_closes_before_request():
    """seqlens [384, 256], 2 parts, c = 2: blocks [6, 4]; total = 8 + 6 =
    14, payload = 7 + 2 = 9.  Part 0: request 0 (8), 1 left <= c: not one
    block of request 1 fits, the part closes at the boundary.  Part 1:
    request 1 (6)."""
    parts, ns = oracle.plan([384, 256], 2, 2)
    assert parts.tolist() == [[0, 0, 0, 6, 0, 0, 0, 0], [1, 1, 0, 4, 1, 0, 0, 0]]
    assert ns.tolist() == [0, 1, 2]


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
    check_greedy_fill(seqlens, parts, num_parts, c)


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


def test_tiny_share_fills_the_first_part():
    """One block, many parts: total 3, payload = 1 + 2 = 3; part 0 takes the
    request and every other part stays empty."""
    parts, ns = oracle.plan([64], 152, 2)
    check_plan_invariants([64], parts, ns, 152, 2)
    check_greedy_fill([64], parts, 152, 2)
    assert parts[0].tolist() == [0, 0, 0, 1, 0, 0, 0, 0]
    assert all(parts[p][0] == 1 for p in range(1, 152))
