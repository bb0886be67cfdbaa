"""Pins of the schedule oracle (CPU only): the pages' printed orders, full coverage of
the mask, the pages' qualitative claims (conflict-free shift schedules, shorter critical
paths), and symmetric-shift balance."""
import os

import pytest

from oracle import schedule as sc

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def read_golden(name):
    rows = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            w, qs = line.split(":")
            rows[int(w)] = [int(x) for x in qs.split()]
    return rows


def test_shift_matches_pages_cyclic_example():
    gold = read_golden("shift_full_N4.txt")
    for u, qs in gold.items():
        assert [q for _, q in sc.visits(sc.SHIFT, False, 4, u)] == qs
        assert all(kv == u for kv, _ in sc.visits(sc.SHIFT, False, 4, u))


def test_descending_matches_pages_reversal():
    gold = read_golden("descending_full_N4.txt")
    for u, qs in gold.items():
        assert [q for _, q in sc.visits(sc.DESCENDING, False, 4, u)] == qs
    assert sc.reduction_order(sc.DESCENDING, False, 4) == sc.reduction_order(sc.SERIAL, False, 4)


CASES = [(s, c, n) for n in (1, 2, 3, 4, 5, 6, 7, 8, 9, 16, 17) for s, c in
         ((sc.SERIAL, False), (sc.SERIAL, True), (sc.DESCENDING, False), (sc.DESCENDING, True),
          (sc.SHIFT, False), (sc.SYMSHIFT, True))]


@pytest.mark.parametrize("sched,causal,N", CASES)
def test_every_allowed_tile_visited_once(sched, causal, N):
    seen = []
    for u in range(sc.num_workers(sched, causal, N)):
        seen += sc.visits(sched, causal, N, u)
    want = [(kv, q) for kv in range(N) for q in range(N) if sc.allowed(causal, q, kv)]
    assert sorted(seen) == sorted(want)
    order = sc.reduction_order(sched, causal, N)
    for q in range(N):
        assert sorted(order[q]) == [kv for kv in range(N) if sc.allowed(causal, q, kv)]


@pytest.mark.parametrize("sched,causal,N", CASES)
def test_conflict_freedom(sched, causal, N):
    """Shift schedules are conflict-free in lock step (section 2.2 B); the serialized
    orders are not (every worker wants the same tile at the same step; a single tile is
    trivially conflict-free)."""
    assert sc.conflict_free(sched, causal, N) == (sched in (sc.SHIFT, sc.SYMSHIFT) or N == 1)


@pytest.mark.parametrize("N", [2, 3, 4, 5, 8, 9, 16, 17])
def test_critical_paths(N):
    """Unit-step critical paths.  Serialized baseline: 2N-1 (the pipeline bubbles of
    section 1).  Descending helps causal masks only (section 2.2 A); Shift reaches the
    lower bound N for full masks; Symmetric Shift needs N+1 steps on ceil(N/2) workers
    (odd N: the padded schedule, its dropped steps closed up by the waits)."""
    assert sc.critical_path(sc.SERIAL, False, N) == 2 * N - 1
    assert sc.critical_path(sc.DESCENDING, False, N) == 2 * N - 1
    assert sc.critical_path(sc.SHIFT, False, N) == N
    assert sc.critical_path(sc.SERIAL, True, N) == 2 * N - 1
    assert sc.critical_path(sc.DESCENDING, True, N) == N
    assert sc.critical_path(sc.SYMSHIFT, True, N) == N + 1


@pytest.mark.parametrize("N", [2, 4, 8, 16, 32])
def test_symshift_balanced_and_one_block_at_a_time(N):
    """Folding the triangle into a square (section 2.2 B): every worker does N+1 tile
    steps, and finishes KV block c before it starts block N-1-c."""
    for c in range(N // 2):
        seq = sc.visits(sc.SYMSHIFT, True, N, c)
        assert len(seq) == N + 1
        kvs = [kv for kv, _ in seq]
        first_other = kvs.index(N - 1 - c)
        assert all(kv == c for kv in kvs[:first_other])
        assert all(kv == N - 1 - c for kv in kvs[first_other:])
        assert kvs[:N // 2] == [c] * (N // 2)
        assert all(q >= N // 2 for _, q in seq[:N // 2])      # phase 1: lower-left rectangle


@pytest.mark.parametrize("N", [1, 3, 5, 7, 9, 31])
def test_odd_symshift_balanced_and_one_block_at_a_time(N):
    """Odd N: (N+1)/2 workers of N steps each (N(N+1)/2 tiles in all); worker 0 runs block
    0 alone, worker c >= 1 finishes block c before it starts block N-c."""
    W = sc.num_workers(sc.SYMSHIFT, True, N)
    assert W == (N + 1) // 2
    for c in range(W):
        kvs = [kv for kv, _ in sc.visits(sc.SYMSHIFT, True, N, c)]
        assert len(kvs) == N
        if c == 0:
            assert kvs == [0] * N
        else:
            assert kvs == [c] * (N - c) + [N - c] * c


def test_odd_symshift_matches_hand_worked_example():
    gold = {}
    with open(os.path.join(GOLDEN, "symshift_causal_N5.txt")) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                w, rest = line.split(":")
                gold[int(w)] = [tuple(int(x) for x in p.split(",")) for p in rest.split()]
    assert set(gold) == {0, 1, 2}
    for c, pairs in gold.items():
        assert sc.visits(sc.SYMSHIFT, True, 5, c) == pairs
    order = sc.reduction_order(sc.SYMSHIFT, True, 5)
    # lock-step slots (padding steps idle): tile 4 gets kv 1, 0, 2 in phase 1, then 3, 4
    assert order[1] == [1, 0] and order[3] == [0, 2, 1, 3] and order[4] == [1, 0, 2, 3, 4]


def test_symshift_rejects_full():
    with pytest.raises(ValueError):
        sc.visits(sc.SYMSHIFT, False, 4, 0)


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("N,heads,P", [(8, 5, 12), (8, 3, 8), (16, 4, 24), (4, 9, 10), (32, 3, 38),
                                       (5, 4, 7), (9, 3, 10)])
def test_packed_shift_is_conflict_free_and_reduces_to_shift(causal, N, heads, P):
    sched = sc.SYMSHIFT if causal else sc.SHIFT
    order = sc.packed_reduction_order(sched, causal, N, heads, P)
    W = sc.num_workers(sched, causal, N)
    rounds = sc.packed_rounds(sched, causal, N, heads, P)
    for hd in range(heads):
        for q in range(N):
            assert sorted(order[(hd, q)]) == [kv for kv in range(N) if sc.allowed(causal, q, kv)]
        if len({rounds[(hd, w)] for w in range(W)}) == 1:     # a head inside one round
            plain = sc.reduction_order(sched, causal, N)
            assert all(order[(hd, q)] == plain[q] for q in range(N))


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("Ns,P", [([2, 4, 1, 9], 7), ([8] * 5, 12), ([3, 16, 5, 1, 1, 7, 12], 10),
                                  ([32, 2, 31], 38), ([1] * 9, 4)])
def test_mixed_packing_keeps_each_heads_shift_order(causal, Ns, P):
    """Heads of different lengths packed together: every tile's order is a permutation of its
    allowed blocks, a head inside one round keeps its plain shift order, and a head's order
    depends only on where its workers fall in the rounds -- equal lengths give the uniform
    packing's order exactly."""
    sched = sc.SYMSHIFT if causal else sc.SHIFT
    order = sc.packed_reduction_order_mixed(sched, causal, Ns, P)
    base = 0
    for hd, N in enumerate(Ns):
        W = sc.num_workers(sched, causal, N)
        for q in range(N):
            assert sorted(order[(hd, q)]) == [kv for kv in range(N) if sc.allowed(causal, q, kv)]
        if base // P == (base + W - 1) // P:
            plain = sc.reduction_order(sched, causal, N)
            assert all(order[(hd, q)] == plain[q] for q in range(N))
        # the same head alone, at the same offset within a round (padding heads of 1 tile
        # in front shift it there): the order depends on nothing else
        pad = base % P
        alone = sc.packed_reduction_order_mixed(sched, causal, [1] * pad + [N], P)
        assert sc.num_workers(sched, causal, 1) == 1
        assert all(alone[(pad, q)] == order[(hd, q)] for q in range(N))
        base += W
    if len(set(Ns)) == 1:
        uni = sc.packed_reduction_order(sched, causal, Ns[0], len(Ns), P)
        assert uni == order
