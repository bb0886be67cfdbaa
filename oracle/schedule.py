"""Oracle for the tile schedules of the DASH pages (test infrastructure only).

A head of length S is cut into N = S/128 query tiles and N KV blocks.  The backward is
KV-stationary: one worker ("SM" on the pages, a persistent CTA on the GPU) owns a KV
block, keeps its dK/dV on chip and visits query tiles one after another, adding one dQ
partial to each visited dQ tile (gist.science technical summary, section 2.1
"Problem formulation": the operations of one KV tile run back to back on one SM).
Determinism fixes, for every dQ tile, the order in which the KV blocks' partials are
added (section 1 "Problem statement").  This module restates each schedule of the pages
as plain lists:

* ``visits(sched, causal, N, u)``: the (kv, q) pairs worker ``u`` processes, in order;
* ``reduction_order(sched, causal, N)``: for every dQ tile q the KV blocks in the order
  their partials are added;
* ``critical_path(...)``: the length of the longest dependency chain when every tile
  step costs one time unit (the DAG of section 2.1: compute nodes chained per worker,
  plus the forced accumulation order edges between consecutive contributors of a tile);
* ``conflict_free(...)``: in lock-step execution no two workers touch the same dQ tile
  at the same step and each tile's accumulation order equals its step order -- the
  property that Lemma 1 (section 2.2 B) asks of the shift schedules.

Readings of the pages (where they are silent or loose):

* SERIAL is the deterministic FlashAttention-3 baseline the pages improve on: worker j
  visits query tiles in ascending order and every dQ tile adds KV blocks 0, 1, ... in
  ascending order (section 1: gradient reductions serialised in a fixed order).
* DESCENDING (section 2.2 A) only reverses the traversal (N-1 down to 0); the
  accumulation order stays ascending in kv.
* SHIFT, full mask (section 2.2 B): the text says SM i processes "i, i+1, ..., N-1, 0,
  ..., i-1".  Because the operations of one KV tile must stay on one SM (section 2.1),
  the listed indices are read as the *query tiles* visited by the worker that owns KV
  block i.  The accumulation order of a tile is its lock-step order.
* SYMSHIFT, causal mask (section 2.2 B, "Symmetric Shift"): worker c owns KV blocks c
  and N-1-c (the pages' pairing), h = N/2.  Phase 1 covers the dense lower-left
  rectangle (q >= h, kv < h) cyclically; phase 2 covers the folded triangle.  The
  pages give no exact step order, so the one below is constructed to be conflict-free
  and to finish block c before starting block N-1-c.  The accumulation order of a tile
  is its lock-step order.
* SYMSHIFT with an odd N (the pages pair blocks i and N-1-i, which needs an even N; they
  say nothing of odd N): append an empty KV block and query tile N, lay out the even
  schedule of N+1 tiles, and drop every step that touches the padding.  The dropped
  steps stay idle slots of the lock step, so a tile's accumulation order is still its
  lock-step order.  Worker 0 is left with block 0 alone and worker c >= 1 with the pair
  (c, N-c); each has N steps.
"""
from __future__ import annotations

SERIAL, DESCENDING, SHIFT, SYMSHIFT = "serial", "descending", "shift", "symshift"
SCHEDULES = (SERIAL, DESCENDING, SHIFT, SYMSHIFT)


def allowed(causal: bool, q: int, kv: int) -> bool:
    """Tile (q, kv) holds at least one unmasked element (causal: kv block <= q tile)."""
    return (kv <= q) if causal else True


def num_workers(sched: str, causal: bool, N: int) -> int:
    return (N + 1) // 2 if sched == SYMSHIFT else N


def _symshift_even(N: int, c: int) -> list[tuple[int, int]]:
    """Worker c's (kv, q) steps of the Symmetric Shift for an even N."""
    h = N // 2
    out = [(c, h + (c + t) % h) for t in range(h)]               # phase 1: rectangle
    for t in range(h + 1):                                       # phase 2: folded triangle
        p = (c + 1 + t) % (h + 1)
        out.append((c, p - 1) if p >= c + 1 else (N - 1 - c, N - 1 - p))
    return out


def timed_visits(sched: str, causal: bool, N: int, u: int) -> list[tuple[int, int, int]]:
    """(slot, kv, q) for worker u in processing order: slot is the lock-step time."""
    if sched == SERIAL:
        seq = [(u, q) for q in range(N) if allowed(causal, q, u)]
    elif sched == DESCENDING:
        seq = [(u, q) for q in reversed(range(N)) if allowed(causal, q, u)]
    elif sched == SHIFT:
        if causal:
            raise ValueError("cyclic shift is the full-mask schedule; causal uses symshift")
        seq = [(u, (u + t) % N) for t in range(N)]
    elif sched == SYMSHIFT:
        if not causal:
            raise ValueError("symmetric shift is the causal-mask schedule")
        if N % 2 == 0:
            seq = _symshift_even(N, u)
        else:  # odd N: the even schedule of N+1 tiles; padding steps become idle slots
            return [(t, kv, q) for t, (kv, q) in enumerate(_symshift_even(N + 1, u))
                    if kv < N and q < N]
    else:
        raise ValueError(sched)
    return [(t, kv, q) for t, (kv, q) in enumerate(seq)]


def visits(sched: str, causal: bool, N: int, u: int) -> list[tuple[int, int]]:
    """(kv, q) pairs processed by worker u, in processing order."""
    return [(kv, q) for _, kv, q in timed_visits(sched, causal, N, u)]


def _arrivals(sched: str, causal: bool, N: int) -> dict[int, list[tuple[int, int]]]:
    arrivals: dict[int, list[tuple[int, int]]] = {q: [] for q in range(N)}
    for u in range(num_workers(sched, causal, N)):
        for t, kv, q in timed_visits(sched, causal, N, u):
            arrivals[q].append((t, kv))
    return arrivals


def reduction_order(sched: str, causal: bool, N: int) -> dict[int, list[int]]:
    """dQ tile q -> KV blocks in the order their partials are added."""
    if sched in (SERIAL, DESCENDING):
        return {q: [kv for kv in range(N) if allowed(causal, q, kv)] for q in range(N)}
    return {q: [kv for _, kv in sorted(a)] for q, a in _arrivals(sched, causal, N).items()}


def rank_table(sched: str, causal: bool, N: int) -> dict[tuple[int, int], int]:
    """(q, kv) -> position of KV block kv in dQ tile q's accumulation order."""
    return {(q, kv): r for q, kvs in reduction_order(sched, causal, N).items()
            for r, kv in enumerate(kvs)}


def conflict_free(sched: str, causal: bool, N: int) -> bool:
    arrivals = _arrivals(sched, causal, N)
    order = reduction_order(sched, causal, N)
    for q, a in arrivals.items():
        a.sort()
        if len({t for t, _ in a}) != len(a):        # two workers on tile q at one step
            return False
        if [kv for _, kv in a] != order[q]:         # step order != accumulation order
            return False
    return True


def critical_path(sched: str, causal: bool, N: int) -> int:
    """Finish time of the last tile step when each step costs 1 and a step starts once
    the worker's previous step and the tile's previous contributor have finished."""
    W = num_workers(sched, causal, N)
    seq = [visits(sched, causal, N, u) for u in range(W)]
    rank = rank_table(sched, causal, N)
    order = reduction_order(sched, causal, N)
    owner = {}
    for u in range(W):
        for p, (kv, q) in enumerate(seq[u]):
            owner[(kv, q)] = (u, p)
    finish: dict[tuple[int, int], int] = {}
    pending = [(u, p) for u in range(W) for p in range(len(seq[u]))]
    while pending:
        progressed, rest = False, []
        for u, p in pending:
            kv, q = seq[u][p]
            deps = []
            if p > 0:
                deps.append((u, p - 1))
            r = rank[(q, kv)]
            if r > 0:
                deps.append(owner[(order[q][r - 1], q)])
            if all(d in finish for d in deps):
                finish[(u, p)] = 1 + max((finish[d] for d in deps), default=0)
                progressed = True
            else:
                rest.append((u, p))
        if not progressed:
            raise RuntimeError("schedule deadlocks in the unit-step model")
        pending = rest
    return max(finish.values())


# ---------------------------------------------------------------------------------------
# Packed shift: the shift workers of all heads are laid out one after another (head-major)
# and dealt round-robin to P processors; processor p runs its workers in order, one per
# round, every round taking the same time (lock step).  A head whose workers fall into two
# rounds runs as two phases.  The accumulation order of every dQ tile is the time order of
# its contributions (round, then step); the visiting order of each worker is the shift
# order of its head.  This is the shift schedule of the pages for a processor count that
# is not a multiple of the workers per head.
def packed_rounds(sched: str, causal: bool, N: int, heads: int, P: int):
    """(head, worker) -> round index."""
    W = num_workers(sched, causal, N)
    return {(hd, w): (hd * W + w) // P for hd in range(heads) for w in range(W)}


def packed_reduction_order(sched: str, causal: bool, N: int, heads: int, P: int):
    """(head, q) -> KV blocks in the order their partials are added."""
    W = num_workers(sched, causal, N)
    rounds = packed_rounds(sched, causal, N, heads, P)
    steps_per_round = 1 + max(t for w in range(W) for t, _, _ in timed_visits(sched, causal, N, w))
    arrivals: dict = {}
    for (hd, w), r in rounds.items():
        for t, kv, q in timed_visits(sched, causal, N, w):
            arrivals.setdefault((hd, q), []).append((r * steps_per_round + t, kv))
    out = {}
    for key, a in arrivals.items():
        a.sort()
        times = [t for t, _ in a]
        assert len(set(times)) == len(times), "two contributions to one tile at one time"
        out[key] = [kv for _, kv in a]
    return out


# A packed batch of heads with different tile counts (variable-length sequences): head i has
# Ns[i] tiles and its own shift workers; the workers of all heads are laid out one after
# another in the given head order and dealt round-robin to P processors as above.  The pages
# treat one length at a time; the reading taken is that every head keeps the shift order of
# its own length and the accumulation order of its tiles is again the time order of their
# contributions.  Only contributions of one head are ever compared, so the time of a
# contribution is its (round, step) pair.
def packed_reduction_order_mixed(sched: str, causal: bool, Ns: list[int], P: int):
    """(head, q) -> KV blocks in the order their partials are added, head i of Ns[i] tiles."""
    arrivals: dict = {}
    base = 0
    for hd, N in enumerate(Ns):
        W = num_workers(sched, causal, N)
        for w in range(W):
            rnd = (base + w) // P
            for t, kv, q in timed_visits(sched, causal, N, w):
                arrivals.setdefault((hd, q), []).append(((rnd, t), kv))
        base += W
    out = {}
    for key, a in arrivals.items():
        a.sort()
        times = [t for t, _ in a]
        assert len(set(times)) == len(times), "two contributions to one tile at one time"
        out[key] = [kv for _, kv in a]
    return out
