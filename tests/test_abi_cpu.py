"""The C-ABI library without a GPU: it builds, loads, exports every symbol the header
declares, rejects bad arguments synchronously, and its schedule tables equal the schedule
oracle's (host logic only; no compute calls)."""
import ctypes
import os
import re

import pytest

import deterministic_attention_backward_gb300 as dash
from deterministic_attention_backward_gb300 import _build
from oracle import schedule as sc

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    _build.build()
    return dash.lib()


def header_functions():
    text = open(os.path.join(ROOT, "include", "dash_attn.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(dash_\w+)\s*\(", text)))


def test_exports_every_declared_symbol(L):
    names = header_functions()
    assert len(names) >= 10
    for n in names:
        assert hasattr(L, n), n
    assert sorted(dash.EXPORTS) == names


def test_workspace_sizes(L):
    """Status block, room for two semaphores per dQ tile, two row vectors and a two-strand
    fp32 accumulator, each part 256-byte aligned."""
    B, S, H, D = 2, 1024, 4, 128
    n = dash.bwd_workspace_bytes(B, S, H, D)
    rows = B * H * S
    need = 256 + 2 * B * H * (S // 128) * 4 + 2 * rows * 4 + 2 * rows * D * 4
    assert need <= n < need + 4 * 256
    # a partial last tile is padded to whole tiles: S = 1000 needs the space of S = 1024
    assert dash.bwd_workspace_bytes(B, 1000, H, D) == dash.bwd_workspace_bytes(B, 1024, H, D)
    assert dash.bwd_workspace_bytes(B, S, H, 96) == 0            # unsupported head dim
    assert dash.fwd_workspace_bytes(B, S, H, 64) == 256


def test_argument_errors_are_synchronous(L):
    null = None
    c = L.dash_attn_bwd(null, null, null, null, null, null, null, null, null,
                        1, 512, 2, 1, 64, 0.0, 0, 1, null, 0, null)
    assert c == 1                                                # DASH_ERR_INVALID
    c = L.dash_attn_bwd(null, null, null, null, null, null, null, null, null,
                        1, 512, 2, 1, 96, 0.0, 0, 1, null, 0, null)
    assert c == 2                                                # head dim 96
    c = L.dash_attn_bwd(null, null, null, null, null, null, null, null, null,
                        1, 512, 3, 2, 64, 0.0, 0, 1, null, 0, null)
    assert c == 1                                                # H % group
    fake = 1 << 20                                               # never dereferenced
    c = L.dash_attn_bwd(*([fake] * 9), 1, 384, 2, 1, 64, 0.0, 1, 7, fake, 1 << 30, null)
    assert c == 1                                                # unknown schedule
    c = L.dash_attn_bwd_stages(*([fake] * 9), 1, 384, 2, 1, 64, 0.0, 1, 1, fake, 1 << 30, 8,
                               null)
    assert c == 1                                                # unknown stage bit
    c = L.dash_attn_bwd_order_log(*([fake] * 9), 1, 384, 2, 1, 64, 0.0, 1, 1, fake, 1 << 30,
                                  null, null)
    assert c == 1                                                # no order log
    c = L.dash_attn_bwd(*([fake] * 9), 1, 512, 2, 1, 64, 0.0, 1, 3, fake, 16, null)
    assert c == 5                                                # workspace too small
    c = L.dash_attn_bwd(*([fake + 4] + [fake] * 8), 1, 512, 2, 1, 64, 0.0, 1, 3, fake, 1 << 30,
                        null)
    assert c == 1                                                # misaligned pointer
    assert L.dash_status_string(4) == b"device-side wait timed out"


SCHEDS = [("serial", sc.SERIAL), ("descending", sc.DESCENDING), ("atomic", None),
          ("shift", None), ("shift_fill", None), ("shift_dual", None)]


@pytest.mark.parametrize("N", [1, 2, 3, 4, 5, 6, 7, 8, 9, 16, 33, 64, 127, 128])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("name,oracle_name", SCHEDS)
def test_library_schedule_equals_oracle(L, name, oracle_name, causal, N):
    if oracle_name is None:  # shift (and the fill mode's shift heads); atomic borrows it
        oracle_name = sc.SYMSHIFT if causal else sc.SHIFT
    table = dash.sched_table(name, causal, N)
    assert len(table) == sc.num_workers(oracle_name, causal, N)
    ranks = sc.rank_table(oracle_name, causal, N)
    for w, segs in enumerate(table):
        flat = [(kv, q) for seg in segs for kv, q, _ in seg]
        assert flat == sc.visits(oracle_name, causal, N, w)
        for seg in segs:
            assert len({kv for kv, _, _ in seg}) == 1           # one KV block per segment
            for kv, q, r in seg:
                assert r == ranks[(q, kv)]


def test_odd_symmetric_shift_segments(L):
    """Odd N: worker 0 has one segment (block 0), every other worker two (c, then N-c),
    all of N steps."""
    N = 7
    table = dash.sched_table("shift", True, N)
    assert len(table) == 4
    assert len(table[0]) == 1 and [kv for kv, _, _ in table[0][0]] == [0] * N
    for c in range(1, 4):
        assert [len(seg) for seg in table[c]] == [N - c, c]
        assert {kv for kv, _, _ in table[c][1]} == {N - c}


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("N,heads,P", [(8, 5, 12), (8, 3, 8), (16, 4, 24), (4, 9, 10), (32, 3, 38),
                                       (32, 64, 152), (64, 8, 152), (16, 20, 152),
                                       (16, 3, 5), (32, 2, 10), (64, 1, 31), (24, 2, 7),
                                       (5, 7, 4), (9, 3, 5), (33, 5, 38), (127, 3, 152),
                                       (3, 40, 152), (31, 2, 7)])
def test_packed_ranks_equal_oracle(L, causal, N, heads, P):
    """The library's packed-shift ranks equal the oracle's lock-step simulation of the
    workers dealt round-robin to P CTAs, also when a head has more workers than CTAs."""
    W = (N + 1) // 2 if causal else N
    if P > heads * W:
        P = heads * W
    order = sc.packed_reduction_order(sc.SYMSHIFT if causal else sc.SHIFT, causal, N, heads, P)
    for (hd, q), kvs in order.items():
        for r, kv in enumerate(kvs):
            assert dash.packed_rank(causal, N, heads, P, hd, q, kv) == r


@pytest.mark.parametrize("causal", [False, True])
def test_grid_sizes(L, causal):
    N, heads, sms = 32, 64, 152
    W = N // 2 if causal else N
    for name in ("serial", "descending", "shift", "shift_fill", "shift_dual", "atomic"):
        w = W if name in ("shift", "shift_fill", "shift_dual", "atomic") else N
        assert dash.sched_grid(name, causal, N, heads, sms) == min(heads * w, sms)
    assert dash.sched_grid("shift_fill", causal, N, 1, sms) == W
    with pytest.raises(ValueError):
        dash.sched_grid("shift", False, 160, 1, 152)
    assert dash.sched_grid("serial", False, 160, 1, 152) == 152
    # the packed schedule (and AUTO) take heads wider than the grid in several rounds
    assert dash.sched_grid("shift_fill", False, 160, 1, 152) == 152
    assert dash.sched_grid("auto", True, 320, 1, 152) == 152


def test_schedule_query_rejects_bad_arguments(L):
    assert L.dash_sched_workers(3, 1, 0) == -1
    assert L.dash_sched_workers(3, 1, 5) == 3                   # odd N: ceil(N/2) workers
    assert L.dash_sched_workers(7, 0, 4) == -1
    assert L.dash_sched_step(1, 0, 4, 0, 0, 4, None, None, None) == -1


def auto_table(causal, D, N, G):
    """The measured choice the header documents for DASH_SCHED_AUTO (one winner everywhere)."""
    return "shift_dual"


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("N", [1, 2, 3, 4, 7, 8, 16, 63, 64, 128])
@pytest.mark.parametrize("causal", [False, True])
def test_auto_schedule_resolution(L, causal, N, D):
    """AUTO runs the measured table's schedule; other schedules pass through, and the table
    queries (which do not know D) see the packed shift traversal both packed schedules
    share."""
    for G in (1, 4):
        want = auto_table(causal, D, N, G)
        assert dash.sched_resolve("auto", causal, N, D, group=G) == want
        assert dash.sched_grid("auto", causal, N, 64, 152) == dash.sched_grid(want, causal, N, 64, 152)
    for name in ("atomic", "serial", "descending", "shift", "shift_fill", "shift_dual"):
        assert dash.sched_resolve(name, causal, N, D) == name
    assert dash.sched_table("auto", causal, N) == dash.sched_table("shift_fill", causal, N)
    assert dash.sched_table("shift_dual", causal, N) == dash.sched_table("shift_fill", causal, N)
    assert L.dash_sched_resolve(7, int(causal), D, N, 1) == -1
    assert L.dash_sched_resolve(5, int(causal), 96, N, 1) == -1


def test_varlen_arguments_and_workspace(L):
    """Packed-batch entry points: offsets are checked before anything runs, and the shared
    workspace is the packed launch's need (per-tile arrays for every tile of the batch plus
    the 1024-entry sequence table: 16 bytes and 4 bytes per entry, each part 256-aligned),
    at least the longest sequence's."""
    import ctypes as ct
    arr = lambda xs: (ct.c_int * len(xs))(*xs)
    fake = 1 << 20
    cu = arr([0, 200, 712, 749])
    table = 16 * 1024 + (4 * 1025 + 255) // 256 * 256
    # 2 + 4 + 1 tiles per head, 4 heads: the arrays of 7 tiles of a B = 1 call
    assert L.dash_attn_bwd_varlen_workspace_bytes(cu, 3, 4, 64) == \
        dash.bwd_workspace_bytes(1, 7 * 128, 4, 64) + table
    assert L.dash_attn_bwd_varlen_workspace_bytes(arr([0, 0, 300, 300]), 3, 2, 128) == \
        dash.bwd_workspace_bytes(1, 300, 2, 128) + table
    assert L.dash_attn_bwd_varlen_workspace_bytes(arr([0, 5, 3]), 2, 4, 64) == 0   # decreasing
    assert L.dash_attn_bwd_varlen_workspace_bytes(arr([1, 5]), 1, 4, 64) == 0      # cu[0] != 0
    args = [fake] * 9
    assert L.dash_attn_bwd_varlen(*args, arr([0, 5, 3]), 2, 4, 1, 64, 0.0, 0, 1, fake, 1 << 30,
                                  None) == 1
    assert L.dash_attn_bwd_varlen(*args, cu, 3, 4, 3, 64, 0.0, 0, 1, fake, 1 << 30, None) == 1
    assert L.dash_attn_bwd_varlen(*args, cu, 3, 4, 1, 64, 0.0, 0, 9, fake, 1 << 30, None) == 1
    assert L.dash_attn_bwd_varlen(*args, cu, 3, 4, 1, 64, 0.0, 0, 7, fake, 1 << 30, None) == 1
    assert L.dash_attn_fwd_varlen(*([fake] * 5), arr([2, 4]), 1, 4, 1, 64, 0.0, 0, fake, 256,
                                  None) == 1
    # the audit form wants its log
    assert L.dash_attn_bwd_varlen_order_log(*args, cu, 3, 4, 1, 64, 0.0, 0, 4, fake, 1 << 30,
                                            None, None) == 1


def test_wait_limit_setting(L):
    """The device-side wait limit is a process-wide setting with a checked range."""
    assert dash.wait_limit() == pytest.approx(2.0)
    try:
        dash.set_wait_limit(0.25)
        assert dash.wait_limit() == pytest.approx(0.25)
        for bad in (0.0, -1.0, 1e-4, 4000.0, float("nan")):
            assert L.dash_attn_set_wait_limit(bad) == 1
        assert dash.wait_limit() == pytest.approx(0.25)
    finally:
        dash.set_wait_limit(2.0)


def test_varlen_workspace_spans_the_largest_packed_launch(L):
    """More than 1024 non-empty sequences run as several packed launches that share the
    workspace: its size is the largest launch's need (its tiles' arrays plus the table),
    empty sequences taking no place in a launch."""
    import ctypes as ct
    table = 16 * 1024 + (4 * 1025 + 255) // 256 * 256
    H, D = 2, 64
    lens = [300] * 1024 + [0] * 5 + [3000] * 3   # launch 1: 1024 x 3 tiles; launch 2: 3 x 24
    cu = [0]
    for n in lens:
        cu.append(cu[-1] + n)
    arr = (ct.c_int * len(cu))(*cu)
    first = dash.bwd_workspace_bytes(1, 1024 * 3 * 128, H, D) + table
    assert L.dash_attn_bwd_varlen_workspace_bytes(arr, len(lens), H, D) == first
    lens2 = [300] * 10 + [0] * 2000 + [16000] * 2   # one launch: 10 x 3 + 2 x 125 tiles
    cu2 = [0]
    for n in lens2:
        cu2.append(cu2[-1] + n)
    arr2 = (ct.c_int * len(cu2))(*cu2)
    want = dash.bwd_workspace_bytes(1, (10 * 3 + 2 * 125) * 128, H, D) + table
    assert L.dash_attn_bwd_varlen_workspace_bytes(arr2, len(lens2), H, D) == want
