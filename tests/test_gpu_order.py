"""The accumulation order the GPU executes, against the schedule oracle, bit for bit: the
tile kernel records, for every (query tile, KV block) pair it visits, the rank at which the
block's dQ partial was added into the tile (the semaphore count the addition waited for),
and that rank must equal the position of the block in the tile's order as the oracle
restates the schedule -- plain lock step for the single-round schedules, the round-robin
packing of the workers onto the GPU's SMs for the packed ones (heads split across rounds
included, whose ranks the kernel derives in closed form from the head's phase)."""
import numpy as np
import pytest
import torch

from dash_inputs import make_qkv_do
from oracle import schedule as sc

pytestmark = pytest.mark.gpu

ORDERED = ["serial", "descending", "shift", "shift_fill", "shift_dual"]


@pytest.fixture(scope="module")
def dash():
    from deterministic_attention_backward_gb300 import _build
    _build.build()
    import deterministic_attention_backward_gb300 as d
    return d


def oracle_ranks(dash, sched, causal, B, H, Hkv, N):
    """[B, H, N, N] rank of (q, kv) in tile q's order per the oracle; -1 where skipped."""
    G = H // Hkv
    want = np.full((B, H, N, N), -1, dtype=np.int32)
    if sched == "shift_dual":  # the packed shift's ranks, split into strands by parity
        sched = "shift_fill"
    if sched in ("serial", "descending"):
        for q in range(N):
            for kv in range(N):
                if sc.allowed(causal, q, kv):
                    want[:, :, q, kv] = kv
        return want
    name = sc.SYMSHIFT if causal else sc.SHIFT
    if sched == "shift":
        for (q, kv), r in sc.rank_table(name, causal, N).items():
            want[:, :, q, kv] = r
        return want
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    heads = B * Hkv
    grid = dash.sched_grid(sched, causal, N, heads, sms)
    for (hd, q), kvs in sc.packed_reduction_order(name, causal, N, heads, grid).items():
        b, g = divmod(hd, Hkv)
        for r, kv in enumerate(kvs):
            want[b, g * G:(g + 1) * G, q, kv] = r
    return want


ORDER_CASES = [  # (B, S, H, Hkv, D, causal)
    (1, 1024, 2, 2, 64, False),     # N = 8
    (1, 1024, 2, 2, 128, False),
    (2, 4096, 16, 16, 128, True),   # 32 heads of 16 pairs: heads split across rounds
    (1, 16384, 2, 2, 128, False),
    (1, 640, 2, 2, 128, True),      # odd N = 5: padded Symmetric Shift
    (2, 1024, 8, 2, 128, True),     # GQA 4:1
    (4, 4096, 32, 32, 64, True),    # 128 heads of 16 pairs: heads split across rounds
    (1, 16384, 2, 2, 64, False),    # N = 128: two heads of 128 workers over two rounds
    (1, 16384, 2, 2, 64, True),
]


@pytest.mark.parametrize("case", ORDER_CASES, ids=lambda c: "B{}S{}H{}-{}D{}{}".format(
    c[0], c[1], c[2], c[3], c[4], "c" if c[5] else "f"))
@pytest.mark.parametrize("sched", ORDERED)
def test_executed_order_equals_oracle(dash, sched, case):
    B, S, H, Hkv, D, causal = case
    N = (S + 127) // 128
    if sched == "shift" and dash.sched_grid("shift_fill", causal, N, 1, 10 ** 6) > \
            torch.cuda.get_device_properties(0).multi_processor_count:
        pytest.skip("plain SHIFT needs a head's workers resident at once")
    q, k, v, do = (t.cuda() for t in make_qkv_do(B, S, H, Hkv, D, seed=11))
    o, lse = dash.fwd(q, k, v, causal=causal, check=True)
    *_, order = dash.bwd_order_log(q, k, v, o, do, lse, causal=causal, schedule=sched)
    got = order.cpu().numpy()
    want = oracle_ranks(dash, sched, causal, B, H, Hkv, N)
    bad = np.argwhere(got != want)
    assert bad.size == 0, f"{len(bad)} pairs differ, first (b,h,q,kv)={tuple(bad[0])}: " \
                          f"got {got[tuple(bad[0])]} want {want[tuple(bad[0])]}"

