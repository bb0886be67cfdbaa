"""Parity at the benchmark's full sizes, in the launch configuration bench.py times: the
largest point of each configuration, the CUDA path (forward, then the backward with every
schedule the bench times, ordered and atomic) against the fp64 oracle on sampled rows of
three (batch, kv head) groups -- the first, the last, and one whose workers the packed
schedules split across two rounds of the grid -- every row the oracle restates computed
from the definitions at full length (LSE and Dvec over all rows, then the sampled dQ, dK, dV
rows)."""
import numpy as np
import pytest
import torch

import oracle
from dash_inputs import make_qkv_do

pytestmark = pytest.mark.gpu

REL_FRO = 1e-2
MAX_ABS = 2e-2
SCHEDULES = ["atomic", "serial", "descending", "shift", "shift_fill", "shift_dual"]
CONFIGS = [  # (name, B, S, H, Hkv, D, causal, schedule timed by bench.py)
    ("full_h16_d128", 1, 16384, 16, 16, 128, False, "shift_fill"),
    ("causal_h32_d128", 1, 16384, 32, 32, 128, True, "shift_fill"),
    ("causal_h32_d64", 1, 16384, 32, 32, 64, True, "shift_fill"),
    ("gqa_causal_8b", 2, 8192, 32, 8, 128, True, "shift_fill"),
]


@pytest.fixture(scope="module")
def dash():
    from deterministic_attention_backward_gb300 import _build
    _build.build()
    import deterministic_attention_backward_gb300 as d
    return d


def sample_rows(S, seed):
    rng = np.random.default_rng(seed)
    fixed = [0, 1, 127, 128, S // 2, S - 129, S - 1]
    return sorted(set(fixed + [int(x) for x in rng.integers(0, S, 5)]))


def close(name, got, ref):
    diff = got - ref
    rel = np.linalg.norm(diff) / max(np.linalg.norm(ref), 1e-30)
    mx = np.abs(diff).max() / max(np.abs(ref).max(), 1e-30)
    assert rel <= REL_FRO and mx <= MAX_ABS, f"{name}: rel_fro={rel:.3e} max={mx:.3e}"


def sampled_groups(dash, causal, N, B, Hkv):
    """(b, g) groups to compare: the first, the last, and a head the packed schedule splits
    across rounds of the grid (if any)."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    heads = B * Hkv
    W = dash.sched_workers("shift_fill", causal, N)
    grid = dash.sched_grid("shift_fill", causal, N, heads, sms)
    split = [hd for hd in range(1, heads - 1) if (hd * W) // grid != (hd * W + W - 1) // grid]
    picks = [0, heads - 1] + split[:1]
    return [divmod(hd, Hkv) for hd in dict.fromkeys(picks)]


@pytest.mark.parametrize("cfg", CONFIGS, ids=[c[0] for c in CONFIGS])
def test_full_size_sampled_rows_match_oracle(dash, cfg):
    name, B, S, H, Hkv, D, causal, _ = cfg
    host = make_qkv_do(B, S, H, Hkv, D, seed=0)
    q, k, v, do = (t.cuda() for t in host)
    o, lse = dash.fwd(q, k, v, causal=causal, check=True)
    ws = torch.empty(dash.bwd_workspace_bytes(B, S, H, D), dtype=torch.uint8, device="cuda")
    G = H // Hkv
    groups = sampled_groups(dash, causal, S // 128, B, Hkv)
    assert len(groups) >= 2
    qr, kr = sample_rows(S, 1), sample_rows(S, 2)
    refs = {bg: oracle.attn_bwd_rows(*host, causal, bg[0], bg[1], qr, kr) for bg in groups}
    for s in SCHEDULES:
        grads = dash.bwd(q, k, v, o, do, lse, causal=causal, schedule=s, workspace=ws)
        dash.status(ws)
        for b, g in groups:
            sq, sk, sv = refs[(b, g)]
            rows_q = grads[0][b, qr][:, g * G:(g + 1) * G].to(torch.float64).cpu().numpy()
            close(f"{name} {s} ({b},{g}) dQ", rows_q, sq)
            close(f"{name} {s} ({b},{g}) dK", grads[1][b, kr, g].to(torch.float64).cpu().numpy(), sk)
            close(f"{name} {s} ({b},{g}) dV", grads[2][b, kr, g].to(torch.float64).cpu().numpy(), sv)


@pytest.mark.parametrize("causal,S", [(False, 160 * 128), (True, 320 * 128), (True, 319 * 128)])
def test_heads_wider_than_the_grid(dash, causal, S):
    """More shift workers per head than SMs (full: N = 160; causal: 160 pairs, also for
    the odd N = 319): the packed schedules (single and two strands, and AUTO) run the head in
    several rounds; sampled rows match the oracle, and AUTO gives the bits of the schedule
    it resolves to."""
    B, H, Hkv, D = 1, 2, 1, 64
    host = make_qkv_do(B, S, H, Hkv, D, seed=4)
    q, k, v, do = (t.cuda() for t in host)
    o, lse = dash.fwd(q, k, v, causal=causal, check=True)
    resolved = dash.sched_resolve("auto", causal, S // 128, D, H // Hkv)
    runs = {s: [t.clone() for t in dash.bwd(q, k, v, o, do, lse, causal=causal, schedule=s,
                                            check=True)]
            for s in ("shift_fill", "shift_dual")}
    again = dash.bwd(q, k, v, o, do, lse, causal=causal, schedule="auto", check=True)
    for a, b in zip(runs[resolved], again):
        assert torch.equal(a, b)
    qr, kr = sample_rows(S, 5), sample_rows(S, 6)
    sq, sk, sv = oracle.attn_bwd_rows(*host, causal, 0, 0, qr, kr)
    for s, grads in runs.items():
        dq, dk, dv = (t.detach().to(torch.float64).cpu().numpy() for t in grads)
        close(f"{s} dQ", dq[0, qr], sq)
        close(f"{s} dK", dk[0, kr, 0], sk)
        close(f"{s} dV", dv[0, kr, 0], sv)
