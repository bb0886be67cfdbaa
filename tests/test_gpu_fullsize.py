"""Parity at the benchmark's full sizes, in the launch configuration bench.py times: the
largest point of each configuration, the CUDA path (forward, then the backward with the
bench's schedule and with the atomic variant) against the fp64 oracle on sampled rows of one
(batch, kv head) group -- every row the oracle restates is computed from the definitions at
full length (LSE and Dvec over all rows, then the sampled dQ, dK, dV rows)."""
import numpy as np
import pytest
import torch

import oracle
from dash_inputs import make_qkv_do

pytestmark = pytest.mark.gpu

REL_FRO = 1e-2
MAX_ABS = 2e-2
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


@pytest.mark.parametrize("cfg", CONFIGS, ids=[c[0] for c in CONFIGS])
def test_full_size_sampled_rows_match_oracle(dash, cfg):
    name, B, S, H, Hkv, D, causal, sched = cfg
    host = make_qkv_do(B, S, H, Hkv, D, seed=0)
    q, k, v, do = (t.cuda() for t in host)
    o, lse = dash.fwd(q, k, v, causal=causal, check=True)
    ws = torch.empty(dash.bwd_workspace_bytes(B, S, H, D), dtype=torch.uint8, device="cuda")
    outs = {}
    for s in (sched, "atomic"):
        grads = dash.bwd(q, k, v, o, do, lse, causal=causal, schedule=s, workspace=ws)
        dash.status(ws)
        outs[s] = [t.detach().to(torch.float64).cpu().numpy() for t in grads]
    G = H // Hkv
    b, g = B - 1, Hkv - 1  # the last group: every earlier batch/head precedes it in memory
    qr, kr = sample_rows(S, 1), sample_rows(S, 2)
    sq, sk, sv = oracle.attn_bwd_rows(*host, causal, b, g, qr, kr)
    for s, (dq, dk, dv) in outs.items():
        close(f"{name} {s} dQ", dq[b, qr][:, g * G:(g + 1) * G], sq)
        close(f"{name} {s} dK", dk[b, kr, g], sk)
        close(f"{name} {s} dV", dv[b, kr, g], sv)


@pytest.mark.parametrize("causal,S", [(False, 160 * 128), (True, 320 * 128), (True, 319 * 128)])
def test_heads_wider_than_the_grid(dash, causal, S):
    """More shift workers per head than SMs (full: N = 160; causal: 160 pairs, also for
    the odd N = 319): the packed schedule (and AUTO) runs the head in several rounds;
    sampled rows match the oracle and repeats are bit-identical."""
    B, H, Hkv, D = 1, 2, 1, 64
    host = make_qkv_do(B, S, H, Hkv, D, seed=4)
    q, k, v, do = (t.cuda() for t in host)
    o, lse = dash.fwd(q, k, v, causal=causal, check=True)
    first = [t.clone() for t in dash.bwd(q, k, v, o, do, lse, causal=causal,
                                         schedule="shift_fill", check=True)]
    again = dash.bwd(q, k, v, o, do, lse, causal=causal, schedule="auto", check=True)
    for a, b in zip(first, again):
        assert torch.equal(a, b)
    qr, kr = sample_rows(S, 5), sample_rows(S, 6)
    sq, sk, sv = oracle.attn_bwd_rows(*host, causal, 0, 0, qr, kr)
    dq, dk, dv = (t.detach().to(torch.float64).cpu().numpy() for t in first)
    close("dQ", dq[0, qr], sq)
    close("dK", dk[0, kr, 0], sk)
    close("dV", dv[0, kr, 0], sv)
