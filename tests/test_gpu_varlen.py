"""Variable-length (packed) batches: the forward and backward over a packed batch against
the fp64 oracle per sequence, bit-identity with the B = 1 call on each sequence's slices
and across repeats, and empty / ragged sequences."""
import numpy as np
import pytest
import torch

import oracle
from dash_inputs import make_qkv_do

pytestmark = pytest.mark.gpu

REL_FRO = 1e-2
MAX_ABS = 2e-2


@pytest.fixture(scope="module")
def dash():
    from deterministic_attention_backward_gb300 import _build
    _build.build()
    import deterministic_attention_backward_gb300 as d
    return d


def close(name, got, ref):
    got = got.detach().to(torch.float64).cpu().numpy()
    diff = got - ref
    rel = np.linalg.norm(diff) / max(np.linalg.norm(ref), 1e-30)
    mx = np.abs(diff).max() / max(np.abs(ref).max(), 1e-30)
    assert rel <= REL_FRO and mx <= MAX_ABS, f"{name}: rel_fro={rel:.3e} max={mx:.3e}"


def packed(lengths, H, Hkv, D, seed):
    """Per-sequence inputs from the seeded generator, concatenated along the token axis."""
    seqs = [make_qkv_do(1, S, H, Hkv, D, seed + b) if S else None for b, S in enumerate(lengths)]
    cat = []
    for n in range(4):
        parts = [s[n][0] for s in seqs if s is not None]
        cat.append(torch.cat(parts, 0).cuda())
    cu = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32)
    return seqs, cat, cu


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
def test_varlen_matches_oracle_and_single_calls(dash, causal, D):
    H, Hkv = 4, 2
    lengths = [200, 512, 37, 0, 1030]
    seqs, (q, k, v, do), cu = packed(lengths, H, Hkv, D, seed=3)
    o, lse = dash.fwd_varlen(q, k, v, cu, causal=causal, check=True)
    grads = {}
    for sched in ("auto", "serial", "atomic"):
        grads[sched] = dash.bwd_varlen(q, k, v, o, do, lse, cu, causal=causal, schedule=sched,
                                       check=True)
    again = dash.bwd_varlen(q, k, v, o, do, lse, cu, causal=causal, schedule="auto", check=True)
    for a, b in zip(again, grads["auto"]):
        assert torch.equal(a, b)
    for b, S in enumerate(lengths):
        if S == 0:
            continue
        s0 = int(cu[b])
        host = seqs[b]
        o_ref, lse_ref = oracle.attn_fwd(*host[:3], causal)
        close(f"O seq{b}", o[s0:s0 + S][None], o_ref)
        lse_b = lse[s0 * H:(s0 + S) * H].view(1, H, S).cpu().numpy()
        assert np.abs(lse_b - lse_ref).max() <= 1e-3
        dq_r, dk_r, dv_r, _, _ = oracle.attn_bwd(*host, causal)
        for sched, (dq, dk, dv) in grads.items():
            close(f"dQ seq{b} {sched}", dq[s0:s0 + S][None], dq_r)
            close(f"dK seq{b} {sched}", dk[s0:s0 + S][None], dk_r)
            close(f"dV seq{b} {sched}", dv[s0:s0 + S][None], dv_r)
        # the packed call runs exactly the B = 1 call on the sequence's slices
        sl = lambda t: t[s0:s0 + S][None].contiguous()
        lse1 = lse[s0 * H:(s0 + S) * H].view(1, H, S).contiguous()
        one = dash.bwd(sl(q), sl(k), sl(v), sl(o), sl(do), lse1, causal=causal,
                       schedule="auto", check=True)
        for a, g in zip(one, grads["auto"]):
            assert torch.equal(a[0], g[s0:s0 + S])
