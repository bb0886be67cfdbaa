"""Failure detection on the GPU without a fault: a dQ ordering semaphore that no worker will
ever release makes the deterministic backward's bounded wait run out.  The kernel must stop
by itself (no hang), report DASH_ERR_TIMEOUT through the workspace status word, and leave
the CUDA context usable for the next call."""
import time

import pytest
import torch

from dash_inputs import make_qkv_do

pytestmark = pytest.mark.gpu

DASH_ERR_TIMEOUT = 4


@pytest.fixture(scope="module")
def dash():
    from deterministic_attention_backward_gb300 import _build
    _build.build()
    import deterministic_attention_backward_gb300 as d
    return d


@pytest.mark.parametrize("limit", [None, 0.25])
@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("schedule", ["serial", "shift_fill", "shift_dual"])
def test_unreleased_semaphore_times_out_and_context_survives(dash, schedule, D, limit):
    """The poller hands each turn to the epilogue through a ring of mbarriers; when the
    semaphore never reaches its count the poller's bounded wait runs out and every role
    gives up through the same abort flag, after the default limit (2 s) or the one set with
    dash_attn_set_wait_limit."""
    B, S, H = 1, 512, 2
    q, k, v, do = (t.cuda() for t in make_qkv_do(B, S, H, H, D, seed=0))
    o, lse = dash.fwd(q, k, v, causal=False, check=True)
    ws = torch.empty(dash.bwd_workspace_bytes(B, S, H, D), dtype=torch.uint8, device="cuda")
    args = dict(causal=False, schedule=schedule, workspace=ws)
    dash.bwd(q, k, v, o, do, lse, stages=dash.PROLOGUE, **args)
    # everything after the 256-byte status block: semaphores, row vectors and accumulator.
    # Every semaphore now holds 0x7F7F7F7F, a count no contributor waits for.
    ws[256:].fill_(0x7F)
    try:
        if limit is not None:
            dash.set_wait_limit(limit)
        t0 = time.time()
        dash.bwd(q, k, v, o, do, lse, stages=dash.TILES, **args)
        with pytest.raises(dash.DashError) as err:
            dash.status(ws)
        elapsed = time.time() - t0
    finally:
        dash.set_wait_limit(2.0)
    assert err.value.code == DASH_ERR_TIMEOUT
    if limit is None:
        assert 1.0 < elapsed < 60.0, elapsed
    else:
        assert 0.5 * limit < elapsed < 1.0, elapsed
    # the context is still usable: a clean call on a fresh workspace succeeds and matches
    # the atomic variant to the parity tolerance
    dq, dk, dv = dash.bwd(q, k, v, o, do, lse, causal=False, schedule=schedule, check=True)
    rq, rk, rv = dash.bwd(q, k, v, o, do, lse, causal=False, schedule="atomic", check=True)
    for got, ref in ((dq, rq), (dk, rk), (dv, rv)):
        rel = (got.float() - ref.float()).norm() / ref.float().norm()
        assert rel < 1e-2
