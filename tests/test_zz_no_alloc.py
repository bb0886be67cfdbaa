"""dash_attn_bwd_noalloc: the backward for callers that cannot provide a workspace.

It runs the same kernels as dash_attn_bwd but keeps its workspace in a fixed device array
inside the library.  Checked here through the C ABI: two calls in a row must each match the
ordinary entry point (with a caller workspace) within the parity tolerance used for the
oracle comparisons, and sizes beyond the array's limit must be refused up front.  This file
is collected last so that a stop-at-first-failure run has already run everything else."""
import ctypes

import pytest
import torch

from dash_inputs import make_qkv_do

pytestmark = pytest.mark.gpu

REL_FRO = 1e-2
MAX_ABS = 2e-2
DASH_ERR_WORKSPACE = 5
SCRATCH_BYTES = 64 << 20


def within(got, ref):
    g, r = got.double(), ref.double()
    rel = (g - r).norm() / r.norm().clamp_min(1e-30)
    mx = (g - r).abs().max() / r.abs().max().clamp_min(1e-30)
    return rel.item() <= REL_FRO and mx.item() <= MAX_ABS, (rel.item(), mx.item())


def test_noalloc_matches_workspace_entry_point():
    from deterministic_attention_backward_gb300 import _build
    _build.build()
    import deterministic_attention_backward_gb300 as dash
    L = dash.lib()

    B, S, H, Hkv, D = 1, 512, 4, 2, 64
    causal, sched = True, "shift"
    q, k, v, do = (t.cuda() for t in make_qkv_do(B, S, H, Hkv, D, seed=7))
    o, lse = dash.fwd(q, k, v, causal=causal, check=True)
    ref = dash.bwd(q, k, v, o, do, lse, causal=causal, schedule=sched, check=True)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)

    outs = []
    for _ in range(2):
        dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
        code = L.dash_attn_bwd_noalloc(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                                       do.data_ptr(), lse.data_ptr(), dq.data_ptr(),
                                       dk.data_ptr(), dv.data_ptr(), B, S, H, H // Hkv, D, 0.0,
                                       int(causal), dash.SCHEDULES[sched], stream)
        assert code == 0, dash.STATUS.get(code, code)
        torch.cuda.synchronize()
        outs.append((dq, dk, dv))
        for name, got, want in zip(("dQ", "dK", "dV"), (dq, dk, dv), ref):
            ok, errs = within(got, want)
            assert ok, f"{name}: rel_fro={errs[0]:.3e} max={errs[1]:.3e}"
    # a deterministic schedule gives the same bits on both calls
    for a, b in zip(*outs):
        assert torch.equal(a, b)


def test_noalloc_rejects_sizes_beyond_its_array():
    import deterministic_attention_backward_gb300 as dash
    L = dash.lib()
    B, S, H, D = 8, 8192, 16, 128
    assert dash.bwd_workspace_bytes(B, S, H, D) > SCRATCH_BYTES
    fake = 1 << 20  # refused before any pointer is used
    code = L.dash_attn_bwd_noalloc(*([fake] * 9), B, S, H, 1, D, 0.0, 0, 1, None)
    assert code == DASH_ERR_WORKSPACE
