"""dash_attn_bwd_noalloc: the backward for callers that cannot provide a workspace.

It runs the same kernels as dash_attn_bwd but keeps its workspace in a fixed device array
inside the library.  Checked here through the C ABI: two calls in a row must each match the
ordinary entry point (with a caller workspace) within the parity tolerance used for the
oracle comparisons -- at both head dims, both masks, and a size that fills nearly the whole
array -- its device status must read clean through dash_attn_noalloc_status, and sizes
beyond the array's limit must be refused up front.  This file is collected last so that a
stop-at-first-failure run has already run everything else."""
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


def run_noalloc(dash, q, k, v, o, do, lse, causal, sched):
    B, S, H, D = q.shape
    Hkv = k.shape[2]
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    code = dash.lib().dash_attn_bwd_noalloc(q.data_ptr(), k.data_ptr(), v.data_ptr(),
                                            o.data_ptr(), do.data_ptr(), lse.data_ptr(),
                                            dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), B, S, H,
                                            H // Hkv, D, 0.0, int(causal),
                                            dash.SCHEDULES[sched], stream)
    assert code == 0, dash.STATUS.get(code, code)
    # the device status of the call, read from the scratch array
    assert dash.lib().dash_attn_noalloc_status(stream) == 0
    return dq, dk, dv


# (B, S, H, Hkv, D, causal, schedule): both head dims, both masks, GQA, and one shape whose
# workspace needs nearly all of the 64 MiB array (B*H*S = 61440 rows at D = 128), so that the
# parts carved at its top are used
CASES = [
    (1, 512, 4, 2, 64, True, "shift"),
    (1, 512, 4, 2, 64, False, "auto"),
    (2, 1024, 4, 2, 128, True, "shift_fill"),
    (2, 1024, 4, 4, 128, False, "shift_dual"),
    (1, 7680, 8, 8, 128, False, "auto"),
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "B{}S{}H{}-{}D{}{}-{}".format(
    c[0], c[1], c[2], c[3], c[4], "c" if c[5] else "f", c[6]))
def test_noalloc_matches_workspace_entry_point(case):
    from deterministic_attention_backward_gb300 import _build
    _build.build()
    import deterministic_attention_backward_gb300 as dash

    B, S, H, Hkv, D, causal, sched = case
    assert dash.bwd_workspace_bytes(B, S, H, D) <= SCRATCH_BYTES
    q, k, v, do = (t.cuda() for t in make_qkv_do(B, S, H, Hkv, D, seed=7))
    o, lse = dash.fwd(q, k, v, causal=causal, check=True)
    ref = dash.bwd(q, k, v, o, do, lse, causal=causal, schedule=sched, check=True)

    outs = []
    for _ in range(2):
        got = run_noalloc(dash, q, k, v, o, do, lse, causal, sched)
        torch.cuda.synchronize()
        outs.append(got)
        for name, g, want in zip(("dQ", "dK", "dV"), got, ref):
            ok, errs = within(g, want)
            assert ok, f"{name}: rel_fro={errs[0]:.3e} max={errs[1]:.3e}"
    # a deterministic schedule gives the same bits on both calls, and the bits of the call
    # with a caller workspace
    for a, b, c in zip(outs[0], outs[1], ref):
        assert torch.equal(a, b)
        assert torch.equal(a, c)


def test_noalloc_rejects_sizes_beyond_its_array():
    import deterministic_attention_backward_gb300 as dash
    L = dash.lib()
    B, S, H, D = 8, 8192, 16, 128
    assert dash.bwd_workspace_bytes(B, S, H, D) > SCRATCH_BYTES
    fake = 1 << 20  # refused before any pointer is used
    code = L.dash_attn_bwd_noalloc(*([fake] * 9), B, S, H, 1, D, 0.0, 0, 1, None)
    assert code == DASH_ERR_WORKSPACE
