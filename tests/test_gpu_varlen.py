"""Variable-length (packed) batches.  The forward and backward over a packed batch against
the fp64 oracle per sequence; the packed schedules run every sequence in one tile-kernel
launch, and the accumulation order the GPU executes there equals the oracle's packing of
heads of mixed lengths (sequence-major, then kv head, dealt round-robin to the grid; one
launch per group of at most 1024 non-empty sequences); where every head's workers fall in
one round the packed call gives the bits of the B = 1 call on the sequence's slices;
repeats are bit-identical, idle and under load; empty, one-token, whole-tile and ragged
sequences."""
import numpy as np
import pytest
import torch

import oracle
from oracle import schedule as sc
from dash_inputs import make_qkv_do

pytestmark = pytest.mark.gpu

REL_FRO = 1e-2
MAX_ABS = 2e-2
MAX_SEQS = 1024  # non-empty sequences per packed launch


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


def check_grads(name, host, causal, dq, dk, dv):
    """dQ, dK, dV of one sequence ([S, heads, D] slices) against the oracle.  A one-token
    sequence is degenerate: the softmax of a single score is constant, so dQ and dK are zero
    in exact arithmetic (the oracle's are rounding noise) and only their size is checked:
    what is left must be rounding, far below the terms dP and rowsum(dO o O) that cancel."""
    dq_r, dk_r, dv_r, _, _ = oracle.attn_bwd(*host, causal)
    close(f"dV {name}", dv[None], dv_r)
    if host[0].shape[1] > 1:
        close(f"dQ {name}", dq[None], dq_r)
        close(f"dK {name}", dk[None], dk_r)
        return
    q, k, v, do = (t.double() for t in host)
    G = q.shape[2] // k.shape[2]
    vv = v.repeat_interleave(G, dim=2)
    dp = (do * vv).sum(-1).abs().max().item()
    size = dp * max(q.abs().max().item(), k.abs().max().item()) / q.shape[-1] ** 0.5
    for n, t in (("dQ", dq), ("dK", dk)):
        got = t.detach().double().abs().max().item()
        assert got <= 1e-3 * size, f"{n} {name}: {got:.3e} (terms of size {size:.3e})"


def packed(lengths, H, Hkv, D, seed):
    """Per-sequence inputs from the seeded generator, concatenated along the token axis."""
    seqs = [make_qkv_do(1, S, H, Hkv, D, seed + b) if S else None for b, S in enumerate(lengths)]
    cat = []
    for n in range(4):
        parts = [s[n][0] for s in seqs if s is not None]
        cat.append(torch.cat(parts, 0).cuda())
    cu = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32)
    return seqs, cat, cu


def tiles(S):
    return (S + 127) // 128


def workers(causal, N):
    return sc.num_workers(sc.SYMSHIFT if causal else sc.SHIFT, causal, N)


def groups(lengths):
    """The packed launches: lists of the non-empty sequences' indices."""
    out, cur = [], []
    for b, S in enumerate(lengths):
        if S == 0:
            continue
        cur.append(b)
        if len(cur) == MAX_SEQS:
            out.append(cur)
            cur = []
    return out + ([cur] if cur else [])


def one_round(lengths, Hkv, causal, sms):
    """True when, in the packed layout and alone, every head's workers share one round."""
    for g in groups(lengths):
        base = 0
        for b in g:
            W = workers(causal, tiles(lengths[b]))
            for _ in range(Hkv):
                if base // sms != (base + W - 1) // sms or W > sms:
                    return False
                base += W
    return True


def sequence(lengths, cu, b, t):
    s0, S = int(cu[b]), lengths[b]
    return t[s0:s0 + S]


def single_call(dash, q, k, v, o, do, lse, cu, lengths, b, H, causal, sched):
    sl = lambda t: sequence(lengths, cu, b, t)[None].contiguous()
    s0, S = int(cu[b]), lengths[b]
    lse1 = lse[s0 * H:(s0 + S) * H].view(1, H, S).contiguous()
    return dash.bwd(sl(q), sl(k), sl(v), sl(o), sl(do), lse1, causal=causal, schedule=sched,
                    check=True)


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
def test_varlen_matches_oracle_and_single_calls(dash, causal, D):
    H, Hkv = 4, 2
    lengths = [200, 512, 37, 0, 1030, 1, 128]
    seqs, (q, k, v, do), cu = packed(lengths, H, Hkv, D, seed=3)
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    assert one_round(lengths, Hkv, causal, sms)
    o, lse = dash.fwd_varlen(q, k, v, cu, causal=causal, check=True)
    grads = {}
    for sched in ("auto", "serial", "atomic", "shift_fill", "shift_dual"):
        grads[sched] = dash.bwd_varlen(q, k, v, o, do, lse, cu, causal=causal, schedule=sched,
                                       check=True)
    # AUTO is resolved once, with the longest sequence's tile count
    want = dash.sched_resolve("auto", causal, tiles(max(lengths)), D, H // Hkv)
    for a, b in zip(grads["auto"], grads[want]):
        assert torch.equal(a, b), want
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
        for sched, (dq, dk, dv) in grads.items():
            check_grads(f"seq{b} {sched}", host, causal, dq[s0:s0 + S], dk[s0:s0 + S],
                        dv[s0:s0 + S])
        # every head inside one round: the packed launch adds each tile's partials in the
        # order of the B = 1 call, and the per-sequence schedules run exactly that call
        for sched in ("serial", "shift_fill", "shift_dual"):
            one = single_call(dash, q, k, v, o, do, lse, cu, lengths, b, H, causal, sched)
            for a, g in zip(one, grads[sched]):
                assert torch.equal(a[0], sequence(lengths, cu, b, g)), (sched, b)


def oracle_log(dash, lengths, H, Hkv, causal, sched):
    """[tiles, Nmax] expected order log (-1 where no partial is added)."""
    G = H // Hkv
    nmax = max(tiles(S) for S in lengths)
    rows = []
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    name = sc.SYMSHIFT if causal else sc.SHIFT
    for g in groups(lengths):
        Ns = [tiles(lengths[b]) for b in g for _ in range(Hkv)]
        units = sum(workers(causal, n) for n in Ns)
        if sched in ("shift_fill", "shift_dual"):
            order = sc.packed_reduction_order_mixed(name, causal, Ns, min(units, sms))
        for i, b in enumerate(g):
            N = tiles(lengths[b])
            for h in range(H):
                for q in range(N):
                    row = np.full(nmax, -1, dtype=np.int32)
                    if sched == "serial":
                        for kv in range(N):
                            if sc.allowed(causal, q, kv):
                                row[kv] = kv
                    else:
                        for r, kv in enumerate(order[(i * Hkv + h // G, q)]):
                            row[kv] = r
                    rows.append(row)
    return np.stack(rows)


def mixed_lengths(n, lo, hi, seed, extra=()):
    rng = np.random.default_rng(seed)
    return [int(x) for x in rng.integers(lo, hi + 1, size=n)] + list(extra)


ORDER_CASES = [  # (lengths, H, Hkv, D)
    (mixed_lengths(24, 1, 3000, 1, extra=(0, 128, 4096)), 4, 2, 128),   # heads straddle rounds
    (mixed_lengths(40, 100, 9000, 2), 2, 2, 64),
    (mixed_lengths(MAX_SEQS + 6, 1, 400, 3), 2, 2, 64),                 # two packed launches
]


@pytest.mark.parametrize("case", ORDER_CASES, ids=["mixed24", "long40", "two_launches"])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("sched", ["shift_fill", "shift_dual", "serial"])
def test_varlen_executed_order_equals_oracle(dash, sched, causal, case):
    lengths, H, Hkv, D = case
    if sched == "serial" and len(lengths) > 64:
        pytest.skip("one launch per sequence: covered by the shorter batches")
    T = sum(lengths)
    g = torch.Generator(device="cpu").manual_seed(7)
    q, do = (torch.randn(T, H, D, generator=g).to("cuda", torch.bfloat16) for _ in range(2))
    k, v = (torch.randn(T, Hkv, D, generator=g).to("cuda", torch.bfloat16) for _ in range(2))
    cu = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32)
    o, lse = dash.fwd_varlen(q, k, v, cu, causal=causal, check=True)
    *_, order = dash.bwd_varlen_order_log(q, k, v, o, do, lse, cu, causal=causal, schedule=sched)
    got = order.cpu().numpy()
    want = oracle_log(dash, lengths, H, Hkv, causal, sched)
    assert got.shape == want.shape
    bad = np.argwhere(got != want)
    assert bad.size == 0, f"{len(bad)} entries differ, first (tile, kv)={tuple(bad[0])}: " \
                          f"got {got[tuple(bad[0])]} want {want[tuple(bad[0])]}"


@pytest.mark.parametrize("causal", [False, True])
def test_varlen_many_sequences_parity_and_repeats(dash, causal):
    """48 sequences of 1 to 2500 tokens (GQA 4:1, D = 128) in one launch: sampled sequences
    against the oracle for every packed schedule, and 100 repeats of the ordered ones
    bit-identical while matrix products load the GPU from a second stream."""
    H, Hkv, D = 8, 2, 128
    lengths = mixed_lengths(45, 1, 2500, 5, extra=(128, 1, 2048))
    seqs, (q, k, v, do), cu = packed(lengths, H, Hkv, D, seed=100)
    o, lse = dash.fwd_varlen(q, k, v, cu, causal=causal, check=True)
    grads = {s: dash.bwd_varlen(q, k, v, o, do, lse, cu, causal=causal, schedule=s, check=True)
             for s in ("atomic", "shift_fill", "shift_dual")}
    order = np.argsort(lengths)
    sample = sorted({int(order[0]), int(order[len(order) // 2]), int(order[-1]),
                     45, 46, 47, 3})
    for b in sample:
        for sched, (dq, dk, dv) in grads.items():
            check_grads(f"seq{b} {sched}", seqs[b], causal, sequence(lengths, cu, b, dq),
                        sequence(lengths, cu, b, dk), sequence(lengths, cu, b, dv))
    side = torch.cuda.Stream()
    a = torch.randn(4096, 4096, device="cuda", dtype=torch.bfloat16)
    sink = torch.empty_like(a)
    ws = torch.empty(dash.bwd_varlen_workspace_bytes(cu, H, D), dtype=torch.uint8, device="cuda")
    outs = [torch.empty_like(t) for t in (q, k, v)]
    for sched in ("shift_fill", "shift_dual"):
        ref = grads[sched]
        for i in range(100):
            if i % 2:
                with torch.cuda.stream(side):
                    for _ in range(4):
                        torch.matmul(a, a, out=sink)
            out = dash.bwd_varlen(q, k, v, o, do, lse, cu, causal=causal, schedule=sched,
                                  dq=outs[0], dk=outs[1], dv=outs[2], workspace=ws)
            for x, y in zip(out, ref):
                assert torch.equal(x, y), (sched, i)
        torch.cuda.synchronize()
        dash.status(ws)


def test_varlen_two_launches_match_oracle(dash):
    """More than 1024 non-empty sequences: two packed launches sharing the workspace."""
    H, Hkv, D = 2, 2, 64
    lengths = mixed_lengths(MAX_SEQS + 6, 1, 300, 9)
    lengths[500] = 0
    seqs, (q, k, v, do), cu = packed(lengths, H, Hkv, D, seed=20)
    o, lse = dash.fwd_varlen(q, k, v, cu, causal=True, check=True)
    dq, dk, dv = dash.bwd_varlen(q, k, v, o, do, lse, cu, causal=True, schedule="shift_dual",
                                 check=True)
    for b in (0, 499, 501, MAX_SEQS - 1, MAX_SEQS, MAX_SEQS + 1, MAX_SEQS + 5):
        check_grads(f"seq{b}", seqs[b], True, sequence(lengths, cu, b, dq),
                    sequence(lengths, cu, b, dk), sequence(lengths, cu, b, dv))
