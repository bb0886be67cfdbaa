"""Pins of the fp64 oracle to facts independent of it (CPU only).

Each test fixes part of the oracle against something other than its own formula:
library routines (torch SDPA and autograd in float64), central finite differences of
its own forward, closed forms for Q = 0, exact causal special cases, and invariants of
softmax attention.  Together they fail on a dropped term, a wrong sign, a wrong scale
placement, a transposed operand or a wrong GQA head mapping.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from dash_inputs import make_qkv_do

CASES = [  # (B, S, H, Hkv, D)
    (1, 1, 2, 2, 3),
    (1, 5, 2, 2, 4),
    (1, 8, 2, 1, 4),
    (2, 7, 4, 2, 5),
]


def rand(shape, seed):
    return np.random.default_rng(seed).standard_normal(shape)


def qkvdo(B, S, H, Hkv, D, seed=0):
    return (rand((B, S, H, D), seed), rand((B, S, Hkv, D), seed + 1),
            rand((B, S, Hkv, D), seed + 2), rand((B, S, H, D), seed + 3))


def torch_attn(q, k, v, causal, scale):
    """torch SDPA in float64 on [B,S,H,D] inputs; K/V heads repeated for GQA."""
    G = q.shape[2] // k.shape[2]
    qt = q.transpose(1, 2)
    kt = k.repeat_interleave(G, dim=2).transpose(1, 2)
    vt = v.repeat_interleave(G, dim=2).transpose(1, 2)
    o = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, is_causal=causal, scale=scale)
    return o.transpose(1, 2)


def relerr(a, b):
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-300))


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("shape", CASES)
def test_fwd_matches_torch_sdpa(shape, causal):
    q, k, v, _ = qkvdo(*shape)
    o, lse = oracle.attn_fwd(q, k, v, causal)
    D = shape[-1]
    ref = torch_attn(*(torch.from_numpy(x) for x in (q, k, v)), causal, 1 / math.sqrt(D)).numpy()
    assert relerr(o, ref) < 1e-12


@pytest.mark.parametrize("causal", [False, True])
def test_lse_matches_torch_logsumexp(causal):
    B, S, H, Hkv, D = 2, 9, 4, 2, 6
    q, k, v, _ = qkvdo(B, S, H, Hkv, D, seed=5)
    _, lse = oracle.attn_fwd(q, k, v, causal)
    G = H // Hkv
    qt = torch.from_numpy(q).transpose(1, 2)                                  # B H S D
    kt = torch.from_numpy(k).repeat_interleave(G, dim=2).transpose(1, 2)
    s = torch.matmul(qt, kt.transpose(-1, -2)) / math.sqrt(D)
    if causal:
        s = s.masked_fill(torch.ones(S, S, dtype=torch.bool).triu(1), float("-inf"))
    ref = torch.logsumexp(s, dim=-1).numpy()
    assert np.max(np.abs(lse - ref)) < 1e-12


def test_explicit_scale_matches_torch():
    q, k, v, _ = qkvdo(1, 6, 2, 2, 4, seed=9)
    o, _ = oracle.attn_fwd(q, k, v, True, scale=0.37)
    ref = torch_attn(*(torch.from_numpy(x) for x in (q, k, v)), True, 0.37).numpy()
    assert relerr(o, ref) < 1e-12


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("shape", [(1, 1, 2, 2, 3), (1, 5, 2, 2, 3), (1, 8, 2, 1, 4), (1, 5, 2, 1, 4)])
def test_grad_central_finite_differences(shape, causal):
    """Gradient of f = sum(O * W) with W = dO, by central differences of the oracle's own
    forward; relative Frobenius error <= 1e-6."""
    q, k, v, w = qkvdo(*shape, seed=11)
    dq, dk, dv, _, _ = oracle.attn_bwd(q, k, v, w, causal)

    def f(q_, k_, v_):
        return float(np.sum(oracle.attn_fwd(q_, k_, v_, causal)[0] * w))

    eps = 1e-5
    for which, x, g in (("q", q, dq), ("k", k, dk), ("v", v, dv)):
        num = np.zeros_like(x)
        for idx in np.ndindex(x.shape):
            xp, xm = x.copy(), x.copy()
            xp[idx] += eps
            xm[idx] -= eps
            args_p = {"q": q, "k": k, "v": v}
            args_m = dict(args_p)
            args_p[which], args_m[which] = xp, xm
            num[idx] = (f(**{k_ + "_": a for k_, a in args_p.items()})
                        - f(**{k_ + "_": a for k_, a in args_m.items()})) / (2 * eps)
        if np.linalg.norm(num) == 0:
            assert np.max(np.abs(g)) < 1e-12
        else:
            assert relerr(g, num) <= 1e-6, which


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("shape", CASES + [(1, 33, 4, 1, 16)])
def test_grad_matches_torch_autograd(shape, causal):
    q, k, v, do = qkvdo(*shape, seed=21)
    dq, dk, dv, o, _ = oracle.attn_bwd(q, k, v, do, causal)
    ts = [torch.from_numpy(x).requires_grad_(True) for x in (q, k, v)]
    ot = torch_attn(*ts, causal, 1 / math.sqrt(shape[-1]))
    ot.backward(torch.from_numpy(do))
    assert relerr(o, ot.detach().numpy()) < 1e-12
    for mine, t in zip((dq, dk, dv), ts):
        assert relerr(mine, t.grad.numpy()) < 1e-10


@pytest.mark.parametrize("causal", [False, True])
def test_dk_sums_to_zero(causal):
    """Every row of dS sums to zero, so the keys' gradients of one head sum to zero."""
    q, k, v, do = qkvdo(2, 12, 4, 2, 8, seed=3)
    _, dk, _, _, _ = oracle.attn_bwd(q, k, v, do, causal)
    total = dk.sum(axis=1)                                  # [B, Hkv, D]
    assert np.max(np.abs(total)) <= 1e-12 * np.max(np.abs(dk)) * dk.shape[1]


@pytest.mark.parametrize("causal", [False, True])
def test_key_shift_invariance(causal):
    """Adding one vector c to every key shifts each score row by a constant: O, dQ, dK,
    dV are unchanged (dQ because the rows of dS sum to zero) and LSE_i moves by
    scale * q_i . c."""
    B, S, H, Hkv, D = 1, 10, 2, 1, 6
    q, k, v, do = qkvdo(B, S, H, Hkv, D, seed=4)
    c = rand((D,), 99)
    a = oracle.attn_bwd(q, k, v, do, causal)
    b = oracle.attn_bwd(q, k + c, v, do, causal)
    for x, y in zip(a[:4], b[:4]):
        assert relerr(y, x) < 1e-10
    shift = np.einsum("bshd,d->bhs", q, c) / math.sqrt(D)
    assert np.max(np.abs(b[4] - a[4] - shift)) < 1e-10


def test_full_mask_key_permutation_equivariance():
    B, S, H, Hkv, D = 1, 9, 2, 2, 4
    q, k, v, do = qkvdo(B, S, H, Hkv, D, seed=6)
    perm = np.random.default_rng(1).permutation(S)
    dq, dk, dv, o, lse = oracle.attn_bwd(q, k, v, do, False)
    dq2, dk2, dv2, o2, lse2 = oracle.attn_bwd(q, k[:, perm], v[:, perm], do, False)
    assert relerr(o2, o) < 1e-12 and np.max(np.abs(lse2 - lse)) < 1e-12
    assert relerr(dq2, dq) < 1e-10
    assert relerr(dk2, dk[:, perm]) < 1e-10 and relerr(dv2, dv[:, perm]) < 1e-10


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("G", [1, 2])
def test_q_zero_closed_forms(causal, G):
    """Q = 0 makes every allowed score equal: P_ij = 1/n_i with n_i = S (full) or i+1
    (causal).  Then LSE_i = ln n_i, O_i = mean of the allowed V_j, dK = 0,
    dV_j = sum over the rows i that see key j (and the group's heads) of dO_i / n_i, and
    dQ_i = (scale / n_i) sum_j (dO_i . (V_j - O_i)) K_j."""
    B, S, Hkv, D = 1, 7, 2, 4
    H = Hkv * G
    _, k, v, do = qkvdo(B, S, H, Hkv, D, seed=8)
    q = np.zeros((B, S, H, D))
    dq, dk, dv, o, lse = oracle.attn_bwd(q, k, v, do, causal)
    scale = 1 / math.sqrt(D)
    n = np.array([(i + 1) if causal else S for i in range(S)])
    assert np.max(np.abs(lse - np.log(n)[None, None, :])) < 1e-14
    assert np.max(np.abs(dk)) < 1e-14
    for h in range(H):
        g = h // G
        for i in range(S):
            vis = slice(0, n[i])
            o_ref = v[0, vis, g].mean(axis=0)
            assert np.max(np.abs(o[0, i, h] - o_ref)) < 1e-13
            coef = (v[0, vis, g] - o_ref) @ do[0, i, h]
            dq_ref = scale / n[i] * (coef @ k[0, vis, g])
            assert np.max(np.abs(dq[0, i, h] - dq_ref)) < 1e-13
    for g in range(Hkv):
        for j in range(S):
            rows = [i for i in range(S) if (not causal or i >= j)]
            ref = sum(do[0, i, g * G + hh] / n[i] for i in rows for hh in range(G))
            assert np.max(np.abs(dv[0, j, g] - ref)) < 1e-13


def test_causal_first_row_and_sparsity():
    """Causal: row 0 sees key 0 only, so P_00 = 1, O_0 = V_0, dS_00 = 0 and dQ_0 = 0
    exactly.  Queries/dO rows before j never reach dK_j/dV_j; keys after i never reach
    dQ_i, O_i or LSE_i (checked bit-exactly by perturbation)."""
    B, S, H, Hkv, D = 1, 8, 2, 2, 4
    q, k, v, do = qkvdo(B, S, H, Hkv, D, seed=12)
    dq, dk, dv, o, lse = oracle.attn_bwd(q, k, v, do, True)
    assert np.all(dq[:, 0] == 0.0)
    assert np.array_equal(o[:, 0], v[:, 0])
    j = 5
    q2, do2 = q.copy(), do.copy()
    q2[:, :j] += 1.0
    do2[:, :j] -= 0.5
    _, dk2, dv2, _, _ = oracle.attn_bwd(q2, k, v, do2, True)
    assert np.array_equal(dk2[:, j:], dk[:, j:]) and np.array_equal(dv2[:, j:], dv[:, j:])
    i = 3
    k2, v2 = k.copy(), v.copy()
    k2[:, i + 1:] += 2.0
    v2[:, i + 1:] *= 3.0
    dq3, _, _, o3, lse3 = oracle.attn_bwd(q, k2, v2, do, True)
    assert np.array_equal(dq3[:, :i + 1], dq[:, :i + 1])
    assert np.array_equal(o3[:, :i + 1], o[:, :i + 1])
    assert np.array_equal(lse3[:, :, :i + 1], lse[:, :, :i + 1])


def test_group_slice_equals_whole():
    B, S, H, Hkv, D = 2, 6, 4, 2, 4
    q, k, v, do = qkvdo(B, S, H, Hkv, D, seed=14)
    dq, dk, dv, _, _ = oracle.attn_bwd(q, k, v, do, True)
    gq, gk, gv, _, _ = oracle.attn_bwd_group(q, k, v, do, True, b=1, g=1)
    assert np.array_equal(gq[0], dq[1, :, 2:4]) and np.array_equal(gk[0], dk[1, :, 1:2])
    assert np.array_equal(gv[0], dv[1, :, 1:2])


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("B,S,H,Hkv,D", [(2, 37, 4, 2, 16), (1, 64, 2, 2, 8), (1, 50, 4, 1, 12)])
def test_sampled_rows_equal_the_full_backward(B, S, H, Hkv, D, causal):
    """The sampled-row oracle (used for parity at full sizes) restates the same definitions
    row by row: its rows equal the full backward's rows to rounding."""
    q, k, v, do = make_qkv_do(B, S, H, Hkv, D, seed=11)
    dq, dk, dv, _, _ = oracle.attn_bwd(q, k, v, do, causal)
    G = H // Hkv
    rng = np.random.default_rng(0)
    for b in range(B):
        for g in range(Hkv):
            qr = sorted(set([0, S - 1] + list(rng.integers(0, S, 5))))
            kr = sorted(set([0, S - 1] + list(rng.integers(0, S, 5))))
            sq, sk, sv = oracle.attn_bwd_rows(q, k, v, do, causal, b, g, qr, kr)
            ref_q = dq[b, qr][:, g * G:(g + 1) * G]
            np.testing.assert_allclose(sq, ref_q, rtol=1e-10, atol=1e-12)
            np.testing.assert_allclose(sk, dk[b, kr, g], rtol=1e-10, atol=1e-12)
            np.testing.assert_allclose(sv, dv[b, kr, g], rtol=1e-10, atol=1e-12)
