"""A synthetic transformer block, shaped like one decoder layer of an 8B-parameter model
(hidden 4096, 32 query heads, 8 KV heads of 128, SwiGLU MLP of 14336, RMSNorm), timed
forward + backward with this library's attention under each backward schedule.

It gives the end-to-end effect of deterministic attention an in-repo analogue: the DASH
pages report the block-level speedup of their schedules over the deterministic baseline
(technical summary, section 4).  Weights and inputs are random (seeded); there is no
dataset, no rotary embedding and no optimizer step.  The dense layers use torch matrix
products (plumbing around the measured path); the attention forward and backward run in
this library's kernels.

    python -m deterministic_attention_backward_gb300.block [--seq 8192] [--batch 1]
"""
from __future__ import annotations

import argparse
import json
import statistics


def _attention_function():
    import torch
    import deterministic_attention_backward_gb300 as dash

    class DashAttention(torch.autograd.Function):
        @staticmethod
        def forward(ctx, q, k, v, causal, schedule):
            o, lse = dash.fwd(q, k, v, causal=causal)
            ctx.save_for_backward(q, k, v, o, lse)
            ctx.causal, ctx.schedule = causal, schedule
            return o

        @staticmethod
        def backward(ctx, do):
            q, k, v, o, lse = ctx.saved_tensors
            dq, dk, dv = dash.bwd(q, k, v, o, do.contiguous(), lse, causal=ctx.causal,
                                  schedule=ctx.schedule)
            return dq, dk, dv, None, None

    return DashAttention


class Block:
    """Pre-norm decoder block: x + Wo·attn(norm(x)), then + W2·(silu(W1 h) * W3 h)."""

    def __init__(self, hidden=4096, heads=32, kv_heads=8, head_dim=128, ffn=14336,
                 device="cuda", seed=0):
        import torch
        g = torch.Generator(device="cpu").manual_seed(seed)

        def w(n_in, n_out):
            t = torch.randn(n_in, n_out, generator=g, dtype=torch.float32) / n_in ** 0.5
            return t.to(device=device, dtype=torch.bfloat16).requires_grad_()

        self.h, self.hk, self.d = heads, kv_heads, head_dim
        self.wqkv = w(hidden, (heads + 2 * kv_heads) * head_dim)
        self.wo = w(heads * head_dim, hidden)
        self.w1, self.w3, self.w2 = w(hidden, ffn), w(hidden, ffn), w(ffn, hidden)
        self.n1 = torch.ones(hidden, device=device, dtype=torch.bfloat16, requires_grad=True)
        self.n2 = torch.ones(hidden, device=device, dtype=torch.bfloat16, requires_grad=True)
        self.attn = _attention_function()
        # when a dict: the attention's inputs and output of the last call are kept there, with
        # their gradients retained (q/k/v.grad = dQ/dK/dV, o.grad = the upstream dO)
        self.capture = None

    @staticmethod
    def _rms(x, weight):
        import torch
        xf = x.float()
        return (xf * torch.rsqrt(xf.square().mean(-1, keepdim=True) + 1e-5)).to(x.dtype) * weight

    def __call__(self, x, schedule, causal=True):
        B, S, _ = x.shape
        qkv = self._rms(x, self.n1) @ self.wqkv
        q, k, v = qkv.split([self.h * self.d, self.hk * self.d, self.hk * self.d], dim=-1)
        q = q.reshape(B, S, self.h, self.d).contiguous()
        k = k.reshape(B, S, self.hk, self.d).contiguous()
        v = v.reshape(B, S, self.hk, self.d).contiguous()
        o = self.attn.apply(q, k, v, causal, schedule)
        if self.capture is not None:
            for t in (q, k, v, o):
                t.retain_grad()
            self.capture.update(q=q, k=k, v=v, o=o)
        a = o.reshape(B, S, self.h * self.d)
        x = x + a @ self.wo
        hid = self._rms(x, self.n2)
        import torch.nn.functional as F
        return x + (F.silu(hid @ self.w1) * (hid @ self.w3)) @ self.w2

    def parameters(self):
        return [self.wqkv, self.wo, self.w1, self.w3, self.w2, self.n1, self.n2]


def time_block(seq=8192, batch=1, schedules=("atomic", "serial", "shift_fill", "auto"),
               steps=10, warmup=3, causal=True, seed=0):
    """Median forward+backward time (ms) of one block per schedule, and each
    deterministic schedule's slowdown against ``atomic``."""
    import torch
    blk = Block(seed=seed)
    g = torch.Generator(device="cpu").manual_seed(seed + 1)
    x = (torch.randn(batch, seq, 4096, generator=g) * 0.5).to("cuda", torch.bfloat16)
    x.requires_grad_()
    gout = torch.randn(batch, seq, 4096, generator=g).to("cuda", torch.bfloat16)

    def step(sched):
        for p in blk.parameters() + [x]:
            p.grad = None
        out = blk(x, sched, causal)
        out.backward(gout)

    res = {}
    for sched in schedules:
        for _ in range(warmup):
            step(sched)
        torch.cuda.synchronize()
        ts = []
        for _ in range(steps):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            step(sched)
            b.record()
            torch.cuda.synchronize()
            ts.append(a.elapsed_time(b))
        res[sched] = statistics.median(ts)
    out = {"block_ms": {k: round(v, 3) for k, v in res.items()}}
    if "atomic" in res:
        out["slowdown_vs_atomic"] = {k: round(v / res["atomic"] - 1, 4)
                                     for k, v in res.items() if k != "atomic"}
    if "serial" in res:
        out["speedup_vs_serial"] = {k: round(res["serial"] / v, 4)
                                    for k, v in res.items() if k not in ("serial", "atomic")}
    out["config"] = {"seq": seq, "batch": batch, "causal": causal, "hidden": 4096,
                     "heads": 32, "kv_heads": 8, "head_dim": 128, "ffn": 14336,
                     "steps": steps, "warmup": warmup}
    return out


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--seq", type=int, default=8192)
    ap.add_argument("--batch", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    args = ap.parse_args()
    print(json.dumps(time_block(args.seq, args.batch, steps=args.steps, warmup=args.warmup)))


if __name__ == "__main__":
    main()
