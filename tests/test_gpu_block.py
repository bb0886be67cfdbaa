"""The synthetic transformer block runs forward and backward through the library's
attention; its parameter gradients are finite, and the attention gradients agree between
the atomic and a deterministic schedule to the parity tolerance."""
import pytest
import torch

pytestmark = pytest.mark.gpu


def test_block_forward_backward_small():
    from deterministic_attention_backward_gb300 import _build
    _build.build()
    from deterministic_attention_backward_gb300.block import Block, time_block
    blk = Block(hidden=512, heads=4, kv_heads=2, head_dim=128, ffn=1024, seed=0)
    x = torch.randn(1, 512, 512, device="cuda", dtype=torch.bfloat16, requires_grad=True)
    grads = {}
    for sched in ("atomic", "shift_fill"):
        for p in blk.parameters() + [x]:
            p.grad = None
        blk(x, sched).float().square().mean().backward()
        grads[sched] = [p.grad.float().clone() for p in blk.parameters() + [x]]
        assert all(torch.isfinite(g).all() for g in grads[sched])
    for a, b in zip(grads["atomic"], grads["shift_fill"]):
        assert ((a - b).norm() / b.norm().clamp_min(1e-30)).item() < 1e-2
    out = time_block(seq=512, batch=1, schedules=("atomic", "shift_fill"), steps=2, warmup=1)
    assert set(out["block_ms"]) == {"atomic", "shift_fill"}
