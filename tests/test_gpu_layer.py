"""GPU: the whole-layer check ("A transformer in PTX", §Three ways to run it: every
fast kernel is checked against its naive twin, and then the whole model; §The model
for the layer).

The attention half of a decoder layer: RMSNorm of the fp32 residual stream, one
fused matmul for q, k and v into a [B, T, Hq+2*Hkv, d] bf16 buffer, RoPE on q and k,
causal grouped-query attention, and the output projection added into the residual
stream. The norm and the matmuls are torch (cuBLAS) here: they are not this
library's work, only the frame the attention is checked in. The attention runs two
ways behind one autograd function each:

* fast: attn_fwd_rope / attn_bwd_rope on views of the fused buffer (the rotation
  inside the attention kernels, the gradients written into one fused dqkv buffer);
* naive: attn_rope, then the naive twin (attn_fwd_naive / attn_bwd_naive, the whole
  score matrix in memory), then attn_rope's inverse on dq and dk.

Both are compared with the f64 oracle layer (oracle.layer_attn, pinned by finite
differences in test_oracle_layer.py) on the same parameters and upstream gradient:
the attention's contribution to the output and every gradient (residual stream,
norm gain, both weight matrices) within a relative Frobenius error of 2e-2, which
covers the bf16 roundings of the normalised input, the projections, the attention
output and the weight gradients; and the fast path no further from the oracle than
the naive twin (within 10%)."""
import pytest
import torch

import causal_gqa_flash_gb300 as gqa
import oracle

from _helpers import f64, rel_fro

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")
BASE = 10000.0
EPS = 1e-5
TOL = 2e-2


@pytest.fixture(scope="module", autouse=True)
def _built():
    gqa.build()
    gqa.load()


def split(qkv, Hq, Hkv):
    return qkv[:, :, :Hq], qkv[:, :, Hq:Hq + Hkv], qkv[:, :, Hq + Hkv:]


class FastRopeAttention(torch.autograd.Function):
    @staticmethod
    def forward(ctx, qkv, Hq, Hkv):
        q, k, v = split(qkv, Hq, Hkv)
        o, lse, q_rot, k_rot = gqa.attn_fwd_rope(q, k, v, base=BASE)
        ctx.save_for_backward(q_rot, k_rot, v, o, lse)
        ctx.heads = (Hq, Hkv)
        return o

    @staticmethod
    def backward(ctx, do):
        q_rot, k_rot, v, o, lse = ctx.saved_tensors
        Hq, Hkv = ctx.heads
        dqkv = torch.empty(q_rot.shape[:2] + (Hq + 2 * Hkv, q_rot.shape[3]), dtype=o.dtype, device=o.device)
        dq, dk, dv = split(dqkv, Hq, Hkv)
        gqa.attn_bwd_rope(q_rot, k_rot, v, o, lse, do.contiguous(), base=BASE, dq=dq, dk=dk, dv=dv)
        return dqkv, None, None


class NaiveRopeAttention(torch.autograd.Function):
    @staticmethod
    def forward(ctx, qkv, Hq, Hkv):
        q, k, v = split(qkv, Hq, Hkv)
        table = gqa.attn_rope_table(qkv.shape[1], qkv.shape[3], base=BASE)
        q_rot = gqa.attn_rope(q, table, y=torch.empty(q.shape, dtype=q.dtype, device=q.device))
        k_rot = gqa.attn_rope(k, table, y=torch.empty(k.shape, dtype=k.dtype, device=k.device))
        v = v.contiguous()
        o, lse = gqa.attn_fwd_naive(q_rot, k_rot, v)
        ctx.save_for_backward(q_rot, k_rot, v, o, lse, table)
        ctx.heads = (Hq, Hkv)
        return o

    @staticmethod
    def backward(ctx, do):
        q_rot, k_rot, v, o, lse, table = ctx.saved_tensors
        dq_rot, dk_rot, dv = gqa.attn_bwd_naive(q_rot, k_rot, v, o, lse, do.contiguous())
        dq = gqa.attn_rope(dq_rot, table, inverse=True, y=torch.empty_like(dq_rot))
        dk = gqa.attn_rope(dk_rot, table, inverse=True, y=torch.empty_like(dk_rot))
        return torch.cat([dq, dk, dv], dim=2), None, None


def gpu_layer(attn, x, g, w_qkv, w_o, dx2, Hq, Hkv, d):
    """Forward and backward of the layer on the GPU; returns x2 and the gradients."""
    x = x.clone().requires_grad_(True)
    g = g.clone().requires_grad_(True)
    w_qkv = w_qkv.clone().requires_grad_(True)
    w_o = w_o.clone().requires_grad_(True)
    B, T, C = x.shape
    r = torch.rsqrt(x.pow(2).mean(-1, keepdim=True) + EPS)
    xn = (x * r * g).to(torch.bfloat16)
    qkv = (xn @ w_qkv.t()).view(B, T, Hq + 2 * Hkv, d)
    o = attn.apply(qkv, Hq, Hkv)
    x2 = x + (o.reshape(B, T, Hq * d) @ w_o.t()).float()
    (x2 * dx2).sum().backward()
    assert gqa.attn_sync_status() == gqa.GQA_OK, gqa.attn_last_error()
    return dict(x2=x2.detach(), dx=x.grad, dg=g.grad, dw_qkv=w_qkv.grad, dw_o=w_o.grad)


def layer_errors(out, ref, x):
    err = {"attn_out": rel_fro(f64(out["x2"]) - f64(x), ref["x2"] - f64(x))}
    for name in ("dx", "dg", "dw_qkv", "dw_o"):
        err[name] = rel_fro(f64(out[name]), ref[name])
    return err


@pytest.mark.parametrize("B,T,C,Hq,Hkv,d", [
    (2, 333, 384, 6, 2, 64),     # the pages' dev head layout, ragged T
    (1, 300, 256, 4, 2, 128),    # d = 128, ragged T
    (2, 256, 192, 3, 3, 64),     # no grouping (Hq = Hkv)
])
def test_whole_layer_against_oracle_and_naive_twin(B, T, C, Hq, Hkv, d):
    gen = torch.Generator().manual_seed(B * 7919 + T + C + d)
    x = torch.randn((B, T, C), generator=gen)
    g = 1.0 + 0.2 * torch.randn((C,), generator=gen)
    w_qkv = (torch.randn(((Hq + 2 * Hkv) * d, C), generator=gen) / C ** 0.5).to(torch.bfloat16)
    w_o = (torch.randn((C, Hq * d), generator=gen) / (Hq * d) ** 0.5).to(torch.bfloat16)
    dx2 = torch.randn((B, T, C), generator=gen)
    ref = oracle.layer_attn(x.double().numpy(), g.double().numpy(), w_qkv.double().numpy(),
                            w_o.double().numpy(), Hq, Hkv, d, dx2.double().numpy(), base=BASE, eps=EPS)
    dev = [t.to(DEV) for t in (x, g, w_qkv, w_o, dx2)]
    fast = layer_errors(gpu_layer(FastRopeAttention, *dev, Hq, Hkv, d), ref, x)
    naive = layer_errors(gpu_layer(NaiveRopeAttention, *dev, Hq, Hkv, d), ref, x)
    print(f"B={B} T={T} C={C} Hq={Hq} Hkv={Hkv} d={d}: fast {fast}, naive {naive}")
    for name, e in fast.items():
        assert e <= TOL, f"fast {name}: rel-F {e:.3e} against the oracle layer"
        assert naive[name] <= TOL, f"naive {name}: rel-F {naive[name]:.3e} against the oracle layer"
        assert e <= 1.1 * naive[name] + 1e-4, f"fast {name} {e:.3e} vs naive {naive[name]:.3e}"
