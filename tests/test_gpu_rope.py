"""GPU: the rotary embedding (attn_rope_table, attn_rope) against oracle.rope.

The rotation of one bf16 pair is computed in fp32 from fp32 cos/sin and rounded
once to bf16, so each output may differ from the f64 oracle by half a bf16 ulp
of the oracle value plus the fp32 work (a few 2^-24 of |x0| + |x1|; bounded
here by 1e-6 (|x0| + |x1|)). The table itself must be the f64 cos/sin rounded
to fp32 (within 2^-24 relative, up to 1.2e-7 absolute). Positions reach 8191
(angles up to 8191 radians). Then the trainer's order, rotation -> attention ->
inverse rotation of dq and dk, is checked end to end against the oracle.
"""
import numpy as np
import pytest
import torch

import causal_gqa_flash_gb300 as gqa
import oracle
from causal_gqa_flash_gb300.inputs import make_inputs

from _helpers import check_against_oracle, f64, half_ulp_bf16

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")
SENTINEL = -3.25


@pytest.fixture(scope="module", autouse=True)
def _built():
    gqa.build()
    gqa.load()


@pytest.mark.parametrize("T,d,base", [(8192, 128, 10000.0), (1000, 64, 10000.0), (77, 64, 500.0)])
def test_table_matches_f64_angles(T, d, base):
    table = gqa.attn_rope_table(T, d, base=base)
    torch.cuda.synchronize()
    ang = oracle.rope_angles(T, d, base)
    tab = table.double().cpu().numpy()
    assert np.max(np.abs(tab[..., 0] - np.cos(ang))) <= 1.2e-7
    assert np.max(np.abs(tab[..., 1] - np.sin(ang))) <= 1.2e-7


def rope_error_ok(y_gpu, ref, x):
    """|y - ref| <= half a bf16 ulp of ref + 1e-6 (|x0| + |x1|), per element."""
    y, xa = f64(y_gpu), np.abs(f64(x))
    pair = xa[..., 0::2] + xa[..., 1::2]
    bound = half_ulp_bf16(ref) + 1e-6 * np.repeat(pair, 2, axis=-1) + 1e-30
    excess = np.abs(y - ref) - bound
    return float(np.max(excess)), np.unravel_index(np.argmax(excess), excess.shape)


@pytest.mark.parametrize("B,T,H,d", [(2, 300, 8, 64), (1, 8192, 2, 128), (3, 129, 5, 128)])
def test_rope_matches_oracle_out_of_place_and_in_place(B, T, H, d):
    g = torch.Generator().manual_seed(B * 1000 + T + d)
    x = torch.randn((B, T, H, d), generator=g).to(torch.bfloat16)
    table = gqa.attn_rope_table(T, d)
    xd = x.to(DEV)
    y = torch.full_like(xd, SENTINEL)
    gqa.attn_rope(xd, table, y=y)
    ref = oracle.rope(x)
    err, where = rope_error_ok(y, ref, x)
    assert err <= 0.0, f"rotation beyond its bound by {err:.3e} at {where}"
    # inverse
    z = gqa.attn_rope(y.clone(), table, inverse=True)
    ref_inv = oracle.rope(y, inverse=True)
    err, where = rope_error_ok(z, ref_inv, y)
    assert err <= 0.0, f"inverse rotation beyond its bound by {err:.3e} at {where}"
    # in place gives the same bits as out of place
    xi = xd.clone()
    gqa.attn_rope(xi, table)
    torch.cuda.synchronize()
    assert torch.equal(xi.view(torch.int16), y.view(torch.int16))


def test_rope_on_fused_qkv_view_leaves_v_alone():
    """One call rotates q and k of a fused [B, T, Hq+2*Hkv, d] projection (its first Hq+Hkv
    heads); v and an extra padding head keep their bits."""
    B, T, Hq, Hkv, d = 2, 260, 6, 2, 64
    H3 = Hq + 2 * Hkv
    g = torch.Generator().manual_seed(11)
    qkv = torch.randn((B, T, H3 + 1, d), generator=g).to(torch.bfloat16).to(DEV)
    before = qkv.clone()
    table = gqa.attn_rope_table(T, d)
    gqa.attn_rope(qkv[:, :, :Hq + Hkv], table)
    torch.cuda.synchronize()
    assert torch.equal(qkv[:, :, Hq + Hkv:].view(torch.int16), before[:, :, Hq + Hkv:].view(torch.int16))
    ref = oracle.rope(before[:, :, :Hq + Hkv].cpu())
    err, where = rope_error_ok(qkv[:, :, :Hq + Hkv], ref, before[:, :, :Hq + Hkv].cpu())
    assert err <= 0.0, f"beyond bound by {err:.3e} at {where}"


@pytest.mark.parametrize("d", [64, 128])
def test_rope_attention_pipeline_against_oracle(d):
    """rotate q, k -> attn_fwd -> attn_bwd -> inverse-rotate dq, dk, against the oracle's
    rope, attention and inverse rope composed in f64 (on the same bf16 rotated inputs the
    kernels saw, so only attention and the final rotation are compared)."""
    B, T, Hq, Hkv = 2, 333, 6, 2
    q, k, v, dout = make_inputs(B, T, Hq, Hkv, d, seed=500 + d)
    table = gqa.attn_rope_table(T, d)
    qr = gqa.attn_rope(q.to(DEV), table, y=torch.empty((B, T, Hq, d), dtype=torch.bfloat16, device=DEV))
    kr = gqa.attn_rope(k.to(DEV), table, y=torch.empty((B, T, Hkv, d), dtype=torch.bfloat16, device=DEV))
    vd, dod = v.to(DEV), dout.to(DEV)
    o, lse = gqa.attn_fwd(qr, kr, vd)
    dqr, dkr, dv = gqa.attn_bwd(qr, kr, vd, o, lse, dod)
    dq = gqa.attn_rope(dqr, table, inverse=True, y=torch.empty_like(dqr))
    dk = gqa.attn_rope(dkr, table, inverse=True, y=torch.empty_like(dkr))
    assert gqa.attn_sync_status() == gqa.GQA_OK, gqa.attn_last_error()
    ref = oracle.bwd(qr.cpu(), kr.cpu(), v, dout)
    ref = dict(ref, dq=oracle.rope(ref["dq"], inverse=True), dk=oracle.rope(ref["dk"], inverse=True))
    check_against_oracle(dict(o=o, lse=lse, dq=dq, dk=dk, dv=dv), ref, f"rope + attention d={d}")
