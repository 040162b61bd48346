"""GPU: attention with the rotary embedding fused in (attn_fwd_rope, attn_bwd_rope).

The fused kernels take their angles in registers: the turn count t * f_i is
reduced exactly in fixed point and the hardware sine and cosine give cos and sin
within ~1e-6, so a rotated element is within half a bf16 ulp of the oracle's
rotation plus 2e-6 (|x0| + |x1|) (attn_rope's table path: 1e-6). Given the
rotated q_rot and k_rot, the attention is the plain kernels' arithmetic: o and lse
are bit-identical to attn_fwd(q_rot, k_rot), and dv to attn_bwd's. dq and dk are
the fp32 gradients of q_rot and k_rot turned back before their one rounding, and
are checked against the oracle's gradients on the same rotated inputs composed
with the oracle's inverse rotation in f64.
"""
import numpy as np
import pytest
import torch

import causal_gqa_flash_gb300 as gqa
import oracle
from causal_gqa_flash_gb300.inputs import WORKLOADS, make_inputs, workload_inputs

from _helpers import check_against_oracle, f64, half_ulp_bf16, rel_fro

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")
BASE = 10000.0


@pytest.fixture(scope="module", autouse=True)
def _built():
    gqa.build()
    gqa.load()


def bits(t):
    return t.contiguous().view(torch.int16) if t.dtype == torch.bfloat16 else t.contiguous().view(torch.int32)


def rotation_excess(y_gpu, x, base=BASE):
    """max over elements of |y - oracle.rope(x)| - (half a bf16 ulp + 2e-6 (|x0| + |x1|))."""
    ref = oracle.rope(x, base=base)
    y, xa = f64(y_gpu), np.abs(f64(x))
    pair = np.repeat(xa[..., 0::2] + xa[..., 1::2], 2, axis=-1)
    return float(np.max(np.abs(y - ref) - half_ulp_bf16(ref) - 2e-6 * pair - 1e-30))


def fused(q, k, v, dout, causal, base=BASE):
    o, lse, qr, kr = gqa.attn_fwd_rope(q, k, v, base=base, causal=causal)
    dq, dk, dv = gqa.attn_bwd_rope(qr, kr, v, o, lse, dout, base=base, causal=causal)
    return dict(o=o, lse=lse, q_rot=qr, k_rot=kr, dq=dq, dk=dk, dv=dv)


def plain_on(fus, v, dout, causal):
    """The plain kernels on the fused path's rotated q and k."""
    o, lse = gqa.attn_fwd(fus["q_rot"], fus["k_rot"], v, causal=causal)
    dqr, dkr, dv = gqa.attn_bwd(fus["q_rot"], fus["k_rot"], v, o, lse, dout, causal=causal)
    return dict(o=o, lse=lse, dq_rot=dqr, dk_rot=dkr, dv=dv)


CASES = [
    # B, T, Hq, Hkv, d, causal
    (1, 1, 2, 1, 64, True),
    (2, 333, 6, 2, 64, True),      # ragged tail
    (2, 333, 6, 2, 128, True),
    (1, 200, 4, 2, 64, False),     # full attention, ragged
    (1, 256, 8, 2, 128, False),
    (4, 1024, 12, 4, 64, True),    # 384 items: several per persistent CTA at d = 64
]


@pytest.mark.parametrize("B,T,Hq,Hkv,d,causal", CASES, ids=lambda x: str(x))
def test_fused_against_oracle(B, T, Hq, Hkv, d, causal):
    q, k, v, dout = make_inputs(B, T, Hq, Hkv, d, seed=900 + T + d)
    qd, kd, vd, dod = (x.to(DEV) for x in (q, k, v, dout))
    fus = fused(qd, kd, vd, dod, causal)
    pl = plain_on(fus, vd, dod, causal)
    assert gqa.attn_sync_status() == gqa.GQA_OK, gqa.attn_last_error()
    assert rotation_excess(fus["q_rot"], q) <= 0.0, "q_rot beyond its bound"
    assert rotation_excess(fus["k_rot"], k) <= 0.0, "k_rot beyond its bound"
    for name in ("o", "lse", "dv"):
        assert torch.equal(bits(fus[name]), bits(pl[name])), f"{name} differs from the plain kernels on q_rot, k_rot"
    if B * T * Hq > 40000:
        # too large for the oracle in seconds: against the plain gradients turned back in f64
        for name in ("dq", "dk"):
            ref = oracle.rope(pl[name + "_rot"].cpu(), base=BASE, inverse=True)
            err = rel_fro(f64(fus[name]), ref)
            assert err <= 4e-3, f"{name}: rel-F {err:.2e} from the plain gradients turned back"
        return
    ref = oracle.bwd(fus["q_rot"].cpu(), fus["k_rot"].cpu(), v, dout, causal=causal)
    ref = dict(ref, dq=oracle.rope(ref["dq"], base=BASE, inverse=True), dk=oracle.rope(ref["dk"], base=BASE,
                                                                                        inverse=True))
    check_against_oracle(fus, ref, f"fused rope B={B} T={T} Hq={Hq} Hkv={Hkv} d={d} causal={causal}")
    # one rounding instead of two: no further from the oracle than rotating the plain
    # kernel's bf16 gradients back with attn_rope
    table = gqa.attn_rope_table(T, d, base=BASE)
    for name in ("dq", "dk"):
        sep = gqa.attn_rope(pl[name + "_rot"], table, inverse=True, y=torch.empty_like(pl[name + "_rot"]))
        e_f, e_s = rel_fro(f64(fus[name]), ref[name]), rel_fro(f64(sep), ref[name])
        assert e_f <= e_s * 1.05 + 1e-6, f"{name}: fused {e_f:.3e} vs rotated afterwards {e_s:.3e}"


@pytest.mark.parametrize("d,base", [(64, 10000.0), (128, 500000.0)])
def test_query_and_key_rotations_agree(d, base):
    """The forward kernel's query rotation and the key pass use the same angles: the same
    tensor given as q and as k (Hq = Hkv) comes out with the same bits, and a token at
    position 0 is not moved."""
    B, T, H = 2, 700, 3
    g = torch.Generator().manual_seed(d)
    x = torch.randn((B, T, H, d), generator=g).to(torch.bfloat16).to(DEV)
    v = torch.randn((B, T, H, d), generator=g).to(torch.bfloat16).to(DEV)
    _, _, qr, kr = gqa.attn_fwd_rope(x, x, v, base=base)
    assert gqa.attn_sync_status() == gqa.GQA_OK, gqa.attn_last_error()
    assert torch.equal(bits(qr), bits(kr))
    assert torch.equal(bits(qr[:, 0]), bits(x[:, 0]))
    assert rotation_excess(qr, x.cpu(), base=base) <= 0.0


def test_fused_in_place_on_a_qkv_buffer():
    """q_rot = q and k_rot = k as views of one fused [B, T, Hq+2*Hkv, d] projection:
    rotated in place, with the same bits as out of place; v and a padding head keep theirs."""
    B, T, Hq, Hkv, d = 2, 300, 6, 2, 64
    g = torch.Generator().manual_seed(21)
    qkv = torch.randn((B, T, Hq + 2 * Hkv + 1, d), generator=g).to(torch.bfloat16).to(DEV)
    before = qkv.clone()
    q, k, v = qkv[:, :, :Hq], qkv[:, :, Hq:Hq + Hkv], qkv[:, :, Hq + Hkv:Hq + 2 * Hkv]
    o_ref, lse_ref, qr_ref, kr_ref = gqa.attn_fwd_rope(q.contiguous(), k.contiguous(), v.contiguous())
    o, lse, qr, kr = gqa.attn_fwd_rope(q, k, v, q_rot=q, k_rot=k)
    assert gqa.attn_sync_status() == gqa.GQA_OK, gqa.attn_last_error()
    assert qr.data_ptr() == q.data_ptr() and kr.data_ptr() == k.data_ptr()
    for a, b in ((o, o_ref), (lse, lse_ref), (qkv[:, :, :Hq], qr_ref), (qkv[:, :, Hq:Hq + Hkv], kr_ref)):
        assert torch.equal(bits(a), bits(b))
    assert torch.equal(bits(qkv[:, :, Hq + Hkv:]), bits(before[:, :, Hq + Hkv:]))


@pytest.mark.parametrize("name", ["c3", "c4"])
def test_fused_full_size(name):
    """Full-size workloads in the launch configuration the benchmark times: o, lse and dv
    bit-identical to the plain kernels on q_rot, k_rot; dq and dk within the rounding of
    rotating those kernels' bf16 gradients back; sampled rotated rows against the oracle;
    repeated runs give the same bits."""
    w = WORKLOADS[name]
    q, k, v, dout = workload_inputs(w)
    qd, kd, vd, dod = (x.to(DEV) for x in (q, k, v, dout))
    fus = fused(qd, kd, vd, dod, w.causal)
    again = fused(qd, kd, vd, dod, w.causal)
    pl = plain_on(fus, vd, dod, w.causal)
    assert gqa.attn_sync_status() == gqa.GQA_OK, gqa.attn_last_error()
    for key in ("o", "lse", "dv"):
        assert torch.equal(bits(fus[key]), bits(pl[key])), f"{key} differs from the plain kernels"
    for key in fus:
        assert torch.equal(bits(fus[key]), bits(again[key])), f"{key} not bit-identical across runs"
    table = gqa.attn_rope_table(w.T, w.d, base=BASE)
    for key in ("dq", "dk"):
        sep = gqa.attn_rope(pl[key + "_rot"], table, inverse=True, y=torch.empty_like(pl[key + "_rot"]))
        err = rel_fro(f64(fus[key]), f64(sep))
        assert err <= 4e-3, f"{key}: rel-F {err:.2e} from the plain gradients rotated back"
    # rotation of sampled batches/tokens (the oracle on all of q would take minutes)
    rows = torch.tensor([0, 1, 127, 128, w.T // 2, w.T - 1])
    for src, got in ((q, fus["q_rot"]), (k, fus["k_rot"])):
        x = src[:, :, :2].contiguous()
        y = got[:, :, :2].cpu()
        full = rotation_excess_rows(y, x, rows)
        assert full <= 0.0, f"rotated rows beyond their bound by {full:.3e}"


def rotation_excess_rows(y, x, rows):
    ref = oracle.rope(x, base=BASE)[:, rows]
    yy, xa = f64(y)[:, rows], np.abs(f64(x))[:, rows]
    pair = np.repeat(xa[..., 0::2] + xa[..., 1::2], 2, axis=-1)
    return float(np.max(np.abs(yy - ref) - half_ulp_bf16(ref) - 2e-6 * pair - 1e-30))
