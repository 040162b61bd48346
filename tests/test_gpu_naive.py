"""GPU: the naive attention (plain kernels that write the whole score matrix,
"A transformer in PTX", §Three ways to run it) and the flash kernels against it.

First the naive path is tied to the f64 oracle element by element on small
shapes, with the oracle tolerances. Then, at the full workload sizes, the flash
kernels are compared with it on every element of every (batch, head) — where the
oracle can only check sampled groups. Both paths round P (and dS) to bf16 and
return bf16, so they differ by bf16-level rounding; the bar is the oracle
tolerances (O: 1e-2, LSE: 1e-3, gradients: relative Frobenius 1e-2), checked per
(batch, head) for O and LSE and per tensor for the gradients, plus per-group
gradient errors below 2e-2. Against the oracle O may differ by half a bf16 ulp
before the 1e-2 applies (one rounding); here both sides are rounded bf16 values,
so two correct results may differ by a full ulp before it applies.
"""
import numpy as np
import pytest
import torch

import causal_gqa_flash_gb300 as gqa
import oracle
from causal_gqa_flash_gb300.inputs import WORKLOADS, make_inputs, workload_inputs

from _helpers import TOL_GRAD, TOL_LSE, TOL_O, check_against_oracle

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")


@pytest.fixture(scope="module", autouse=True)
def _built():
    gqa.build()
    gqa.load()


def run_naive(q, k, v, dout, causal):
    o, lse = gqa.attn_fwd_naive(q, k, v, causal=causal)
    dq, dk, dv = gqa.attn_bwd_naive(q, k, v, o, lse, dout, causal=causal)
    assert gqa.attn_sync_status() == gqa.GQA_OK, gqa.attn_last_error()
    return dict(o=o, lse=lse, dq=dq, dk=dk, dv=dv)


@pytest.mark.parametrize("case", [
    (1, 128, 6, 2, 64, True), (2, 300, 4, 1, 128, True), (1, 200, 4, 2, 64, False), (1, 1, 2, 1, 64, True),
    (1, 77, 3, 3, 128, False),
], ids=lambda c: "B{}_T{}_Hq{}_Hkv{}_d{}_{}".format(c[0], c[1], c[2], c[3], c[4], "causal" if c[5] else "full"))
def test_naive_against_oracle(case):
    B, T, Hq, Hkv, d, causal = case
    q, k, v, dout = make_inputs(B, T, Hq, Hkv, d, seed=900 + T + d)
    out = run_naive(*(x.to(DEV) for x in (q, k, v, dout)), causal)
    check_against_oracle(out, oracle.bwd(q, k, v, dout, causal=causal), f"naive {case}")


def ulp_bf16(r):
    """Spacing of bf16 numbers at |r| (8 significant bits)."""
    mag = torch.clamp(r.abs(), min=2.0 ** -126)
    return torch.ldexp(torch.ones_like(mag), torch.floor(torch.log2(mag)).to(torch.int32) - 7)


def rel_fro(a, r):
    a, r = a.double(), r.double()
    return float(torch.linalg.vector_norm(a - r) / torch.linalg.vector_norm(r))


@pytest.mark.parametrize("name", ["c3", "c4", "c5"])
def test_flash_against_naive_full_size(name):
    w = WORKLOADS[name]
    q, k, v, dout = (x.to(DEV) for x in workload_inputs(w))
    B, T, Hq, d = q.shape
    Hkv = k.shape[2]
    G = Hq // Hkv
    o, lse = gqa.attn_fwd(q, k, v, causal=w.causal)
    dq, dk, dv = gqa.attn_bwd(q, k, v, o, lse, dout, causal=w.causal)
    assert gqa.attn_sync_status() == gqa.GQA_OK, gqa.attn_last_error()
    ref = run_naive(q, k, v, dout, w.causal)
    torch.cuda.synchronize()
    # O and LSE of every (batch, head)
    of, on = o.float(), ref["o"].float()
    e_o = (of - on).abs() - ulp_bf16(on)
    e_o_bh = e_o.amax(dim=(1, 3))                       # [B, Hq]
    e_l_bh = (lse - ref["lse"]).abs().amax(dim=2)       # [B, Hq]
    worst_o = np.unravel_index(int(e_o_bh.argmax()), e_o_bh.shape)
    worst_l = np.unravel_index(int(e_l_bh.argmax()), e_l_bh.shape)
    msg = (f"{name}: O {float(e_o_bh.max()):.2e} beyond one bf16 ulp at (b, h) {worst_o}, "
           f"LSE {float(e_l_bh.max()):.2e} at {worst_l}")
    # gradients: whole tensors and every (batch, kv group)
    errs = {nm: rel_fro(a, ref[nm]) for nm, a in (("dq", dq), ("dk", dk), ("dv", dv))}
    grp = []
    for b in range(B):
        for g in range(Hkv):
            hs = slice(g * G, (g + 1) * G)
            grp.append(max(rel_fro(dq[b, :, hs], ref["dq"][b, :, hs]), rel_fro(dk[b, :, g], ref["dk"][b, :, g]),
                           rel_fro(dv[b, :, g], ref["dv"][b, :, g])))
    msg += f", dQ {errs['dq']:.2e} dK {errs['dk']:.2e} dV {errs['dv']:.2e}, worst group {max(grp):.2e}"
    print(msg)
    assert bool(torch.isfinite(of).all()) and bool(torch.isfinite(lse).all()), msg
    assert float(e_o_bh.max()) <= TOL_O and float(e_l_bh.max()) <= TOL_LSE, msg
    assert max(errs.values()) <= TOL_GRAD and max(grp) <= 2 * TOL_GRAD, msg


@pytest.mark.parametrize("case", [(1, 32767, 2, 1, 128, True), (1, 16385, 4, 1, 64, True)],
                         ids=lambda c: "B{}_T{}_Hq{}_Hkv{}_d{}".format(*c[:5]))
def test_flash_against_naive_long_context(case):
    """Sequences far beyond what the CPU oracle can hold (a T x T f64 matrix per head):
    256 key tiles per row at T = 32767, so the running max is rescaled across hundreds
    of tiles; ragged ends one row past and one row short of a tile boundary."""
    B, T, Hq, Hkv, d, causal = case
    q, k, v, dout = (x.to(DEV) for x in make_inputs(B, T, Hq, Hkv, d, seed=T))
    o, lse = gqa.attn_fwd(q, k, v, causal=causal)
    dq, dk, dv = gqa.attn_bwd(q, k, v, o, lse, dout, causal=causal)
    assert gqa.attn_sync_status() == gqa.GQA_OK, gqa.attn_last_error()
    ref = run_naive(q, k, v, dout, causal)
    e_o = float(((o.float() - ref["o"].float()).abs() - ulp_bf16(ref["o"].float())).max())
    e_l = float((lse - ref["lse"]).abs().max())
    errs = {nm: rel_fro(a, ref[nm]) for nm, a in (("dq", dq), ("dk", dk), ("dv", dv))}
    msg = f"{case}: O {e_o:.2e} beyond one bf16 ulp, LSE {e_l:.2e}, " + ", ".join(
        f"{nm} {e:.2e}" for nm, e in errs.items())
    print(msg)
    assert e_o <= TOL_O and e_l <= TOL_LSE and max(errs.values()) <= TOL_GRAD, msg
