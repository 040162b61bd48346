"""GPU parity at the full benchmark sizes, in the launch configuration the
benchmark times. The whole problem runs on the GPU; the oracle then checks
whole (batch, kv-head) groups — each an independent slice of the problem with
all of its query heads — element by element: O and LSE of every group against the
oracle's forward, and the gradients of the first and last group against its
backward. Every output is checked for finiteness, guard bytes and bit-identical
repeat runs.
"""
import numpy as np
import pytest
import torch

import causal_gqa_flash_gb300 as gqa
import oracle
from causal_gqa_flash_gb300.inputs import WORKLOADS, workload_inputs

from _helpers import TOL_GRAD, TOL_LSE, TOL_O, Guarded, f64, max_abs, o_err, rel_fro

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")


@pytest.fixture(scope="module", autouse=True)
def _built():
    gqa.build()
    gqa.load()


@pytest.mark.parametrize("name", ["c3", "c4", "c5"])
def test_fullsize_groups(name):
    w = WORKLOADS[name]
    q, k, v, dout = workload_inputs(w)
    B, T, Hq, d = q.shape
    Hkv = k.shape[2]
    G = Hq // Hkv
    qd, kd, vd, dod = (x.to(DEV) for x in (q, k, v, dout))
    go = Guarded((B, T, Hq, d), torch.bfloat16, DEV)
    gl = Guarded((B, Hq, T), torch.float32, DEV)
    gdq = Guarded((B, T, Hq, d), torch.bfloat16, DEV)
    gdk = Guarded((B, T, Hkv, d), torch.bfloat16, DEV)
    gdv = Guarded((B, T, Hkv, d), torch.bfloat16, DEV)
    gqa.attn_fwd(qd, kd, vd, causal=w.causal, o=go.tensor, lse=gl.tensor)
    gqa.attn_bwd(qd, kd, vd, go.tensor, gl.tensor, dod, causal=w.causal, dq=gdq.tensor, dk=gdk.tensor,
                 dv=gdv.tensor)
    assert gqa.attn_sync_status() == gqa.GQA_OK, gqa.attn_last_error()
    outs = [g.tensor.clone() for g in (go, gl, gdq, gdk, gdv)]
    for g in (go, gl, gdq, gdk, gdv):
        assert g.intact()
        assert torch.isfinite(g.tensor.float()).all()
    # repeat: identical bytes
    gqa.attn_fwd(qd, kd, vd, causal=w.causal, o=go.tensor, lse=gl.tensor)
    gqa.attn_bwd(qd, kd, vd, go.tensor, gl.tensor, dod, causal=w.causal, dq=gdq.tensor, dk=gdk.tensor,
                 dv=gdv.tensor)
    torch.cuda.synchronize()
    for a, g in zip(outs, (go, gl, gdq, gdk, gdv)):
        assert torch.equal(a.view(torch.uint8), g.tensor.view(torch.uint8))

    o, lse, dq, dk, dv = outs
    worst_o = worst_l = 0.0
    for b in range(B):
        for kv in range(Hkv):
            hs = slice(kv * G, (kv + 1) * G)
            ro, rl = oracle.fwd(q[b:b + 1, :, hs], k[b:b + 1, :, kv:kv + 1], v[b:b + 1, :, kv:kv + 1],
                                causal=w.causal)
            worst_o = max(worst_o, o_err(f64(o[b:b + 1, :, hs]), ro))
            worst_l = max(worst_l, max_abs(f64(lse[b:b + 1, hs]), rl))
    print(f"{name} every group: O {worst_o:.2e} beyond the bf16 half-ulp, LSE {worst_l:.2e}")
    assert worst_o <= TOL_O and worst_l <= TOL_LSE, (worst_o, worst_l)
    for b, kv in ((0, 0), (B - 1, Hkv - 1)):
        hs = slice(kv * G, (kv + 1) * G)
        ref = oracle.bwd(q[b:b + 1, :, hs], k[b:b + 1, :, kv:kv + 1], v[b:b + 1, :, kv:kv + 1],
                         dout[b:b + 1, :, hs], causal=w.causal)
        og = f64(o[b:b + 1, :, hs])
        e_o = o_err(og, ref["o"])
        raw_o = max_abs(og, ref["o"])
        e_l = max_abs(f64(lse[b:b + 1, hs]), ref["lse"])
        e_dq = rel_fro(f64(dq[b:b + 1, :, hs]), ref["dq"])
        e_dk = rel_fro(f64(dk[b:b + 1, :, kv:kv + 1]), ref["dk"])
        e_dv = rel_fro(f64(dv[b:b + 1, :, kv:kv + 1]), ref["dv"])
        msg = f"{name} b={b} kv={kv}: O {e_o:.2e} (raw {raw_o:.2e}) LSE {e_l:.2e} dQ {e_dq:.2e} dK {e_dk:.2e} dV {e_dv:.2e}"
        print(msg)
        assert e_o <= TOL_O and e_l <= TOL_LSE, msg
        assert max(e_dq, e_dk, e_dv) <= TOL_GRAD, msg
