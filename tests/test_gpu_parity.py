"""GPU parity: the CUDA path (through the C ABI) against the f64 CPU oracle,
element by element, on seeded bf16 inputs at sizes the oracle finishes in
seconds: several tiles, ragged tails, T = 1, several GQA ratios, both head
dims, causal and full attention. Guard bytes around every output catch
stores outside it; repeated calls must give identical bytes.

Tolerances (fixed by the method's target): O max abs error <= 1e-2, LSE max
abs error <= 1e-3, dQ/dK/dV relative Frobenius error <= 1e-2.
"""
import pytest
import torch

import causal_gqa_flash_gb300 as gqa
import oracle
from causal_gqa_flash_gb300.inputs import WORKLOADS, make_inputs, workload_inputs

from _helpers import Guarded, check_against_oracle

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")


@pytest.fixture(scope="module", autouse=True)
def _built():
    gqa.build()
    gqa.load()


def run_gpu(q, k, v, dout, causal):
    B, T, Hq, d = q.shape
    Hkv = k.shape[2]
    qd, kd, vd, dod = (x.to(DEV).contiguous() for x in (q, k, v, dout))
    go = Guarded((B, T, Hq, d), torch.bfloat16, DEV)
    gl = Guarded((B, Hq, T), torch.float32, DEV)
    gdq = Guarded((B, T, Hq, d), torch.bfloat16, DEV)
    gdk = Guarded((B, T, Hkv, d), torch.bfloat16, DEV)
    gdv = Guarded((B, T, Hkv, d), torch.bfloat16, DEV)
    gqa.attn_fwd(qd, kd, vd, causal=causal, o=go.tensor, lse=gl.tensor)
    gqa.attn_bwd(qd, kd, vd, go.tensor, gl.tensor, dod, causal=causal, dq=gdq.tensor, dk=gdk.tensor,
                 dv=gdv.tensor)
    assert gqa.attn_sync_status() == gqa.GQA_OK, gqa.attn_last_error()
    for name, g in (("o", go), ("lse", gl), ("dq", gdq), ("dk", gdk), ("dv", gdv)):
        assert g.intact(), f"store outside {name}"
    return dict(o=go.tensor, lse=gl.tensor, dq=gdq.tensor, dk=gdk.tensor, dv=gdv.tensor)


CASES = [
    # B, T, Hq, Hkv, d, causal, qk_std
    (1, 128, 6, 2, 64, True, 1.0),     # one tile, the trainer's head layout
    (1, 1, 2, 1, 64, True, 1.0),       # a single token
    (1, 2, 4, 4, 64, True, 1.0),       # plain multi-head, two tokens
    (2, 127, 4, 2, 64, True, 1.0),     # ragged single tile
    (1, 129, 4, 1, 128, True, 1.0),    # one row into a second tile, d=128, G=4
    (1, 255, 8, 1, 64, True, 1.0),     # G=8
    (2, 300, 4, 1, 128, True, 2.0),    # ragged, large logits
    (1, 384, 6, 2, 64, True, 1.0),     # three full tiles
    (1, 640, 4, 2, 128, True, 1.0),    # five tiles, d=128
    (1, 200, 4, 2, 64, False, 1.0),    # full attention, ragged
    (1, 256, 2, 2, 128, False, 1.0),   # full attention, d=128
    (1, 333, 6, 3, 64, False, 2.0),    # full attention, ragged, large logits
    # more 128-query items than the d = 64 forward's persistent CTAs (2 per SM), so
    # CTAs run several items back to back
    (4, 1500, 8, 2, 64, True, 1.0),    # causal, ragged, 384 items
    (4, 1000, 12, 4, 64, False, 1.0),  # full attention, ragged, 384 items of equal cost
    # runs of short items (one or two key tiles) back to back: a CTA's next item can
    # start before its query tile has landed in the other buffer
    (48, 256, 8, 2, 64, True, 1.0),    # 768 items of 1-2 tiles
    (64, 128, 8, 2, 64, False, 1.0),   # 512 single-tile items
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "B{}_T{}_Hq{}_Hkv{}_d{}_{}_s{}".format(
    c[0], c[1], c[2], c[3], c[4], "causal" if c[5] else "full", c[6]))
def test_parity_small(case):
    B, T, Hq, Hkv, d, causal, std = case
    q, k, v, dout = make_inputs(B, T, Hq, Hkv, d, seed=17 + T + d, qk_std=std)
    out = run_gpu(q, k, v, dout, causal)
    ref = oracle.bwd(q, k, v, dout, causal=causal)
    check_against_oracle(out, ref, str(case))


@pytest.mark.parametrize("name", ["c1", "c2"])
def test_parity_workload(name):
    """The small workloads in full, element by element."""
    w = WORKLOADS[name]
    q, k, v, dout = workload_inputs(w)
    out = run_gpu(q, k, v, dout, w.causal)
    ref = oracle.bwd(q, k, v, dout, causal=w.causal)
    check_against_oracle(out, ref, name)


@pytest.mark.parametrize("name", ["c1", "c2"])
def test_bit_identical_across_runs(name):
    """No float atomics: three calls give the same bytes (fwd and bwd). The larger
    workloads repeat in test_gpu_fullsize.py."""
    w = WORKLOADS[name]
    q, k, v, dout = (x.to(DEV) for x in workload_inputs(w))
    outs = []
    for _ in range(3):
        o, lse = gqa.attn_fwd(q, k, v, causal=w.causal)
        dq, dk, dv = gqa.attn_bwd(q, k, v, o, lse, dout, causal=w.causal)
        torch.cuda.synchronize()
        outs.append([t.clone() for t in (o, lse, dq, dk, dv)])
    for other in outs[1:]:
        for a, b in zip(outs[0], other):
            assert torch.equal(a.view(torch.uint8), b.view(torch.uint8))


def test_user_stream_and_outputs_overwritten():
    """Work goes on the caller's stream; stale output contents never leak in."""
    q, k, v, dout = (x.to(DEV) for x in make_inputs(1, 300, 4, 2, 64, seed=5))
    s = torch.cuda.Stream()
    o = torch.full_like(q, 7.0)
    lse = torch.full((1, 4, 300), 3.0, device=DEV)
    dq, dk, dv = torch.full_like(q, 9.0), torch.full_like(k, 9.0), torch.full_like(v, 9.0)
    with torch.cuda.stream(s):
        gqa.attn_fwd(q, k, v, o=o, lse=lse, stream=s)
        gqa.attn_bwd(q, k, v, o, lse, dout, dq=dq, dk=dk, dv=dv, stream=s)
    s.synchronize()
    o2, lse2 = gqa.attn_fwd(q, k, v)
    dq2, dk2, dv2 = gqa.attn_bwd(q, k, v, o2, lse2, dout)
    torch.cuda.synchronize()
    for a, b in ((o, o2), (lse, lse2), (dq, dq2), (dk, dk2), (dv, dv2)):
        assert torch.equal(a, b)


def test_bad_arguments_on_gpu():
    q, k, v, dout = (x.to(DEV) for x in make_inputs(1, 128, 6, 2, 64, seed=1))
    with pytest.raises(gqa.AttnError) as e:
        gqa.attn_fwd(q[:, :, :5].contiguous(), k, v)  # Hq=5 over Hkv=2
    assert e.value.code == gqa.GQA_ERR_INVALID_ARG
    assert gqa.attn_sync_status() == gqa.GQA_OK


@pytest.mark.parametrize("name", ["c2", "c5"])
def test_repeated_steps_no_timeout(name):
    """Pipeline barriers under repetition: 40 fwd+bwd steps, every one must end with
    a clean status word and the same bytes (a phase race shows up as a timeout or
    as different bits)."""
    w = WORKLOADS[name]
    q, k, v, dout = (x.to(DEV) for x in workload_inputs(w))
    ref = None
    for i in range(40):
        o, lse = gqa.attn_fwd(q, k, v, causal=True)
        dq, dk, dv = gqa.attn_bwd(q, k, v, o, lse, dout, causal=True)
        assert gqa.attn_sync_status() == gqa.GQA_OK, f"step {i}: {gqa.attn_last_error()}"
        cur = [t.clone() for t in (o, lse, dq, dk, dv)]
        if ref is None:
            ref = cur
        else:
            for a, b in zip(ref, cur):
                assert torch.equal(a.view(torch.uint8), b.view(torch.uint8)), f"step {i}"


@pytest.mark.parametrize("B,T,Hq,Hkv,d,causal", [
    (2, 1000, 6, 2, 64, True),
    (1, 2048, 8, 2, 128, True),
    (3, 700, 9, 3, 64, False),
])
def test_task_orders_give_identical_bits(B, T, Hq, Hkv, d, causal):
    """The backward's task order (tile-major, group-major, or chosen by size) only moves
    the time: every output element has one owner and a fixed summation order."""
    q, k, v, dout = (x.to(DEV) for x in make_inputs(B, T, Hq, Hkv, d, seed=4242 + T))
    o, lse = gqa.attn_fwd(q, k, v, causal=causal)
    outs = []
    try:
        for order in (1, 2, 0):
            gqa.attn_set_task_order(order)
            outs.append([t.clone() for t in gqa.attn_bwd(q, k, v, o, lse, dout, causal=causal)])
    finally:
        gqa.attn_set_task_order(0)
    assert gqa.attn_sync_status() == gqa.GQA_OK, gqa.attn_last_error()
    for other in outs[1:]:
        for a, b in zip(outs[0], other):
            assert torch.equal(a.view(torch.int16), b.view(torch.int16))
