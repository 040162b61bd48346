"""GPU: the strided entry points (attn_fwd_strided, attn_bwd_strided) on views.

q, k and v are read straight out of one fused [B, T, Hq + 2*Hkv, d] projection
buffer ("A transformer in PTX", §The model: one fused matmul computes queries,
keys and values) or out of sequence-first [T, B, H, d] tensors; o and the
gradients are written into parts of wider buffers. Every output must be
bit-identical to the contiguous entry points on the same values, and every
element of the wider buffers outside the views must keep its sentinel. One case
is also checked against the f64 oracle.
"""
import pytest
import torch

import causal_gqa_flash_gb300 as gqa
import oracle
from causal_gqa_flash_gb300.inputs import make_inputs

from _helpers import check_against_oracle

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")
SENTINEL = -3.25  # exact in bf16


@pytest.fixture(scope="module", autouse=True)
def _built():
    gqa.build()
    gqa.load()


def contiguous_reference(q, k, v, dout, causal):
    o, lse = gqa.attn_fwd(q, k, v, causal=causal)
    dq, dk, dv = gqa.attn_bwd(q, k, v, o, lse, dout, causal=causal)
    torch.cuda.synchronize()
    return o, lse, dq, dk, dv


def same_bits(a, b):
    return torch.equal(a.contiguous().view(torch.int16), b.contiguous().view(torch.int16))


CASES = [
    # B, T, Hq, Hkv, d, causal
    (2, 300, 6, 2, 64, True),     # ragged, the trainer's head layout
    (1, 520, 4, 1, 128, True),    # d = 128 (pointer-store backward epilogue), G = 4
    (3, 200, 4, 2, 64, False),    # full attention
    (2, 129, 2, 2, 128, False),   # plain multi-head, d = 128, a row into a second tile
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "B{}_T{}_Hq{}_Hkv{}_d{}_{}".format(
    c[0], c[1], c[2], c[3], c[4], "causal" if c[5] else "full"))
def test_fused_qkv_views_bit_identical(case):
    B, T, Hq, Hkv, d, causal = case
    q, k, v, dout = (x.to(DEV) for x in make_inputs(B, T, Hq, Hkv, d, seed=31 + T + d))
    ref = contiguous_reference(q, k, v, dout, causal)

    # fused projection [B, T, Hq + 2*Hkv + 1, d]: q | k | v | one unused head
    H3 = Hq + 2 * Hkv
    qkv = torch.full((B, T, H3 + 1, d), SENTINEL, dtype=torch.bfloat16, device=DEV)
    qkv[:, :, :Hq] = q
    qkv[:, :, Hq:Hq + Hkv] = k
    qkv[:, :, Hq + Hkv:H3] = v
    qv, kv_, vv = qkv[:, :, :Hq], qkv[:, :, Hq:Hq + Hkv], qkv[:, :, Hq + Hkv:H3]
    # o into heads [1, Hq + 1) of a [B, T, Hq + 2, d] buffer; dO read from a wider buffer too
    obuf = torch.full((B, T, Hq + 2, d), SENTINEL, dtype=torch.bfloat16, device=DEV)
    ov = obuf[:, :, 1:Hq + 1]
    dobuf = torch.full((B, T, Hq + 1, d), SENTINEL, dtype=torch.bfloat16, device=DEV)
    dobuf[:, :, 1:] = dout
    dov = dobuf[:, :, 1:]
    # gradients into one fused [B, T, Hq + 2*Hkv + 1, d] buffer
    dqkv = torch.full((B, T, H3 + 1, d), SENTINEL, dtype=torch.bfloat16, device=DEV)
    dqv, dkv_, dvv = dqkv[:, :, :Hq], dqkv[:, :, Hq:Hq + Hkv], dqkv[:, :, Hq + Hkv:H3]

    o, lse = gqa.attn_fwd_strided(qv, kv_, vv, ov, causal=causal)
    gqa.attn_bwd_strided(qv, kv_, vv, ov, lse, dov, dqv, dkv_, dvv, causal=causal)
    assert gqa.attn_sync_status() == gqa.GQA_OK, gqa.attn_last_error()

    for name, a, r in (("o", ov, ref[0]), ("dq", dqv, ref[2]), ("dk", dkv_, ref[3]), ("dv", dvv, ref[4])):
        assert same_bits(a, r), f"{name} differs from the contiguous path"
    assert torch.equal(lse, ref[1])
    for name, buf, untouched in (("o", obuf, [obuf[:, :, 0], obuf[:, :, Hq + 1]]), ("dqkv", dqkv, [dqkv[:, :, H3]]),
                                 ("qkv", qkv, [qkv[:, :, H3]])):
        for u in untouched:
            assert bool((u == SENTINEL).all()), f"a store outside the views of {name}"


@pytest.mark.parametrize("d", [64, 128])
def test_sequence_first_views_bit_identical(d):
    """[T, B, H, d] tensors read and written in place (batch stride H*d, token stride B*H*d)."""
    B, T, Hq, Hkv = 3, 260, 4, 2
    q, k, v, dout = (x.to(DEV) for x in make_inputs(B, T, Hq, Hkv, d, seed=77 + d))
    ref = contiguous_reference(q, k, v, dout, True)

    def seq_first(x):
        return x.transpose(0, 1).contiguous().transpose(0, 1)  # [B,T,H,d] view of a [T,B,H,d] buffer

    qs, ks, vs, dos = (seq_first(x) for x in (q, k, v, dout))
    assert qs.stride(0) == Hq * d and qs.stride(1) == B * Hq * d
    os_ = seq_first(torch.full_like(q, SENTINEL))
    dqs, dks, dvs = (seq_first(torch.full_like(x, SENTINEL)) for x in (q, k, v))
    _, lse = gqa.attn_fwd_strided(qs, ks, vs, os_, causal=True)
    gqa.attn_bwd_strided(qs, ks, vs, os_, lse, dos, dqs, dks, dvs, causal=True)
    assert gqa.attn_sync_status() == gqa.GQA_OK, gqa.attn_last_error()
    for name, a, r in (("o", os_, ref[0]), ("dq", dqs, ref[2]), ("dk", dks, ref[3]), ("dv", dvs, ref[4])):
        assert same_bits(a, r), f"{name} differs from the contiguous path"
    assert torch.equal(lse, ref[1])


def test_fused_views_against_oracle():
    """The strided path on a fused buffer, element by element against the f64 oracle."""
    B, T, Hq, Hkv, d = 2, 333, 6, 2, 64
    q, k, v, dout = make_inputs(B, T, Hq, Hkv, d, seed=404)
    H3 = Hq + 2 * Hkv
    qkv = torch.cat([q, k, v], dim=2).to(DEV)
    qv, kv_, vv = qkv[:, :, :Hq], qkv[:, :, Hq:Hq + Hkv], qkv[:, :, Hq + Hkv:H3]
    dqkv = torch.empty((B, T, H3, d), dtype=torch.bfloat16, device=DEV)
    o = torch.empty((B, T, Hq, d), dtype=torch.bfloat16, device=DEV)
    _, lse = gqa.attn_fwd_strided(qv, kv_, vv, o, causal=True)
    gqa.attn_bwd_strided(qv, kv_, vv, o, lse, dout.to(DEV), dqkv[:, :, :Hq], dqkv[:, :, Hq:Hq + Hkv],
                         dqkv[:, :, Hq + Hkv:], causal=True)
    assert gqa.attn_sync_status() == gqa.GQA_OK, gqa.attn_last_error()
    out = dict(o=o, lse=lse, dq=dqkv[:, :, :Hq], dk=dqkv[:, :, Hq:Hq + Hkv], dv=dqkv[:, :, Hq + Hkv:])
    ref = oracle.bwd(q, k, v, dout, causal=True)
    check_against_oracle(out, ref, "fused qkv views")


def test_strided_rejects_unpacked_heads():
    q, k, v, _ = (x.to(DEV) for x in make_inputs(1, 128, 4, 2, 64, seed=3))
    with pytest.raises(ValueError):
        gqa.attn_fwd_strided(q.transpose(1, 2).contiguous().transpose(1, 2), k, v, torch.empty_like(q))
