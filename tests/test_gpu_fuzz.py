"""GPU: seeded random shapes against the f64 oracle.

The parity cases of test_gpu_parity.py are chosen by hand; these are drawn: batch
1-8, T from 1 to 1000 (mostly ragged), kv heads 1-4 with 1, 2, 3, 4 or 8 query heads
each, head dim 64 or 128, causal or full attention, and query/key scale 1 or 2. Each
shape runs the forward and the backward through the C ABI with guard bytes around
every output, is compared element by element with the oracle (the tolerances of the
parity tests), and is run a second time to check that the bytes repeat. The shapes
land on every pipeline path of the kernels: one item or task per CTA and several,
ring stages wrapping within and across tasks, single-tile and ragged last tiles.
"""
import random

import pytest
import torch

import causal_gqa_flash_gb300 as gqa
import oracle
from causal_gqa_flash_gb300.inputs import make_inputs

from _helpers import Guarded, check_against_oracle

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")


def shapes(n=24, seed=20260):
    rng = random.Random(seed)
    out = []
    for i in range(n):
        B = rng.randint(1, 8)
        T = rng.choice([1, rng.randint(2, 127), 128, rng.randint(129, 600), rng.randint(129, 600),
                        rng.randint(600, 1000)])
        Hkv = rng.randint(1, 4)
        G = rng.choice([1, 2, 3, 4, 8])
        d = rng.choice([64, 128])
        causal = rng.random() < 0.7
        std = rng.choice([1.0, 2.0])
        out.append((B, T, G * Hkv, Hkv, d, causal, std, 7000 + i))
    return out


@pytest.fixture(scope="module", autouse=True)
def _built():
    gqa.build()
    gqa.load()


def run(q, k, v, dout, causal):
    B, T, Hq, d = q.shape
    Hkv = k.shape[2]
    qd, kd, vd, dod = (x.to(DEV).contiguous() for x in (q, k, v, dout))
    g = {name: Guarded(shape, dt, DEV) for name, shape, dt in (
        ("o", (B, T, Hq, d), torch.bfloat16), ("lse", (B, Hq, T), torch.float32),
        ("dq", (B, T, Hq, d), torch.bfloat16), ("dk", (B, T, Hkv, d), torch.bfloat16),
        ("dv", (B, T, Hkv, d), torch.bfloat16))}
    gqa.attn_fwd(qd, kd, vd, causal=causal, o=g["o"].tensor, lse=g["lse"].tensor)
    gqa.attn_bwd(qd, kd, vd, g["o"].tensor, g["lse"].tensor, dod, causal=causal, dq=g["dq"].tensor,
                 dk=g["dk"].tensor, dv=g["dv"].tensor)
    assert gqa.attn_sync_status() == gqa.GQA_OK, gqa.attn_last_error()
    for name, buf in g.items():
        assert buf.intact(), f"store outside {name}"
    return {name: buf.tensor.clone() for name, buf in g.items()}


@pytest.mark.parametrize("case", shapes(), ids=lambda c: "B{}_T{}_Hq{}_Hkv{}_d{}_{}_s{}".format(
    c[0], c[1], c[2], c[3], c[4], "causal" if c[5] else "full", c[6]))
def test_random_shape_against_oracle(case):
    B, T, Hq, Hkv, d, causal, std, seed = case
    q, k, v, dout = make_inputs(B, T, Hq, Hkv, d, seed=seed, qk_std=std)
    first = run(q, k, v, dout, causal)
    check_against_oracle(first, oracle.bwd(q, k, v, dout, causal=causal), str(case))
    again = run(q, k, v, dout, causal)
    for name in first:
        assert torch.equal(first[name].view(torch.uint8), again[name].view(torch.uint8)), name
