"""The backward entry point that allocates nothing (attn_bwd_noalloc).

It is for callers that may not allocate device memory where they run the
backward, so its scratch is a fixed array inside the library. It runs the
preprocess and the dQ and dK/dV task launch (attn_bwd_preprocess and
attn_bwd_dq_dkv), whose scratch is small. Called through the C ABI twice in a
row (different shapes, so the second call meets the first call's leftovers in
the shared array), its dQ/dK/dV must equal those of the same two stages given
a caller workspace (the same kernels on the same inputs: the same bytes), and
agree with attn_bwd within the tolerance of the parity tests. A warmed-up call
must leave the device's free memory unchanged.
This file is collected last on purpose.
"""
import ctypes

import pytest
import torch

import causal_gqa_flash_gb300 as gqa
from causal_gqa_flash_gb300.inputs import make_inputs

from _helpers import TOL_GRAD, f64, rel_fro

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")


@pytest.fixture(scope="module")
def lib():
    gqa.build()
    return gqa.load()


def _p(t):
    return ctypes.c_void_p(t.data_ptr())


@pytest.mark.parametrize("shapes", [[(2, 700, 6, 2, 64, 11), (1, 300, 4, 1, 128, 12)]])
def test_noalloc_matches_workspace_backward(lib, shapes):
    for B, T, Hq, Hkv, d, seed in shapes:
        q, k, v, dout = (x.to(DEV) for x in make_inputs(B, T, Hq, Hkv, d, seed=seed))
        o, lse = gqa.attn_fwd(q, k, v, causal=True)
        full = gqa.attn_bwd(q, k, v, o, lse, dout, causal=True)  # caller-provided workspace
        ws = torch.empty(gqa.attn_bwd_workspace_bytes(B, T, Hq), dtype=torch.uint8, device=DEV)
        ref = tuple(torch.empty_like(x) for x in (q, k, v))
        gqa.attn_bwd_preprocess(o, lse, dout, ws)
        gqa.attn_bwd_dq_dkv(q, k, v, dout, *ref, ws, causal=True)
        dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
        stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
        rc = lib.attn_bwd_noalloc(_p(q), _p(k), _p(v), _p(o), _p(lse), _p(dout), _p(dq), _p(dk), _p(dv), B, T, Hq,
                                  Hkv, d, 1, stream)
        assert rc == gqa.GQA_OK, gqa.attn_last_error()
        assert gqa.attn_sync_status() == gqa.GQA_OK, gqa.attn_last_error()
        for i, (name, a) in enumerate((("dq", dq), ("dk", dk), ("dv", dv))):
            err = rel_fro(f64(a), f64(full[i]))
            print(f"B={B} T={T} Hq={Hq} Hkv={Hkv} d={d} {name}: rel-F {err:.2e} against attn_bwd")
            assert err <= TOL_GRAD, (name, err)
            assert torch.equal(a.view(torch.int16), ref[i].view(torch.int16)), name


def test_noalloc_allocates_no_device_memory(lib):
    B, T, Hq, Hkv, d = 2, 513, 6, 2, 64
    q, k, v, dout = (x.to(DEV) for x in make_inputs(B, T, Hq, Hkv, d, seed=21))
    o, lse = gqa.attn_fwd(q, k, v, causal=True)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    args = (_p(q), _p(k), _p(v), _p(o), _p(lse), _p(dout), _p(dq), _p(dk), _p(dv), B, T, Hq, Hkv, d, 1, stream)
    assert lib.attn_bwd_noalloc(*args) == gqa.GQA_OK, gqa.attn_last_error()  # warm-up (symbol lookup)
    torch.cuda.synchronize()
    free0 = torch.cuda.mem_get_info(DEV)[0]
    assert lib.attn_bwd_noalloc(*args) == gqa.GQA_OK, gqa.attn_last_error()
    torch.cuda.synchronize()
    free1 = torch.cuda.mem_get_info(DEV)[0]
    assert gqa.attn_sync_status() == gqa.GQA_OK, gqa.attn_last_error()
    assert free1 == free0, (free0, free1)


def test_noalloc_rejects_problems_beyond_its_scratch(lib):
    fake = ctypes.c_void_p(0x100000)  # never dereferenced: the size check comes first
    B, T, Hq = 1, 1 << 17, 16        # needs 2 * 16 * 131072 * 4 bytes = 16 MiB > 8 MiB
    assert gqa.attn_bwd_workspace_bytes(B, T, Hq) > gqa.NOALLOC_SCRATCH_BYTES
    rc = lib.attn_bwd_noalloc(*([fake] * 9), B, T, Hq, 2, 64, 1, None)
    assert rc == gqa.GQA_ERR_INVALID_ARG
    msg = gqa.attn_last_error()
    assert "more than the library's fixed" in msg
    # the row limit it states leaves room for the 256 bytes of task counters
    assert f"<= {(gqa.NOALLOC_SCRATCH_BYTES - 256) // 8}" in msg, msg
