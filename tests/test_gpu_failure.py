"""Failure detection without a GPU fault: a kernel whose wait runs out of budget
records GQA_ERR_TIMEOUT in the device status word and returns; the host reads
it, the word is cleared, and the context stays usable."""
import pytest
import torch

import causal_gqa_flash_gb300 as gqa
from causal_gqa_flash_gb300.inputs import make_inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    gqa.build()
    gqa.load()


def test_wait_timeout_is_reported_and_cleared():
    assert gqa.attn_sync_status() == gqa.GQA_OK
    gqa.attn_selftest_timeout(2_000_000)  # 2 ms budget on a barrier nobody arrives at
    assert gqa.attn_sync_status() == gqa.GQA_ERR_TIMEOUT
    assert "selftest" in gqa.attn_last_error()
    assert gqa.attn_sync_status() == gqa.GQA_OK  # read-and-clear


def test_context_usable_after_timeout():
    gqa.attn_selftest_timeout(1_000_000)
    assert gqa.attn_sync_status() == gqa.GQA_ERR_TIMEOUT
    q, k, v, dout = (x.cuda() for x in make_inputs(1, 256, 4, 2, 64, seed=3))
    o, lse = gqa.attn_fwd(q, k, v)
    dq, dk, dv = gqa.attn_bwd(q, k, v, o, lse, dout)
    assert gqa.attn_sync_status() == gqa.GQA_OK
    assert torch.isfinite(o.float()).all() and torch.isfinite(dq.float()).all()
