"""The rate probes run on every SM and report plausible rates: the tcgen05 MMA
chain between 1/8 of and the nominal dense bf16 rate per SM (8192 FLOP per cycle at
M = 128 with N >= 128), wider N never slower per FLOP than N = 64, the ex2 unit
between 4 and 128 lanes per cycle per SM, and an SM clock of a few hundred MHz to
a few GHz while the probes ran."""
import pytest

import causal_gqa_flash_gb300 as gqa

pytestmark = pytest.mark.gpu


def test_probe_rates():
    gqa.build()
    r = gqa.probe_rates(iters=1024)
    print(r)
    for key, rate in r["mma"].items():
        assert 1024 < rate <= 8192 * 1.02, (key, rate)
    assert r["mma"]["ss_n128_one_acc"] >= 0.98 * r["mma"]["ss_n64_one_acc"]
    assert 4 <= r["ex2_lanes_per_clk"] <= 128
    assert 300 < r["sm_mhz_during_mma"] < 3000
    assert gqa.attn_sync_status() == gqa.GQA_OK


def test_probe_tma():
    """TMA tile loads: from a buffer that fits the L2 at least as fast as from one
    that does not, HBM between 1 and 12 TB/s, and a load latency between 0.1 and 20
    microseconds."""
    gqa.build()
    res = gqa.probe_tma(sizes_mb=(32, 1024), iters=500)
    print(res)
    by = {(r["buffer_mb"], r["ctas_per_sm"]): r for r in res}
    for cps in (1, 2):
        assert by[(32, cps)]["tbps"] >= 0.9 * by[(1024, cps)]["tbps"], by
        assert 1.0 < by[(1024, cps)]["tbps"] < 12.0, by
    for r in res:
        assert 0.1 < r["latency_us"] < 20.0, r
    assert gqa.attn_sync_status() == gqa.GQA_OK
