"""Measured rates of this GPU's tensor core and ex2 unit (one CTA per SM).

    python -m causal_gqa_flash_gb300.probe [--iters N]

prints one JSON line: tcgen05 bf16 MMA FLOP per cycle per SM for N = 64, 128, 256
with A in shared memory ("ss") or tensor memory ("ts"), ex2 lanes per cycle per SM,
the SM clock seen during the MMA probes, the best MMA rate at that clock over
all SMs in TFLOP/s, and the TMA tile-load rate from the L2 and from HBM with the
load latency it implies ("tma"). "Talking to the GPU", §The real tensor core peak: measure the
unit's real rate with enough independent work per SM instead of trusting the data
sheet. The kernels are attn_probe_mma / attn_probe_ex2 / attn_probe_tma of the library.
"""
from __future__ import annotations

import argparse
import json


def main() -> int:
    ap = argparse.ArgumentParser()
    ap.add_argument("--iters", type=int, default=4096)
    args = ap.parse_args()
    import causal_gqa_flash_gb300 as gqa
    gqa.build()
    res = gqa.probe_rates(iters=args.iters)
    res["tma"] = gqa.probe_tma()
    print(json.dumps(res), flush=True)
    return 0


if __name__ == "__main__":
    raise SystemExit(main())
