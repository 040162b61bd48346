#!/usr/bin/env python3
"""Benchmark of causal grouped-query flash attention, forward + backward, on GB300.

One step = one forward (attn_fwd) and one backward (preprocess, then dQ and dK/dV
in one launch) over
one batch of the workload, with inputs resident in HBM. The metric is causal
TFLOP/s of fwd+bwd with the standard count: fwd = 4*B*Hq*T^2*d/2 and
bwd = 2.5 * fwd (five matmuls; the dQ and dK/dV kernels actually run seven).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload c4|c1..c5|all] [--impl ours|reference]

The default workload is c4 (B=2 T=8192 Hq=32 Hkv=8 d=128, the largest): the
throughput targets are stated at T >= 4096. --workload all prints one line per
workload, c1, c2, c3 and c5 first and the c4 line last.

Under torchrun (N > 1) every rank runs its own replica of the workload on its
own GPU (the (batch, kv-head) units are independent: no collective is needed);
the time is the max over ranks and the value is the work of all ranks over it.

--impl reference times the f64 CPU oracle (the only reference this project has)
on the host cores, on a bounded sample of the same workload.

Rank 0 prints one JSON line.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "causal GQA flash-attn fwd+bwd TFLOP/s (bf16) and % of GB300 dense bf16 peak"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
L2_FLUSH_BYTES = 256 << 20  # twice the 129 MB L2


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--workload", default="c4",
                    help="c1..c5 or all (default c4, B=2 T=8192 Hq=32 Hkv=8 d=128, the largest single-GPU workload)")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true", help="skip the oracle timing leg")
    ap.add_argument("--layout", default="separate", choices=["separate", "fused"],
                    help="fused: q, k, v are views of one [B,T,Hq+2*Hkv,d] projection buffer and the gradients "
                         "go to one such buffer (attn_fwd_strided / attn_bwd_strided)")
    ap.add_argument("--rope", nargs="?", const="fused", default="none", choices=["none", "fused", "separate"],
                    help="with --layout fused: each step also applies the rotary embedding to q and k. fused (the "
                         "default of a bare --rope): attn_fwd_rope / attn_bwd_rope, the rotation inside the "
                         "attention kernels (keys in one pass); separate: attn_rope before attention and its "
                         "inverse on dq and dk after it")
    ap.add_argument("--profile-run", action="store_true",
                    help="timed steps only (no clock soak, e2e or oracle leg): the command profiled under ncu")
    return ap.parse_args()


def causal_pairs(T: int, causal: bool) -> float:
    return T * T / 2.0 if causal else float(T * T)


def fwd_flops(w) -> float:
    return 4.0 * w.B * w.Hq * causal_pairs(w.T, w.causal) * w.d


def step_flops(w) -> float:
    return 3.5 * fwd_flops(w)


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return json.load(f), "measured"
    except (OSError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


def config_dict(w, extra=None):
    d = {"workload": f"{w.name}: {w.describe()}", "B": w.B, "seq_len": w.T, "Hq": w.Hq, "Hkv": w.Hkv, "d": w.d,
         "causal": w.causal, "flop_convention": "fwd=4*B*Hq*T^2*d/2, bwd=2.5*fwd"}
    if extra:
        d.update(extra)
    return d


# ----------------------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi sampling of SM clock and throttle reasons while the GPU is busy."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    NAMES = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")

    def __init__(self, bus_id: str | None):
        self.bus_id = bus_id
        self.proc = None
        self.lines = []

    def start(self):
        cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "100"]
        if self.bus_id:
            cmd += ["-i", self.bus_id]
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        self.lines = [ln for ln in out.splitlines() if ln.strip()]

    def summary(self):
        sm, mx, reasons = [], [], set()
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for name, val in zip(self.NAMES, parts[5:9]):
                if val.lower() == "active":
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


def gpu_bus_id(torch, dev):
    try:
        p = torch.cuda.get_device_properties(dev)
        return f"{p.pci_domain_id:08X}:{p.pci_bus_id:02X}:{p.pci_device_id:02X}.0"
    except Exception:
        return None


# ----------------------------------------------------------------------------- traffic record
def max_over_ranks(torch, dist, value: float, world: int, device=None) -> float:
    """The largest `value` over all ranks (the slowest rank's time); the value
    itself when there is one rank. Works with NCCL on CUDA tensors and with
    gloo on CPU tensors."""
    if world <= 1:
        return float(value)
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_tflops(world: int, flops_per_step: float, steps: int, ms_total: float) -> float:
    """Work of all ranks (weak scaling: every rank runs the same steps) over the
    slowest rank's total time, in TFLOP/s."""
    return world * flops_per_step * steps / (ms_total * 1e-3) / 1e12


def packed_buffer(torch, specs, device=None, pin=False):
    """One flat uint8 buffer holding tensors of the given (shape, dtype), each at a
    256-byte aligned offset; returns the buffer and the tensor views."""
    offs, total = [], 0
    for shape, dt in specs:
        nbytes = int(torch.Size(shape).numel()) * torch.empty((), dtype=dt).element_size()
        offs.append((total, nbytes))
        total += (nbytes + 255) // 256 * 256
    buf = torch.empty(total, dtype=torch.uint8, device=device, pin_memory=pin)
    views = [buf[o:o + n].view(dt).view(shape) for (o, n), (shape, dt) in zip(offs, specs)]
    return buf, views


def kernel_source_hash(files):
    """Hash of the kernel sources' code: comments, blank lines and indentation
    are left out, so an edit to comments alone keeps the recorded counters."""
    h = hashlib.sha256()
    for f in files:
        with open(os.path.join(ROOT, "causal_gqa_flash_gb300", "csrc", f), encoding="utf-8") as fh:
            text = re.sub(r"/\*.*?\*/", "", fh.read(), flags=re.S)
        for line in text.splitlines():
            code = line.split("//", 1)[0].strip()
            if code:
                h.update(code.encode() + b"\n")
    return h.hexdigest()[:16]


KERNEL_SOURCES = {
    "attn_fwd_kernel": ["attn_fwd.cu", "attn_common.cuh", "sm103_ptx.cuh"],
    "bwd_pre_kernel": ["attn_bwd.cu", "attn_common.cuh", "sm103_ptx.cuh"],
    "bwd_main_kernel": ["attn_bwd.cu", "attn_common.cuh", "sm103_ptx.cuh"],
}


def recorded_counters(kernel: str, workload: str):
    """The committed ncu record of a kernel on a workload (DRAM bytes per launch and,
    where captured, the tensor pipe's active share), or None once the kernel's source
    has changed since the capture."""
    path = os.path.join(ROOT, "profiles", "dram_traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f)
    except (OSError, ValueError):
        return None
    ent = rec.get(kernel, {}).get(workload)
    if not ent or ent.get("source_sha256_16") != kernel_source_hash(KERNEL_SOURCES[kernel]):
        return None
    return ent


def recorded_traffic(kernel: str, workload: str):
    """DRAM bytes per launch from the committed ncu summary, if the kernel source is unchanged since."""
    ent = recorded_counters(kernel, workload)
    return None if ent is None else ent.get("dram_bytes_per_launch")


# ----------------------------------------------------------------------------- CPU oracle leg
def oracle_sample(w, min_seconds: float, max_seconds: float):
    """Time the f64 oracle (fwd+bwd) on whole (batch, kv-head) groups of the workload."""
    import oracle
    from causal_gqa_flash_gb300.inputs import workload_inputs

    q, k, v, dout = workload_inputs(w)
    G = w.Hq // w.Hkv
    groups = [(b, kv) for b in range(w.B) for kv in range(w.Hkv)]
    sl = []
    for b, kv in groups:
        hs = slice(kv * G, (kv + 1) * G)
        sl.append(tuple(x.double().numpy()[b:b + 1, :, s].copy() for x, s in
                        ((q, hs), (k, slice(kv, kv + 1)), (v, slice(kv, kv + 1)), (dout, hs))))
    group_flops = 3.5 * 4.0 * 1 * G * causal_pairs(w.T, w.causal) * w.d
    done = 0
    t0 = time.perf_counter()
    while True:
        qs, ks, vs, ds = sl[done % len(sl)]
        oracle.bwd(qs, ks, vs, ds, causal=w.causal)
        done += 1
        el = time.perf_counter() - t0
        if el >= min_seconds or el >= max_seconds:
            break
    return {"value": group_flops * done / el / 1e12, "seconds": el, "groups": done,
            "cores": oracle.max_threads(),
            "sample": f"{done} (batch, kv-head) groups of {w.name} (each {G} query heads x T={w.T}), "
                      f"f64 oracle fwd+bwd, {el:.1f} s"}


# ----------------------------------------------------------------------------- reference arm
def run_reference(args, w):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    import oracle
    from causal_gqa_flash_gb300.inputs import workload_inputs
    q, k, v, dout = workload_inputs(w)
    G = w.Hq // w.Hkv
    qs, ks, vs, ds = (x.double().numpy()[0:1, :, s].copy() for x, s in
                      ((q, slice(0, G)), (k, slice(0, 1)), (v, slice(0, 1)), (dout, slice(0, G))))
    sample_flops = 3.5 * 4.0 * G * causal_pairs(w.T, w.causal) * w.d
    for _ in range(args.warmup):
        oracle.bwd(qs, ks, vs, ds, causal=w.causal)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle.bwd(qs, ks, vs, ds, causal=w.causal)
    el = time.perf_counter() - t0
    value = sample_flops * args.steps / el / 1e12
    sample = (f"each step: one (batch, kv-head) group of {w.name} ({G} query heads x T={w.T}), "
              f"f64 oracle fwd+bwd on the host cores")
    line = {"metric": METRIC, "value": value, "unit": "TFLOP/s", "impl": "reference", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": el / args.steps * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": config_dict(w, {"sample": "one (batch, kv-head) group per step"}),
            "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": oracle.max_threads(), "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


# ----------------------------------------------------------------------------- our arm
# Matmuls (over the causal pairs of all heads) each kernel is credited with, by the
# standard count: the forward two (S = QK^T, O = PV), the backward five (S, dP, dV,
# dK, dQ). EXECUTED_MATMULS is what the kernels run: the backward's dQ tasks compute
# S and dP a second time.
CREDITED_MATMULS = {"attn_fwd_kernel": 2, "bwd_main_kernel": 5, "bwd_pre_kernel+bwd_main_kernel": 5}
EXECUTED_MATMULS = {"attn_fwd_kernel": 2, "bwd_main_kernel": 7, "bwd_pre_kernel+bwd_main_kernel": 7}


class Context:
    """Per-process state shared by the workloads of one run."""

    def __init__(self, args):
        import torch
        import torch.distributed as dist

        import causal_gqa_flash_gb300 as gqa

        self.torch, self.dist, self.gqa = torch, dist, gqa
        self.world = int(os.environ.get("WORLD_SIZE", "1"))
        self.rank = int(os.environ.get("RANK", "0"))
        local = int(os.environ.get("LOCAL_RANK", "0"))
        if self.world > 1:
            dist.init_process_group("nccl")
        torch.cuda.set_device(local)
        self.dev = torch.device("cuda", local)
        gqa.build()
        gqa.load()
        self.peaks, self.peak_src = load_peaks()
        self.flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=self.dev)

    def barrier(self):
        if self.world > 1:
            self.dist.barrier()


def run_workload(args, ctx, w, cpu_seconds):
    """Time the step on workload w; returns the JSON line (rank 0) or None."""
    torch, dist, gqa = ctx.torch, ctx.dist, ctx.gqa
    from causal_gqa_flash_gb300.inputs import workload_inputs

    world, rank, dev, peaks, peak_src = ctx.world, ctx.rank, ctx.dev, ctx.peaks, ctx.peak_src
    flush = ctx.flush

    # Inputs and outputs each live in one contiguous buffer (views at 256-byte
    # aligned offsets), so the end-to-end leg moves them with one copy each way.
    # Two of each on the device: the end-to-end leg alternates between them.
    q_c, k_c, v_c, do_c = workload_inputs(w)
    in_specs = [(x.shape, x.dtype) for x in (q_c, k_c, v_c, do_c)]
    out_specs = [(q_c.shape, torch.bfloat16), ((w.B, w.Hq, w.T), torch.float32), (q_c.shape, torch.bfloat16),
                 (k_c.shape, torch.bfloat16), (v_c.shape, torch.bfloat16)]
    fused = args.layout == "fused"
    H3 = w.Hq + 2 * w.Hkv
    if fused:
        # one [B,T,Hq+2*Hkv,d] projection buffer in, one gradient buffer of that shape out
        qkv_shape = (w.B, w.T, H3, w.d)
        in_specs = [(qkv_shape, torch.bfloat16), (do_c.shape, do_c.dtype)]
        out_specs = [(q_c.shape, torch.bfloat16), ((w.B, w.Hq, w.T), torch.float32), (qkv_shape, torch.bfloat16)]
    in_h, host_in = packed_buffer(torch, in_specs, pin=True)
    if fused:
        host_in[0][:, :, :w.Hq].copy_(q_c)
        host_in[0][:, :, w.Hq:w.Hq + w.Hkv].copy_(k_c)
        host_in[0][:, :, w.Hq + w.Hkv:].copy_(v_c)
        host_in[1].copy_(do_c)
    else:
        for dst, src in zip(host_in, (q_c, k_c, v_c, do_c)):
            dst.copy_(src)
    del q_c, k_c, v_c, do_c
    rope = args.rope if fused else "none"
    if args.rope != "none" and not fused:
        raise SystemExit("--rope needs --layout fused")
    rope = None if rope == "none" else rope
    table = gqa.attn_rope_table(w.T, w.d, device=dev) if rope == "separate" else None
    qk_rot = torch.empty((w.B, w.T, w.Hq + w.Hkv, w.d), dtype=torch.bfloat16, device=dev) if rope else None
    cut = (slice(0, w.Hq), slice(w.Hq, w.Hq + w.Hkv), slice(w.Hq + w.Hkv, H3))

    def make_set():
        """Device buffers of one step and their views."""
        in_d, in_views = packed_buffer(torch, in_specs, device=dev)
        out_d, out_views = packed_buffer(torch, out_specs, device=dev)
        sv = {"in": in_d, "out": out_d}
        if fused:
            qkv, sv["dout"] = in_views
            sv["o"], sv["lse"], dqkv = out_views
            sv["q"], sv["k"], sv["v"] = (qkv[:, :, c] for c in cut)
            sv["dq"], sv["dk"], sv["dv"] = (dqkv[:, :, c] for c in cut)
            if rope == "separate":
                # q and k rotated out of the projection buffer into their own buffer; dq and dk
                # rotated back in place in the gradient buffer
                sv["qk_raw"] = qkv[:, :, :w.Hq + w.Hkv]
                sv["q"], sv["k"] = qk_rot[:, :, :w.Hq], qk_rot[:, :, w.Hq:]
                sv["dqk"] = dqkv[:, :, :w.Hq + w.Hkv]
            elif rope == "fused":
                # the forward rotates q and k of the projection buffer into their own buffer,
                # the backward takes those and writes dq, dk of the unrotated q, k
                sv["q_rot"], sv["k_rot"] = qk_rot[:, :, :w.Hq], qk_rot[:, :, w.Hq:]
        else:
            sv["q"], sv["k"], sv["v"], sv["dout"] = in_views
            sv["o"], sv["lse"], sv["dq"], sv["dk"], sv["dv"] = out_views
        return sv

    sets = [make_set(), make_set()]
    for sv in sets:
        sv["in"].copy_(in_h)
    ws = torch.empty(gqa.attn_bwd_workspace_bytes(w.B, w.T, w.Hq), dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    causal = w.causal
    sv0 = sets[0]

    def step(sv, ev=None, rev=None, public=False):
        """One fwd + bwd on the buffers sv. ev: events between the kernels; public: the
        calls a user makes (attn_fwd, attn_bwd) instead of the backward's two stages."""
        q, k, v, o, lse, dout, dq, dk, dv = (sv[n] for n in ("q", "k", "v", "o", "lse", "dout", "dq", "dk", "dv"))
        if fused and rope == "fused":
            if ev is not None:
                ev[0].record(stream)
            gqa.attn_fwd_rope(q, k, v, causal=causal, o=o, lse=lse, q_rot=sv["q_rot"], k_rot=sv["k_rot"],
                              stream=stream)
            if ev is not None:
                ev[1].record(stream)
                ev[2].record(stream)
            gqa.attn_bwd_rope(sv["q_rot"], sv["k_rot"], v, o, lse, dout, causal=causal, dq=dq, dk=dk, dv=dv,
                              workspace=ws, stream=stream)
            if ev is not None:
                ev[3].record(stream)
            return
        if fused:
            if rope:
                if rev is not None:
                    rev[0].record(stream)
                gqa.attn_rope(sv["qk_raw"], table, y=qk_rot, stream=stream)
                if rev is not None:
                    rev[1].record(stream)
            # the strided backward is one call: its preprocess and main kernel share one interval
            if ev is not None:
                ev[0].record(stream)
            gqa.attn_fwd_strided(q, k, v, o, causal=causal, lse=lse, stream=stream)
            if ev is not None:
                ev[1].record(stream)
                ev[2].record(stream)
            gqa.attn_bwd_strided(q, k, v, o, lse, dout, dq, dk, dv, causal=causal, workspace=ws, stream=stream)
            if ev is not None:
                ev[3].record(stream)
            if rope:
                if rev is not None:
                    rev[2].record(stream)
                gqa.attn_rope(sv["dqk"], table, inverse=True, stream=stream)
                if rev is not None:
                    rev[3].record(stream)
            return
        if ev is not None:
            ev[0].record(stream)
        gqa.attn_fwd(q, k, v, causal=causal, o=o, lse=lse, stream=stream)
        if ev is not None:
            ev[1].record(stream)
        if public:
            gqa.attn_bwd(q, k, v, o, lse, dout, causal=causal, dq=dq, dk=dk, dv=dv, workspace=ws, stream=stream)
            return
        gqa.attn_bwd_preprocess(o, lse, dout, ws, stream=stream)
        if ev is not None:
            ev[2].record(stream)
        gqa.attn_bwd_dq_dkv(q, k, v, dout, dq, dk, dv, ws, causal=causal, stream=stream)
        if ev is not None:
            ev[3].record(stream)

    for _ in range(max(args.warmup, 3)):
        step(sv0)
    torch.cuda.synchronize(dev)
    if gqa.attn_sync_status(stream) != gqa.GQA_OK:
        raise RuntimeError(gqa.attn_last_error())

    sampler = ClockSampler(gpu_bus_id(torch, dev)) if rank == 0 and not args.profile_run else None
    if sampler:
        sampler.start()
        time.sleep(0.3)
    # Timed region: one event pair per step (kernels back to back, so each kernel's
    # launch and prologue can overlap the previous kernel's tail).
    step_ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(args.steps)]
    ctx.barrier()
    torch.cuda.synchronize(dev)
    wall0 = time.perf_counter()
    for i in range(args.steps):
        flush.zero_()  # L2 flush between timed steps, outside the events
        step_ev[i][0].record(stream)
        step(sv0)
        step_ev[i][1].record(stream)
    ctx.barrier()
    torch.cuda.synchronize(dev)
    wall = time.perf_counter() - wall0
    # Per-kernel breakdown (events between the kernels) for the roofline, same workload.
    events = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(args.steps)]
    rope_ev = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(args.steps)]
    for i in range(args.steps):
        flush.zero_()
        step(sv0, events[i], rope_ev[i])
    torch.cuda.synchronize(dev)
    # The end-to-end leg next, while the GPU is in the state the device-timed steps saw
    # (after a long soak a power-capped part runs slower, which would charge the copies
    # with a clock drop they did not cause); the clock sampler keeps running through it.
    e2e = e2e_leg(args, ctx, w, sets, in_h, out_specs, step)
    # keep the GPU busy with identical untimed steps so the 100 ms clock sampler sees
    # at least 1.5 s of load
    while sampler and time.perf_counter() - wall0 < 1.5:
        for _ in range(20):
            flush.zero_()
            step(sv0)
        torch.cuda.synchronize(dev)
    if sampler:
        sampler.stop()
    if gqa.attn_sync_status(stream) != gqa.GQA_OK:
        raise RuntimeError(gqa.attn_last_error())

    names = ["attn_fwd_kernel", "bwd_pre_kernel", "bwd_main_kernel"]
    per_kernel = {n: sum(events[i][j].elapsed_time(events[i][j + 1]) for i in range(args.steps))
                  for j, n in enumerate(names)}
    if fused:  # one strided backward call: its two kernels are timed as one interval
        per_kernel = {"attn_fwd_kernel": per_kernel["attn_fwd_kernel"],
                      "bwd_pre_kernel+bwd_main_kernel": per_kernel["bwd_main_kernel"]}
    rope_info = None
    if rope == "fused":
        # extra HBM bytes of the fused rotation per step: k read and k_rot written, q_rot
        # written by the forward (the angles are computed in registers)
        extra = (2 * w.Hkv + w.Hq) * w.B * w.T * w.d * 2
        rope_info = {"mode": "fused", "calls_per_step": 2,
                     "kernels": "rope_kernel on k (in the forward interval); q rotated inside attn_fwd_kernel, "
                                "dq and dk inverse-rotated inside bwd_main_kernel",
                     "extra_bytes_per_step": extra}
    elif rope:
        rope_ms = sum(rope_ev[i][0].elapsed_time(rope_ev[i][1]) + rope_ev[i][2].elapsed_time(rope_ev[i][3])
                      for i in range(args.steps)) / args.steps
        # per step: q, k read and written, dq, dk read and written (bf16), and 32 table bytes
        # per 16-byte chunk of a token in each of the two calls
        rope_bytes = 4 * w.B * w.T * (w.Hq + w.Hkv) * w.d * 2 + 2 * w.B * w.T * w.d * 4
        rope_info = {"mode": "separate", "kernel": "rope_kernel", "calls_per_step": 2, "ms_per_step": rope_ms,
                     "bytes_per_step": rope_bytes, "bound": "hbm",
                     "achieved_gbs": rope_bytes / (rope_ms * 1e-3) / 1e9, "peak_gbs": peaks["hbm_gbs"],
                     "frac": rope_bytes / (rope_ms * 1e-3) / 1e9 / peaks["hbm_gbs"]}
    step_ms = sorted(step_ev[i][0].elapsed_time(step_ev[i][1]) for i in range(args.steps))
    ms_median = statistics.median(step_ms)
    step_ms_total = max_over_ranks(torch, dist, sum(step_ms), world, dev)
    ms_per_step = step_ms_total / args.steps
    value = whole_job_tflops(world, step_flops(w), args.steps, step_ms_total)
    per_gpu = value / world

    # roofline of the dominant kernel (largest share of the step)
    pairs = causal_pairs(w.T, w.causal)
    mm = 2.0 * w.B * w.Hq * pairs * w.d  # one causal matmul over all heads
    pre_bytes = 2 * w.B * w.T * w.Hq * w.d * 2 + w.B * w.Hq * w.T * 4 + 2 * w.B * w.Hq * w.T * 4
    dom = max(per_kernel, key=per_kernel.get)
    avg_ms = per_kernel[dom] / args.steps
    if dom == "bwd_pre_kernel":
        achieved = pre_bytes / (avg_ms * 1e-3) / 1e9
        roof = {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s"}
    else:
        achieved = CREDITED_MATMULS[dom] * mm / (avg_ms * 1e-3) / 1e12
        roof = {"bound": "tensor", "achieved": achieved, "peak": peaks["bf16_tflops"], "unit": "TFLOP/s"}
    roof["frac"] = roof["achieved"] / roof["peak"]
    roof["kernel"] = dom
    roof["peak_source"] = f"{peak_src} burst" if roof["bound"] == "tensor" else peak_src
    rec = None if fused else recorded_counters(dom, w.name)
    roof["traffic"] = None if rec is None else rec.get("dram_bytes_per_launch")
    if roof["bound"] == "tensor":
        # the same kernel time with the matmuls it runs, and against the sustained peak
        roof["credited_matmuls"] = CREDITED_MATMULS[dom]
        roof["executed_matmuls"] = EXECUTED_MATMULS[dom]
        roof["executed_frac"] = EXECUTED_MATMULS[dom] * mm / (avg_ms * 1e-3) / 1e12 / roof["peak"]
        sus = peaks.get("bf16_tflops_sustained")
        roof["frac_of_sustained"] = roof["achieved"] / sus if sus else None
        roof["tensor_active_pct_ncu"] = None if rec is None else rec.get("tensor_active_pct")
    kernel_ms = {n: t / args.steps for n, t in per_kernel.items()}
    bwd_ms = kernel_ms["bwd_pre_kernel+bwd_main_kernel"] if fused else (
        kernel_ms["bwd_pre_kernel"] + kernel_ms["bwd_main_kernel"])
    fwd_tf = fwd_flops(w) / (kernel_ms["attn_fwd_kernel"] * 1e-3) / 1e12
    bwd_tf = 2.5 * fwd_flops(w) / (bwd_ms * 1e-3) / 1e12

    cpu = None
    if rank == 0 and world == 1 and cpu_seconds > 0 and not (args.no_cpu_baseline or args.profile_run):
        s = oracle_sample(w, min_seconds=cpu_seconds, max_seconds=3 * cpu_seconds)
        cpu = {"value": s["value"], "unit": "TFLOP/s", "cores": s["cores"], "kind": "oracle", "sample": s["sample"]}

    del sets, ws
    if rank != 0:
        return None
    clocks = sampler.summary() if sampler else None
    peak = peaks["bf16_tflops"]
    return {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "ms_per_step_median": ms_median,
        "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": config_dict(w, {"l2": "flushed between timed steps (256 MB write, outside the events)",
                                  "rope": {"fused": "rotary embedding inside the attention kernels (in the step)",
                                           "separate": "q, k rotated before and dq, dk after attention (in the step)",
                                           None: "none"}[rope],
                                  "layout": "fused qkv / dqkv buffers, strided views" if fused
                                  else "separate contiguous q, k, v, dq, dk, dv",
                                  "parallelism": f"replicas x{world}" if world > 1 else "single GPU"}),
        # the same step counted with the exact number of causal pairs, T(T+1)/2
        "value_exact_pairs": value * ((w.T + 1) / w.T if w.causal else 1.0),
        "pct_of_peak": 100.0 * per_gpu / peak,
        "peak_tflops": peak, "peak_source": f"{peak_src} burst",
        "fwd_tflops": fwd_tf, "fwd_pct_of_peak": 100.0 * fwd_tf / peak,
        "bwd_tflops": bwd_tf, "bwd_pct_of_peak": 100.0 * bwd_tf / peak,
        "kernel_ms": kernel_ms,
        "roofline": roof,
        "cpu_baseline": cpu,
        "e2e": e2e,
        "gpu_launches": {"fused": 4, "separate": 5, None: 3}[rope] * args.steps,
        "rope": rope_info,
        "clocks": clocks,
        "wall_s_timed": wall,
    }


def e2e_leg(args, ctx, w, sets, in_h, out_specs, step):
    """The metric end to end through the public calls (attn_fwd, attn_bwd), with every
    step's inputs copied in from pinned host memory and its outputs copied back out.
    Two device buffer sets and two pinned output buffers alternate, and the copies run
    on two copy streams (one each way), so step i+1's upload and step i-1's download
    overlap step i's kernels, as a trainer feeding the GPU would overlap them."""
    torch, dist = ctx.torch, ctx.dist
    if args.profile_run:
        return {"value": None, "unit": "TFLOP/s", "h2d_bytes_per_step": in_h.numel(),
                "d2h_bytes_per_step": None}
    dev, stream = ctx.dev, torch.cuda.current_stream(ctx.dev)
    outs_h = [packed_buffer(torch, out_specs, pin=True)[0] for _ in range(2)]
    up, down = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    Ev = lambda: torch.cuda.Event(enable_timing=True)  # noqa: E731

    def run(n):
        ev_in, ev_used, ev_out = [Ev(), Ev()], [Ev(), Ev()], [Ev(), Ev()]
        e0, e1 = Ev(), Ev()
        e0.record(up)
        with torch.cuda.stream(up):
            sets[0]["in"].copy_(in_h, non_blocking=True)
        ev_in[0].record(up)
        for i in range(n):
            b = i & 1
            if i + 1 < n:
                # next step's inputs into the other set, once step i-1 no longer reads them
                if i >= 1:
                    up.wait_event(ev_used[1 - b])
                with torch.cuda.stream(up):
                    sets[1 - b]["in"].copy_(in_h, non_blocking=True)
                ev_in[1 - b].record(up)
            stream.wait_event(ev_in[b])
            if i >= 2:
                stream.wait_event(ev_out[b])  # outputs of step i-2 are out of this set
            step(sets[b], public=True)
            ev_used[b].record(stream)
            down.wait_event(ev_used[b])
            with torch.cuda.stream(down):
                outs_h[b].copy_(sets[b]["out"], non_blocking=True)
            ev_out[b].record(down)
        e1.record(down)  # the last download comes after every other copy and kernel
        torch.cuda.synchronize(dev)
        return e0.elapsed_time(e1)

    run(3)
    # the first upload and the last download are not overlapped with anything: timing
    # as many steps as the device-timed region spreads them as thinly
    n = max(3, args.steps)
    ctx.barrier()
    torch.cuda.synchronize(dev)
    te_ms = max_over_ranks(torch, dist, run(n), ctx.world, dev)
    return {"value": whole_job_tflops(ctx.world, step_flops(w), n, te_ms), "unit": "TFLOP/s",
            "h2d_bytes_per_step": in_h.numel(), "d2h_bytes_per_step": outs_h[0].numel(),
            "ms_per_step": te_ms / n,
            "overlap": "double-buffered: uploads and downloads on their own streams, beside the kernels"}


def run_ours(args, names):
    ctx = Context(args)
    from causal_gqa_flash_gb300.inputs import WORKLOADS
    for i, name in enumerate(names):
        last = i + 1 == len(names)
        line = run_workload(args, ctx, WORKLOADS[name], cpu_seconds=10.0 if last else 5.0)
        if line is not None:
            print(json.dumps(line), flush=True)
        ctx.torch.cuda.empty_cache()
    if ctx.world > 1:
        ctx.barrier()
        ctx.dist.destroy_process_group()
    return 0


ALL_ORDER = ["c1", "c2", "c3", "c5", "c4"]  # the headline workload last


def main():
    args = parse_args()
    from causal_gqa_flash_gb300.inputs import WORKLOADS
    names = ALL_ORDER if args.workload == "all" else [args.workload]
    for n in names:
        if n not in WORKLOADS:
            raise SystemExit(f"unknown workload {n!r} (c1..c5 or all)")
    if args.impl == "reference":
        return run_reference(args, WORKLOADS[names[-1]])
    return run_ours(args, names)


if __name__ == "__main__":
    sys.exit(main())
