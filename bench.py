#!/usr/bin/env python3
"""Benchmark of the KDA hot path on one GB300 (or N replicas under torchrun).

One step = one pass of the whole hot path on synthetic K3-shaped inputs:
  prefill leg:  gate + chunked prefill, B=1, T=4096, H=96, d=128 (the headline
                tokens/s workload), as one launch of the chunked kernel that
                computes the gate itself (kda_chunk_prefill_gated);
  decode leg:   gate + recurrent decode, 256 sequences x 96 heads, fp32 states
                [256, 96, 128, 128] (1.61 GB) updated in place (kda_gate_fused on
                the new token, then kda_recurrent_decode: 3 % faster than the
                one-launch kda_recurrent_decode_gated, which is timed too).
`value` is prefill sequence tokens/s over all ranks; the decode leg reports
state GB/s against the measured HBM peak.  The unfused prefill pair (bit-exact
gate kernel, then kda_chunk_prefill) and the gated decode are timed in a second
loop and reported too.  Inputs are larger than L2 (129 MB):
the prefill leg reads ~0.6 GB and the decode leg streams 3.2 GB per step.

`--impl reference` times the CPU oracle (fp64 recurrence + fp32 gate spec) on
the host cores, on a bounded sample of the same prefill workload.
"""
from __future__ import annotations

import argparse
import datetime
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import torch  # noqa: E402

T_PREFILL = 4096
H = 96
D = 128
CHUNK = 64
B_DECODE = 256
WORKLOAD = (f"KDA gate+chunked prefill B=1 T={T_PREFILL} H={H} d={D} (chunk {CHUNK}); "
            f"gate+recurrent decode B={B_DECODE} H={H} d={D} fp32 state in place")
METRIC = "KDA prefill tokens/s (H=96,d=128,T=4096); decode state GB/s vs HBM peak"


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as fh:
            p = json.load(fh)
        return {"hbm_gbs": float(p["hbm_gbs"]), "bf16_tflops": float(p["bf16_tflops"]),
                "bf16_tflops_sustained": float(p.get("bf16_tflops_sustained", p["bf16_tflops"])),
                "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
            "source": "fallback"}


# --- algorithmic work --------------------------------------------------------------------

def prefill_flops_per_head(lengths, K=D, V=D, C=CHUNK):
    """Algorithmic flops of the chunked form for one head (triangular products
    counted as triangular): per chunk of L tokens, A_kk (strict lower) and A_qk
    (lower) inner products over K, the UT inverse (L^3/3), W = T beta Kbar and
    Ut = T beta V, U = Ut - W S, O = Qbar S + A_qk U, S update."""
    total = 0
    for n in lengths:
        for c0 in range(0, n, C):
            L = min(C, n - c0)
            tri_lo, tri = L * (L - 1) // 2, L * (L + 1) // 2
            total += 2 * K * tri_lo + 2 * K * tri          # A_kk, A_qk
            total += L ** 3 // 3                           # UT inverse
            total += 2 * K * tri + 2 * V * tri             # W, Ut
            total += 2 * L * K * V * 3                     # U, Qbar S, S update
            total += 2 * V * tri                           # A_qk U
    return total


def chunk_backward_flops_per_head(lengths, K=D, V=D, C=CHUNK):
    """Algorithmic flops of the chunked backward for one head: the forward pass
    that keeps the chunk-start states (prefill_flops_per_head), then per chunk of
    L tokens the recomputed products (A_qk and A_kk, W, U-tilde, U = U-tilde - W S)
    and the gradient products (dU, dS, dA_qk, dQbar, dW, dKhat, dT, d(beta K),
    d(beta V), the two dA_kk products, dKtilde and dK), each counted as a dense
    product of its operand shapes (2 flops per multiply-add)."""
    total = prefill_flops_per_head(lengths, K, V, C)
    for n in lengths:
        for c0 in range(0, n, C):
            L = min(C, n - c0)
            macs = (2 * L * L * K            # [Qt; Kr] Ks^T
                    + L * L * (K + V)        # W', U-tilde
                    + L * K * V              # U
                    + L * L * V + L * K * V  # dU
                    + 2 * L * K * V          # dS
                    + L * L * V              # dA_qk
                    + L * K * V + L * L * K  # dQt
                    + L * K * V              # dW'
                    + L * K * V              # dKh
                    + L * L * (K + V)        # dT
                    + L * L * (K + V)        # d(beta Kr), d(beta V)
                    + 2 * L * L * L          # T^T dT T^T
                    + 2 * L * L * K          # dKs
                    + L * L * K)             # dA_kk Ks
            total += 2 * macs
    return total


def prefill_io_bytes(T, Hh=H, K=D, V=D, o_bytes=2):
    """Minimal HBM bytes of gate+prefill: f (bf16) read by the gate, g (fp32)
    written by the gate and read by prefill, b/beta, q/k/v (bf16) read, o written."""
    per_token_head = 2 * K + 4 * K * 2 + 4 * 2 + 2 * K * 2 + 2 * V + o_bytes * V
    return T * Hh * per_token_head


def prefill_kernel_bytes(T, Hh=H, K=D, V=D, o_bytes=2):
    """Minimal HBM bytes of the prefill kernel alone: q, k, v (bf16), g (fp32),
    beta (fp32) read, o written (zero initial state, final state written)."""
    return T * Hh * (2 * K * 2 + 2 * V + 4 * K + 4 + o_bytes * V) + Hh * K * V * 4


def decode_bytes(B=B_DECODE, Hh=H, K=D, V=D, state_bytes=4, gated=False):
    """Decode kernel: every state (fp32, or bf16 with state_bytes=2) read once
    and written once, plus the token (q, k, v bf16; g and beta fp32, or with
    gated=True the bf16 gate pre-activation and fp32 beta logit) and the
    output (bf16)."""
    gate = 2 * K + 4 if gated else 4 * K + 4
    return B * Hh * (2 * K * V * state_bytes + 2 * K * 2 + 2 * V + gate + 2 * V)


# DRAM read+write bytes per benchmark launch, from the ncu captures summarised
# in profiles/ (dram__bytes_read.sum + dram__bytes_write.sum), with the SHA-256
# of the kernel source they were taken on: a changed source reports null.
NCU_TRAFFIC = {
    "chunk_unfused": {"src": ["kda_chunk.cu", "kda_chunk_common.cuh", "kda_sm100.cuh", "kda_f32x2.cuh"],
                     "bytes": 4 * 138.82e6,
                     "sha256": ["1dc515dc5e3ccbdf95b753842424885a65626cc9722c56b2c2bb356b6a3c1a47",
                             "17d6fd9cfa56e1c3a45045394b09808f9856c13fe0200ad23e45cd6bc4b02399",
                             "8881aa469733f65a4c014ed9f4f0aa68c6f6518704b09fe54617047b32840e72",
                             "c5455d461a5735fe8529d24adc80e51f03cd6f12a6b4cb7c406826b40c47bd2d"],
                     "note": "T=1024 capture x 4 (profiles/chunk_prefill_T1024_H96.md)"},
    "chunk_gated": {"src": ["kda_chunk.cu", "kda_chunk_common.cuh", "kda_sm100.cuh", "kda_f32x2.cuh"],
                   "bytes": 4 * 110.78e6,
                   "sha256": ["1dc515dc5e3ccbdf95b753842424885a65626cc9722c56b2c2bb356b6a3c1a47",
                           "17d6fd9cfa56e1c3a45045394b09808f9856c13fe0200ad23e45cd6bc4b02399",
                           "8881aa469733f65a4c014ed9f4f0aa68c6f6518704b09fe54617047b32840e72",
                           "c5455d461a5735fe8529d24adc80e51f03cd6f12a6b4cb7c406826b40c47bd2d"],
                   "note": "T=1024 capture x 4 (profiles/chunk_prefill_gated_T1024_H96.md)"},
    "decode": {"src": ["kda_decode.cu", "kda_gate_spec.cuh"], "bytes": 4 * 754.03e6,
               "sha256": ["68f5f05ba5aab124309cb1ad3f458a194b6ceada7c9f575cd296d72aa540af8c",
                          "8aed1e00efe29355e1843f1ca8a41b9485b9cc3ac211f3cdca9a9c6f7ba36816"],
               "note": "B=64 capture x 4 (profiles/decode_B64_H96.md)"},
    "decode_pool": {"src": ["kda_decode.cu", "kda_gate_spec.cuh"], "bytes": 4 * 350.96e6,
                    "sha256": ["68f5f05ba5aab124309cb1ad3f458a194b6ceada7c9f575cd296d72aa540af8c",
                               "8aed1e00efe29355e1843f1ca8a41b9485b9cc3ac211f3cdca9a9c6f7ba36816"],
                    "note": "B=64 capture x 4 (profiles/decode_bf16_pool_B64_H96.md)"},
    "gate": {"src": ["kda_gate.cu", "kda_gate_spec.cuh", "kda_gate_spec_x2.cuh", "kda_f32x2.cuh"],
             "bytes": 246.59e6,
             "sha256": ["b2531cbc98d87995bf0d28e746d0b8e2bc9fe32797688b40f6fbf14c0f35f229",
                        "8aed1e00efe29355e1843f1ca8a41b9485b9cc3ac211f3cdca9a9c6f7ba36816",
                        "778d78a20aa1906029a458cd4637581380c9c9720ad6861eb5dfc943faf9199d",
                        "c5455d461a5735fe8529d24adc80e51f03cd6f12a6b4cb7c406826b40c47bd2d"],
             "note": "T=4096 capture (profiles/gate_T4096_H96.md)"},
    "short_conv": {"src": ["kda_shortconv.cu"], "bytes": 552.45e6,
                   "sha256": ["d69ef349b594f9f5be7de9855c96ce080dc0c0fb1d58e2a9aa31d2fd7cc2d4a6"],
                   "note": "T=4096 capture (profiles/short_conv_T4096_H96.md)"},
    "backward": {"src": ["kda_backward.cu"], "bytes": 16 * 2.067e9,
                 "sha256": ["58f242b881fc2d1b1acb1532ced68f7c8a83e5dd92b3b19f71833997525eacc1"],
                 "note": "T=256 capture x 16 (per-token state scratch; profiles/backward_T256_H96.md)"},
    "backward_chunked": {"src": ["kda_chunk_bwd.cu"], "bytes": None, "sha256": [],
                         "note": "T=256 capture (profiles/chunk_backward_T256_H96.md): the per-CTA "
                                 "scratch stays in L2 at T=4096, so its traffic does not scale "
                                 "with the tokens"},
}


def measured_traffic(kernel_id):
    """(bytes, note) of the ncu capture of one kernel, or (None, why) when a
    source file of the kernel has changed since the capture."""
    import hashlib
    ent = NCU_TRAFFIC.get(kernel_id)
    if ent is None:
        return None, "not captured"
    if ent["bytes"] is None:
        return None, ent["note"]
    digests = []
    for name in ent["src"]:
        path = os.path.join(ROOT, "gated_delta_rule_33_gb300", "csrc", name)
        if not os.path.exists(path):
            return None, "source missing"
        with open(path, "rb") as fh:
            digests.append(hashlib.sha256(fh.read()).hexdigest())
    if digests != ent["sha256"]:
        return None, "kernel changed since the ncu capture"
    return ent["bytes"], ent["note"]


# --- clocks ----------------------------------------------------------------------------

class ClockSampler:
    """nvidia-smi clocks and throttle reasons, sampled every 20 ms.  start()
    returns once the first sample has arrived; stop() keeps only the samples
    whose timestamps fall inside the marked window."""
    QUERY = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.proc = None
        self.lines = []
        self.window = None
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={gpu_index}", f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "20"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            first = self.proc.stdout.readline()  # the sampler is running
            if first:
                self.lines.append(first)
        except (FileNotFoundError, OSError):
            self.proc = None

    def mark(self, t0: float, t1: float):
        self.window = (t0, t1)

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        sms, maxes, reasons, all_sms = [], [], set(), []
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in (self.lines + out.strip().splitlines()):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                ts = datetime.datetime.strptime(parts[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
                sm, mx = float(parts[1]), float(parts[2])
            except ValueError:
                continue
            all_sms.append(sm)
            if self.window is not None and not (self.window[0] - 0.03 <= ts <= self.window[1] + 0.03):
                continue
            sms.append(sm)
            maxes.append(mx)
            for name, val in zip(names, parts[5:9]):
                if val.lower() == "active":
                    reasons.add(name)
        if not sms:
            return {"sm_mhz": None, "sm_max_mhz": None, "samples": 0, "reasons": [],
                    "note": f"timed region shorter than the 20 ms sampling interval; "
                            f"{len(all_sms)} samples around it, median "
                            f"{statistics.median(all_sms) if all_sms else None} MHz"}
        return {"sm_mhz": statistics.median(sms), "sm_max_mhz": max(maxes),
                "samples": len(sms), "reasons": sorted(reasons)}


# --- distributed helpers -----------------------------------------------------------------
# Each rank runs its own sequences (weak scaling; no data-path exchange): the
# helpers live in gated_delta_rule_33_gb300/sharding.py.

def dist_setup(n_gpus):
    from gated_delta_rule_33_gb300.sharding import dist_setup as _setup
    return _setup()


def barrier(world):
    from gated_delta_rule_33_gb300.sharding import barrier as _barrier
    _barrier(world)


def max_over_ranks(x: float, world: int, device) -> float:
    from gated_delta_rule_33_gb300.sharding import max_over_ranks as _max
    return _max(x, world, device)


def host_affinity_for(dev_index: int) -> dict:
    """Restrict this process to the CPUs next to the GPU (its PCI device's
    local_cpulist in sysfs), so that pinned host buffers allocated afterwards
    sit in the memory nearest to the GPU; returns what was found."""
    info = {}
    try:
        bus = None
        props = torch.cuda.get_device_properties(dev_index)
        if all(hasattr(props, a) for a in ("pci_domain_id", "pci_bus_id", "pci_device_id")):
            bus = f"{props.pci_domain_id:04x}:{props.pci_bus_id:02x}:{props.pci_device_id:02x}.0"
        else:
            out = subprocess.run(["nvidia-smi", "--query-gpu=pci.bus_id", "--format=csv,noheader",
                                  "-i", str(dev_index)], capture_output=True, text=True, timeout=20)
            raw = out.stdout.strip().lower()          # e.g. 00000009:01:00.0
            if raw:
                dom, rest = raw.split(":", 1)
                bus = f"{int(dom, 16):04x}:{rest}"
        if bus is None:
            return {"note": "no PCI bus id"}
        base = f"/sys/bus/pci/devices/{bus}"
        info["pci"] = bus
        with open(base + "/numa_node") as fh:
            info["numa_node"] = int(fh.read().strip())
        with open(base + "/local_cpulist") as fh:
            cpulist = fh.read().strip()
        cpus = set()
        for part in cpulist.split(","):
            if "-" in part:
                a, b = part.split("-")
                cpus.update(range(int(a), int(b) + 1))
            elif part:
                cpus.add(int(part))
        allowed = os.sched_getaffinity(0)
        near = cpus & allowed
        if near and near != allowed:
            os.sched_setaffinity(0, near)
            info["cpus"] = cpulist
        else:
            info["cpus"] = "unchanged"
    except Exception as exc:  # best effort: the measurement still runs
        info["note"] = f"affinity not set: {type(exc).__name__}"
    return info


# --- reference arm (the CPU oracle) --------------------------------------------------------

def run_reference(args):
    rank, world, _ = dist_setup(args.gpus)
    if rank != 0:
        return 0
    import numpy as np
    import oracle
    from gated_delta_rule_33_gb300 import synth

    oracle.build()
    cores = oracle.default_threads()
    heads = args.ref_heads
    x = synth.make_inputs(T_PREFILL, H=H, D=D, seed=0)
    sel = list(range(heads))
    f = x.f[:, sel].float().numpy()
    b = x.b[:, sel].numpy()
    dt = x.dt_bias[sel].numpy()
    q, k, v = (t[:, sel].double().numpy() for t in (x.q, x.k, x.v))

    def step():
        g, beta = oracle.gate(f, b, x.A_log.numpy(), dt, x.alog_mode)
        oracle.recurrent(q, k, v, g, beta, nthreads=cores)

    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step()
    dt_s = (time.perf_counter() - t0) / args.steps
    # tokens/s of the full 96-head workload = sampled token-heads/s / 96
    value = T_PREFILL * heads / H / dt_s
    sample = (f"gate + fp64 recurrence on {heads} of {H} heads, T={T_PREFILL}, d={D}; "
              f"tokens/s scaled to all {H} heads")
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": dt_s * 1e3, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": WORKLOAD, "sample": sample},
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cores,
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line))
    return 0


def cpu_baseline(heads: int):
    """The oracle, as it stands, on the host cores: gate + fp64 recurrence on a
    sample of heads of the T=4096 workload."""
    import oracle
    from gated_delta_rule_33_gb300 import synth

    oracle.build()
    cores = oracle.default_threads()
    x = synth.make_inputs(T_PREFILL, H=H, D=D, seed=0)
    sel = list(range(heads))
    f, b, dt = x.f[:, sel].float().numpy(), x.b[:, sel].numpy(), x.dt_bias[sel].numpy()
    q, k, v = (t[:, sel].double().numpy() for t in (x.q, x.k, x.v))
    t0 = time.perf_counter()
    g, beta = oracle.gate(f, b, x.A_log.numpy(), dt, x.alog_mode)
    oracle.recurrent(q, k, v, g, beta, nthreads=cores)
    elapsed = time.perf_counter() - t0
    # one thread, on a sample of 4 heads
    t1 = time.perf_counter()
    g1, b1 = oracle.gate(f[:, :4], b[:, :4], x.A_log.numpy(), dt[:4], x.alog_mode)
    oracle.recurrent(q[:, :4], k[:, :4], v[:, :4], g1, b1, nthreads=1)
    one = time.perf_counter() - t1
    return {"value": T_PREFILL * heads / H / elapsed, "unit": "tokens/s", "cores": cores,
            "kind": "oracle",
            "sample": f"gate + fp64 recurrence on {heads} of {H} heads, T={T_PREFILL}, d={D} "
                      f"({elapsed:.1f} s); tokens/s scaled to all {H} heads",
            "one_thread": {"value": T_PREFILL * 4 / H / one, "unit": "tokens/s", "cores": 1,
                           "sample": f"4 of {H} heads ({one:.1f} s), scaled to all {H} heads"}}


# --- our arm -------------------------------------------------------------------------------

def run_ours(args):
    import gated_delta_rule_33_gb300 as kda
    from gated_delta_rule_33_gb300 import synth

    rank, world, local_rank = dist_setup(args.gpus)
    if not torch.cuda.is_available():
        raise RuntimeError("bench.py needs a CUDA GPU")
    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    kda.load()
    stream = torch.cuda.current_stream(dev)

    # prefill leg inputs (resident in HBM before timing)
    x = synth.make_inputs(T_PREFILL, H=H, D=D, seed=rank)
    q, k, v, f = (t.to(dev) for t in (x.q, x.k, x.v, x.f))
    b, A_log, dt_bias = x.b.to(dev), x.A_log.to(dev), x.dt_bias.to(dev)
    g = torch.empty(T_PREFILL, H, D, device=dev)
    beta = torch.empty(T_PREFILL, H, device=dev)
    o = torch.empty(T_PREFILL, H, D, dtype=torch.bfloat16, device=dev)
    Sf = torch.empty(1, H, D, D, device=dev)
    ws = torch.empty(max(kda.kda_chunk_prefill_workspace_size(T_PREFILL, 1, H), 16),
                     dtype=torch.uint8, device=dev)
    # decode leg inputs
    d = synth.make_decode_inputs(B_DECODE, H=H, D=D, seed=rank, state_device=dev)
    dq, dk, dv, df = (t.to(dev) for t in (d.q, d.k, d.v, d.f))
    db, dA, ddt = d.b.to(dev), d.A_log.to(dev), d.dt_bias.to(dev)
    dg = torch.empty(B_DECODE, H, D, device=dev)
    dbeta = torch.empty(B_DECODE, H, device=dev)
    dout = torch.empty(B_DECODE, H, D, dtype=torch.bfloat16, device=dev)
    state = d.state


    launches_per_step = 3

    def step(record=None):
        if record is not None:
            record[0].record(stream)
        kda.kda_chunk_prefill_gated(q, k, v, f, b, A_log, x.alog_mode, dt_bias, None, 1.0, None,
                                    Sf, o, ws, stream)
        if record is not None:
            record[1].record(stream)
        kda.kda_gate_fused(df, db, dA, d.alog_mode, ddt, dg, dbeta, stream)
        if record is not None:
            record[2].record(stream)
        kda.kda_recurrent_decode(dq, dk, dv, dg, dbeta, state, 1.0, dout, stream)
        if record is not None:
            record[3].record(stream)

    def unfused_step(record):
        record[0].record(stream)
        kda.kda_gate_fused(f, b, A_log, x.alog_mode, dt_bias, g, beta, stream)
        record[1].record(stream)
        kda.kda_chunk_prefill(q, k, v, g, beta, None, 1.0, None, Sf, o, ws, stream)
        record[2].record(stream)
        kda.kda_recurrent_decode_gated(dq, dk, dv, df, db, dA, d.alog_mode, ddt, state, None, 1.0,
                                       dout, stream)
        record[3].record(stream)

    for _ in range(max(args.warmup, 3) if args.warmup >= 3 else args.warmup):
        step()
    torch.cuda.synchronize(dev)
    if kda.kda_get_last_device_error(stream) != 0:
        raise RuntimeError("device error during warm-up")

    sampler = ClockSampler(dev.index if dev.index is not None else 0)
    per_step = []
    barrier(world)
    torch.cuda.synchronize(dev)
    wall0 = time.time()
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    t_start.record(stream)
    step_events = []
    for _ in range(args.steps):
        evs = [torch.cuda.Event(enable_timing=True) for _ in range(4)]
        step(evs)
        step_events.append(evs)
    t_end.record(stream)
    torch.cuda.synchronize(dev)
    sampler.mark(wall0, time.time())
    barrier(world)
    clocks = sampler.stop()
    total_ms = t_start.elapsed_time(t_end)
    for evs in step_events:
        per_step.append([evs[i].elapsed_time(evs[i + 1]) for i in range(3)])
    fused_ms = statistics.mean(p[0] for p in per_step)
    dgate_ms = statistics.mean(p[1] for p in per_step)
    decode_ms = statistics.mean(p[2] for p in per_step)
    step_ms = total_ms / args.steps

    # the unfused pair, same inputs, its own timed loop (not part of `value`)
    for _ in range(max(args.warmup, 1)):
        unfused_step([torch.cuda.Event(enable_timing=True) for _ in range(4)])
    torch.cuda.synchronize(dev)
    uf = []
    for _ in range(args.steps):
        evs = [torch.cuda.Event(enable_timing=True) for _ in range(4)]
        unfused_step(evs)
        uf.append(evs)
    torch.cuda.synchronize(dev)
    gate_ms = statistics.mean(e[0].elapsed_time(e[1]) for e in uf)
    prefill_ms = statistics.mean(e[1].elapsed_time(e[2]) for e in uf)
    gdecode_ms = statistics.mean(e[2].elapsed_time(e[3]) for e in uf)

    def timed(fn, steps):
        """Mean CUDA-event time of fn() on the stream after one untimed call."""
        fn()
        torch.cuda.synchronize(dev)
        evs = []
        for _ in range(steps):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            fn()
            e1.record(stream)
            evs.append((e0, e1))
        torch.cuda.synchronize(dev)
        return statistics.mean(a.elapsed_time(b) for a, b in evs)

    def protocol(fn, warmup=20, iters=100, repeats=3):
        """The timing protocol of the pages' FlashKDA measurements
        (K3_ARTIFACT_AUDIT.md section 7.4): `warmup` untimed calls, then `repeats`
        runs of `iters` calls, each call bracketed by CUDA events on the stream;
        mean and 95th percentile over all calls, and the spread of the repeat
        means (max / min)."""
        for _ in range(warmup):
            fn()
        torch.cuda.synchronize(dev)
        times, means = [], []
        for _ in range(repeats):
            evs = []
            for _ in range(iters):
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                fn()
                e1.record(stream)
                evs.append((e0, e1))
            torch.cuda.synchronize(dev)
            rep = [a.elapsed_time(b) for a, b in evs]
            times += rep
            means.append(statistics.mean(rep))
        times.sort()
        return {"mean_ms": statistics.mean(times),
                "p95_ms": times[min(len(times) - 1, int(0.95 * len(times)))],
                "repeat_spread": max(means) / min(means), "calls": len(times),
                "protocol": f"warm-up {warmup}, {repeats} x {iters} calls, CUDA events"}

    proto = {}
    proto["prefill_gated"] = protocol(lambda: kda.kda_chunk_prefill_gated(
        q, k, v, f, b, A_log, x.alog_mode, dt_bias, None, 1.0, None, Sf, o, ws, stream))
    proto["prefill_unfused"] = protocol(lambda: kda.kda_chunk_prefill(
        q, k, v, g, beta, None, 1.0, None, Sf, o, ws, stream))
    proto["gate"] = protocol(lambda: kda.kda_gate_fused(f, b, A_log, x.alog_mode, dt_bias, g, beta,
                                                        stream))
    proto["decode"] = protocol(lambda: kda.kda_recurrent_decode(dq, dk, dv, dg, dbeta, state, 1.0,
                                                                dout, stream))

    # decode from a bf16 state pool addressed by slot (reversed order); its own
    # timed loop, not part of `value`
    pool = state.to(torch.bfloat16)
    slots = torch.arange(B_DECODE - 1, -1, -1, dtype=torch.int32, device=dev)
    pool_ms = timed(lambda: kda.kda_recurrent_decode_indexed(dq, dk, dv, dg, dbeta, pool, slots,
                                                             1.0, dout, stream), args.steps)
    del pool

    # the pre-step (ShortConv + SiLU + L2 norm on q, k, v) at the prefill size
    sx = synth.make_shortconv_inputs(T_PREFILL, H=H, D=D, seed=rank)
    sxs = [t.to(dev) for t in sx.x]
    sws = [t.to(dev) for t in sx.w]
    souts = [torch.empty_like(t) for t in sxs]
    sfin = torch.empty(1, 3, 3, H * D, dtype=torch.bfloat16, device=dev)
    conv_ms = timed(lambda: kda.kda_short_conv_qkv(*sxs, *sws, None, None, sfin, *souts, stream),
                    args.steps)
    del sx, sxs, souts

    # the backward (training regime) of the prefill workload
    kda.kda_gate_fused(f, b, A_log, x.alog_mode, dt_bias, g, beta, stream)
    bgen = torch.Generator(device=dev).manual_seed(rank + 77)
    bdO = torch.randn(T_PREFILL, H, D, device=dev, generator=bgen).to(torch.bfloat16)
    bgrads = [torch.empty(T_PREFILL, H, D, device=dev) for _ in range(4)]
    bdbeta = torch.empty(T_PREFILL, H, device=dev)
    bws = torch.empty(kda.kda_recurrent_backward_workspace_size(T_PREFILL, 1, H),
                      dtype=torch.uint8, device=dev)
    bwd_ms = timed(lambda: kda.kda_recurrent_backward(q, k, v, g, beta, None, 1.0, None, bdO, None,
                                                      *bgrads, bdbeta, None, bws, stream),
                   max(args.steps // 3, 1))
    cws = torch.empty(kda.kda_chunk_backward_workspace_size(T_PREFILL, 1, H), dtype=torch.uint8,
                      device=dev)
    proto["backward_chunked"] = protocol(
        lambda: kda.kda_chunk_backward(q, k, v, g, beta, None, 1.0, None, bdO, None, *bgrads,
                                       bdbeta, None, cws, stream), warmup=3, iters=10, repeats=3)
    del cws
    # the training pair: the prefill that keeps the chunk-start states, and the
    # backward that reads them instead of running the forward again
    ckpt = torch.empty(kda.kda_chunk_checkpoints_size(T_PREFILL, 1, H), dtype=torch.uint8,
                       device=dev)
    proto["prefill_checkpointed"] = protocol(
        lambda: kda.kda_chunk_prefill_checkpointed(q, k, v, g, beta, None, 1.0, None, Sf, o, ckpt,
                                                   ws, stream), warmup=3, iters=20, repeats=3)
    kws = torch.empty(kda.kda_chunk_backward_checkpointed_workspace_size(T_PREFILL, 1, H),
                      dtype=torch.uint8, device=dev)
    proto["backward_checkpointed"] = protocol(
        lambda: kda.kda_chunk_backward_checkpointed(q, k, v, g, beta, None, 1.0, ckpt, bdO, None,
                                                    *bgrads, bdbeta, None, kws, stream),
        warmup=3, iters=10, repeats=3)
    del bgrads, bws, bdO, ckpt, kws

    # the other prefill configurations of the hot path: a varlen batch of 8
    # sequences (lengths uniform in [512, 8192], partial tail chunks) and one
    # long sequence (T = 65536, nonzero initial state) followed by 128
    # one-token decode steps from its final state
    vx = synth.make_inputs(lengths=synth.varlen_lengths(8, 512, 8192, seed=3), H=H, D=D,
                           seed=rank + 5, device=dev)
    vo = torch.empty(vx.N, H, D, dtype=torch.bfloat16, device=dev)
    vS = torch.empty(vx.B, H, D, D, device=dev)
    vws = torch.empty(max(kda.kda_chunk_prefill_workspace_size(vx.N, vx.B, H), 16),
                      dtype=torch.uint8, device=dev)
    proto["prefill_varlen"] = protocol(
        lambda: kda.kda_chunk_prefill_gated(vx.q, vx.k, vx.v, vx.f, vx.b, vx.A_log, vx.alog_mode,
                                            vx.dt_bias, vx.cu_seqlens, 1.0, None, vS, vo, vws,
                                            stream), warmup=3, iters=10, repeats=3)
    varlen = {"sequences": vx.B, "tokens": vx.N,
              "lengths": [int(a) for a in (vx.cu_seqlens[1:] - vx.cu_seqlens[:-1]).tolist()],
              "ms": proto["prefill_varlen"]["mean_ms"],
              "tokens_per_s": world * vx.N / (proto["prefill_varlen"]["mean_ms"] * 1e-3),
              "protocol": proto["prefill_varlen"]}
    del vx, vo, vS, vws
    T_LONG = 65536
    lx = synth.make_inputs(T_LONG, H=H, D=D, seed=rank + 6, s0_std=0.05, device=dev)
    lo_ = torch.empty(T_LONG, H, D, dtype=torch.bfloat16, device=dev)
    lS = torch.empty(1, H, D, D, device=dev)
    lws = torch.empty(max(kda.kda_chunk_prefill_workspace_size(T_LONG, 1, H), 16),
                      dtype=torch.uint8, device=dev)
    proto["prefill_long"] = protocol(
        lambda: kda.kda_chunk_prefill_gated(lx.q, lx.k, lx.v, lx.f, lx.b, lx.A_log, lx.alog_mode,
                                            lx.dt_bias, None, 1.0, lx.initial_state, lS, lo_,
                                            lws, stream), warmup=2, iters=5, repeats=3)
    ld = synth.make_inputs(128, H=H, D=D, seed=rank + 7, device=dev)
    lg = torch.empty(128, H, D, device=dev)
    lbeta = torch.empty(128, H, device=dev)
    kda.kda_gate_fused(ld.f, ld.b, ld.A_log, ld.alog_mode, ld.dt_bias, lg, lbeta, stream)
    ldo = torch.empty(1, H, D, dtype=torch.bfloat16, device=dev)

    def decode_128():
        for t in range(128):
            kda.kda_recurrent_decode(ld.q[t:t + 1], ld.k[t:t + 1], ld.v[t:t + 1], lg[t:t + 1],
                                     lbeta[t:t + 1], lS, 1.0, ldo, stream)

    proto["decode_after_long"] = protocol(decode_128, warmup=2, iters=3, repeats=3)
    long_context = {"tokens": T_LONG, "ms": proto["prefill_long"]["mean_ms"],
                    "tokens_per_s": world * T_LONG / (proto["prefill_long"]["mean_ms"] * 1e-3),
                    "decode_steps": 128,
                    "decode_ms_per_step": proto["decode_after_long"]["mean_ms"] / 128,
                    "decode_note": "B=1: the 6.3 MB state stays in L2, so this is latency, "
                                   "not an HBM figure",
                    "protocol": {"prefill": proto["prefill_long"],
                                 "decode_128_steps": proto["decode_after_long"]}}
    del lx, lo_, lS, lws, ld, lg, lbeta, ldo

    prefill_leg_ms = max_over_ranks(fused_ms, world, dev)
    step_ms_max = max_over_ranks(step_ms, world, dev)
    decode_ms_max = max_over_ranks(decode_ms, world, dev)
    value = world * T_PREFILL / (prefill_leg_ms * 1e-3)

    # e2e: through the same C ABI, every step copies its inputs from pinned host
    # memory and reads its outputs (o and the final state) back to pinned host
    # memory.  Steps are pipelined as a serving loop would run them: two device
    # buffer sets, host-to-device copies on one stream, the prefill on the
    # compute stream, device-to-host copies on a third, so that step i+1's
    # inputs and step i-1's outputs move while step i computes.  Events order
    # each buffer set's reuse; every step still moves all of its bytes.
    cpus_before = os.sched_getaffinity(0)
    host_numa = host_affinity_for(local_rank)
    host_in = [t.pin_memory() for t in (x.q, x.k, x.v, x.f, x.b)]
    h2d = sum(t.numel() * t.element_size() for t in host_in)
    slots = []
    for _ in range(2):
        slots.append({
            "in": [torch.empty_like(t, device=dev) for t in host_in],
            "o": torch.empty_like(o), "S": torch.empty_like(Sf),
            "host_o": torch.empty(o.shape, dtype=o.dtype).pin_memory(),
            "host_S": torch.empty(Sf.shape, dtype=Sf.dtype).pin_memory(),
            "h2d_done": torch.cuda.Event(), "compute_done": torch.cuda.Event(),
            "d2h_done": torch.cuda.Event(), "used": False,
        })
    d2h = o.numel() * o.element_size() + Sf.numel() * Sf.element_size()
    os.sched_setaffinity(0, cpus_before)   # the buffers stay where they were placed
    h2d_stream = torch.cuda.Stream(dev)
    d2h_stream = torch.cuda.Stream(dev)

    def e2e_step(i):
        sl = slots[i % 2]
        with torch.cuda.stream(h2d_stream):
            if sl["used"]:
                h2d_stream.wait_event(sl["compute_done"])   # step i-2 has read this set
            for hsrc, ddst in zip(host_in, sl["in"]):
                ddst.copy_(hsrc, non_blocking=True)
            sl["h2d_done"].record(h2d_stream)
        stream.wait_event(sl["h2d_done"])
        if sl["used"]:
            stream.wait_event(sl["d2h_done"])              # step i-2's outputs are out
        eq, ek, evv, ef, eb = sl["in"]
        kda.kda_chunk_prefill_gated(eq, ek, evv, ef, eb, A_log, x.alog_mode, dt_bias, None, 1.0,
                                    None, sl["S"], sl["o"], ws, stream)
        sl["compute_done"].record(stream)
        with torch.cuda.stream(d2h_stream):
            d2h_stream.wait_event(sl["compute_done"])
            sl["host_o"].copy_(sl["o"], non_blocking=True)
            sl["host_S"].copy_(sl["S"], non_blocking=True)
            sl["d2h_done"].record(d2h_stream)
        sl["used"] = True

    for i in range(max(args.warmup, 1)):
        e2e_step(i)
    torch.cuda.synchronize(dev)
    barrier(world)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(h2d_stream)
    for i in range(args.steps):
        e2e_step(i)
    d2h_stream.wait_event(slots[(args.steps - 1) % 2]["compute_done"])
    e1.record(d2h_stream)
    torch.cuda.synchronize(dev)
    e2e_ms = max_over_ranks(e0.elapsed_time(e1) / args.steps, world, dev)
    e2e_value = world * T_PREFILL / (e2e_ms * 1e-3)
    # the last step's read-back equals a direct read of its outputs
    last = slots[(args.steps - 1) % 2]
    if not (torch.equal(last["host_o"], last["o"].cpu()) and torch.equal(last["host_S"], last["S"].cpu())):
        raise RuntimeError("e2e read-back does not match the device outputs")

    if kda.kda_get_last_device_error(stream) != 0:
        raise RuntimeError("device error during the timed region")

    if rank != 0:
        return 0
    peaks = measured_peaks()
    hbm = peaks["hbm_gbs"]
    # tf32 dense peak = measured bf16 peak x the ratio of NVIDIA's published dense
    # rates for GB300 (tf32 1.1, bf16 2.25 PFLOP/s per GPU; the per-8-GPU figures of
    # 18 and 36 PFLOP/s are with 2:4 sparsity)
    tf32_peak = peaks["bf16_tflops"] * (1.1 / 2.25)
    pf_flops = H * prefill_flops_per_head([T_PREFILL])
    pf_tflops = pf_flops / (fused_ms * 1e-3) / 1e12
    # fused kernel bytes: q, k, v, f (bf16) and beta logits read, o written, final state
    pf_bytes = T_PREFILL * H * (2 * D * 4 + 4 + 2 * D) + H * D * D * 4
    rl_prefill = {"kernel": "kda chunked prefill with in-kernel gate (tcgen05 kind::tf32)",
                  "bound": "tensor", "achieved": pf_tflops, "peak": tf32_peak, "unit": "TFLOP/s",
                  "frac": pf_tflops / tf32_peak, "traffic": None,
                  "peak_source": f"{peaks['source']} bf16 burst x nominal tf32/bf16 ratio 1.1/2.25",
                  "algorithmic_flops_per_launch": pf_flops,
                  "hbm_achieved_gbs": pf_bytes / (fused_ms * 1e-3) / 1e9,
                  "hbm_frac": pf_bytes / (fused_ms * 1e-3) / 1e9 / hbm,
                  "algorithmic_bytes_per_launch": pf_bytes}
    # the fraction of the binding roof: the time the kernel would take at the
    # slower of its two roofs (tf32 tensor or HBM), over the measured time
    t_tensor_ms = pf_flops / (tf32_peak * 1e12) * 1e3
    t_hbm_ms = pf_bytes / (hbm * 1e9) * 1e3
    roof_ms = max(t_tensor_ms, t_hbm_ms)
    rl_prefill["binding_roof"] = "tensor" if t_tensor_ms >= t_hbm_ms else "hbm"
    rl_prefill["roof_ms"] = {"tensor_tf32": t_tensor_ms, "hbm": t_hbm_ms}
    rl_prefill["binding_roof_frac"] = roof_ms / fused_ms
    rl_prefill["frac_of_bf16_peak"] = pf_tflops / peaks["bf16_tflops"]
    rl_prefill["protocol"] = proto["prefill_gated"]
    up_bytes = prefill_kernel_bytes(T_PREFILL)
    rl_prefill_unfused = {"kernel": "kda chunked prefill, precomputed g and beta",
                          "bound": "tensor",
                          "achieved": pf_flops / (prefill_ms * 1e-3) / 1e12, "peak": tf32_peak,
                          "unit": "TFLOP/s",
                          "frac": pf_flops / (prefill_ms * 1e-3) / 1e12 / tf32_peak,
                          "traffic": None, "algorithmic_flops_per_launch": pf_flops,
                          "hbm_frac": up_bytes / (prefill_ms * 1e-3) / 1e9 / hbm,
                          "algorithmic_bytes_per_launch": up_bytes,
                          "protocol": proto["prefill_unfused"]}
    dec_bytes = decode_bytes()
    dec_gbs = dec_bytes / (decode_ms_max * 1e-3) / 1e9
    rl_decode = {"kernel": "kda recurrent decode", "bound": "hbm",
                 "achieved": dec_gbs, "peak": hbm, "unit": "GB/s", "frac": dec_gbs / hbm,
                 "traffic": None, "peak_source": peaks["source"],
                 "algorithmic_bytes_per_launch": dec_bytes, "protocol": proto["decode"]}
    pool_bytes = decode_bytes(state_bytes=2) + B_DECODE * 4
    pool_gbs = pool_bytes / (pool_ms * 1e-3) / 1e9
    rl_pool = {"kernel": "kda recurrent decode, bf16 state pool by slot", "bound": "hbm",
               "achieved": pool_gbs, "peak": hbm, "unit": "GB/s", "frac": pool_gbs / hbm,
               "traffic": None, "traffic_note": "not captured", "ms": pool_ms,
               "peak_source": peaks["source"], "algorithmic_bytes_per_launch": pool_bytes}
    conv_bytes = 3 * (T_PREFILL * H * D * 4 + H * D * 16 + 3 * H * D * 2)
    conv_gbs = conv_bytes / (conv_ms * 1e-3) / 1e9
    rl_conv = {"kernel": "kda short conv + SiLU + L2 norm pre-step (q, k, v)", "bound": "hbm",
               "achieved": conv_gbs, "peak": hbm, "unit": "GB/s", "frac": conv_gbs / hbm,
               "traffic": None, "traffic_note": "not captured", "ms": conv_ms,
               "peak_source": peaks["source"], "algorithmic_bytes_per_launch": conv_bytes}
    # backward: per token-head one forward step (5 K V flops: decay, column sum,
    # rank-1 update) and one reverse step (18 K V: G += q do^T, du, S', w, four
    # row sums, G update), against the fp32 FMA rate of the CUDA cores (SMs x 128
    # lanes x 2 flops x the median SM clock sampled in the timed region)
    bwd_flops = T_PREFILL * H * 23 * D * D
    sm_mhz = clocks.get("sm_mhz") or peaks.get("sm_max_mhz") or 2070.0
    fp32_peak = (torch.cuda.get_device_properties(dev).multi_processor_count * 128 * 2 *
                 sm_mhz * 1e6 / 1e12)
    bwd_tflops = bwd_flops / (bwd_ms * 1e-3) / 1e12
    rl_bwd = {"kernel": "kda recurrent backward (token by token, CUDA cores)", "bound": "alu",
              "achieved": bwd_tflops, "peak": fp32_peak, "unit": "TFLOP/s",
              "frac": bwd_tflops / fp32_peak, "traffic": None, "traffic_note": "not captured",
              "peak_source": "fp32 FMA lanes x median SM clock of the timed region",
              "algorithmic_flops_per_launch": bwd_flops, "ms": bwd_ms,
              "tokens_per_s": T_PREFILL / (bwd_ms * 1e-3)}
    gate_bytes = T_PREFILL * H * (2 * D + 4 * D + 8)
    gate_gbs = gate_bytes / (gate_ms * 1e-3) / 1e9
    rl_gate = {"kernel": "kda gate", "bound": "hbm", "achieved": gate_gbs, "peak": hbm,
               "unit": "GB/s", "frac": gate_gbs / hbm, "traffic": None,
               "peak_source": peaks["source"], "algorithmic_bytes_per_launch": gate_bytes,
               "protocol": proto["gate"]}
    cb_ms = proto["backward_chunked"]["mean_ms"]
    cb_flops = H * chunk_backward_flops_per_head([T_PREFILL])
    cb_tflops = cb_flops / (cb_ms * 1e-3) / 1e12
    rl_cbwd = {"kernel": "kda chunked backward (tcgen05 bf16 high/low products; with its "
                         "checkpointing forward pass)", "bound": "tensor",
               "achieved": cb_tflops, "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
               "frac": cb_tflops / peaks["bf16_tflops"], "traffic": None,
               "peak_source": f"{peaks['source']} bf16 burst",
               "algorithmic_flops_per_launch": cb_flops, "ms": cb_ms,
               "tokens_per_s": T_PREFILL / (cb_ms * 1e-3),
               "protocol": proto["backward_chunked"]}
    kb_ms = proto["backward_checkpointed"]["mean_ms"]
    kb_flops = cb_flops - H * prefill_flops_per_head([T_PREFILL])
    kb_tflops = kb_flops / (kb_ms * 1e-3) / 1e12
    training = {"prefill_checkpointed_ms": proto["prefill_checkpointed"]["mean_ms"],
                "backward_checkpointed_ms": kb_ms,
                "backward_checkpointed_tflops": kb_tflops,
                "backward_checkpointed_frac": kb_tflops / peaks["bf16_tflops"],
                "checkpoint_bytes": kda.kda_chunk_checkpoints_size(T_PREFILL, 1, H),
                "protocol": {"prefill_checkpointed": proto["prefill_checkpointed"],
                             "backward_checkpointed": proto["backward_checkpointed"]}}
    for rl, kid in ((rl_prefill, "chunk_gated"), (rl_prefill_unfused, "chunk_unfused"),
                    (rl_decode, "decode"), (rl_pool, "decode_pool"), (rl_gate, "gate"),
                    (rl_conv, "short_conv"), (rl_bwd, "backward"), (rl_cbwd, "backward_chunked")):
        rl["traffic"], rl["traffic_note"] = measured_traffic(kid)
    # the dominant kernel is the one with the largest share of the step
    roofline = rl_prefill if fused_ms >= decode_ms_max else rl_decode
    cpu = cpu_baseline(args.cpu_heads) if not args.no_cpu_baseline else None
    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": step_ms_max,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "tf32",
        "data": "synthetic",
        "config": {"workload": WORKLOAD, "inputs_exceed_l2": True, "l2_flush": False,
                   "prefill_T": T_PREFILL, "heads": H, "d": D, "decode_batch": B_DECODE,
                   "parallelism": f"replicas x{world}"},
        "prefill_gated_ms": fused_ms, "decode_gate_ms": dgate_ms, "decode_ms": decode_ms_max,
        "unfused": {"gate_ms": gate_ms, "prefill_ms": prefill_ms,
                    "tokens_per_s": T_PREFILL / ((gate_ms + prefill_ms) * 1e-3)},
        "decode_gated_ms": gdecode_ms,
        "decode_state_gbs": dec_gbs, "decode_frac_of_hbm": dec_gbs / hbm,
        "roofline": roofline,
        "rooflines": {"gate": rl_gate, "prefill_gated": rl_prefill,
                      "prefill_unfused": rl_prefill_unfused, "decode": rl_decode,
                      "decode_bf16_pool": rl_pool, "short_conv": rl_conv, "backward": rl_bwd,
                      "backward_chunked": rl_cbwd},
        "training": training,
        "prefill_varlen": varlen,
        "prefill_long_context": long_context,
        "e2e": {"value": e2e_value, "unit": "tokens/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms,
                "schedule": "steps pipelined over two buffer sets: H2D, prefill and D2H "
                            "on three streams", "host_memory": host_numa},
        "gpu_launches": launches_per_step * args.steps,
        "clocks": clocks,
        "peaks": peaks,
        "cpu_baseline": cpu,
    }
    print(json.dumps(line))
    return 0


def run_profile_case(args):
    """A few launches of one kernel at a chosen size, for ncu captures
    (`ncu -k regex:<kernel> -s <warm-up launches> -c 1 python bench.py --profile ...`).
    Prints one line; its timings are not bench values."""
    import gated_delta_rule_33_gb300 as kda
    from gated_delta_rule_33_gb300 import synth
    dev = torch.device("cuda", 0)
    kda.load()
    if args.profile == "short_conv":
        sx = synth.make_shortconv_inputs(args.size, H=H, D=D, seed=0)
        xs = [t.to(dev) for t in sx.x]
        ws = [t.to(dev) for t in sx.w]
        for _ in range(args.warmup + 1):
            kda.short_conv(*xs, *ws)
    elif args.profile in ("gate", "prefill", "prefill_gated", "backward", "backward_chunked"):
        x = synth.make_inputs(args.size, H=H, D=D, seed=0, device=dev)
        g, beta = kda.gate(x.f, x.b, x.A_log, x.dt_bias, x.alog_mode)
        dO = torch.randn_like(x.q) if args.profile.startswith("backward") else None
        for _ in range(args.warmup + 1):
            if args.profile == "gate":
                kda.gate(x.f, x.b, x.A_log, x.dt_bias, x.alog_mode)
            elif args.profile == "prefill":
                kda.prefill(x.q, x.k, x.v, g, beta)
            elif args.profile == "prefill_gated":
                kda.prefill_gated(x.q, x.k, x.v, x.f, x.b, x.A_log, x.dt_bias, x.alog_mode)
            elif args.profile == "backward":
                kda.backward(x.q, x.k, x.v, g, beta, dO, want_dS0=False)
            else:
                kda.backward_chunked(x.q, x.k, x.v, g, beta, dO, want_dS0=False)
    else:
        d = synth.make_decode_inputs(args.size, H=H, D=D, seed=0, state_device=dev)
        q, k, v, f, b = (t.to(dev) for t in (d.q, d.k, d.v, d.f, d.b))
        g, beta = kda.gate(f, b, d.A_log.to(dev), d.dt_bias.to(dev), d.alog_mode)
        if args.profile == "decode_pool":
            pool = d.state.to(torch.bfloat16)
            slots = torch.arange(args.size - 1, -1, -1, dtype=torch.int32, device=dev)
            del d
        for _ in range(args.warmup + 1):
            if args.profile == "decode":
                kda.decode(q, k, v, g, beta, d.state)
            else:
                kda.decode_indexed(q, k, v, g, beta, pool, slots)
    torch.cuda.synchronize()
    st = kda.kda_get_last_device_error()
    print(json.dumps({"profile": args.profile, "size": args.size, "device_error": st}))
    return 0 if st == 0 else 1


def main():
    ap = argparse.ArgumentParser(description=__doc__)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--ref-heads", type=int, default=8,
                    help="heads of the T=4096 workload per reference-arm step")
    ap.add_argument("--cpu-heads", type=int, default=96,
                    help="heads of the T=4096 workload timed for cpu_baseline")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--profile", choices=["gate", "prefill", "prefill_gated", "decode",
                                          "decode_pool", "short_conv", "backward",
                                          "backward_chunked"], default=None,
                    help="run only this kernel (warm-up + 1 launch) for an ncu capture")
    ap.add_argument("--size", type=int, default=1024,
                    help="--profile size: tokens (gate, prefill) or sequences (decode)")
    args = ap.parse_args()
    if args.profile is not None:
        return run_profile_case(args)
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
