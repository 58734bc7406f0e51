#!/usr/bin/env python
"""Throughput of the groupwise low-bit linear layer on one GB300 (or N replicas).

Workload (default): the Llama-3.1-8B decode linears at M = 1, group 64, bit
widths 1..7 -- (K, N) = (4096, 6144) qkv, (4096, 4096) o, (4096, 28672)
gate+up, (14336, 4096) down -- 28 layers.  One step is one call of every
layer: 28 launches of the qmv kernel over ~0.9 GB of packed weights, scales
and zeros, more than the 129 MB L2, so every launch reads its weights cold.

  value      algorithmic HBM bytes of a step / device time of a step, GB/s,
             with all inputs resident in HBM; the step is replayed from a
             CUDA graph of 28 C-ABI calls.
  e2e        the same metric with every input copied from pinned host memory
             and y copied back, through the public Python binding, per step
             (the step's inputs in one pinned arena, copied in four chunks that
             overlap the previous chunk's layers; host-to-device bandwidth on
             this machine, ~210 GB/s, bounds it).
  roofline   the qmv kernel alone: per-layer time (CUDA graphs of flush + call
             minus flush alone), summed over the 28 layers.
  qmm_m128   the batched form: the same shapes at M = 128, b = 4, g = 128 on the
             tensor-core kernel, TFLOP/s against the measured bf16 peak.
  quantize   the GPU quantiser on the gate+up weight (bf16, b = 4, g = 64),
             GB/s against the measured HBM peak.
  int4wo_128 the int4wo-128 configuration (b = 4, g = 128) of the same linears
             at M = 1 (per call, L2 flushed) and M = 128 (the qmm_m128
             numbers), summed over the 8B model's 32 decoder layers.
  swiglu_gate_up  the fused gate+up call (silu(gate) * up, F = 14336 outputs)
             on the gate+up weights of the step, per bit width, beside the
             plain linear on the same weight.
  cpu_baseline  the fp64 CPU oracle on a bounded sample of output rows.

``--impl reference`` times the CPU oracle instead (the method's plain
definition; no GPU work).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time
from pathlib import Path

import numpy as np

ROOT = Path(__file__).resolve().parent
sys.path.insert(0, str(ROOT))

import synth  # noqa: E402

METRIC = "qmv µs & achieved HBM GB/s (M=1, b=1..7) vs 8 TB/s; qmm TFLOP/s at M=128"
GROUP = 64
BITS = tuple(range(1, 8))
WORKLOAD = "llama3.1-8b decode linears: M=1, g=64, b=1..7, (K,N) in qkv/o/gate_up/down"


def layer_list():
    return [(name, K, N, b) for b in BITS for name, (K, N) in synth.LLAMA_8B.items()]


def algorithmic_bytes(M, K, N, bits, group, bias=False, rows=None):
    """Bytes the method must move: packed codes + fp16 scale and zero + x + y (+ bias)."""
    n = N if rows is None else rows
    return n * K * bits // 8 + 4 * n * (K // group) + 2 * M * K + 2 * M * n + (2 * n if bias else 0)


def measured_peaks():
    p = ROOT / "MEASURED_PEAKS.json"
    if p.exists():
        d = json.loads(p.read_text())
        return float(d["hbm_gbs"]), float(d.get("bf16_tflops", 0.0)), "measured"
    return 6800.0, 1900.0, "fallback"


# ---------------------------------------------------------------------------
# Distributed plumbing (replicas; no collective on the data path).
# ---------------------------------------------------------------------------

def whole_job_gbs(world: int, step_bytes: int, steps: int, ms_total_max: float) -> float:
    """Weak scaling: every rank streams step_bytes per step; the job's rate is
    all ranks' bytes over the slowest rank's time."""
    return world * step_bytes * steps / (ms_total_max / 1e3) / 1e9


def dist_env():
    return int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")), \
        int(os.environ.get("LOCAL_RANK", "0"))


class Dist:
    def __init__(self, backend):
        import torch.distributed as dist
        self.rank, self.world, self.local = dist_env()
        self.dist = dist if self.world > 1 else None
        if self.dist is not None:
            dist.init_process_group(backend=backend)

    def barrier(self):
        if self.dist is not None:
            self.dist.barrier()

    def max(self, v: float) -> float:
        if self.dist is None:
            return v
        import torch
        dev = "cuda" if self.dist.get_backend() == "nccl" else "cpu"
        t = torch.tensor([v], dtype=torch.float64, device=dev)
        self.dist.all_reduce(t, op=self.dist.ReduceOp.MAX)
        return float(t.item())

    def close(self):
        if self.dist is not None:
            self.dist.destroy_process_group()


# ---------------------------------------------------------------------------
# Clocks during the timed region (nvidia-smi, sampled in the background).
# ---------------------------------------------------------------------------

class ClockSampler:
    FIELDS = ("index,pci.bus_id,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, bus_id: str | None):
        self.bus_id = bus_id
        self.proc = None
        self.lines: list[str] = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "50"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.thread.join(timeout=2)
        rows = [r.split(", ") for r in self.lines if r.count(",") >= 9]
        if self.bus_id:
            mine = [r for r in rows if r[1].lower().endswith(self.bus_id.lower()[-12:])]
            rows = mine or rows
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
        idx = rows[0][0]
        rows = [r for r in rows if r[0] == idx]

        def num(s):
            try:
                return float(s)
            except ValueError:
                return None
        sm = [num(r[2]) for r in rows if num(r[2]) is not None]
        reasons = set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            for name, v in zip(names, r[6:10]):
                if v.strip().lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": num(rows[0][3]), "reasons": sorted(reasons), "samples": len(rows),
                "power_w_max": max((num(r[4]) or 0.0) for r in rows)}


# ---------------------------------------------------------------------------
# The CPU oracle on a sample of output rows (reference arm and cpu_baseline).
# ---------------------------------------------------------------------------

class OracleSample:
    """Host inputs for a sample of rows of every layer, packed by the oracle."""

    def __init__(self, rows_per_layer: int, seed: int = 0):
        import oracle
        self.o = oracle.Oracle()
        self.items = []
        for name, K, N, b in layer_list():
            key = (b, GROUP)
            r = np.random.default_rng([seed, K, N, b]).choice(N, rows_per_layer, replace=False)
            r.sort()
            x = synth.make_x(seed, 1, K, False, key)
            codes = synth.make_codes(seed, N, K, b, key)[r]
            s, z = synth.make_scale_zero(seed, N, K // GROUP, (K, b, GROUP))
            self.items.append(dict(K=K, b=b, x=x, packed=self.o.pack(codes, b), s=s[r], z=z[r],
                                   rows=np.arange(r.size), bytes=algorithmic_bytes(
                                       1, K, N, b, GROUP, rows=r.size)))
        self.bytes = sum(i["bytes"] for i in self.items)

    def run(self):
        for i in self.items:
            self.o.linear_rows(i["x"], i["packed"], i["s"], i["z"], None, i["K"], i["b"], GROUP,
                               i["rows"])


def calibrate_oracle(seconds: float):
    """Rows per layer such that one pass over all 28 layers takes about ``seconds``."""
    probe = OracleSample(2)
    t = time.perf_counter()
    probe.run()
    dt = max(time.perf_counter() - t, 1e-6)
    rows = int(max(1, min(4096, 2 * seconds / dt)))
    return OracleSample(rows), rows


def time_oracle(sample: OracleSample, reps: int = 1):
    t = time.perf_counter()
    for _ in range(reps):
        sample.run()
    dt = time.perf_counter() - t
    return sample.bytes * reps / dt / 1e9, dt


# ---------------------------------------------------------------------------
# Arms.
# ---------------------------------------------------------------------------

def base_config():
    return {"workload": WORKLOAD, "M": 1, "group": GROUP, "bits": list(BITS),
            "shapes_KN": {k: list(v) for k, v in synth.LLAMA_8B.items()},
            "layers_per_step": len(layer_list()), "bias": False,
            "l2": "inputs larger than L2 (each step streams ~0.9 GB of distinct weights)",
            "seed": 0}


def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return 0
    total = args.steps + args.warmup
    per_step = min(5.0, 90.0 / max(total, 1))
    sample, rows = calibrate_oracle(per_step)
    for _ in range(args.warmup):
        sample.run()
    gbs, dt = time_oracle(sample, args.steps)
    ms = dt / args.steps * 1e3
    line = {
        "impl": "reference", "metric": METRIC, "value": gbs, "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": base_config(),
        "cpu_baseline": {"value": gbs, "unit": "GB/s", "cores": 1, "kind": "oracle",
                         "sample": f"{rows} output rows of each of the 28 layers per step"},
        "e2e": {"value": gbs, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def kernel_source_hash():
    h = hashlib.sha256()
    for p in sorted((ROOT / "bit_groupwise_weight_gb300" / "csrc").glob("*")):
        if p.name in ("qmv.cu", "common.cuh"):
            h.update(p.read_bytes())
    return h.hexdigest()[:16]


def profiled_traffic():
    """Per-launch DRAM bytes (read + write) of the qmv kernel from the committed ncu
    summary, if that summary was taken on the current kernel source; else None."""
    p = ROOT / "profiles" / "qmv_stream_llama8b_decode.md"
    if not p.exists():
        return None
    fields = {}
    for line in p.read_text().splitlines():
        if line.startswith("- ") and ": " in line:
            k, v = line[2:].split(": ", 1)
            fields[k.strip()] = v.strip().strip("`")
    if fields.get("kernel_source_sha256_16") != kernel_source_hash():
        return None
    try:
        return float(fields["dram_bytes_per_launch"])
    except (KeyError, ValueError):
        return None


def measure_qmm(torch, lb, dev, stream, M=128, bits=4, group=128, reps=10):
    """The batched form: the same four Llama-3.1-8B shapes at M = 128, b = 4, g = 128, with
    bias and 1% outlier columns in x, on the tensor-core kernel.  Each layer is timed as a
    CUDA graph of `reps` calls; TFLOP/s = 2*M*N*K / time."""
    out = []
    for name, (K, N) in synth.LLAMA_8B.items():
        L = synth.make_layer(0, M, K, N, bits, group, bias=True, outliers=True)
        w = lb.pack_weights(torch.from_numpy(L.codes).to(dev), bits)
        x = torch.from_numpy(L.x.view(np.int16)).view(torch.bfloat16).to(dev)
        s = torch.from_numpy(L.scales.view(np.int16)).view(torch.float16).to(dev)
        z = torch.from_numpy(L.zeros.view(np.int16)).view(torch.float16).to(dev)
        b = torch.from_numpy(L.bias.view(np.int16)).view(torch.float16).to(dev)
        y = torch.empty((M, N), dtype=torch.bfloat16, device=dev)

        def call():
            lb.linear_ptr(x.data_ptr(), w.data_ptr(), s.data_ptr(), z.data_ptr(), b.data_ptr(),
                          y.data_ptr(), M, K, N, bits, group, stream.cuda_stream, lb.PATH_QMM)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(stream):
            call()
            stream.synchronize()
            with torch.cuda.graph(g, stream=stream):
                for _ in range(reps):
                    call()
        stream.synchronize()
        best = float("inf")
        for _ in range(5):
            a = torch.cuda.Event(enable_timing=True)
            c = torch.cuda.Event(enable_timing=True)
            with torch.cuda.stream(stream):
                a.record(stream)
                g.replay()
                c.record(stream)
            stream.synchronize()
            best = min(best, a.elapsed_time(c) * 1e3 / reps)
        out.append({"layer": name, "K": K, "N": N, "us": round(best, 2),
                    "TFLOPs": round(2 * M * N * K / best / 1e6, 1)})
        del w, x, s, z, b, y, g
    total_flop = sum(2 * M * o["N"] * o["K"] for o in out)
    total_us = sum(o["us"] for o in out)
    tflops = total_flop / total_us / 1e6
    _, tc_peak, kind = measured_peaks()
    return {"M": M, "bits": bits, "group": group, "TFLOPs": round(tflops, 1),
            "roofline": {"bound": "tensor", "achieved": round(tflops, 1), "peak": tc_peak,
                         "unit": "TFLOP/s", "frac": round(tflops / tc_peak, 4),
                         "peak_kind": f"{kind} bf16_tflops (burst)"},
            "layers": out, "timing": "CUDA graph of 10 calls per layer; weights 4-59 MB, L2-warm"}


def measure_quantize(torch, lb, dev, stream, bits=4, group=64, reps=5):
    """The quantiser on the largest Llama-3.1-8B weight (gate+up, K=4096, N=28672) in bf16:
    235 MB read per call, more than L2, so back-to-back calls stream from HBM.
    GB/s = (weights read + packed codes, scales and zeros written) / time."""
    K, N = synth.LLAMA_8B["gate_up"]
    w32 = synth.make_weights(0, N, K)
    w = torch.from_numpy(synth.f32_to_bf16_bits(w32).view(np.int16)).view(torch.bfloat16).to(dev)
    packed = torch.empty((N, K * bits // 8), dtype=torch.uint8, device=dev)
    sc = torch.empty((N, K // group), dtype=torch.float16, device=dev)
    ze = torch.empty((N, K // group), dtype=torch.float16, device=dev)
    with torch.cuda.stream(stream):
        lb.quantize_weights(w, bits, group, packed, sc, ze)
        stream.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for _ in range(reps):
                lb.quantize_weights(w, bits, group, packed, sc, ze)
    stream.synchronize()
    best = float("inf")
    for _ in range(5):
        a = torch.cuda.Event(enable_timing=True)
        c = torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            a.record(stream)
            g.replay()
            c.record(stream)
        stream.synchronize()
        best = min(best, a.elapsed_time(c) * 1e3 / reps)
    nbytes = N * K * 2 + N * K * bits // 8 + 4 * N * (K // group)
    gbs = nbytes / best / 1e3
    hbm_peak, _, kind = measured_peaks()
    return {"layer": "gate_up", "K": K, "N": N, "bits": bits, "group": group, "w_dtype": "bf16",
            "us": round(best, 2), "bytes": nbytes,
            "roofline": {"bound": "hbm", "achieved": round(gbs, 1), "peak": hbm_peak,
                         "unit": "GB/s", "frac": round(gbs / hbm_peak, 4),
                         "peak_kind": f"{kind} hbm_gbs (burst copy)"},
            "timing": f"CUDA graph of {reps} calls; 235 MB of weights per call (> L2)"}


def run_ours(args):
    import torch
    import bit_groupwise_weight_gb300 as lb
    from bit_groupwise_weight_gb300 import build as lbuild

    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    dist = Dist("nccl")
    lbuild.build()
    dev = torch.device("cuda", local)
    stream = torch.cuda.Stream(dev)

    # --- inputs: host (pinned) and device copies of every layer -----------------
    layers = []
    for name, K, N, b in layer_list():
        key = (b, GROUP)
        x = synth.make_x(0, 1, K, False, key)
        codes = synth.make_codes(0, N, K, b, key)
        s, z = synth.make_scale_zero(0, N, K // GROUP, (K, b, GROUP))
        d_codes = torch.from_numpy(codes).to(dev)
        with torch.cuda.stream(stream):
            packed = lb.pack_weights(d_codes, b)
        stream.synchronize()
        del d_codes
        t = dict(name=name, K=K, N=N, b=b,
                 x=torch.from_numpy(x.view(np.int16)).view(torch.bfloat16).to(dev),
                 w=packed,
                 s=torch.from_numpy(s.view(np.int16)).view(torch.float16).to(dev),
                 z=torch.from_numpy(z.view(np.int16)).view(torch.float16).to(dev),
                 y=torch.empty((1, N), dtype=torch.bfloat16, device=dev),
                 bytes=algorithmic_bytes(1, K, N, b, GROUP))
        layers.append(t)
    step_bytes = sum(t["bytes"] for t in layers)

    def call(t, st):
        lb.linear_ptr(t["x"].data_ptr(), t["w"].data_ptr(), t["s"].data_ptr(), t["z"].data_ptr(),
                      None, t["y"].data_ptr(), 1, t["K"], t["N"], t["b"], GROUP, st)

    # --- CUDA graph of one step --------------------------------------------------
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        for t in layers:           # one eager pass first (module load, first-call setup)
            call(t, stream.cuda_stream)
        stream.synchronize()
        with torch.cuda.graph(graph, stream=stream):
            for t in layers:
                call(t, stream.cuda_stream)
    stream.synchronize()

    bus = None
    try:
        bus = torch.cuda.get_device_properties(dev).pci_bus_id
    except AttributeError:
        bus = None

    with torch.cuda.stream(stream):
        for _ in range(max(args.warmup, 3)):
            graph.replay()
    stream.synchronize()

    ev0 = torch.cuda.Event(enable_timing=True)
    ev1 = torch.cuda.Event(enable_timing=True)
    clocks = ClockSampler(bus)
    clocks.start()
    time.sleep(0.15)
    dist.barrier()
    torch.cuda.synchronize(dev)
    with torch.cuda.stream(stream):
        ev0.record(stream)
        for _ in range(args.steps):
            graph.replay()
        ev1.record(stream)
    torch.cuda.synchronize(dev)
    dist.barrier()
    clk = clocks.stop()
    ms_total = ev0.elapsed_time(ev1)
    ms_total = dist.max(ms_total)
    ms_per_step = ms_total / args.steps
    value = whole_job_gbs(world, step_bytes, args.steps, ms_total)

    # --- per-layer kernel time, cold L2 (roofline of the qmv kernel) -------------
    # CUDA-event timestamps are coarse on this platform (about 2 us), so each layer is
    # timed as a difference of two CUDA graphs: n x (L2 flush + call) minus n x flush.
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    flush = torch.empty(int(2 * l2), dtype=torch.uint8, device=dev)

    def graph_us(fn, reps=5):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(stream):
            fn()
            stream.synchronize()
            with torch.cuda.graph(g, stream=stream):
                fn()
        stream.synchronize()
        best = float("inf")
        for _ in range(reps):
            a = torch.cuda.Event(enable_timing=True)
            c = torch.cuda.Event(enable_timing=True)
            with torch.cuda.stream(stream):
                a.record(stream)
                g.replay()
                c.record(stream)
            stream.synchronize()
            best = min(best, a.elapsed_time(c) * 1e3)
        return best

    nrep = 10
    flush_us = graph_us(lambda: [flush.fill_(i) for i in range(nrep)])
    per_layer = []
    for t in layers:
        def with_call(t=t):
            for i in range(nrep):
                flush.fill_(i)
                call(t, stream.cuda_stream)
        # A difference at or below zero (possible under a profiler) counts as 1 ns.
        us = max(graph_us(with_call) - flush_us, 1e-2) / nrep
        per_layer.append({"layer": t["name"], "bits": t["b"], "K": t["K"], "N": t["N"],
                          "us": round(us, 3), "GBps": round(t["bytes"] / us / 1e3, 1), "_us": us})
    # --- the fused gate+up call (silu(gate) * up) on the same gate+up weights ----
    swiglu = []
    if not args.no_swiglu:
        for t in layers:
            if t["name"] != "gate_up":
                continue
            F = t["N"] // 2
            h = torch.empty((1, F), dtype=torch.bfloat16, device=dev)

            def with_glu(t=t, h=h, F=F):
                for i in range(nrep):
                    flush.fill_(i)
                    lb.linear_swiglu_ptr(t["x"].data_ptr(), t["w"].data_ptr(), t["s"].data_ptr(),
                                         t["z"].data_ptr(), None, h.data_ptr(), 1, t["K"], F, t["b"],
                                         GROUP, stream.cuda_stream)
            us = max(graph_us(with_glu) - flush_us, 1e-2) / nrep
            plain = next(p for p in per_layer if p["layer"] == "gate_up" and p["bits"] == t["b"])
            nbytes = algorithmic_bytes(1, t["K"], t["N"], t["b"], GROUP) - 2 * F   # y holds F outputs
            swiglu.append({"bits": t["b"], "K": t["K"], "F": F, "us": round(us, 3),
                           "plain_linear_us": plain["us"], "GBps": round(nbytes / us / 1e3, 1)})
    # --- the int4wo-128 configuration (b = 4, g = 128) at M = 1 ------------------
    int4_m1 = []
    if not args.no_int4wo:
        for t in layers:
            if t["b"] != 4:
                continue
            sc, zc = synth.make_scale_zero(0, t["N"], t["K"] // 128, (t["K"], 4, 128))
            s128 = torch.from_numpy(sc.view(np.int16)).view(torch.float16).to(dev)
            z128 = torch.from_numpy(zc.view(np.int16)).view(torch.float16).to(dev)

            def with_int4(t=t, s128=s128, z128=z128):
                for i in range(nrep):
                    flush.fill_(i)
                    lb.linear_ptr(t["x"].data_ptr(), t["w"].data_ptr(), s128.data_ptr(), z128.data_ptr(),
                                  None, t["y"].data_ptr(), 1, t["K"], t["N"], 4, 128, stream.cuda_stream)
            us = max(graph_us(with_int4) - flush_us, 1e-2) / nrep
            nbytes = algorithmic_bytes(1, t["K"], t["N"], 4, 128)
            int4_m1.append({"layer": t["name"], "K": t["K"], "N": t["N"], "us": round(us, 3),
                            "GBps": round(nbytes / us / 1e3, 1)})
    del flush
    kern_us = sum(p.pop("_us") for p in per_layer)
    achieved = step_bytes / kern_us / 1e3
    hbm_peak, tc_peak, peak_kind = measured_peaks()

    # --- e2e: host buffers through the public API --------------------------------
    # A step's inputs live in one pinned host arena (each tensor 256-byte
    # aligned) and are copied in E2E_CHUNKS large copies on a copy stream; the
    # layers of chunk c run on the compute stream as soon as chunk c has landed,
    # while chunk c + 1 is still in flight.  The outputs land in one device
    # arena and come back in one copy.  Timed from the first copy to the end of
    # the last.
    e2e_steps = max(1, min(args.steps, 10))
    align = 256
    offs, size = [], 0
    for t in layers:
        o = {}
        for k in ("x", "w", "s", "z"):
            o[k] = size
            size += (t[k].numel() * t[k].element_size() + align - 1) // align * align
        offs.append(o)
    host_arena = torch.empty(size, dtype=torch.uint8).pin_memory()
    dev_arena = torch.empty(size, dtype=torch.uint8, device=dev)
    views = []
    for t, o in zip(layers, offs):
        v = {}
        for k in ("x", "w", "s", "z"):
            nb = t[k].numel() * t[k].element_size()
            host_arena[o[k]:o[k] + nb].copy_(t[k].reshape(-1).view(torch.uint8).cpu())
            v[k] = dev_arena[o[k]:o[k] + nb].view(t[k].dtype).view(t[k].shape)
        views.append(v)
    y_sizes = [t["N"] for t in layers]
    y_dev = torch.empty(sum(y_sizes), dtype=torch.bfloat16, device=dev)
    y_host = torch.empty(sum(y_sizes), dtype=torch.bfloat16).pin_memory()
    y_views, yo = [], 0
    for n in y_sizes:
        y_views.append(y_dev[yo:yo + n].view(1, n))
        yo += n
    E2E_CHUNKS = 4
    bounds = [round(i * len(layers) / E2E_CHUNKS) for i in range(E2E_CHUNKS + 1)]
    copy_stream = torch.cuda.Stream(dev)
    h2d = size
    d2h = y_host.numel() * 2
    torch.cuda.synchronize(dev)
    dist.barrier()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    landed = [torch.cuda.Event() for _ in range(E2E_CHUNKS)]
    with torch.cuda.stream(stream):
        e0.record(stream)
        for _ in range(e2e_steps):
            copy_stream.wait_stream(stream)           # the previous step is done with the arena
            with torch.cuda.stream(copy_stream):
                for c in range(E2E_CHUNKS):
                    lo = offs[bounds[c]]["x"]
                    hi = offs[bounds[c + 1]]["x"] if bounds[c + 1] < len(layers) else size
                    dev_arena[lo:hi].copy_(host_arena[lo:hi], non_blocking=True)
                    landed[c].record(copy_stream)
            for c in range(E2E_CHUNKS):
                stream.wait_event(landed[c])
                for i in range(bounds[c], bounds[c + 1]):
                    t, v = layers[i], views[i]
                    lb.linear(v["x"], v["w"], v["s"], v["z"], None, t["b"], GROUP, out=y_views[i])
            y_host.copy_(y_dev, non_blocking=True)
        e1.record(stream)
    torch.cuda.synchronize(dev)
    e2e_ms = dist.max(e0.elapsed_time(e1)) / e2e_steps
    e2e_value = world * step_bytes / (e2e_ms / 1e3) / 1e9
    # The arena round trip must reproduce the device-resident results.
    for i, t in enumerate(layers):
        ref = lb.linear(t["x"], t["w"], t["s"], t["z"], None, t["b"], GROUP)
        assert torch.equal(y_views[i], ref), f"e2e output of layer {i} differs"
    del dev_arena, host_arena

    qmm = None if args.no_qmm else measure_qmm(torch, lb, dev, stream)
    int4wo = None
    if int4_m1:
        # The 8B model has 32 decoder layers of these four linears.
        stack1 = 32 * sum(r["us"] for r in int4_m1)
        int4wo = {"bits": 4, "group": 128, "M1": {"layers": int4_m1, "stack_us": round(stack1, 1),
                                                  "linear_tokens_per_s": round(1e6 / stack1, 1),
                                                  "timing": "per call, L2 flushed, CUDA-graph differences"}}
        if qmm is not None:
            stack128 = 32 * sum(r["us"] for r in qmm["layers"])
            int4wo["M128"] = {"layers": qmm["layers"], "stack_us": round(stack128, 1),
                              "linear_tokens_per_s": round(128 * 1e6 / stack128, 1),
                              "timing": qmm["timing"]}
        int4wo["what"] = ("the int4wo-128 configuration (4-bit codes, groups of 128) on the Llama-3.1-8B "
                          "linears; stack_us = 32 decoder layers x (qkv + o + gate_up + down), the linear "
                          "layers' share of one decode step (no attention, norms, embeddings or lm_head)")
    quant = None if args.no_quantize else measure_quantize(torch, lb, dev, stream)

    line = {
        "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": base_config() | {"parallelism": f"replicas{world}" if world > 1 else "single",
                                   "step_bytes": step_bytes},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": hbm_peak, "unit": "GB/s",
                     "frac": achieved / hbm_peak, "traffic": profiled_traffic(),
                     "kernel": "qmv_stream (all 28 layers; per-launch time from CUDA graphs, L2 flushed)",
                     "peak_kind": f"{peak_kind} hbm_gbs (burst copy)"},
        "e2e": {"value": e2e_value, "unit": "GB/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h},
        "gpu_launches": len(layers) * args.steps,
        "clocks": clk,
        "layers": per_layer,
    }
    if qmm is not None:
        line["qmm_m128"] = qmm
    if quant is not None:
        line["quantize"] = quant
    if int4wo is not None:
        line["int4wo_128"] = int4wo
    if swiglu:
        line["swiglu_gate_up"] = {
            "M": 1, "group": GROUP, "layers": swiglu,
            "what": "lowbit_linear_swiglu: silu(gate) * up from the 8B gate+up weight in one call "
                    "(F = 14336 outputs); plain_linear_us is lowbit_linear on the same weight",
            "timing": "per call, L2 flushed, CUDA-graph differences"}

    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        sample, rows = calibrate_oracle(args.cpu_seconds)
        gbs, _ = time_oracle(sample)
        line["cpu_baseline"] = {"value": gbs, "unit": "GB/s", "cores": 1, "kind": "oracle",
                                "sample": f"{rows} output rows of each of the 28 layers "
                                          f"(fp64, one thread)"}
    if rank == 0:
        print(json.dumps(line), flush=True)
    dist.close()
    return 0


def run_profile_layer(spec: str, calls: int):
    """Call one layer `calls` times through lowbit_linear, nothing timed: a small, fixed
    workload for ncu captures.  spec = name:bits:M[:group], name one of qkv/o/gate_up/down."""
    import torch
    import bit_groupwise_weight_gb300 as lb
    from bit_groupwise_weight_gb300 import build as lbuild
    lbuild.build()
    parts = spec.split(":")
    name, bits, M = parts[0], int(parts[1]), int(parts[2])
    group = int(parts[3]) if len(parts) > 3 else (64 if M <= 2 else 128)
    K, N = synth.LLAMA_8B[name]
    L = synth.make_layer(0, M, K, N, bits, group, bias=M > 2, outliers=M > 2)
    dev = torch.device("cuda", 0)
    w = lb.pack_weights(torch.from_numpy(L.codes).to(dev), bits)
    x = torch.from_numpy(L.x.view(np.int16)).view(torch.bfloat16).to(dev)
    s = torch.from_numpy(L.scales.view(np.int16)).view(torch.float16).to(dev)
    z = torch.from_numpy(L.zeros.view(np.int16)).view(torch.float16).to(dev)
    b = None if L.bias is None else torch.from_numpy(L.bias.view(np.int16)).view(torch.float16).to(dev)
    y = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
    for _ in range(calls):
        lb.linear(x, w, s, z, b, bits, group, out=y)
    torch.cuda.synchronize()
    print(json.dumps({"profile_layer": spec, "calls": calls, "path": lb.select_path(M, K, N, bits, group),
                      "wait_timeouts": lb.wait_timeouts()}))
    return 0


def run_profile_quantize(spec: str, calls: int):
    """Quantise the gate+up weight (bf16) `calls` times, nothing timed: a fixed
    workload for ncu captures.  spec = bits:group."""
    import torch
    import bit_groupwise_weight_gb300 as lb
    from bit_groupwise_weight_gb300 import build as lbuild
    lbuild.build()
    bits, group = (int(v) for v in spec.split(":"))
    K, N = synth.LLAMA_8B["gate_up"]
    w = torch.from_numpy(synth.f32_to_bf16_bits(synth.make_weights(0, N, K)).view(np.int16))
    w = w.view(torch.bfloat16).to("cuda:0")
    for _ in range(calls):
        lb.quantize_weights(w, bits, group)
    torch.cuda.synchronize()
    print(json.dumps({"profile_quantize": spec, "calls": calls}))
    return 0


def main():
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-qmm", action="store_true", help="skip the secondary M=128 qmm measurement")
    ap.add_argument("--no-int4wo", action="store_true",
                    help="skip the secondary int4wo-128 (b = 4, g = 128) configuration")
    ap.add_argument("--no-swiglu", action="store_true",
                    help="skip the secondary fused gate+up (silu * up) measurement")
    ap.add_argument("--no-quantize", action="store_true",
                    help="skip the secondary quantiser measurement")
    ap.add_argument("--profile-layer", default=None,
                    help="name:bits:M[:group] -- only call that layer (for ncu captures)")
    ap.add_argument("--profile-quantize", default=None,
                    help="bits:group -- only run the quantiser on the gate+up weight (for ncu captures)")
    ap.add_argument("--profile-calls", type=int, default=2)
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.profile_layer:
        return run_profile_layer(args.profile_layer, args.profile_calls)
    if args.profile_quantize:
        return run_profile_quantize(args.profile_quantize, args.profile_calls)
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
