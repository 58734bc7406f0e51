#!/usr/bin/env python
"""Throughput of the groupwise low-bit linear layer on one GB300 (or N replicas).

Workload (default): the Llama-3.1-8B decode linears at M = 1, group 64, bit
widths 1..7 -- (K, N) = (4096, 6144) qkv, (4096, 4096) o, (4096, 28672)
gate+up, (14336, 4096) down -- 28 layers.  One step is one call of every
layer: 28 launches of the decode kernel over ~0.86 GB of packed weights,
scales and zeros, more than the 129 MB L2, so every launch reads its weights
cold.

  value       algorithmic HBM bytes of a step / device time of a step, GB/s,
              with all inputs resident in HBM; the step is replayed from a
              CUDA graph of 28 C-ABI calls.
  roofline    the decode kernel inside the timed step: algorithmic bytes per
              launch / average launch time of the timed region (every launch
              of a step is that kernel), against the measured HBM copy peak.
  roofline_isolated  the same kernel called alone, L2 flushed before every
              call (CUDA graphs of flush + call minus flush alone), summed over
              the 28 layers: the cost of a call with nothing to overlap.
  layers      per layer and bit width: the in-stream time (calls of that layer
              back to back over rotating copies of its weights, together more
              than twice L2) with GB/s and roofline fraction, and the isolated
              time.
  e2e         the same metric with every input copied from pinned host memory
              and y copied back, through the public Python binding, per step
              (the step's inputs in one pinned arena, copied in four chunks that
              overlap the previous chunk's layers); host-to-device bandwidth
              bounds it.
  single_qmv  one K = N = 4096, b = 4, g = 64 call at M = 1.
  llama3_small_decode  the Llama-3.2-3B and -1B decode linears at M = 1,
              b in {2, 3, 4, 6}, g in {32, 64, 128, 256}, in-stream.
  small_batch the Llama-3.1-8B linears at b = 4, g = 128, M in {2..32}, bias
              on qkv: the dispatched call and both kernels forced, in-stream.
  qmm         the batched form: the same shapes at M in {128, 2048}, b in
              {4, 5}, g = 128, bias, 1% outlier columns in x, on the
              tensor-core kernel, TFLOP/s against the measured bf16 peak
              (qmm_m128 repeats the M = 128, b = 4 entry).
  quantize    the GPU quantiser on the gate+up weight (bf16, b = 4, g = 64).
  int4wo_128  b = 4, g = 128 on the same linears at M = 1 and M = 128, summed
              over the 8B model's 32 decoder layers.
  swiglu_gate_up  the fused gate+up call (silu(gate) * up) per bit width.
  cpu_baseline  the fp64 CPU oracle on a bounded sample of output rows of the
              step's layers, on all host cores (one thread per core, rows
              split between them); cpu_baseline_1thread on one core.

``--impl reference`` times the CPU oracle instead (the method's plain
definition; no GPU work).
"""
from __future__ import annotations

import argparse
import concurrent.futures
import hashlib
import json
import math
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
DTYPE = "bf16"      # x and y bf16, b-bit codes, fp16 scales/zeros; fp32 accumulation
L2_RULE = ("inputs larger than L2: a step streams ~0.86 GB of distinct weights; per-layer "
           "figures use rotating copies of the layer's weights totalling > 2.5 x L2, or an "
           "L2 flush before every call (isolated)")


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


def host_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


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
    """Host inputs for `rows_per_layer` output rows of every layer of the step,
    drawn from the step's distributions (x of the layer, uniform codes, the
    step's scale and zero recipe; the rows are a sample of the workload, not
    the GPU's exact rows), packed by the oracle.

    run(threads) splits every layer's rows into `threads` contiguous chunks and
    calls the oracle on each chunk from its own thread (the oracle is plain C
    called through ctypes, which releases the interpreter lock for the call,
    and keeps no state between calls); the arithmetic of every row is the
    oracle's, unchanged."""

    def __init__(self, rows_per_layer: int, seed: int = 0):
        import oracle
        self.o = oracle.Oracle()
        self.rows_per_layer = rows_per_layer
        self.items = []
        R = rows_per_layer
        for name, K, N, b in layer_list():
            key = (b, GROUP, N, R)
            x = synth.make_x(seed, 1, K, False, (b, GROUP))
            codes = synth.make_codes(seed, R, K, b, key)
            s, z = synth.make_scale_zero(seed, R, K // GROUP, (K,) + key)
            self.items.append(dict(K=K, b=b, x=x, packed=self.o.pack(codes, b), s=s, z=z,
                                   rows=np.arange(R), bytes=algorithmic_bytes(1, K, N, b, GROUP, rows=R)))
        self.bytes = sum(i["bytes"] for i in self.items)

    def _one(self, i, rows):
        self.o.linear_rows(i["x"], i["packed"], i["s"], i["z"], None, i["K"], i["b"], GROUP, rows,
                           N=i["packed"].shape[0])

    def run(self, threads: int = 1, pool=None):
        if threads <= 1 or pool is None:
            for i in self.items:
                self._one(i, i["rows"])
            return
        futs = [pool.submit(self._one, i, chunk) for i in self.items
                for chunk in np.array_split(i["rows"], threads) if chunk.size]
        for f in futs:
            f.result()


def time_oracle(sample: OracleSample, reps: int = 1, threads: int = 1, pool=None):
    t = time.perf_counter()
    for _ in range(reps):
        sample.run(threads, pool)
    dt = time.perf_counter() - t
    return sample.bytes * reps / dt / 1e9, dt


def cpu_baseline(seconds: float, threads: int):
    """The oracle on a bounded sample of the step's rows (32 rows of every layer
    per thread), on `threads` threads, repeated for about `seconds`."""
    rows = 32 * threads
    with concurrent.futures.ThreadPoolExecutor(max_workers=threads) as pool:
        sample = OracleSample(rows)
        _, dt1 = time_oracle(sample, 1, threads, pool)
        reps = max(1, round(seconds / max(dt1, 1e-6)))
        gbs, dt = time_oracle(sample, reps, threads, pool)
    return {"value": gbs, "unit": "GB/s", "cores": threads, "kind": "oracle",
            "sample": f"{rows} output rows of each of the 28 layers, {reps} passes "
                      f"(fp64 oracle, {threads} thread{'s' if threads > 1 else ''}, {dt:.1f} s)"}


# ---------------------------------------------------------------------------
# Arms.
# ---------------------------------------------------------------------------

def base_config(world: int = 1):
    """The step's configuration; both arms print the same dict."""
    return {"workload": WORKLOAD, "M": 1, "group": GROUP, "bits": list(BITS),
            "shapes_KN": {k: list(v) for k, v in synth.LLAMA_8B.items()},
            "layers_per_step": len(layer_list()), "bias": False, "l2": L2_RULE, "seed": 0,
            "parallelism": f"replicas{world}" if world > 1 else "single",
            "step_bytes": sum(algorithmic_bytes(1, K, N, b, GROUP) for _, K, N, b in layer_list())}


def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return 0
    threads = host_cores()
    rows = 32 * threads
    with concurrent.futures.ThreadPoolExecutor(max_workers=threads) as pool:
        sample = OracleSample(rows)
        for _ in range(args.warmup):
            sample.run(threads, pool)
        gbs, dt = time_oracle(sample, args.steps, threads, pool)
    ms = dt / args.steps * 1e3
    line = {
        "impl": "reference", "metric": METRIC, "value": gbs, "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": base_config(world),
        "cpu_baseline": {"value": gbs, "unit": "GB/s", "cores": threads, "kind": "oracle",
                         "sample": f"{rows} output rows of each of the 28 layers per step "
                                   f"(fp64 oracle, {threads} threads)"},
        "e2e": {"value": gbs, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


KERNEL_FILES = ("qmv_mma.cuh", "qmv_mma_host.cu", "ptx.cuh", "common.cuh")


def kernel_source_hash():
    """Hash of the decode kernel's sources (the profile summary records it)."""
    h = hashlib.sha256()
    csrc = ROOT / "bit_groupwise_weight_gb300" / "csrc"
    for p in sorted(csrc.glob("*")):
        if p.name in KERNEL_FILES or (p.name.startswith("qmv_mma_b") and p.suffix == ".cu"):
            h.update(p.name.encode())
            h.update(p.read_bytes())
    return h.hexdigest()[:16]


def profiled_traffic():
    """Per-launch DRAM bytes (read + write, averaged over the 28 launches of a step)
    of the decode kernel from the committed ncu summary, if that summary was taken
    on the current kernel source; else None."""
    p = ROOT / "profiles" / "qmv_mma_llama8b_decode.md"
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


class Gpu:
    """Device tensors and CUDA-graph timing on one stream."""

    def __init__(self, torch, lb, dev, stream):
        self.torch, self.lb, self.dev, self.stream = torch, lb, dev, stream
        self.l2 = torch.cuda.get_device_properties(dev).L2_cache_size
        self.flush = torch.empty(int(2 * self.l2), dtype=torch.uint8, device=dev)
        self._flush_us = None

    # -- inputs ------------------------------------------------------------------
    def bits16(self, a, dtype):
        return self.torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(dtype).to(self.dev)

    def pack(self, codes, bits):
        torch = self.torch
        d = torch.from_numpy(codes).to(self.dev)
        with torch.cuda.stream(self.stream):
            w = self.lb.pack_weights(d, bits)
        self.stream.synchronize()
        return w

    def layer(self, L, codes_packed=None):
        """Device tensors of a synth.Layer (weights packed by the library)."""
        torch = self.torch
        d = {"M": L.M, "K": L.K, "N": L.N, "bits": L.bits, "group": L.group,
             "x": self.bits16(L.x, torch.bfloat16),
             "s": self.bits16(L.scales, torch.float16), "z": self.bits16(L.zeros, torch.float16),
             "bias": None if L.bias is None else self.bits16(L.bias, torch.float16),
             "y": torch.empty((L.M, L.N), dtype=torch.bfloat16, device=self.dev)}
        if codes_packed is not None:
            d["w"] = codes_packed
        else:
            torch_codes = torch.from_numpy(L.codes).to(self.dev)
            with torch.cuda.stream(self.stream):
                d["w"] = self.lb.pack_weights(torch_codes, L.bits)
            self.stream.synchronize()
        return d

    def call(self, d, w, s, z, path=0):
        b = d["bias"]
        self.lb.linear_ptr(d["x"].data_ptr(), w.data_ptr(), s.data_ptr(), z.data_ptr(),
                           None if b is None else b.data_ptr(), d["y"].data_ptr(), d["M"], d["K"],
                           d["N"], d["bits"], d["group"], self.stream.cuda_stream, path)

    # -- timing ------------------------------------------------------------------
    def graph_us(self, fn, reps=5, stat=min):
        """Device time (us) of one replay of a CUDA graph that captures fn()."""
        torch = self.torch
        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(self.stream):
            fn()
            self.stream.synchronize()
            with torch.cuda.graph(g, stream=self.stream):
                fn()
        self.stream.synchronize()
        times = []
        for _ in range(reps):
            a = torch.cuda.Event(enable_timing=True)
            c = torch.cuda.Event(enable_timing=True)
            with torch.cuda.stream(self.stream):
                a.record(self.stream)
                g.replay()
                c.record(self.stream)
            self.stream.synchronize()
            times.append(a.elapsed_time(c) * 1e3)
        del g
        return stat(times)

    def in_stream_us(self, d, path=0, resident_bytes=None):
        """us per call with the calls back to back in one stream (each may overlap
        the previous one's tail, as inside a model step) over rotating copies of
        the weights, scales and zeros that together exceed 2.5 x L2, so every call
        reads its weights from HBM."""
        nb = resident_bytes or (d["w"].numel() + 2 * d["s"].numel() * 2)
        copies = max(2, math.ceil(2.5 * self.l2 / nb))
        sets = [(d["w"], d["s"], d["z"])] + [(d["w"].clone(), d["s"].clone(), d["z"].clone())
                                             for _ in range(copies - 1)]
        calls = max(copies, 16)

        def fn():
            for i in range(calls):
                w, s, z = sets[i % copies]
                self.call(d, w, s, z, path)
        us = self.graph_us(fn, reps=5, stat=statistics.median) / calls
        del sets
        return us

    def flushed_us(self, call_once, nrep=10):
        """us of call_once() with L2 flushed before it: CUDA graphs of nrep x
        (flush + call) minus nrep x flush alone (CUDA-event timestamps are too
        coarse to time a single short launch).  A difference at or below zero
        (possible under a profiler) counts as 10 ns."""
        if self._flush_us is None:
            self._flush_us = self.graph_us(lambda: [self.flush.fill_(i) for i in range(nrep)])

        def fn():
            for i in range(nrep):
                self.flush.fill_(i)
                call_once()
        return max(self.graph_us(fn) - self._flush_us, 1e-2) / nrep

    def isolated_us(self, d, path=0):
        return self.flushed_us(lambda: self.call(d, d["w"], d["s"], d["z"], path))


def hbm_entry(nbytes, us, peak):
    gbs = nbytes / us / 1e3
    return {"us": round(us, 3), "GBps": round(gbs, 1), "frac": round(gbs / peak, 4)}


def measure_single(G, peak):
    """One K = N = 4096, b = 4, g = 64 call at M = 1 (x ~ N(0,1), uniform codes,
    scale U[1e-3, 1e-2], zero = -scale U[6, 9], seed 0)."""
    c = synth.SINGLE_QMV
    L = synth.make_layer(0, c["M"], c["K"], c["N"], c["bits"], c["group"], c["bias"], c["outliers"])
    d = G.layer(L)
    nb = algorithmic_bytes(1, L.K, L.N, L.bits, L.group)
    out = {"K": L.K, "N": L.N, "M": 1, "bits": L.bits, "group": L.group, "bytes": nb}
    out |= hbm_entry(nb, G.in_stream_us(d), peak)
    iso = hbm_entry(nb, G.isolated_us(d), peak)
    out |= {"isolated_us": iso["us"], "isolated_GBps": iso["GBps"], "isolated_frac": iso["frac"]}
    out["timing"] = ("us: in-stream (back to back over rotating weight copies > 2.5 x L2); "
                     "isolated: L2 flushed before the call")
    return out


def measure_llama3_small(G, peak):
    """Llama-3.2-3B and -1B decode linears, M = 1, b in {2, 3, 4, 6}, g in {32..256}.
    The codes of a (shape, b) are shared by its four group sizes; scales, zeros and
    x are drawn per (b, g)."""
    rows = []
    for model, shapes in (("3B", synth.LLAMA_3B), ("1B", synth.LLAMA_1B)):
        for name, (K, N) in shapes.items():
            for b in (2, 3, 4, 6):
                codes = synth.make_codes(0, N, K, b, (3 if model == "3B" else 1, b))
                w = G.pack(codes, b)
                del codes
                for g in (32, 64, 128, 256):
                    s, z = synth.make_scale_zero(0, N, K // g, (K, b, g))
                    L = synth.Layer(M=1, K=K, N=N, bits=b, group=g, x=synth.make_x(0, 1, K, False, (b, g)),
                                    codes=None, scales=s, zeros=z, bias=None)
                    d = G.layer(L, codes_packed=w)
                    nb = algorithmic_bytes(1, K, N, b, g)
                    rows.append({"model": model, "layer": name, "K": K, "N": N, "bits": b, "group": g}
                                | hbm_entry(nb, G.in_stream_us(d), peak))
                    del d
                del w
    fr = [r["frac"] for r in rows]
    return {"M": 1, "layers": rows, "frac_min": min(fr), "frac_median": statistics.median(fr),
            "timing": "in-stream: back to back over rotating weight copies > 2.5 x L2"}


def measure_small_batch(G, peak):
    """Llama-3.1-8B linears, b = 4, g = 128, M in {2, 4, 8, 16, 32}, bias on qkv:
    the dispatched call (lowbit_linear) and each kernel forced."""
    lb = G.lb
    rows = []
    for name, (K, N) in synth.LLAMA_8B.items():
        codes = synth.make_codes(0, N, K, 4, (4, 128))
        w = G.pack(codes, 4)
        del codes
        s, z = synth.make_scale_zero(0, N, K // 128, (K, 4, 128))
        for M in (2, 4, 8, 16, 32):
            L = synth.Layer(M=M, K=K, N=N, bits=4, group=128, x=synth.make_x(0, M, K, False, (4, 128)),
                            codes=None, scales=s, zeros=z,
                            bias=synth.make_bias(0, N, (4, 128)) if name == "qkv" else None)
            d = G.layer(L, codes_packed=w)
            nb = algorithmic_bytes(M, K, N, 4, 128, bias=name == "qkv")
            path = {lb.PATH_QMV: "qmv", lb.PATH_QMM: "qmm"}[lb.select_path(M, K, N, 4, 128)]
            r = {"layer": name, "K": K, "N": N, "M": M, "path": path, "bytes": nb}
            r |= hbm_entry(nb, G.in_stream_us(d), peak)
            r["qmv_us"] = round(G.in_stream_us(d, lb.PATH_QMV), 3)
            r["qmm_us"] = round(G.in_stream_us(d, lb.PATH_QMM), 3)
            rows.append(r)
            del d
        del w
    return {"bits": 4, "group": 128, "layers": rows,
            "timing": "in-stream: back to back over rotating weight copies > 2.5 x L2; "
                      "us/GBps/frac are the dispatched call's"}


def measure_qmm(G, tc_peak, peak_kind, Ms=(128, 2048), bits_list=(4, 5), group=128):
    """The batched form on the tensor-core kernel: the Llama-3.1-8B shapes with bias
    and 1% outlier columns in x, TFLOP/s = 2 M N K / time."""
    lb = G.lb
    out = []
    for bits in bits_list:
        for name, (K, N) in synth.LLAMA_8B.items():
            codes = synth.make_codes(0, N, K, bits, (bits, group))
            w = G.pack(codes, bits)
            del codes
            s, z = synth.make_scale_zero(0, N, K // group, (K, bits, group))
            bias = synth.make_bias(0, N, (bits, group))
            for M in Ms:
                L = synth.Layer(M=M, K=K, N=N, bits=bits, group=group,
                                x=synth.make_x(0, M, K, True, (bits, group)), codes=None,
                                scales=s, zeros=z, bias=bias)
                d = G.layer(L, codes_packed=w)
                us = G.in_stream_us(d, lb.PATH_QMM)
                out.append({"M": M, "bits": bits, "layer": name, "K": K, "N": N, "us": round(us, 2),
                            "TFLOPs": round(2 * M * N * K / us / 1e6, 1)})
                del d
            del w
    res = {}
    for M in Ms:
        for bits in bits_list:
            sel = [o for o in out if o["M"] == M and o["bits"] == bits]
            flop = sum(2 * M * o["N"] * o["K"] for o in sel)
            us = sum(o["us"] for o in sel)
            tf = flop / us / 1e6
            res[f"M{M}_b{bits}"] = {
                "M": M, "bits": bits, "group": group, "TFLOPs": round(tf, 1),
                "roofline": {"bound": "tensor", "achieved": round(tf, 1), "peak": tc_peak,
                             "unit": "TFLOP/s", "frac": round(tf / tc_peak, 4),
                             "peak_kind": f"{peak_kind} bf16_tflops (burst)"},
                "layers": [{k: v for k, v in o.items() if k not in ("M", "bits")} for o in sel]}
    res["timing"] = "in-stream: back to back over rotating weight copies > 2.5 x L2"
    return res


def measure_quantize(G, hbm_peak, peak_kind, bits=4, group=64, reps=5):
    """The quantiser on the largest Llama-3.1-8B weight (gate+up, K=4096, N=28672) in bf16:
    235 MB read per call, more than L2, so back-to-back calls stream from HBM.
    GB/s = (weights read + packed codes, scales and zeros written) / time."""
    torch, lb = G.torch, G.lb
    K, N = synth.LLAMA_8B["gate_up"]
    w = G.bits16(synth.f32_to_bf16_bits(synth.make_weights(0, N, K)), torch.bfloat16)
    packed = torch.empty((N, K * bits // 8), dtype=torch.uint8, device=G.dev)
    sc = torch.empty((N, K // group), dtype=torch.float16, device=G.dev)
    ze = torch.empty((N, K // group), dtype=torch.float16, device=G.dev)

    def fn():
        for _ in range(reps):
            lb.quantize_weights(w, bits, group, packed, sc, ze)
    us = G.graph_us(fn) / reps
    nbytes = N * K * 2 + N * K * bits // 8 + 4 * N * (K // group)
    gbs = nbytes / us / 1e3
    return {"layer": "gate_up", "K": K, "N": N, "bits": bits, "group": group, "w_dtype": "bf16",
            "us": round(us, 2), "bytes": nbytes,
            "roofline": {"bound": "hbm", "achieved": round(gbs, 1), "peak": hbm_peak,
                         "unit": "GB/s", "frac": round(gbs / hbm_peak, 4),
                         "peak_kind": f"{peak_kind} hbm_gbs (copy)"},
            "timing": f"CUDA graph of {reps} calls; 235 MB of weights per call (> L2)"}


def measure_e2e(torch, lb, dev, stream, layers, steps, dist, world, step_bytes):
    """Host buffers through the public API.  A step's inputs live in one pinned
    host arena (each tensor 256-byte aligned) and are copied in E2E_CHUNKS large
    copies on a copy stream; the layers of chunk c run on the compute stream as
    soon as chunk c has landed, while chunk c + 1 is still in flight.  The
    outputs land in one device arena and come back in one copy.  Timed from the
    first copy to the end of the last."""
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
    torch.cuda.synchronize(dev)
    dist.barrier()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    landed = [torch.cuda.Event() for _ in range(E2E_CHUNKS)]
    with torch.cuda.stream(stream):
        e0.record(stream)
        for _ in range(steps):
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
    e2e_ms = dist.max(e0.elapsed_time(e1)) / steps
    # The arena round trip must reproduce the device-resident results.
    for i, t in enumerate(layers):
        ref = lb.linear(t["x"], t["w"], t["s"], t["z"], None, t["b"], GROUP)
        assert torch.equal(y_views[i], ref), f"e2e output of layer {i} differs"
    return {"value": world * step_bytes / (e2e_ms / 1e3) / 1e9, "unit": "GB/s",
            "h2d_bytes_per_step": size, "d2h_bytes_per_step": y_host.numel() * 2}


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
    hbm_peak, tc_peak, peak_kind = measured_peaks()

    # --- inputs: device copies of every layer of the step -----------------------
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

    try:
        bus = torch.cuda.get_device_properties(dev).pci_bus_id
    except AttributeError:
        bus = None

    with torch.cuda.stream(stream):
        for _ in range(max(args.warmup, 3)):
            graph.replay()
    stream.synchronize()

    # --- the timed region ----------------------------------------------------------
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
    ms_rank = ev0.elapsed_time(ev1)
    ms_total = dist.max(ms_rank)
    ms_per_step = ms_total / args.steps
    value = whole_job_gbs(world, step_bytes, args.steps, ms_total)
    # In-step roofline of the decode kernel: every launch in the timed region is
    # one, so its average launch time is this rank's step time / 28.
    n_launch = len(layers)
    avg_launch_us = ms_rank / args.steps * 1e3 / n_launch
    achieved = step_bytes / n_launch / avg_launch_us / 1e3

    G = Gpu(torch, lb, dev, stream)

    # --- per layer: in-stream and isolated ---------------------------------------
    per_layer = []
    for t in layers:
        d = {"M": 1, "K": t["K"], "N": t["N"], "bits": t["b"], "group": GROUP, "x": t["x"],
             "w": t["w"], "s": t["s"], "z": t["z"], "bias": None, "y": t["y"]}
        r = {"layer": t["name"], "bits": t["b"], "K": t["K"], "N": t["N"], "bytes": t["bytes"]}
        r |= hbm_entry(t["bytes"], G.in_stream_us(d), hbm_peak)
        iso = G.isolated_us(d)
        r |= {"isolated_us": round(iso, 3), "_iso": iso}
        per_layer.append(r)
    iso_sum = sum(p.pop("_iso") for p in per_layer)
    iso_gbs = step_bytes / iso_sum / 1e3

    # --- the fused gate+up call (silu(gate) * up) on the same gate+up weights ----
    swiglu = []
    if not args.no_swiglu:
        for t in layers:
            if t["name"] != "gate_up":
                continue
            F = t["N"] // 2
            h = torch.empty((1, F), dtype=torch.bfloat16, device=dev)

            def glu(t=t, h=h, F=F):
                lb.linear_swiglu_ptr(t["x"].data_ptr(), t["w"].data_ptr(), t["s"].data_ptr(),
                                     t["z"].data_ptr(), None, h.data_ptr(), 1, t["K"], F, t["b"],
                                     GROUP, stream.cuda_stream)
            us = G.flushed_us(glu)
            plain = next(p for p in per_layer if p["layer"] == "gate_up" and p["bits"] == t["b"])
            nbytes = algorithmic_bytes(1, t["K"], t["N"], t["b"], GROUP) - 2 * F   # y holds F outputs
            swiglu.append({"bits": t["b"], "K": t["K"], "F": F, "us": round(us, 3),
                           "plain_linear_us": plain["isolated_us"], "GBps": round(nbytes / us / 1e3, 1)})

    # --- the int4wo-128 configuration (b = 4, g = 128) at M = 1 ------------------
    int4_m1 = []
    if not args.no_int4wo:
        for t in layers:
            if t["b"] != 4:
                continue
            sc, zc = synth.make_scale_zero(0, t["N"], t["K"] // 128, (t["K"], 4, 128))
            d = {"M": 1, "K": t["K"], "N": t["N"], "bits": 4, "group": 128, "x": t["x"], "w": t["w"],
                 "s": G.bits16(sc, torch.float16), "z": G.bits16(zc, torch.float16), "bias": None,
                 "y": t["y"]}
            nbytes = algorithmic_bytes(1, t["K"], t["N"], 4, 128)
            int4_m1.append({"layer": t["name"], "K": t["K"], "N": t["N"]}
                           | hbm_entry(nbytes, G.in_stream_us(d), hbm_peak))

    single = None if args.no_configs else measure_single(G, hbm_peak)
    small3 = None if args.no_configs else measure_llama3_small(G, hbm_peak)
    batch = None if args.no_configs else measure_small_batch(G, hbm_peak)
    qmm = None if args.no_qmm else measure_qmm(G, tc_peak, peak_kind,
                                               Ms=(128,) if args.no_configs else (128, 2048))
    quant = None if args.no_quantize else measure_quantize(G, hbm_peak, peak_kind)
    del G

    e2e = measure_e2e(torch, lb, dev, stream, layers, max(1, min(args.steps, 10)), dist, world,
                      step_bytes)

    int4wo = None
    if int4_m1:
        # The 8B model has 32 decoder layers of these four linears.
        stack1 = 32 * sum(r["us"] for r in int4_m1)
        int4wo = {"bits": 4, "group": 128, "M1": {"layers": int4_m1, "stack_us": round(stack1, 1),
                                                  "linear_tokens_per_s": round(1e6 / stack1, 1),
                                                  "timing": "in-stream, rotating weight copies"}}
        if qmm is not None:
            q = qmm["M128_b4"]["layers"]
            stack128 = 32 * sum(r["us"] for r in q)
            int4wo["M128"] = {"layers": q, "stack_us": round(stack128, 1),
                              "linear_tokens_per_s": round(128 * 1e6 / stack128, 1),
                              "timing": qmm["timing"]}
        int4wo["what"] = ("the int4wo-128 configuration (4-bit codes, groups of 128) on the Llama-3.1-8B "
                          "linears; stack_us = 32 decoder layers x (qkv + o + gate_up + down), the linear "
                          "layers' share of one decode step (no attention, norms, embeddings or lm_head)")

    line = {
        "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": DTYPE, "data": "synthetic",
        "config": base_config(world),
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": hbm_peak, "unit": "GB/s",
                     "frac": achieved / hbm_peak, "traffic": profiled_traffic(),
                     "kernel": "qmv_mma_kernel (every launch of the step)",
                     "launches_per_step": n_launch,
                     "algorithmic_bytes_per_launch": step_bytes / n_launch,
                     "avg_launch_us": avg_launch_us,
                     "measured": "CUDA events on the launching stream around the timed region",
                     "peak_kind": f"{peak_kind} hbm_gbs (copy)"},
        "roofline_isolated": {"bound": "hbm", "achieved": iso_gbs, "peak": hbm_peak, "unit": "GB/s",
                              "frac": iso_gbs / hbm_peak, "sum_us": round(iso_sum, 2),
                              "what": "the 28 layers called one at a time, L2 flushed before each "
                                      "call, nothing to overlap with"},
        "e2e": e2e,
        "gpu_launches": n_launch * args.steps,
        "clocks": clk,
        "layers": per_layer,
    }
    if single is not None:
        line["single_qmv"] = single
    if small3 is not None:
        line["llama3_small_decode"] = small3
    if batch is not None:
        line["small_batch"] = batch
    if qmm is not None:
        line["qmm"] = qmm
        line["qmm_m128"] = qmm["M128_b4"]
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
        line["cpu_baseline"] = cpu_baseline(args.cpu_seconds, host_cores())
        line["cpu_baseline_1thread"] = cpu_baseline(args.cpu_seconds, 1)
    if rank == 0:
        print(json.dumps(line), flush=True)
    dist.close()
    return 0


def run_profile_layer(spec: str, calls: int):
    """Call one layer `calls` times through lowbit_linear, nothing timed: a small, fixed
    workload for ncu captures.  spec = name:bits:M[:group], name one of qkv/o/gate_up/down
    or a Llama-3.2 shape as 3b_<name> / 1b_<name>."""
    import torch
    import bit_groupwise_weight_gb300 as lb
    from bit_groupwise_weight_gb300 import build as lbuild
    lbuild.build()
    parts = spec.split(":")
    name, bits, M = parts[0], int(parts[1]), int(parts[2])
    group = int(parts[3]) if len(parts) > 3 else (64 if M <= 2 else 128)
    table = synth.LLAMA_8B
    if name.startswith("3b_"):
        table, name = synth.LLAMA_3B, name[3:]
    elif name.startswith("1b_"):
        table, name = synth.LLAMA_1B, name[3:]
    K, N = table[name]
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
    ap.add_argument("--no-configs", action="store_true",
                    help="skip the single-call, Llama-3.2, small-batch and M = 2048 measurements")
    ap.add_argument("--no-qmm", action="store_true", help="skip the batched (qmm) measurements")
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
