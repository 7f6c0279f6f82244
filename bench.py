#!/usr/bin/env python3
"""Benchmark of the fused low-bit dequantize-and-multiply on GB300.

Default workload: one Llama-7B-shaped decoder layer at decode (M = 1 token),
2-bit Lloyd-Max G=32 weights with 3.5% binary16 anchor columns — the seven
projections (q, k, v, o: 4096x4096; gate, up: 11008x4096; down: 4096x11008)
run as ONE grouped GEMV launch per step.  Eight distinct layer copies (720 MB)
rotate, so every step streams its weights from HBM, not L2.

metric: weight GB/s = algorithmic bytes (codes + scales + offsets + anchor
weights + anchor indices + x + y) / time; `roofline.frac` against the measured
HBM copy bandwidth; equivalent tok/s of a 32-layer stack.

Second figure (`gemm`): prefill of a 14B-shaped layer (q/k/v/o 5120x5120,
gate/up 13824x5120, down 5120x13824) at M = 2048 bf16 tokens, the seven
projections in one lq_gemm_grouped launch, for 2-bit G=32 + anchors and for
NF4 block 64; TFLOP/s =
2*M*N*K summed over the layer / step time, against the measured dense bf16
peak.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl lq|reference]

Under torchrun each rank runs its own replica (the layer needs no exchange);
the slowest rank's time sets the aggregate.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import synth  # noqa: E402

METRIC = "dequant-GEMV weight GB/s (% of GB300 HBM peak); dequant-GEMM TFLOP/s"
WORKLOAD = "llama-7b decoder layer, decode M=1, 2-bit Lloyd-Max G=32 + 3.5% fp16 anchors, 7 projections per launch"
ROTATE = 8          # distinct layer copies in HBM (8 x 90 MB > 129 MB L2)
STACK_LAYERS = 32   # layers of the 7B stack for the tok/s equivalent


def max_over_ranks(value: float, dist, device) -> float:
    """The slowest rank's time: every rank's replica must have finished for the job to be done."""
    import torch
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def _traffic(key):
    """DRAM bytes per launch from the committed ncu summary (profiles/traffic.json)."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        return json.load(f).get(key)


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), float(d.get("bf16_tflops_sustained", d["bf16_tflops"])), "measured"
    return 6800.0, 1900.0, 1700.0, "fallback"


def layer_packs(M: int, copy: int):
    """Host-side packed 2-bit weights and x for one layer copy."""
    from math import floor
    out = []
    for i, (name, N, K) in enumerate(synth.LAYER_SHAPES["7b"]):
        A = int(floor(0.035 * K))
        pk = synth.random_packed_2bit(N, K, A, sigma=0.02, seed=100 + copy, cfg=2, matrix_id=i)
        outl = synth.outlier_channels(K, 0.01, seed=100 + copy, cfg=2)
        xb = synth.activations(M, K, "f16", synth.channel_sigma(K, outl, 20.0), seed=100 + copy, cfg=2, matrix_id=i)
        out.append((name, pk, xb))
    return out


def algorithmic_bytes(packs, M: int) -> int:
    total = 0
    for _, pk, _ in packs:
        N, K, A = pk["N"], pk["K"], pk["A"]
        total += N * K // 4 + 2 * 2 * N * (K // 32) + 2 * N * A + 4 * A + 2 * M * K + 4 * M * N
    return total


class ClockSampler:
    """nvidia-smi SM clock and throttle-reason samples while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.dev = device_index
        self.proc = None
        self.lines: list[str] = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.dev), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self._t = threading.Thread(target=self._read, daemon=True)
            self._t.start()
        except (FileNotFoundError, OSError):
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for nm, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(nm)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


def host_cores() -> int:
    return len(os.sched_getaffinity(0))


def cpu_baseline(packs, seconds: float = 12.0, threads: int = 1):
    """The oracle as it stands (plain C) on a bounded sample of rows: `threads` host threads,
    each computing its own rows of every projection (the oracle's C call releases the
    interpreter lock, so the threads run on separate cores).  Returns (GB/s, sample)."""
    from concurrent.futures import ThreadPoolExecutor
    from oracle import oracle as O
    O.build()
    rows_per = 4

    def worker(tid):
        done_bytes, rows_done = 0, 0
        t0 = time.perf_counter()
        while time.perf_counter() - t0 < seconds:
            for i, (_, pk, xb) in enumerate(packs):
                n0 = ((rows_done * threads + tid) * 37 + i * 101) % (pk["N"] - rows_per)
                O.gemv_2bit_rows(pk, xb, "f16", n0, n0 + rows_per)
                K, A = pk["K"], pk["A"]
                done_bytes += rows_per * (K // 4 + 4 * (K // 32) + 2 * A)
            rows_done += rows_per
        return done_bytes, rows_done

    t0 = time.perf_counter()
    with ThreadPoolExecutor(max_workers=threads) as ex:
        res = list(ex.map(worker, range(threads)))
    wall = time.perf_counter() - t0
    done_bytes = sum(r[0] for r in res)
    rows_done = sum(r[1] for r in res)
    return done_bytes / wall / 1e9, (f"{rows_done} rows of each of the 7 projections on {threads} host thread(s), "
                                     f"{seconds:.0f} s (oracle fmaf dequant + fp64 dot), weight bytes only")


def run_reference(args):
    """The oracle on the host cores, same metric and workload, bounded sample per step."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    packs = layer_packs(1, 0)
    from oracle import oracle as O
    O.build()
    per_step = max(1.0, 60.0 / max(1, args.steps + args.warmup))
    cores = host_cores()
    vals = []
    for s in range(args.warmup + args.steps):
        gbs, sample = cpu_baseline(packs, seconds=min(per_step, 8.0), threads=cores)
        if s >= args.warmup:
            vals.append(gbs)
    v = statistics.median(vals)
    layer_bytes = algorithmic_bytes(packs, 1)
    line = {"impl": "reference", "metric": METRIC, "value": round(v, 4), "unit": "GB/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(layer_bytes / (v * 1e9) * 1e3, 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": WORKLOAD, "sample": sample},
            "cpu_baseline": {"value": round(v, 4), "unit": "GB/s", "cores": cores, "kind": "oracle", "sample": sample},
            "e2e": {"value": round(v, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


SINGLE_LINEAR_SETS = 32768   # distinct 512x256 weight sets of the single-linear workload (1.9 GB, far beyond L2)


def single_linear_batched(lq, torch, h, device: str, steps: int, warmup: int):
    """The 512x256 single linear (2-bit, A = 8) over SINGLE_LINEAR_SETS distinct weight sets in one launch."""
    L, N, K, A = SINGLE_LINEAR_SETS, 512, 256, 8
    big = synth.random_packed_2bit_sets(L, N, K, A, seed=1, cfg=1)
    w = lq.QuantWeights.from_host(big, lq.FMT_2BIT, device=device)
    del big
    x = torch.from_numpy(synth.activations(L, K, "f16", seed=1, cfg=1)).view(torch.float16).to(device).view(L, 1, K)
    y = torch.empty((L, 1, N), dtype=torch.float32, device=device)
    ld = 8
    strides = dict(codes=N * K // 4, scales=N * K // 32 * 2, offsets=N * K // 32 * 2, anchor_idx=4 * A,
                   anchor_w=N * ld * 2, x=K * 2, y=N * 4)
    prob = [h.problem(w, x[0], y[0], batch=L, strides=strides)]
    per_set = N * K // 4 + 2 * 2 * N * (K // 32) + 2 * N * A + 4 * A + 2 * K + 4 * N
    stream = torch.cuda.current_stream()
    for _ in range(warmup):
        h.gemv_grouped(prob, stream=stream)
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(steps):
        h.gemv_grouped(prob, stream=stream)
    e1.record(stream)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / steps
    # one weight set per call: the latency of a single small call, launches back to back
    one = synth.random_packed_2bit(N, K, A, seed=1, cfg=1)
    w1 = lq.QuantWeights.from_host(one, lq.FMT_2BIT, device=device)
    x1 = x[0].clone()
    y1 = torch.empty((1, N), dtype=torch.float32, device=device)
    for _ in range(warmup):
        h.gemv(w1, x1, y1, stream=stream)
    torch.cuda.synchronize()
    calls = 200
    e0.record(stream)
    for _ in range(calls):
        h.gemv(w1, x1, y1, stream=stream)
    e1.record(stream)
    torch.cuda.synchronize()
    single_us = e0.elapsed_time(e1) / calls * 1e3
    return {"workload": f"512x256 single linear, 2-bit G=32 + 8 fp16 anchors, M=1, {L} distinct weight sets in one launch",
            "value": round(L * per_set / (ms * 1e-3) / 1e9, 1), "unit": "GB/s", "ms_per_launch": round(ms, 4),
            "bytes_per_launch": L * per_set, "single_call_us": round(single_us, 2),
            # DRAM bytes of the same kernel over 4096 sets (ncu), scaled to this launch's sets
            "traffic": (lambda t: None if t is None else int(t * L // 4096))(_traffic("gemv_ring_512x256_4096_sets_bytes_per_launch"))}


GEMM_M = 2048
GEMM_WORKLOAD = "14b decoder layer prefill, M=2048 bf16 tokens, 7 projections in one lq_gemm_grouped launch"


def gemm_layer(lq, torch, h, fmt: str, device: str, steps: int, warmup: int):
    """Time the 14B-layer prefill: returns (TFLOP/s, ms per layer, mean ms of the largest projection's launch)."""
    from math import floor
    mats, flops = [], 0
    for i, (name, N, K) in enumerate(synth.LAYER_SHAPES["14b"]):
        if fmt == "2bit":
            pk = synth.random_packed_2bit(N, K, int(floor(0.035 * K)), sigma=0.02, seed=500, cfg=5, matrix_id=i)
            w = lq.QuantWeights.from_host(pk, lq.FMT_2BIT, device=device)
        elif fmt == "int4":
            pk = synth.random_packed_int4(N, K, int(floor(0.01 * K)), sigma=0.02, seed=500, cfg=5, matrix_id=i)
            w = lq.QuantWeights.from_host(pk, lq.FMT_INT4, device=device)
        elif fmt == "nf4_dq":
            pk = synth.random_packed_nf4_dq(N, K, sigma=0.02, seed=500, cfg=5, matrix_id=i)
            w = lq.QuantWeights.from_host(pk, lq.FMT_NF4_DQ, device=device)
        else:
            pk = synth.random_packed_nf4(N, K, sigma=0.02, seed=500, cfg=5, matrix_id=i)
            w = lq.QuantWeights.from_host(pk, lq.FMT_NF4, device=device)
        outl = synth.outlier_channels(K, 0.01, seed=500, cfg=5)
        xb = synth.activations(GEMM_M, K, "bf16", synth.channel_sigma(K, outl, 20.0), seed=500, cfg=5, matrix_id=i)
        x = torch.from_numpy(xb).view(torch.bfloat16).to(device)
        y = torch.empty((GEMM_M, N), dtype=torch.bfloat16, device=device)
        mats.append((name, w, x, y))
        flops += 2 * GEMM_M * N * K
    stream = torch.cuda.current_stream()
    probs = [h.problem(w, x, y) for _, w, x, y in mats]

    def step():
        h.gemm_grouped(probs, stream=stream)

    for _ in range(warmup):
        step()
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    with ClockSampler(torch.cuda.current_device()) as clk:
        time.sleep(0.2)
        e0.record(stream)
        for _ in range(steps):
            step()
        e1.record(stream)
        torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / steps
    # the largest projection alone, for the kernel roofline
    name, w, x, y = max(mats, key=lambda m: m[1].N * m[1].K)
    a0 = torch.cuda.Event(enable_timing=True)
    a1 = torch.cuda.Event(enable_timing=True)
    reps = 10
    a0.record(stream)
    for _ in range(reps):
        h.gemm(w, x, y, stream=stream)
    a1.record(stream)
    torch.cuda.synchronize()
    one_ms = a0.elapsed_time(a1) / reps
    one_flops = 2 * GEMM_M * w.N * w.K
    # 2-bit: bitmap memset + anchor gather + GEMM; INT4: + one x permutation per projection;
    # NF4-DQ: one block-maximum decode per projection + GEMM
    launches = {"2bit": 3, "nf4": 1, "int4": 3 + len(mats), "nf4_dq": 1 + len(mats)}[fmt]
    return {"fmt": fmt, "value": round(flops / (ms * 1e-3) / 1e12, 1), "unit": "TFLOP/s", "ms_per_layer": round(ms, 4),
            "largest": {"name": name, "N": w.N, "K": w.K, "ms": round(one_ms, 4),
                        "tflops": round(one_flops / (one_ms * 1e-3) / 1e12, 1)},
            "launches_per_layer": launches, "clocks": clk.summary()}


QUANT_WORKLOAD = "7b decoder layer (q,k,v,o 4096x4096; gate,up 11008x4096; down 4096x11008), fp32 weights on the device"


def quantizer_layer(lq, torch, h, device: str, reps: int = 3):
    """Time the GPU quantizers over one 7B layer: anchors + 2-bit G=32, and NF4 block 64."""
    from math import floor
    g = torch.Generator(device=device)
    g.manual_seed(77)
    mats = []
    for i, (name, N, K) in enumerate(synth.LAYER_SHAPES["7b"]):
        W = torch.randn((N, K), generator=g, device=device, dtype=torch.float32) * 0.02
        outl = synth.outlier_channels(K, 0.01, seed=77, cfg=2)
        prof = torch.from_numpy(np.sqrt(2.0 / np.pi) * synth.channel_sigma(K, outl, 20.0)).to(device)
        mats.append((W, prof))
    weights = sum(W.numel() for W, _ in mats)
    stream = torch.cuda.current_stream()

    def two_bit():
        for W, prof in mats:
            h.quantize_2bit(W, h.select_anchors(W, profile=prof, stream=stream), stream=stream)

    def nf4():
        for W, _ in mats:
            h.quantize_nf4(W, stream=stream)

    out = {}
    for name, fn in (("2bit", two_bit), ("nf4", nf4)):
        fn()
        torch.cuda.synchronize()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(reps):
            fn()
        e1.record(stream)
        torch.cuda.synchronize()
        ms = e0.elapsed_time(e1) / reps
        out[name] = {"ms_per_layer": round(ms, 3), "gweights_per_s": round(weights / (ms * 1e-3) / 1e9, 2),
                     "fp32_read_gb_s": round(4 * weights / (ms * 1e-3) / 1e9, 1)}
    # the oracle's quantizer on a row sample of the gate projection, for scale
    from oracle import oracle as O
    N, K = 256, 4096
    Wh = synth.weights(N, K, 0.02, seed=77, cfg=2)
    ai = O.select_anchors(Wh, np.ones(K))
    t0 = time.perf_counter()
    O.quantize_2bit(Wh, ai)
    cpu_s = time.perf_counter() - t0
    out["cpu_baseline"] = {"value": round(N * K / cpu_s / 1e9, 4), "unit": "Gweights/s", "cores": 1, "kind": "oracle",
                           "sample": f"oracle 2-bit quantizer on {N}x{K} (anchors given)"}
    out.update({"workload": QUANT_WORKLOAD, "weights_per_layer": weights,
                "bound": "fp64 arithmetic (every decision in fp64 to match the oracle bit for bit)"})
    return out


STREAM_LAYERS = 32


def device_layer(lq, torch, shapes, fmt, g, device, sigma=0.02):
    """One layer of random packed weights made on the device (throughput runs; the contents do not
    change the kernels' work): uniform random codes, scales and offsets of the synthetic
    magnitudes, sorted random anchor columns (2-bit), absmax (NF4), scales, a random
    column permutation and 1 % anchor columns (INT4), or 8-bit float maxima and their
    second-level constants (NF4 with double quantization)."""
    from math import floor
    ws = []
    for name, N, K in shapes:
        if fmt == lq.FMT_2BIT:
            A = int(floor(0.035 * K))
            ld = max(8, (A + 7) // 8 * 8)
            codes = torch.randint(0, 256, (N, K // 4), generator=g, device=device, dtype=torch.uint8)
            scales = (torch.rand((N, K // 32), generator=g, device=device) * sigma + 0.5 * sigma).half()
            offsets = (torch.randn((N, K // 32), generator=g, device=device) * 0.1 * sigma).half()
            aidx = torch.randperm(K, generator=g, device=device)[:A].sort().values.to(torch.int32).contiguous()
            aw = (torch.randn((N, ld), generator=g, device=device) * sigma).half()
            ws.append(lq.QuantWeights(lq.FMT_2BIT, N, K, codes, scales, offsets, aidx, aw, A, ld))
        elif fmt == lq.FMT_INT4:
            A = int(floor(0.01 * K))
            ld = max(8, (A + 7) // 8 * 8)
            codes = torch.randint(0, 256, (N, K // 2), generator=g, device=device, dtype=torch.uint8)
            scales = (torch.rand((N, K // 32), generator=g, device=device) * 0.25 * sigma + 0.125 * sigma).half()
            perm = torch.randperm(K, generator=g, device=device).to(torch.int32).contiguous()
            aidx = torch.randperm(K, generator=g, device=device)[:A].sort().values.to(torch.int32).contiguous()
            aw = (torch.randn((N, ld), generator=g, device=device) * sigma).half()
            ws.append(lq.QuantWeights(lq.FMT_INT4, N, K, codes, scales, perm, aidx, aw, A, ld))
        elif fmt == lq.FMT_NF4_DQ:
            codes = torch.randint(0, 256, (N, K // 2), generator=g, device=device, dtype=torch.uint8)
            acodes = torch.randint(0, 0x7F, (N, K // 64), generator=g, device=device, dtype=torch.uint8)
            nb = (N * (K // 64) + 255) // 256
            second = torch.rand((1 + nb,), generator=g, device=device) * sigma / 448.0
            second[0] = 3 * sigma
            ws.append(lq.QuantWeights(lq.FMT_NF4_DQ, N, K, codes, acodes, second))
        else:
            codes = torch.randint(0, 256, (N, K // 2), generator=g, device=device, dtype=torch.uint8)
            absmax = torch.rand((N, K // 64), generator=g, device=device) * 2 * sigma + sigma
            ws.append(lq.QuantWeights(lq.FMT_NF4, N, K, codes, absmax))
    return ws


def layer_weight_bytes(ws, M: int) -> int:
    total = 0
    for w in ws:
        N, K = w.N, w.K
        if w.format == 1:
            total += N * K // 4 + 2 * 2 * N * (K // 32) + 2 * N * w.A + 4 * w.A
        elif w.format == 3:   # INT4: codes, binary16 scales, anchors, the permutation
            total += N * K // 2 + 2 * N * (K // 32) + 2 * N * w.A + 4 * w.A + 4 * K
        elif w.format == 4:   # NF4 with double quantization: codes, 8-bit maxima, second level
            total += N * K // 2 + N * (K // 64) + 4 * (1 + (N * (K // 64) + 255) // 256)
        else:
            total += N * K // 2 + 4 * N * (K // 64)
        total += 2 * M * K + 4 * M * N
    return total


def decode_workloads(lq, torch, h, device: str, reps: int = 5):
    """Decode throughput of the other listed decode workloads: the 7B layer in NF4 (8 rotating
    copies, bf16 x, M = 1, 4, 16), the same layer in the INT4 format (fp16 x) and in NF4 with
    double quantization (bf16 x), and an 80-layer 70B stack resident in HBM (2-bit + anchors,
    fp16 x, M = 1, 8, 32), one grouped call per layer, one pass captured in a CUDA graph."""
    g = torch.Generator(device=device)
    g.manual_seed(303)
    out = {}
    stream = torch.cuda.current_stream()
    for key, shapes, fmt, layers, Ms, xdt in (
            ("nf4_7b_layer", synth.LAYER_SHAPES["7b"], lq.FMT_NF4, ROTATE, (1, 4, 16), torch.bfloat16),
            ("int4_7b_layer", synth.LAYER_SHAPES["7b"], lq.FMT_INT4, ROTATE, (1, 4, 16), torch.float16),
            ("nf4_dq_7b_layer", synth.LAYER_SHAPES["7b"], lq.FMT_NF4_DQ, ROTATE, (1, 4, 16), torch.bfloat16),
            ("llama70b_80_layer_stack", synth.LAYER_SHAPES["70b"], lq.FMT_2BIT, 80, (1, 8, 32), torch.float16)):
        stack = [device_layer(lq, torch, shapes, fmt, g, device, 0.015 if "70b" in key else 0.02) for _ in range(layers)]
        res = {}
        for M in Ms:
            xs = [torch.randn((M, w.K), generator=g, device=device).to(xdt) for w in stack[0]]
            ys = [torch.empty((M, w.N), dtype=torch.float32, device=device) for w in stack[0]]
            probs = [[h.problem(w, x, y) for w, x, y in zip(ws, xs, ys)] for ws in stack]
            for p in probs[:3]:
                h.gemv_grouped(p, stream=stream)
            torch.cuda.synchronize()
            # one pass over the layers captured in a CUDA graph and replayed, as the headline step is
            g_stream = torch.cuda.Stream()
            g_stream.wait_stream(stream)
            cg = torch.cuda.CUDAGraph()
            with torch.cuda.graph(cg, stream=g_stream):
                for p in probs:
                    h.gemv_grouped(p, stream=g_stream)
            cg.replay()
            torch.cuda.synchronize()
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record()
            for _ in range(reps):
                cg.replay()
            e1.record()
            torch.cuda.synchronize()
            ms = e0.elapsed_time(e1) / (reps * layers)
            del cg
            lb = layer_weight_bytes(stack[0], M)
            res[f"M={M}"] = {"us_per_layer": round(ms * 1e3, 1), "gb_s": round(lb / (ms * 1e-3) / 1e9, 1),
                             "tok_s_stack": round(M * 1e3 / (ms * layers), 1) if layers == 80 else None}
        res["layer_bytes_m1"] = layer_weight_bytes(stack[0], 1)
        res["layers"] = layers
        out[key] = res
        del stack
        torch.cuda.empty_cache()
    h.sync()
    return out


def stream_stack(lq, torch, h, device: str, M: int = 1, reps: int = 3):
    """A 32-layer 7B stack held in pinned host memory, streamed through two device slots
    (lq_stream_run): tokens/s of one decode pass, the host-to-device rate it reached, and
    the plain copy rate of the same bytes for comparison."""
    distinct = 4
    blobs, xs = [], None
    for c in range(distinct):
        packs = layer_packs(M, 100 + c)
        blob, meta = lq.pack_layer([pk for _, pk, _ in packs], lq.FMT_2BIT)
        blobs.append((blob, meta))
        if xs is None:
            xs = [torch.from_numpy(xb).view(torch.float16).to(device) for _, _, xb in packs]
            ys = [torch.empty((M, pk["N"]), dtype=torch.float32, device=device) for _, pk, _ in packs]
    layer_bytes = max(b.nbytes for b, _ in blobs)
    stride = (layer_bytes + 4095) // 4096 * 4096
    host = torch.empty(STREAM_LAYERS * stride, dtype=torch.uint8).pin_memory()
    hv = host.numpy()
    for l in range(STREAM_LAYERS):
        b = blobs[l % distinct][0]
        hv[l * stride:l * stride + b.nbytes] = b
    ls = lq.LayerStream(h, stride)
    meta = blobs[0][1]
    probs = [ls.problem(meta[i], lq.FMT_2BIT, xs[i], ys[i]) for i in range(len(meta))]
    stream = torch.cuda.current_stream()
    ls.run(host, stride, layer_bytes, STREAM_LAYERS, probs, stream=stream)
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(reps):
        ls.run(host, stride, layer_bytes, STREAM_LAYERS, probs, stream=stream)
    e1.record(stream)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / reps
    # the copies alone, the same bytes in the same sized pieces
    dev_buf = torch.empty(layer_bytes, dtype=torch.uint8, device=device)
    c0 = torch.cuda.Event(enable_timing=True)
    c1 = torch.cuda.Event(enable_timing=True)
    c0.record(stream)
    for l in range(STREAM_LAYERS):
        dev_buf.copy_(host[l * stride:l * stride + layer_bytes], non_blocking=True)
    c1.record(stream)
    torch.cuda.synchronize()
    copy_ms = c0.elapsed_time(c1)
    # the kernels reading the pinned host bytes themselves (no copies)
    direct = None
    try:
        ls.run_direct(host, stride, layer_bytes, STREAM_LAYERS, probs, stream=stream)
        torch.cuda.synchronize()
        d0 = torch.cuda.Event(enable_timing=True)
        d1 = torch.cuda.Event(enable_timing=True)
        d0.record(stream)
        for _ in range(reps):
            ls.run_direct(host, stride, layer_bytes, STREAM_LAYERS, probs, stream=stream)
        d1.record(stream)
        torch.cuda.synchronize()
        dms = d0.elapsed_time(d1) / reps
        direct = {"ms_per_token": round(dms, 3), "tok_s": round(1e3 / dms, 1),
                  "host_read_gb_s": round(STREAM_LAYERS * layer_bytes / (dms * 1e-3) / 1e9, 1)}
    except lq.LQError as e:
        direct = {"unavailable": str(e)}
    ls.close()
    weight_bytes = STREAM_LAYERS * layer_bytes
    return {"workload": f"{STREAM_LAYERS}-layer 7B stack, 2-bit + anchors, M={M}, weights in pinned host memory",
            "ms_per_token": round(ms, 3), "tok_s": round(1e3 / ms, 1),
            "h2d_gb_s_achieved": round(weight_bytes / (ms * 1e-3) / 1e9, 1),
            "plain_copy_gb_s": round(weight_bytes / (copy_ms * 1e-3) / 1e9, 1),
            "layer_bytes": layer_bytes, "distinct_layers": distinct, "direct_host_read": direct}


def run_lq(args):
    import torch

    import bit_weight_quantized_dequant_gb300 as lq

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    lq.build()
    M = 1
    hbm, bf16, bf16_sus, peak_kind = peaks()

    h = lq.Handle(local)
    copies = []
    io_bufs = []          # per layer copy: (all x of the layer in one buffer, all y in one buffer)
    host_copy0 = None
    for c in range(ROTATE):
        packs = layer_packs(M, c + 17 * rank)
        if c == 0:
            host_copy0 = packs
        # the layer's x and y each live in one contiguous buffer (every piece starts on 16 bytes:
        # K is a multiple of 256 and N of 16), so a step's inputs and results move in one copy each
        xbuf = torch.empty(sum(M * pk["K"] for _, pk, _ in packs), dtype=torch.float16, device=f"cuda:{local}")
        ybuf = torch.empty(sum(M * pk["N"] for _, pk, _ in packs), dtype=torch.float32, device=f"cuda:{local}")
        mats = []
        xo = yo = 0
        for name, pk, xb in packs:
            w = lq.QuantWeights.from_host(pk, lq.FMT_2BIT, device=f"cuda:{local}")
            x = xbuf[xo:xo + M * pk["K"]].view(M, pk["K"])
            x.copy_(torch.from_numpy(xb).view(torch.float16))
            y = ybuf[yo:yo + M * pk["N"]].view(M, pk["N"])
            xo += M * pk["K"]
            yo += M * pk["N"]
            mats.append((w, x, y))
        copies.append([h.problem(w, x, y) for (w, x, y) in mats] + [mats])
        io_bufs.append((xbuf, ybuf))
    layer_bytes = algorithmic_bytes(host_copy0, M)
    stream = torch.cuda.current_stream()
    prepared = [h.prepare(c[:-1]) for c in copies]   # each layer copy's C problem array, built once

    def step(i):
        h.gemv_grouped(prepared[i % ROTATE], stream=stream)

    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize()

    # direct calls: each step launched from the host, back to back (events only around the loop)
    d0 = torch.cuda.Event(enable_timing=True)
    d1 = torch.cuda.Event(enable_timing=True)
    d0.record(stream)
    for i in range(args.steps):
        step(i)
    d1.record(stream)
    torch.cuda.synchronize()
    h.sync()
    direct_ms = d0.elapsed_time(d1) / args.steps
    # one call alone: an event pair around each call (the events keep consecutive launches apart)
    n_alone = min(args.steps, 50)
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(n_alone)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(n_alone)]
    for i in range(n_alone):
        starts[i].record(stream)
        step(i)
        ends[i].record(stream)
    torch.cuda.synchronize()
    h.sync()
    pair_ms = statistics.mean(s.elapsed_time(e) for s, e in zip(starts, ends))

    # the timed run: the K steps captured once in a CUDA graph (two kernel nodes per step, the same
    # calls on the same 8 rotating layer copies) and replayed; a serving loop replays decode this way
    graph_note = "one CUDA graph holding the K steps (1 kernel node each), replayed once"
    cg = None
    try:
        g_stream = torch.cuda.Stream()
        g_stream.wait_stream(stream)
        cg = torch.cuda.CUDAGraph()
        with torch.cuda.graph(cg, stream=g_stream):
            for i in range(args.steps):
                h.gemv_grouped(prepared[i % ROTATE], stream=g_stream)
        cg.replay()   # untimed: uploads the graph
        torch.cuda.synchronize()
        h.sync()
    except Exception as e:   # capture refused here: time the direct calls instead, and say so
        cg = None
        graph_note = f"direct calls (graph capture unavailable: {type(e).__name__})"

    def timed_pass():
        if cg is not None:
            cg.replay()
        else:
            for i in range(args.steps):
                step(i)

    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    t_all0 = torch.cuda.Event(enable_timing=True)
    t_all1 = torch.cuda.Event(enable_timing=True)
    with ClockSampler(local) as clk:
        time.sleep(0.3)
        t_all0.record()
        timed_pass()
        t_all1.record()
        torch.cuda.synchronize()
        # keep the GPU busy a little longer so the sampler sees the loaded clocks
        extra_until = time.perf_counter() + 0.3
        while time.perf_counter() < extra_until:
            timed_pass()
            torch.cuda.synchronize()
    h.sync()
    total_ms = t_all0.elapsed_time(t_all1)
    if dist:
        total_ms = max_over_ranks(total_ms, dist, f"cuda:{local}")
    ms_per_step = total_ms / args.steps
    value = world * layer_bytes / (ms_per_step * 1e-3) / 1e9
    # the dominant launch pair: its average duration within the timed run (back to back, so the
    # per-step time), and, from the direct calls, the pair bracketed by its own events
    kern_ms = total_ms / args.steps
    achieved = layer_bytes / (kern_ms * 1e-3) / 1e9

    # end to end through the public API: x from pinned host memory in, y back to pinned host memory, every step
    # (one pinned host buffer holds a layer's x, one its y: one copy in and one copy out per step)
    xs_host = io_bufs[0][0].cpu().pin_memory()
    ys_host = torch.empty(io_bufs[0][1].numel(), dtype=torch.float32).pin_memory()
    h2d = xs_host.numel() * xs_host.element_size()
    d2h = ys_host.numel() * ys_host.element_size()

    # Every step copies its x in and its y out; the copies run on their own streams, ordered by
    # events per layer copy, so that step i + 1's copy in and step i's copy out overlap the kernels
    # next to them (a serving loop pipelines its I/O this way).
    copy_in, copy_out = torch.cuda.Stream(), torch.cuda.Stream()
    ev_in = [torch.cuda.Event() for _ in range(ROTATE)]
    ev_k = [torch.cuda.Event() for _ in range(ROTATE)]
    ev_out = [torch.cuda.Event() for _ in range(ROTATE)]
    for r in range(ROTATE):   # (recorded once, so that the first waits on them are satisfied)
        ev_k[r].record(stream)
        ev_out[r].record(stream)

    def e2e_step(i):
        r = i % ROTATE
        xbuf, ybuf = io_bufs[r]
        copy_in.wait_event(ev_k[r])              # the kernel that last read this x buffer is done
        with torch.cuda.stream(copy_in):
            xbuf.copy_(xs_host, non_blocking=True)
            ev_in[r].record(copy_in)
        stream.wait_event(ev_in[r])
        stream.wait_event(ev_out[r])             # this y buffer has been copied out
        h.gemv_grouped(prepared[r], stream=stream)
        ev_k[r].record(stream)
        copy_out.wait_event(ev_k[r])
        with torch.cuda.stream(copy_out):
            ys_host.copy_(ybuf, non_blocking=True)
            ev_out[r].record(copy_out)

    for i in range(args.warmup):
        e2e_step(i)
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    copy_in.wait_event(e0)
    for i in range(args.steps):
        e2e_step(i)
    stream.wait_stream(copy_out)                 # the last copy out is inside the timed region
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = e0.elapsed_time(e1) / args.steps
    e2e_val = world * layer_bytes / (e2e_ms * 1e-3) / 1e9

    single = single_linear_batched(lq, torch, h, f"cuda:{local}", 20, 3)
    single["frac_of_hbm"] = round(single["value"] / hbm, 4)

    gemm = None
    if not args.no_gemm:
        dev = f"cuda:{local}"
        g2 = gemm_layer(lq, torch, h, "2bit", dev, args.gemm_steps, 3)
        g4 = gemm_layer(lq, torch, h, "nf4", dev, args.gemm_steps, 3)
        gi4 = gemm_layer(lq, torch, h, "int4", dev, args.gemm_steps, 3)
        gdq = gemm_layer(lq, torch, h, "nf4_dq", dev, args.gemm_steps, 3)
        gemm = {"workload": GEMM_WORKLOAD, "metric": "dequant-GEMM TFLOP/s", "dtype": "bf16 x bf16 -> f32 accumulate",
                "2bit": g2, "nf4": g4, "int4": gi4, "nf4_dq": gdq,
                "roofline": {"bound": "tensor", "achieved": g2["value"], "peak": bf16, "unit": "TFLOP/s",
                             "frac": round(g2["value"] / bf16, 4), "peak_kind": peak_kind + " bf16 burst",
                             "kernel": "gemm_kernel<2bit>, one lq_gemm_grouped launch over the layer's 7 projections",
                             "traffic": _traffic("gemm_14b_layer_2bit_bytes_per_launch"),
                             "largest_projection_alone_tflops": g2["largest"]["tflops"]},
                "frac_of_bf16_peak": {"2bit": round(g2["value"] / bf16, 4), "nf4": round(g4["value"] / bf16, 4),
                                      "int4": round(gi4["value"] / bf16, 4), "nf4_dq": round(gdq["value"] / bf16, 4)}}

    decode_more = decode_workloads(lq, torch, h, f"cuda:{local}") if not args.no_decode_workloads else None
    quant = quantizer_layer(lq, torch, h, f"cuda:{local}") if not args.no_quant else None
    streamed = stream_stack(lq, torch, h, f"cuda:{local}") if not args.no_stream else None
    if streamed:
        streamed["resident_tok_s"] = round(1e3 / (ms_per_step * STACK_LAYERS), 1)

    traffic = _traffic("gemv_ring_7b_layer_m1_bytes_per_launch")

    if rank == 0:
        cores = host_cores()
        cpu_v, sample = cpu_baseline(host_copy0, seconds=8.0, threads=cores)
        cpu_1, sample_1 = cpu_baseline(host_copy0, seconds=4.0, threads=1)
        line = {
            "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(ms_per_step, 5), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f16", "data": "synthetic",
            "config": {"workload": WORKLOAD, "M": M, "layer_bytes": layer_bytes, "rotated_copies": ROTATE,
                       "l2": f"inputs larger than L2: {ROTATE} distinct layer copies ({ROTATE * layer_bytes / 1e6:.0f} MB)",
                       "parallelism": f"replicas x{world}", "launch": graph_note},
            "frac_of_hbm": round(value / world / hbm, 4),
            "tok_s_32_layer_stack": round(1e3 / (ms_per_step * STACK_LAYERS), 1),
            "roofline": {"bound": "hbm", "achieved": round(achieved, 2), "peak": hbm, "unit": "GB/s",
                         "frac": round(achieved / hbm, 4), "traffic": traffic, "peak_kind": peak_kind,
                         "kernel": "gemv_ring_kernel (each CTA builds its x in shared memory), one grouped call per layer: the timed run's time per step (the launches run back to back)",
                         "launch_alone_direct_call_gb_s": round(layer_bytes / (pair_ms * 1e-3) / 1e9, 2),
                         "algorithmic_bytes_per_launch": layer_bytes},
            "decode_target_workload": {"note": "the 512x256 single linear, where the decode target (75 % of HBM) is quoted",
                                       "value": single["value"], "unit": "GB/s", "frac_of_hbm": single["frac_of_hbm"],
                                       "workload": single["workload"]},
            "cpu_baseline": {"value": round(cpu_v, 4), "unit": "GB/s", "cores": cores, "kind": "oracle", "sample": sample,
                             "one_thread": {"value": round(cpu_1, 4), "unit": "GB/s", "cores": 1, "sample": sample_1}},
            "e2e": {"value": round(e2e_val, 2), "unit": "GB/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                    "note": "every step: x copied in from pinned host memory, the grouped call, y copied out; the "
                            "copies on their own streams, overlapping the neighbouring steps' kernels"},
            "gpu_launches": args.steps,   # one ring-kernel launch per grouped call (no pre-pass: x is built in-kernel)
            "clocks": clk.summary(),
            "direct_calls": {"value": round(world * layer_bytes / (direct_ms * 1e-3) / 1e9, 2), "unit": "GB/s",
                             "ms_per_step": round(direct_ms, 5), "note": "each step launched from the host"},
            "single_linear_512x256_batched": single,
            "gemm": gemm,
            "decode_workloads": decode_more,
            "quantizer": quant,
            "layer_streaming": streamed,
        }
        print(json.dumps(line), flush=True)
    h.close()
    if dist:
        dist.destroy_process_group()


def run_case(args):
    """One workload, three calls, nothing timed: the command line the ncu summaries in profiles/ capture."""
    import torch

    import bit_weight_quantized_dequant_gb300 as lq
    lq.build()
    h = lq.Handle(0)
    if args.case == "quant7b":
        quantizer_layer(lq, torch, h, "cuda", reps=2)
    elif args.case == "gemv7b":
        mats = []
        for name, pk, xb in layer_packs(1, 0):
            w = lq.QuantWeights.from_host(pk, lq.FMT_2BIT)
            x = torch.from_numpy(xb).view(torch.float16).cuda()
            y = torch.empty((1, pk["N"]), dtype=torch.float32, device="cuda")
            mats.append((w, x, y))
        probs = [h.problem(w, x, y) for w, x, y in mats]
        for _ in range(3):
            h.gemv_grouped(probs)
    elif args.case == "gemv512x256":
        # the single 512x256 linear over 4096 distinct weight sets (234 MB, past L2) in one launch
        L, N, K, A = 4096, 512, 256, 8
        big = synth.random_packed_2bit_sets(L, N, K, A, seed=1, cfg=1)
        w = lq.QuantWeights.from_host(big, lq.FMT_2BIT)
        x = torch.from_numpy(synth.activations(L, K, "f16", seed=1, cfg=1)).view(torch.float16).cuda().view(L, 1, K)
        y = torch.empty((L, 1, N), dtype=torch.float32, device="cuda")
        strides = dict(codes=N * K // 4, scales=N * K // 32 * 2, offsets=N * K // 32 * 2, anchor_idx=4 * A,
                       anchor_w=N * 8 * 2, x=K * 2, y=N * 4)
        prob = [h.problem(w, x[0], y[0], batch=L, strides=strides)]
        for _ in range(3):
            h.gemv_grouped(prob)
    else:
        from math import floor
        fmt = args.case.split("-")[1]
        mats = []
        for i, (name, N, K) in enumerate(synth.LAYER_SHAPES["14b"]):
            if fmt == "2bit":
                pk = synth.random_packed_2bit(N, K, int(floor(0.035 * K)), sigma=0.02, seed=500, cfg=5, matrix_id=i)
                w = lq.QuantWeights.from_host(pk, lq.FMT_2BIT)
            else:
                pk = synth.random_packed_nf4(N, K, sigma=0.02, seed=500, cfg=5, matrix_id=i)
                w = lq.QuantWeights.from_host(pk, lq.FMT_NF4)
            xb = synth.activations(GEMM_M, K, "bf16", synth.channel_sigma(K, synth.outlier_channels(K, 0.01, seed=500, cfg=5), 20.0),
                                   seed=500, cfg=5, matrix_id=i)
            x = torch.from_numpy(xb).view(torch.bfloat16).cuda()
            y = torch.empty((GEMM_M, N), dtype=torch.bfloat16, device="cuda")
            mats.append((w, x, y))
        probs = [h.problem(w, x, y) for w, x, y in mats]
        for _ in range(3):
            h.gemm_grouped(probs)
    torch.cuda.synchronize()
    h.close()
    print(json.dumps({"case": args.case, "calls": 3}))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="lq", choices=["lq", "reference"])
    ap.add_argument("--gemm-steps", type=int, default=20)
    ap.add_argument("--no-gemm", action="store_true")
    ap.add_argument("--no-quant", action="store_true")
    ap.add_argument("--no-stream", action="store_true")
    ap.add_argument("--no-decode-workloads", action="store_true")
    ap.add_argument("--case", choices=["gemv7b", "gemv512x256", "gemm14b-2bit", "gemm14b-nf4", "quant7b"],
                    help="run one workload three times, untimed (what the profiles capture)")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.case:
        run_case(args)
    elif args.impl == "reference":
        run_reference(args)
    else:
        run_lq(args)


if __name__ == "__main__":
    main()
