#!/usr/bin/env python
"""Benchmark of the dequantize-fused quantized matmul on GB300.

Default workload: the full decode weight stream of a Llama-2-70B-shaped model
at EXL2 4.0 bpw -- 80 layers x 7 quantized linears (q, k, v, o, gate, up,
down), M = 1. As in the model, q, k and v read one activation vector and
gate and up another, so each layer is four calls: exq_gemv_multi(q, k, v),
exq_gemv(o), exq_gemv_multi(gate, up), exq_gemv(down), each with a fresh
x ~ N(0,1); 320 calls back to back on one stream, captured once in a CUDA
graph (``--ungrouped``: 560 exq_gemv calls, one per linear, each with its
own x). One step = one token = all 560 matmuls; the weights (38.5 GB of
packed codes + fp16 scales) are far larger than L2, so every step streams
them from HBM.

Prints one JSON line. ``value`` is the packed-weight throughput (qweight +
scales bytes per step / time) with everything resident in HBM; ``e2e`` is the
same metric when each step also copies its activation vectors (one per
call) in from pinned host memory and its 560 outputs back; ``roofline`` relates the GEMV
kernel to the measured HBM copy bandwidth; ``cpu_baseline`` is the CPU oracle
on a bounded sample of the same workload.

``--impl reference`` times the CPU oracle instead (one bounded sample per
step) and prints the same metric.
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

# The CPU oracle arm (--impl reference) runs on one thread and says so; BLAS
# reads these when numpy loads, so they are set before the import.
if "--impl=reference" in sys.argv or any(
        a == "--impl" and b == "reference" for a, b in zip(sys.argv, sys.argv[1:])):
    for _v in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
        os.environ.setdefault(_v, "1")

import numpy as np  # noqa: E402

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import synth  # noqa: E402

METRIC = "decode GEMV weight GB/s (% of 8 TB/s); prefill GEMM TFLOPS (% of fp16 peak)"
UNIT = "GB/s"
NOMINAL_HBM_GBS = 8000.0
FALLBACK_HBM_GBS = 6800.0
WORKLOAD = "decode_stream_70b"
LINEARS = list(synth.LLAMA2_70B_SHAPES.items())
# linears of a decoder layer that read the same activations
GROUPS = (("q", "k", "v"), ("o",), ("gate", "up"), ("down",))
GEMV_SOURCES = ["quantized_weight_exq_gb300/csrc/exq_gemv.cu", "quantized_weight_exq_gb300/csrc/exq_device.cuh"]


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="exq", choices=["exq", "reference"])
    ap.add_argument("--layers", type=int, default=80, help="decoder layers in the stream (80 = Llama-2-70B)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--format", default="exl2", choices=["exl2", "exl2_qscale"],
                    help="decode stream format: EXL2 4.0 bpw with fp16 scales (default) or with two-level "
                         "scales (4-bit group-scale codes x per-column fp16 maxima)")
    ap.add_argument("--segment-order", default="random", choices=["random", "sorted"],
                    help="stored order of a layer's EXL2 segments: as drawn, or grouped by width (the row "
                         "remapping lays out equal widths contiguously)")
    ap.add_argument("--ungrouped", action="store_true",
                    help="decode stream as one exq_gemv per linear (each with its own x) instead of grouping "
                         "the linears that share x (q/k/v, gate/up) into exq_gemv_multi calls")
    ap.add_argument("--prefill", action="store_true",
                    help="time the prefill GEMM over the 70B shapes instead (one JSON line, TFLOPS per shape)")
    ap.add_argument("--kv", action="store_true",
                    help="time the quantized KV cache codec (Q4/Q6/Q8 write and read) over a Llama-2-70B cache "
                         "at 32K context instead (one JSON line, GB/s per width and direction)")
    ap.add_argument("--convert", action="store_true",
                    help="time the EXL2 conversion (error table, host solve at 4.0 bpw, RTN quantisation) of the "
                         "Llama-2-70B gate weight instead (one JSON line)")
    ap.add_argument("--kv-groups", type=int, default=80 * 2 * 32768 * 8,
                    help="groups of 128 values for --kv (default: the whole 70B cache at 32K context)")
    ap.add_argument("--dequant", action="store_true",
                    help="time the standalone dequantisation of the 70B gate weight instead (one JSON line)")
    ap.add_argument("--no-prefill", action="store_true", help="leave the prefill record out of the default line")
    ap.add_argument("--decode-sweep", action="store_true",
                    help="time single GEMVs of the GPTQ 4096, GPTQ act-order 7B and EXL2 4.0 7B workloads "
                         "instead (one JSON line, GB/s per shape and M)")
    return ap.parse_args()


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def source_hash(paths) -> str:
    h = hashlib.sha256()
    for p in paths:
        with open(os.path.join(ROOT, p), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def profile_traffic():
    """DRAM traffic per algorithmic byte of the GEMV kernel, from the committed
    ncu summary, or None if that summary was taken on other kernel sources."""
    p = os.path.join(ROOT, "profiles", "gemv_exl2_decode_70b.md")
    if not os.path.exists(p):
        return None
    txt = open(p).read()
    m = re.search(r"bench-traffic: dram_bytes_per_algorithmic_byte=([0-9.]+) source_hash=([0-9a-f]+)", txt)
    if not m or m.group(2) != source_hash(GEMV_SOURCES):
        return None
    return float(m.group(1))


# ----------------------------------------------------------------------------- clocks

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.proc = None
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "100",
                 "-i", str(gpu_index)], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except Exception:
            self.proc.kill()
            out, _ = self.proc.communicate()
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx.append(float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


# ----------------------------------------------------------------------------- workload

def bit_mix(layer: int, lin: int, K: int):
    wid = synth.WORKLOAD_IDS[WORKLOAD]
    return synth.solve_bit_mix(K // 32, 4.0, synth.EXL2_BITS, synth.rng_for(0, wid, 7 * layer + lin, 4))


def build_stream(exq, torch, layers: int, device, grouped: bool = True, two_level: bool = False,
                 sorted_widths: bool = False):
    """Device-resident packed weights for the whole stream, as a list of
    calls (weights, x, outputs). Packed codes are uniform random words (a
    segment column's b words are a bijection of its 32 uniform b-bit codes);
    bits, scales and permutations follow the EXL2 4.0 bpw recipe. Grouped:
    one call (and one x) per group of linears that share activations."""
    wid = synth.WORKLOAD_IDS[WORKLOAD]
    names = [n for n, _ in LINEARS]
    groups = GROUPS if grouped else tuple((n,) for n in names)
    x_total = sum(synth.LLAMA2_70B_SHAPES[grp[0]][0] for grp in groups) * layers
    y_total = sum(N for _, (K, N) in LINEARS) * layers
    x_all = torch.empty(x_total, dtype=torch.float16, device=device)
    y_all = torch.empty(y_total, dtype=torch.float16, device=device)
    xo = yo = 0
    calls = []
    for layer in range(layers):
        for grp in groups:
            ws, ys = [], []
            x = None
            for name in grp:
                i = names.index(name)
                K, N = synth.LLAMA2_70B_SHAPES[name]
                gen = torch.Generator(device=device)
                gen.manual_seed(int(synth.rng_for(0, wid, 7 * layer + i, 0).integers(0, 2 ** 62)))
                bits = bit_mix(layer, i, K)
                if sorted_widths:  # equal widths stored contiguously (the permutation absorbs the order)
                    bits = np.sort(bits)[::-1].copy()
                ws.append(exl2_device_layer(exq, torch, K, N, bits, gen, device, two_level))
                if x is None:  # the group's activations: drawn with its first linear's generator
                    x = x_all[xo:xo + K].view(1, K)
                    x.copy_(torch.randn(1, K, device=device, generator=gen).half())
                    xo += K
                ys.append(y_all[yo:yo + N].view(1, N))
                yo += N
            calls.append((ws, x, ys))
    return calls, x_all, y_all


def issue_call(exq, call, workspace):
    ws, x, ys = call
    if len(ws) == 1:
        exq.exq_gemv(ws[0], x, ys[0], workspace=workspace)
    else:
        exq.exq_gemv_multi(ws, x, ys, workspace=workspace)


def call_workspace_size(exq, call) -> int:
    ws, x, _ = call
    if len(ws) == 1:
        return exq.exq_gemv_workspace_size(ws[0], x.shape[0])
    return exq.exq_gemv_multi_workspace_size(ws, x.shape[0])


def exl2_device_layer(exq, torch, K, N, bits, gen, device, two_level=False, perm=True):
    """An EXL2 layer drawn on the device: uniform packed words (the packing is
    a bijection, so these are uniform codes), fp16 scales ~ U(0.002, 0.03) or
    two-level scales (uniform 4-bit codes, column maxima ~ U(0.02, 0.05)), and
    a random permutation."""
    off = exq.exq_exl2_seg_word_off(bits).astype(np.int64)
    qw = torch.randint(0, 2 ** 32, (int(off[-1]), N), dtype=torch.int64, device=device, generator=gen).to(torch.int32)
    if two_level:
        qs = torch.randint(0, 2 ** 32, (K // 32, N // 8), dtype=torch.int64, device=device,
                           generator=gen).to(torch.int32)
        mx = (torch.rand(N, device=device, generator=gen) * 0.03 + 0.02).half()
    else:
        sc = (torch.rand(K // 32, N, device=device, generator=gen) * 0.028 + 0.002).half()
    pm = torch.randperm(K, device=device, generator=gen).to(torch.int32) if perm else None
    if two_level:
        return exq.exl2_qscale_weight(qw, off.astype(np.int32), qs, mx, pm, K, N, device=device)
    return exq.exl2_weight(qw, off.astype(np.int32), sc, pm, K, N, device=device)


PREFILL_SHAPES = (("q", 8192, 8192), ("k", 8192, 1024), ("gate", 8192, 28672), ("down", 28672, 8192))


def run_prefill(args, device):
    """The prefill GEMM over the Llama-2-70B projection shapes at M = 512 and
    2048, GPTQ g128 (no act-order) and EXL2 2.5 bpw from {2, 3, 4}; at M = 2048
    also EXL2 with two-level scales, GPTQ with act-order and EXL2 with a row
    permutation (x gathered first, inside the timed launch); packed
    words drawn uniformly on the device (the packing is a bijection, so this is
    the distribution of uniform codes). CUDA events around `--steps` launches
    after `--warmup`; TFLOPS = 2 M K N / time."""
    import torch

    import __graft_entry__
    __graft_entry__.build()
    import quantized_weight_exq_gb300 as exq

    torch.cuda.set_device(device)
    peak_bf16 = None
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            peak_bf16 = float(json.load(f)["bf16_tflops"])
    except Exception:
        peak_bf16 = 1900.0
    shapes = {}
    for fmt in ("gptq_g128", "exl2_2.5bpw", "exl2_2.5bpw_two_level", "gptq_g128_act_order", "exl2_2.5bpw_permuted"):
        variant = fmt.endswith(("two_level", "act_order", "permuted"))
        for M in ((2048,) if variant else (512, 2048)):
            for name, K, N in PREFILL_SHAPES:
                gen = torch.Generator(device=device)
                gen.manual_seed(1000 * M + K + N)
                if fmt.startswith("gptq"):
                    qw = torch.randint(0, 2 ** 32, (K // 8, N), dtype=torch.int64, device=device,
                                       generator=gen).to(torch.int32)
                    qz = torch.randint(0, 2 ** 32, (K // 128, N // 8), dtype=torch.int64, device=device,
                                       generator=gen).to(torch.int32)
                    sc = (torch.rand(K // 128, N, device=device, generator=gen) * 0.015 + 0.005).half()
                    pm = torch.randperm(K, device=device, generator=gen).int() if fmt.endswith("act_order") else None
                    w = exq.gptq_weight(qw, qz, sc, pm, K, N, 128, device=device)
                else:
                    bits = synth.solve_bit_mix(K // 32, 2.5, (2, 3, 4), np.random.default_rng(K + N))
                    w = exl2_device_layer(exq, torch, K, N, bits, gen, device,
                                          two_level=fmt.endswith("two_level"), perm=fmt.endswith("permuted"))
                x = torch.randn(M, K, device=device, generator=gen).half()
                y = torch.empty(M, N, device=device, dtype=torch.float16)
                nws = exq.exq_gemm_workspace_size(w, M)
                ws = torch.empty(max(nws, 16), dtype=torch.uint8, device=device) if nws else None
                for _ in range(args.warmup):
                    exq.exq_gemm(w, x, y, ws)
                torch.cuda.synchronize()
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record()
                for _ in range(args.steps):
                    exq.exq_gemm(w, x, y, ws)
                e1.record()
                torch.cuda.synchronize()
                us = e0.elapsed_time(e1) * 1000 / args.steps
                tf = 2 * M * K * N / us / 1e6
                shapes[f"{fmt} M={M} {name} {K}x{N}"] = {"us": round(us, 1), "tflops": round(tf, 1),
                                                          "frac": round(tf / peak_bf16, 4)}
    # linears that read the same x in one launch (exq_gemm_multi): q+k+v and gate+up
    for fmt in ("gptq_g128", "exl2_2.5bpw"):
        for grp in (("q", "k", "v"), ("gate", "up")):
            for M in ((512, 2048) if grp[0] == "q" else (2048,)):
                gen = torch.Generator(device=device)
                gen.manual_seed(2000 * M + len(grp))
                ws_ = []
                for name in grp:
                    K, N = synth.LLAMA2_70B_SHAPES[name]
                    if fmt.startswith("gptq"):
                        qw = torch.randint(0, 2 ** 32, (K // 8, N), dtype=torch.int64, device=device,
                                           generator=gen).to(torch.int32)
                        qz = torch.randint(0, 2 ** 32, (K // 128, N // 8), dtype=torch.int64, device=device,
                                           generator=gen).to(torch.int32)
                        sc = (torch.rand(K // 128, N, device=device, generator=gen) * 0.015 + 0.005).half()
                        ws_.append(exq.gptq_weight(qw, qz, sc, None, K, N, 128, device=device))
                    else:
                        bits = synth.solve_bit_mix(K // 32, 2.5, (2, 3, 4), np.random.default_rng(K + N))
                        ws_.append(exl2_device_layer(exq, torch, K, N, bits, gen, device, perm=False))
                K = ws_[0].K
                x = torch.randn(M, K, device=device, generator=gen).half()
                ys = [torch.empty(M, w.N, device=device, dtype=torch.float16) for w in ws_]
                for _ in range(args.warmup):
                    exq.exq_gemm_multi(ws_, x, ys)
                torch.cuda.synchronize()
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record()
                for _ in range(args.steps):
                    exq.exq_gemm_multi(ws_, x, ys)
                e1.record()
                torch.cuda.synchronize()
                us = e0.elapsed_time(e1) * 1000 / args.steps
                ntot = sum(w.N for w in ws_)
                tf = 2 * M * K * ntot / us / 1e6
                shapes[f"{fmt} M={M} {'+'.join(grp)} grouped {K}x{ntot}"] = {
                    "us": round(us, 1), "tflops": round(tf, 1), "frac": round(tf / peak_bf16, 4)}
                del ws_, x, ys
    if exq.exq_get_last_device_error() != 0:
        raise RuntimeError("device error word set during the prefill sweep")
    best = max(v["tflops"] for v in shapes.values())
    return {
        "metric": "prefill GEMM TFLOPS (fp16 in, fp32 accumulate)",
        "value": best,
        "unit": "TFLOPS",
        "n_gpus": 1,
        "steps": args.steps,
        "warmup": args.warmup,
        "higher_is_better": True,
        "dtype": "f16",
        "data": "synthetic",
        "config": {"workload": "prefill_70b_shapes", "value_is": "best shape"},
        "roofline": {"bound": "tensor", "peak": peak_bf16, "unit": "TFLOPS",
                     "peak_kind": "measured bf16 cuBLAS burst (fp16 runs at the same rate)"},
        "shapes": shapes,
    }


def prefill_record(exq, torch, device, steps: int = 10, warmup: int = 3):
    """The prefill half of the metric, for the default line: exq_gemm on the
    Llama-2-70B gate shape (8192 x 28672) at M = 2048, GPTQ g128 and EXL2 2.5
    bpw; packed words drawn uniformly on the device. CUDA events on the
    launching stream around `steps` launches after `warmup`; TFLOPS =
    2 M K N / average launch time, against the measured bf16 burst peak (fp16
    runs at the same tensor-core rate; each launch is timed alone)."""
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            pk = json.load(f)
        peak, peak_s, kind = float(pk["bf16_tflops"]), float(pk.get("bf16_tflops_sustained", 0) or 0), "measured"
    except Exception:
        peak, peak_s, kind = 1900.0, 1700.0, "fallback"
    M, (K, N) = 2048, synth.LLAMA2_70B_SHAPES["gate"]
    out = {"workload": "prefill_70b_gate_8192x28672_M2048", "M": M, "K": K, "N": N, "peak": peak,
           "peak_kind": f"{kind} bf16 burst (cuBLAS); fp16 runs at the same rate", "unit": "TFLOPS"}
    stream = torch.cuda.Stream(device=device)
    for fmt in ("gptq_g128", "exl2_2.5bpw"):
        gen = torch.Generator(device=device)
        gen.manual_seed(77 + len(fmt))
        if fmt.startswith("gptq"):
            qw = torch.randint(0, 2 ** 32, (K // 8, N), dtype=torch.int64, device=device, generator=gen).to(torch.int32)
            qz = torch.randint(0, 2 ** 32, (K // 128, N // 8), dtype=torch.int64, device=device,
                               generator=gen).to(torch.int32)
            sc = (torch.rand(K // 128, N, device=device, generator=gen) * 0.015 + 0.005).half()
            w = exq.gptq_weight(qw, qz, sc, None, K, N, 128, device=device)
        else:
            bits = synth.solve_bit_mix(K // 32, 2.5, (2, 3, 4), np.random.default_rng(K + N))
            w = exl2_device_layer(exq, torch, K, N, bits, gen, device, perm=False)
        x = torch.randn(M, K, device=device, generator=gen).half()
        y = torch.empty(M, N, device=device, dtype=torch.float16)
        nws = exq.exq_gemm_workspace_size(w, M)
        ws = torch.empty(max(nws, 16), dtype=torch.uint8, device=device) if nws else None
        torch.cuda.synchronize()
        with torch.cuda.stream(stream):
            for _ in range(warmup):
                exq.exq_gemm(w, x, y, ws, stream=stream)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for _ in range(steps):
                exq.exq_gemm(w, x, y, ws, stream=stream)
            e1.record(stream)
        torch.cuda.synchronize()
        us = e0.elapsed_time(e1) * 1000 / steps
        tf = 2 * M * K * N / us / 1e6
        out[fmt] = {"us": round(us, 1), "tflops": round(tf, 1), "frac": round(tf / peak, 4),
                    "frac_of_sustained": round(tf / peak_s, 4) if peak_s else None,
                    "kernel": "gemm_kernel (tcgen05, TMEM accumulator)", "launches": steps}
        del w, x, y, ws
    # the q, k and v projections (8192 x 8192, 1024, 1024) in one exq_gemm_multi launch, GPTQ g128
    gen = torch.Generator(device=device)
    gen.manual_seed(91)
    ws_ = []
    for name in ("q", "k", "v"):
        Kq, Nq = synth.LLAMA2_70B_SHAPES[name]
        qw = torch.randint(0, 2 ** 32, (Kq // 8, Nq), dtype=torch.int64, device=device, generator=gen).to(torch.int32)
        qz = torch.randint(0, 2 ** 32, (Kq // 128, Nq // 8), dtype=torch.int64, device=device,
                           generator=gen).to(torch.int32)
        sc = (torch.rand(Kq // 128, Nq, device=device, generator=gen) * 0.015 + 0.005).half()
        ws_.append(exq.gptq_weight(qw, qz, sc, None, Kq, Nq, 128, device=device))
    x = torch.randn(M, ws_[0].K, device=device, generator=gen).half()
    ys = [torch.empty(M, w.N, device=device, dtype=torch.float16) for w in ws_]
    with torch.cuda.stream(stream):
        for _ in range(warmup):
            exq.exq_gemm_multi(ws_, x, ys, stream=stream)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(steps):
            exq.exq_gemm_multi(ws_, x, ys, stream=stream)
        e1.record(stream)
    torch.cuda.synchronize()
    us = e0.elapsed_time(e1) * 1000 / steps
    ntot = sum(w.N for w in ws_)
    tf = 2 * M * ws_[0].K * ntot / us / 1e6
    out["gptq_g128_qkv_grouped"] = {"us": round(us, 1), "tflops": round(tf, 1), "frac": round(tf / peak, 4),
                                    "shape": f"8192 x (8192 + 1024 + 1024), M = {M}",
                                    "kernel": "gemm_kernel over the three layers' tiles (exq_gemm_multi)",
                                    "launches": steps}
    if exq.exq_get_last_device_error() != 0:
        raise RuntimeError("device error word set during the prefill record")
    return out


def run_dequant(args, device):
    """The standalone dequantisation (exq_dequant) of the Llama-2-70B gate
    weight (8192 x 28672) at EXL2 4.0 bpw (permuted rows), EXL2 4.0 with
    two-level scales and GPTQ g128: packed words drawn uniformly on the device.
    CUDA events around `--steps` launches after `--warmup`; GB/s = (packed
    bytes read + 2 K N bytes written) / time, against the measured HBM copy
    bandwidth (far above L2: 470 MB written per launch)."""
    import torch

    import __graft_entry__
    __graft_entry__.build()
    import quantized_weight_exq_gb300 as exq

    torch.cuda.set_device(device)
    peak, peak_kind = measured_peaks()
    K, N = synth.LLAMA2_70B_SHAPES["gate"]
    res = {}
    for fmt in ("exl2_4.0bpw", "exl2_4.0bpw_two_level", "gptq_g128"):
        gen = torch.Generator(device=device)
        gen.manual_seed(31 + len(fmt))
        if fmt.startswith("gptq"):
            qw = torch.randint(0, 2 ** 32, (K // 8, N), dtype=torch.int64, device=device, generator=gen).to(torch.int32)
            qz = torch.randint(0, 2 ** 32, (K // 128, N // 8), dtype=torch.int64, device=device,
                               generator=gen).to(torch.int32)
            sc = (torch.rand(K // 128, N, device=device, generator=gen) * 0.015 + 0.005).half()
            w = exq.gptq_weight(qw, qz, sc, None, K, N, 128, device=device)
        else:
            bits = synth.solve_bit_mix(K // 32, 4.0, synth.EXL2_BITS, np.random.default_rng(K))
            w = exl2_device_layer(exq, torch, K, N, bits, gen, device, two_level=fmt.endswith("two_level"))
        W = torch.empty(K, N, dtype=torch.float16, device=device)
        for _ in range(args.warmup):
            exq.exq_dequant(w, W)
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(args.steps):
            exq.exq_dequant(w, W)
        e1.record()
        torch.cuda.synchronize()
        us = e0.elapsed_time(e1) * 1000 / args.steps
        moved = w.packed_bytes + 2 * K * N
        gbs = moved / us / 1e3
        res[fmt] = {"us": round(us, 1), "GB/s": round(gbs, 1), "frac": round(gbs / peak, 4),
                    "packed_bytes": w.packed_bytes, "written_bytes": 2 * K * N}
        del w, W
    if exq.exq_get_last_device_error() != 0:
        raise RuntimeError("device error word set during the dequant run")
    return {
        "metric": "standalone dequant GB/s (packed bytes read + fp16 bytes written)",
        "value": min(v["GB/s"] for v in res.values()),
        "unit": UNIT,
        "n_gpus": 1,
        "steps": args.steps,
        "warmup": args.warmup,
        "higher_is_better": True,
        "dtype": "f16",
        "data": "synthetic",
        "config": {"workload": "dequant_70b_gate_8192x28672", "value_is": "slowest format",
                   "l2": "outputs larger than L2 (470 MB of fp16 per launch)"},
        "roofline": {"bound": "hbm", "peak": peak, "unit": UNIT, "peak_kind": peak_kind},
        "formats": res,
    }


def run_decode_sweep(args, device):
    """Single exq_gemv calls of the decode workloads: GPTQ 4-bit g128 4096x4096
    at M = 1 (no act-order); GPTQ act-order on the Llama-2-7B shapes at M in
    {1, 4, 16}; EXL2 4.0 bpw (permuted) on the 7B shapes at M in {1, 8}. Then
    the 7B linears that share x (q+k+v, gate+up) as one exq_gemv_multi call
    each, in both formats.
    Packed words are drawn uniformly on the device (the packing is a
    bijection, so this is the distribution of uniform codes and zeros); each
    timed call uses the next weight copy of a ring larger than twice L2, so
    every call streams its weights from HBM. `--steps` calls (after
    `--warmup`) captured in one CUDA graph and timed with CUDA events around a
    replay; GB/s = packed bytes (codes + scales + zeros) per call / time."""
    import torch

    import __graft_entry__
    __graft_entry__.build()
    import quantized_weight_exq_gb300 as exq

    torch.cuda.set_device(device)
    peak, peak_kind = measured_peaks()
    ring_bytes = 300e6

    def gptq(K, N, act, gen):
        qw = torch.randint(0, 2 ** 32, (K // 8, N), dtype=torch.int64, device=device, generator=gen).to(torch.int32)
        qz = torch.randint(0, 2 ** 32, (K // 128, N // 8), dtype=torch.int64, device=device,
                           generator=gen).to(torch.int32)
        sc = (torch.rand(K // 128, N, device=device, generator=gen) * 0.015 + 0.005).half()
        perm = torch.randperm(K, device=device, generator=gen).int() if act else None
        return exq.gptq_weight(qw, qz, sc, perm, K, N, 128, device=device)

    def exl2(K, N, gen, rng, two_level=False):
        bits = synth.solve_bit_mix(K // 32, 4.0, synth.EXL2_BITS, rng)
        return exl2_device_layer(exq, torch, K, N, bits, gen, device, two_level)

    cases = [("gptq_g128 4096x4096", "gptq", 4096, (4096,), False, (1,))]
    for name, (K, N) in synth.LLAMA2_7B_SHAPES.items():
        if name in ("q", "gate", "down"):
            cases.append((f"gptq_act_order 7b {name} {K}x{N}", "gptq", K, (N,), True, (1, 4, 16)))
    for name, (K, N) in synth.LLAMA2_7B_SHAPES.items():
        if name in ("q", "gate", "down"):
            cases.append((f"exl2_4.0bpw 7b {name} {K}x{N}", "exl2", K, (N,), True, (1, 8)))
    for grp in (("q", "k", "v"), ("gate", "up")):
        K = synth.LLAMA2_7B_SHAPES[grp[0]][0]
        Ns = tuple(synth.LLAMA2_7B_SHAPES[n][1] for n in grp)
        tag = "+".join(grp)
        cases.append((f"gptq_act_order 7b {tag} grouped", "gptq", K, Ns, True, (1, 4, 16)))
        cases.append((f"exl2_4.0bpw 7b {tag} grouped", "exl2", K, Ns, True, (1, 8)))
    # the same EXL2 shapes with two-level scales
    K, N = synth.LLAMA2_7B_SHAPES["gate"]
    cases.append((f"exl2_4.0bpw_two_level 7b gate {K}x{N}", "exl2_qs", K, (N,), True, (1, 8)))
    cases.append(("exl2_4.0bpw_two_level 7b gate+up grouped", "exl2_qs", K, (N, N), True, (1, 8)))
    shapes = {}
    for label, fmt, K, Ns, act, Ms in cases:
        gen = torch.Generator(device=device)
        gen.manual_seed(K * 7 + sum(Ns) + len(Ns) - 1)
        rng = np.random.default_rng(K + sum(Ns) + len(Ns) - 1)
        reps = max(2, int(ring_bytes // (K * sum(Ns) // 2)) + 1)
        ring = [[gptq(K, N, act, gen) if fmt == "gptq" else exl2(K, N, gen, rng, fmt == "exl2_qs") for N in Ns]
                for _ in range(reps)]

        def call(i, x, ys, ws):
            if len(Ns) == 1:
                exq.exq_gemv(ring[i % reps][0], x, ys[0], workspace=ws)
            else:
                exq.exq_gemv_multi(ring[i % reps], x, ys, workspace=ws)

        for M in Ms:
            x = torch.randn(M, K, device=device, generator=gen).half()
            ys = [torch.empty(M, N, device=device, dtype=torch.float16) for N in Ns]
            ws = torch.zeros(exq.exq_gemv_multi_workspace_size(ring[0], M), dtype=torch.uint8, device=device)
            # one CUDA graph of `steps` calls (the host launch cost of a small
            # call exceeds its GPU time; the graph times the GPU)
            stream = torch.cuda.Stream(device=device)
            stream.wait_stream(torch.cuda.current_stream(device))
            graph = torch.cuda.CUDAGraph()
            with torch.cuda.stream(stream):
                for i in range(args.warmup):
                    call(i, x, ys, ws)
                torch.cuda.synchronize(device)
                with torch.cuda.graph(graph, stream=stream):
                    for i in range(args.steps):
                        call(i, x, ys, ws)
            graph.replay()
            torch.cuda.synchronize(device)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            graph.replay()
            e1.record()
            torch.cuda.synchronize(device)
            us = e0.elapsed_time(e1) * 1000 / args.steps
            gbs = sum(w.packed_bytes for w in ring[0]) / us / 1e3
            shapes[f"{label} M={M}"] = {"us": round(us, 2), "GB/s": round(gbs, 1), "frac": round(gbs / peak, 4)}
        del ring
    if exq.exq_get_last_device_error() != 0:
        raise RuntimeError("device error word set during the decode sweep")
    return {
        "metric": "decode GEMV weight GB/s (single calls)",
        "value": max(v["GB/s"] for v in shapes.values()),
        "unit": UNIT,
        "n_gpus": 1,
        "steps": args.steps,
        "warmup": args.warmup,
        "higher_is_better": True,
        "dtype": "f16",
        "data": "synthetic",
        "config": {"workload": "decode_configs_gptq4096_gptq_act_order_7b_exl2_4p0_7b", "value_is": "best case",
                   "l2": "weight ring larger than twice L2", "launch": "CUDA graph of the timed calls"},
        "roofline": {"bound": "hbm", "peak": peak, "unit": UNIT, "peak_kind": peak_kind},
        "shapes": shapes,
    }


def run_kv(args, device):
    """The quantized KV cache codec over a Llama-2-70B cache at 32K context:
    80 layers x K and V x 32768 tokens x 8 KV heads = 41,943,040 groups of
    D = 128 fp16 values (10.7 GB), values N(0, 1) times a per-group power of
    two in 2^-6 .. 2^2. For each width, `--steps` quantize launches and
    `--steps` dequantize launches after `--warmup`, CUDA events around each
    run; GB/s = bytes read + written per launch / time (far above L2)."""
    import torch

    import __graft_entry__
    __graft_entry__.build()
    import quantized_weight_exq_gb300 as exq

    torch.cuda.set_device(device)
    peak, peak_kind = measured_peaks()
    G, D = args.kv_groups, 128
    gen = torch.Generator(device=device)
    gen.manual_seed(11)
    x = torch.empty(G, D, dtype=torch.float16, device=device)
    chunk = 1 << 22
    for i in range(0, G, chunk):  # drawn in slices to bound the fp32 temporaries
        n = min(chunk, G - i)
        x[i:i + n] = (torch.randn(n, D, device=device, generator=gen) *
                      torch.exp2(torch.randint(-6, 3, (n, 1), device=device, generator=gen).float())).half()
    out = torch.empty_like(x)
    widths = {}

    def timed(fn):
        for _ in range(args.warmup):
            fn()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(args.steps):
            fn()
        e1.record()
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) * 1000 / args.steps  # us

    for bits in (4, 6, 8):
        codes = torch.empty(G, D * bits // 32, dtype=torch.int32, device=device)
        scales = torch.empty(G, dtype=torch.float16, device=device)
        q_us = timed(lambda: exq.exq_kv_quantize(x, bits, codes, scales))
        d_us = timed(lambda: exq.exq_kv_dequantize(codes, scales, D, bits, out))
        packed = G * D * bits // 8 + 2 * G
        q_gbs = (2 * G * D + packed) / q_us / 1e3
        d_gbs = (packed + 2 * G * D) / d_us / 1e3
        widths[f"Q{bits}"] = {
            "quantize_us": round(q_us, 1), "quantize_GB/s": round(q_gbs, 1), "quantize_frac": round(q_gbs / peak, 4),
            "dequantize_us": round(d_us, 1), "dequantize_GB/s": round(d_gbs, 1),
            "dequantize_frac": round(d_gbs / peak, 4),
            "cache_bytes": packed, "fp16_bytes": 2 * G * D,
        }
        del codes, scales
    if exq.exq_get_last_device_error() != 0:
        raise RuntimeError("device error word set during the KV codec run")
    return {
        "metric": "quantized KV cache codec GB/s (bytes read + written per pass)",
        "value": min(min(v["quantize_GB/s"], v["dequantize_GB/s"]) for v in widths.values()),
        "unit": UNIT,
        "n_gpus": 1,
        "steps": args.steps,
        "warmup": args.warmup,
        "higher_is_better": True,
        "dtype": "f16",
        "data": "synthetic",
        "config": {"workload": "kv_cache_70b_32k" if G == 80 * 2 * 32768 * 8 else f"kv_cache_{G}_groups",
                   "groups": G, "D": D, "value_is": "slowest width and direction",
                   "l2": f"inputs larger than L2 ({2 * G * D / 1e9:.1f} GB of fp16 per pass)"},
        "roofline": {"bound": "hbm", "peak": peak, "unit": UNIT, "peak_kind": peak_kind},
        "widths": widths,
    }


def run_convert(args, device):
    """EXL2 conversion of one Llama-2-70B gate weight (8192 x 28672 fp16,
    N(0, 0.02) times a per-row power of two in 2^-2 .. 2^2 and a per-segment
    one in 2^-3 .. 2^3, a random input permutation): the RTN error table on the GPU, the bits solve on the host
    for 4.0 bpw, the RTN quantisation on the GPU. CUDA events around `--steps`
    launches after `--warmup` for the two kernels; wall time for the solve."""
    import torch

    import __graft_entry__
    __graft_entry__.build()
    import quantized_weight_exq_gb300 as exq

    torch.cuda.set_device(device)
    peak, peak_kind = measured_peaks()
    K, N = synth.LLAMA2_70B_SHAPES["gate"]
    gen = torch.Generator(device=device)
    gen.manual_seed(5)
    W = (torch.randn(K, N, device=device, generator=gen) * 0.02 *
         torch.exp2(torch.randint(-2, 3, (K, 1), device=device, generator=gen).float())).half()
    perm = torch.randperm(K, device=device, generator=gen).to(torch.int32)
    # loudness per stored segment (its 32 input rows), so that the solve has something to allocate
    loud = torch.exp2(torch.randint(-3, 4, (K // 32,), device=device, generator=gen).float())
    rows = perm.long()
    W[rows] = (W[rows].float() * loud.repeat_interleave(32)[:, None]).half()

    def timed(fn):
        for _ in range(args.warmup):
            fn()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(args.steps):
            fn()
        e1.record()
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) * 1000 / args.steps

    err = exq.exq_measure_exl2(W, perm)
    m_us = timed(lambda: exq.exq_measure_exl2(W, perm))
    t0 = time.perf_counter()
    bits = exq.exq_solve_exl2_bits(err.cpu().numpy().astype(np.float64), 4 * (K // 32))
    solve_ms = (time.perf_counter() - t0) * 1000
    w = exq.exq_quantize_exl2(W, bits, perm)
    q_us = timed(lambda: exq.exq_quantize_exl2(W, bits, perm))
    if exq.exq_get_last_device_error() != 0:
        raise RuntimeError("device error word set during the conversion")
    w_bytes = 2 * K * N
    packed = w.qweight.numel() * 4 + w.scales.numel() * 2
    hist = {int(b): int((bits == b).sum()) for b in synth.EXL2_BITS}
    return {
        "metric": "EXL2 conversion GB/s (fp16 weight bytes read; quantise: + packed bytes written)",
        "value": round((w_bytes + packed) / q_us / 1e3, 1),
        "unit": UNIT,
        "n_gpus": 1,
        "steps": args.steps,
        "warmup": args.warmup,
        "higher_is_better": True,
        "dtype": "f16 in, fp32 decisions",
        "data": "synthetic",
        "config": {"workload": "convert_70b_gate_4p0bpw", "K": K, "N": N, "value_is": "quantise",
                   "l2": "inputs larger than L2 (470 MB of fp16)"},
        "roofline": {"bound": "hbm", "peak": peak, "unit": UNIT, "peak_kind": peak_kind},
        "measure": {"us": round(m_us, 1), "GB/s": round(w_bytes / m_us / 1e3, 1),
                    "frac": round(w_bytes / m_us / 1e3 / peak, 4), "widths_tried": 6},
        "solve": {"ms": round(solve_ms, 2), "segments": K // 32, "budget_bits": 4 * (K // 32), "widths": hist},
        "quantize": {"us": round(q_us, 1), "GB/s": round((w_bytes + packed) / q_us / 1e3, 1),
                     "frac": round((w_bytes + packed) / q_us / 1e3 / peak, 4)},
    }


def max_over_ranks(times, world, device=None):
    """The slowest rank's times: every rank waits for all of them (all-reduce
    MAX over the process group; a CPU tensor under gloo)."""
    if world <= 1:
        return list(times)
    import torch
    import torch.distributed as dist
    t = torch.tensor(list(times), device=device, dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(v) for v in t.cpu()]


def job_throughput(bytes_per_step: int, steps: int, t_ms: float, world: int) -> float:
    """Whole-job GB/s: every replica streams bytes_per_step per step, and the
    job takes the slowest rank's time."""
    return world * bytes_per_step * steps / (t_ms * 1e-3) / 1e9


def run_exq(args, rank, world, device):
    import torch

    import __graft_entry__
    __graft_entry__.build()
    import quantized_weight_exq_gb300 as exq

    torch.cuda.set_device(device)
    grouped = not args.ungrouped
    two_level = args.format == "exl2_qscale"
    calls, x_all, y_all = build_stream(exq, torch, args.layers, device, grouped=grouped, two_level=two_level,
                                       sorted_widths=args.segment_order == "sorted")
    per_layer = len(calls) // args.layers
    bytes_per_step = sum(w.packed_bytes for ws_, _, _ in calls for w in ws_)
    n_linears = sum(len(ws_) for ws_, _, _ in calls)
    n_launch = len(calls)
    # kernels per step: the GEMV, plus one act-order gather of x for a call with a permuted layer
    n_kernels = sum(2 if any(w.perm is not None for w in ws_) else 1 for ws_, _, _ in calls)
    # one zero-filled workspace for the whole stream, sized for its largest call
    ws = torch.zeros(max(call_workspace_size(exq, c) for c in calls[:per_layer]), dtype=torch.uint8, device=device)
    torch.cuda.synchronize()

    stream = torch.cuda.Stream(device=device)
    with torch.cuda.stream(stream):
        for c in calls[:per_layer]:      # settle per-kernel attributes before capture
            issue_call(exq, c, ws)
        stream.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=stream):
            for c in calls:
                issue_call(exq, c, ws)
    torch.cuda.synchronize()
    if exq.exq_get_last_device_error() != 0:
        raise RuntimeError("device error word set after warm-up")

    def barrier():
        if world > 1:
            import torch.distributed as dist
            dist.barrier()

    def timed(step_fn, steps):
        ev0 = torch.cuda.Event(enable_timing=True)
        ev1 = torch.cuda.Event(enable_timing=True)
        barrier()
        torch.cuda.synchronize()
        with torch.cuda.stream(stream):
            ev0.record(stream)
            for _ in range(steps):
                step_fn()
            ev1.record(stream)
        torch.cuda.synchronize()
        barrier()
        return ev0.elapsed_time(ev1)  # ms

    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            graph.replay()
    torch.cuda.synchronize()

    sampler = ClockSampler(torch.cuda.current_device())
    time.sleep(0.3)
    t_ms = timed(graph.replay, args.steps)
    clocks = sampler.stop()

    # end to end: activations in from pinned host memory, outputs back, per step
    x_host = torch.empty_like(x_all, device="cpu").pin_memory()
    x_host.copy_(x_all.cpu())
    y_host = torch.empty_like(y_all, device="cpu").pin_memory()

    def e2e_step():
        x_all.copy_(x_host, non_blocking=True)
        graph.replay()
        y_host.copy_(y_all, non_blocking=True)

    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            e2e_step()
    torch.cuda.synchronize()
    t_e2e_ms = timed(e2e_step, args.steps)

    t_ms, t_e2e_ms = max_over_ranks([t_ms, t_e2e_ms], world, device)

    if exq.exq_get_last_device_error() != 0:
        raise RuntimeError("device error word set during the timed region")

    gbs = job_throughput(bytes_per_step, args.steps, t_ms, world)
    e2e_gbs = job_throughput(bytes_per_step, args.steps, t_e2e_ms, world)
    peak, peak_kind = measured_peaks()
    per_gpu = gbs / world
    traffic_ratio = None if two_level else profile_traffic()
    bytes_per_launch = bytes_per_step / n_launch
    result = {
        "metric": METRIC,
        "value": round(gbs, 2),
        "unit": UNIT,
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(t_ms / args.steps, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f16",
        "data": "synthetic",
        "config": {
            "workload": "decode_stream_70b_exl2_4p0bpw" + ("_two_level_scales" if two_level else ""),
            "model_shape": "Llama-2-70B (80 layers x q,k,v,o,gate,up,down)",
            "scales": "4-bit group-scale codes x fp16 column maxima" if two_level else "fp16 per (segment, column)",
            "segment_order": args.segment_order,
            "layers": args.layers,
            "M": 1,
            "bpw": 4.0,
            "bytes_per_step": bytes_per_step,
            "linears_per_step": n_linears,
            "gemv_calls_per_step": n_launch,
            "grouping": "q+k+v and gate+up share x: exq_gemv_multi" if grouped else "one exq_gemv per linear",
            "tokens_per_s": round(1000.0 / (t_ms / args.steps), 2),
            "pct_of_8TBps": round(100 * per_gpu / NOMINAL_HBM_GBS, 2),
            "l2": f"inputs larger than L2 (the packed stream is {bytes_per_step / 1e9:.1f} GB per step)",
            "launch": "one CUDA graph per step, programmatic dependent launch between GEMVs",
            "parallelism": f"replicas x{world}",
        },
        "roofline": {
            "bound": "hbm",
            "achieved": round(per_gpu, 2),
            "peak": peak,
            "peak_kind": peak_kind,
            "unit": "GB/s",
            "frac": round(per_gpu / peak, 4),
            "traffic": None if traffic_ratio is None else round(traffic_ratio * bytes_per_launch),
            "algorithmic_bytes_per_launch": round(bytes_per_launch),
            "kernel": ("gemv_kernel<EXL2_QSCALE, M<=8>" if two_level else "gemv_kernel<EXL2, M<=8>")
                      + " (+ gather_x_kernel per act-order call)",
        },
        "e2e": {
            "value": round(e2e_gbs, 2),
            "unit": UNIT,
            "h2d_bytes_per_step": x_all.numel() * 2,
            "d2h_bytes_per_step": y_all.numel() * 2,
        },
        "gpu_launches": n_kernels * args.steps,
        "clocks": clocks,
    }
    if not args.no_prefill:
        result["prefill"] = prefill_record(exq, torch, device)
    return result


# ----------------------------------------------------------------------------- oracle

def oracle_sample_gbs(seconds_target: float = 12.0, max_linears: int = 48, first_layer: int = 0):
    """Time the CPU oracle (as it stands) on a bounded sample of the stream:
    whole k / v projections (8192 x 1024) of the layers from `first_layer`,
    packed words drawn exactly as in the GPU stream's recipe (numpy side).
    Runs in this process with numpy; returns (GB/s of packed bytes, seconds,
    sample text, bytes)."""
    import oracle as O

    wid = synth.WORKLOAD_IDS[WORKLOAD]
    done_bytes, elapsed, n = 0, 0.0, 0
    layer = first_layer
    while n == 0 or (elapsed < seconds_target and n < max_linears):
        for i in (1, 2):  # k, v
            K, N = LINEARS[i][1]
            bits = bit_mix(layer, i, K)
            off = O.exl2_seg_word_off(bits)
            qw = synth.uniform_words(int(off[-1]) * N, seed=0, workload=wid, layer=7 * layer + i).reshape(-1, N)
            s = synth.fp16_uniform(synth.rng_for(0, wid, 7 * layer + i, 2), 0.002, 0.03, (K // 32, N))
            perm = synth.rng_for(0, wid, 7 * layer + i, 5).permutation(K).astype(np.int32)
            x = synth.activations(1, K, seed=0, workload=wid, layer=7 * layer + i)
            t0 = time.perf_counter()
            W = O.dequant_exl2(qw, off, bits, s.view(np.uint16), perm)
            O.matmul(x, W)
            elapsed += time.perf_counter() - t0
            done_bytes += qw.nbytes + s.nbytes
            n += 1
            if n >= max_linears:
                break
        layer += 1
    return done_bytes / elapsed / 1e9, elapsed, f"{n} whole 8192x1024 k/v projections (EXL2 4.0 bpw, M=1)", done_bytes


def _oracle_worker(first_layer: int):
    g, t, _, b = oracle_sample_gbs(seconds_target=6.0, max_linears=24, first_layer=first_layer)
    return b, t


def oracle_parallel_gbs(workers: int):
    """The same sample split over `workers` processes (spawned: no process of
    this pool is forked from one that touched a GPU), each on its own layers;
    GB/s = all bytes / wall time of the pool."""
    import multiprocessing as mp
    ctx = mp.get_context("spawn")
    with ctx.Pool(workers) as pool:
        pool.map(_oracle_worker_warm, range(workers))  # interpreters and imports up before the clock
        t0 = time.perf_counter()
        res = pool.map(_oracle_worker, [100 + 12 * i for i in range(workers)])
        wall = time.perf_counter() - t0
    return sum(b for b, _ in res) / wall / 1e9, wall


def _oracle_worker_warm(_):
    import oracle  # noqa: F401
    return 0


def cpu_model() -> str:
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except Exception:
        pass
    import platform
    return platform.processor() or platform.machine()


def cpu_baseline_subprocess():
    """The oracle timing in a fresh process: single-threaded, then one
    single-threaded process per host core."""
    env = dict(os.environ, OMP_NUM_THREADS="1", OPENBLAS_NUM_THREADS="1", MKL_NUM_THREADS="1")
    cores = os.cpu_count() or 1
    code = ("import json,sys; sys.path.insert(0, %r); import bench; "
            "g, t, s, _ = bench.oracle_sample_gbs(); p, w = bench.oracle_parallel_gbs(%d); "
            "print(json.dumps([g, t, s, p, w]))") % (ROOT, cores)
    r = subprocess.run([sys.executable, "-c", code], env=env, capture_output=True, text=True, timeout=900, cwd=ROOT)
    if r.returncode != 0:
        return None
    g, t, s, p, w = json.loads(r.stdout.strip().splitlines()[-1])
    return {"value": round(p, 4), "unit": UNIT, "cores": cores, "kind": "oracle",
            "cpu": cpu_model(), "single_thread_value": round(g, 4),
            "sample": f"{cores} single-threaded processes, each on whole 8192x1024 k/v projections of its own "
                      f"layers for about 6 s ({w:.1f} s wall); single thread: {s}, {t:.1f} s; numpy float64"}


def run_reference(args):
    os.environ.setdefault("OMP_NUM_THREADS", "1")
    res = []
    for _ in range(args.warmup):
        oracle_sample_gbs(seconds_target=0.0, max_linears=1)
    t_total, b_total = 0.0, 0.0
    for _ in range(args.steps):
        g, t, _, _ = oracle_sample_gbs(seconds_target=0.0, max_linears=1)
        t_total += t
        b_total += g * t * 1e9
        res.append(g)
    gbs = b_total / t_total / 1e9
    sample = "1 whole 8192x1024 k projection of the 70B EXL2 4.0 bpw stream per step (M=1)"
    return {
        "impl": "reference",
        "metric": METRIC,
        "value": round(gbs, 4),
        "unit": UNIT,
        "n_gpus": args.gpus,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(1000 * t_total / args.steps, 3),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f64",
        "data": "synthetic",
        "config": {"workload": "decode_stream_70b_exl2_4p0bpw", "sample": sample},
        "cpu_baseline": {"value": round(gbs, 4), "unit": UNIT, "cores": 1, "kind": "oracle", "sample": sample},
        "e2e": {"value": round(gbs, 4), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def main():
    args = parse_args()
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))

    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(run_reference(args)), flush=True)
        return

    import torch
    if args.prefill:
        if rank == 0:
            print(json.dumps(run_prefill(args, torch.device("cuda", local))), flush=True)
        return
    if args.convert:
        if rank == 0:
            print(json.dumps(run_convert(args, torch.device("cuda", local))), flush=True)
        return
    if args.kv:
        if rank == 0:
            print(json.dumps(run_kv(args, torch.device("cuda", local))), flush=True)
        return
    if args.dequant:
        if rank == 0:
            print(json.dumps(run_dequant(args, torch.device("cuda", local))), flush=True)
        return
    if args.decode_sweep:
        if rank == 0:
            print(json.dumps(run_decode_sweep(args, torch.device("cuda", local))), flush=True)
        return
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    device = torch.device("cuda", local)
    result = run_exq(args, rank, world, device)
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        result["cpu_baseline"] = cpu_baseline_subprocess()
    if rank == 0:
        print(json.dumps(result), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
