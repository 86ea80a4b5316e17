#!/usr/bin/env python
"""Benchmark of the quantized decode GEMV/GEMM: achieved GB/s, TFLOP/s and fraction of the HBM roofline.

Default workload (one "step" = one decode token through every linear of an 8B-shaped decoder):
32 layers x {q 4096x4096, k 1024x4096, v 1024x4096, o 4096x4096, gate 14336x4096,
up 14336x4096, down 4096x14336}, M = 1, asymmetric INT4 (uint4 codes, fp16 scale, 4-bit
zero, group 128).  Weights are drawn N(0, 0.02) with 0.1 % outliers x20 on the GPU (seeded),
quantized by the library's GPU quantizer and packed once (untimed); x is bf16 N(0, 1), a fresh
row per linear.  The 224 uq_gemm calls of a step are captured in one CUDA graph.  The packed
weights (3.6 GB) exceed L2 (~129 MB), so no flush is needed between steps.

Metric: algorithmic bytes (packed codes + scales + zeros + x + y, each once) per second.  The
same JSON line carries a `sweep` of the other workloads (the batched-decode M sweep, the
8192 x 8192 format sweep and the 70B-shaped two-level INT4 stack), each timed on its own graph.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl uq|reference] [--workload NAME] [--m M]
                    [--gated] [--no-sweep] [--no-cpu-baseline]

Under torchrun each rank runs an independent replica on its own GPU (the path has no
exchange step); value = bytes of all ranks / max-over-ranks time ("weak" scaling).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "quantized decode GEMV/GEMM GB/s and % of HBM roofline vs M (1 GB300)"
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0

_L8 = [("q", 4096, 4096), ("k", 1024, 4096), ("v", 1024, 4096), ("o", 4096, 4096),
       ("gate", 14336, 4096), ("up", 14336, 4096), ("down", 4096, 14336)]
_L70 = [("q", 8192, 8192), ("k", 1024, 8192), ("v", 1024, 8192), ("o", 8192, 8192),
        ("gate", 28672, 8192), ("up", 28672, 8192), ("down", 8192, 28672)]
WORKLOADS = {
    "llama8b-int4a-decode": dict(fmt="INT4_ASYM", group=128, sigma=0.02, outlier_p=0.001, layers=32,
                                 linears=_L8, m=1,
                                 title="8B-shaped decode linears (32 layers x q,k,v,o,gate,up,down), "
                                       "INT4 asym g128, 0.1% outliers x20"),
    "sweep-int4a": dict(fmt="INT4_ASYM", group=128, sigma=0.02, outlier_p=0.0, layers=48,
                        linears=[("gate", 14336, 4096), ("down", 4096, 14336)], m=1,
                        title="batched decode sweep: 14336x4096 and 4096x14336, INT4 asym g128"),
    "int8s-8192": dict(fmt="INT8_SYM", group=128, sigma=0.02, outlier_p=0.0, layers=40,
                       linears=[("w", 8192, 8192)], m=1, title="8192x8192 INT8 sym g128"),
    "int2a-8192": dict(fmt="INT2_ASYM", group=64, sigma=0.02, outlier_p=0.0, layers=100,
                       linears=[("w", 8192, 8192)], m=1, title="8192x8192 INT2 asym g64"),
    "nf4-8192": dict(fmt="NF4", group=64, sigma=0.02, outlier_p=0.0, layers=60,
                     linears=[("w", 8192, 8192)], m=1, title="8192x8192 NF4 g64"),
    "k4-70b-stack": dict(fmt="K4", group=256, sigma=0.015, outlier_p=0.0, layers=8, linears=_L70, m=1,
                         title="70B-shaped decode linear stack (8 layers x 7), two-level INT4"),
    "w4a8-sweep": dict(fmt="INT4_ASYM", group=128, sigma=0.02, outlier_p=0.0, layers=8,
                       linears=[("gate", 14336, 4096), ("down", 4096, 14336)], m=1, mode="w4a8",
                       title="W4A8 (dynamic per-row int8 x, dp4a): 14336x4096 and 4096x14336, INT4 asym g128"),
    "q4_0-8192": dict(fmt="INT4_SYM", group=32, sigma=0.01, outlier_p=0.0, layers=8, linears=[("w", 8192, 8192)],
                      m=1, source="gguf:Q4_0", title="8192x8192 GGUF Q4_0 blocks (repacked, INT4_SYM g32)"),
}
# The sweep carried in the default line: (workload, layers = weight copies per graph, M values).
# Every graph streams more packed weight bytes than L2 holds, so each replay reads them from HBM.
SWEEP = [("sweep-int4a", 8, (1, 2, 4, 8, 16, 32, 64)),
         ("int8s-8192", 8, (1, 16)), ("int2a-8192", 16, (1, 16)), ("nf4-8192", 8, (1, 16)),
         ("k4-70b-stack", 8, (1, 8, 32)), ("w4a8-sweep", 8, (1, 8)), ("q4_0-8192", 8, (1, 16))]
# the decode step again, with each layer's gate and up linears as one gated op (uq_gemm_gated)
SWEEP_GATED = [("llama8b-int4a-decode", 8, (1, 4))]
# linears that read the same input as the linear before them in a decoder layer
SHARES_INPUT_WITH_PREVIOUS = ("k", "v", "up")
BITS = {"INT4_SYM": 4, "INT4_ASYM": 4, "INT8_SYM": 8, "INT2_ASYM": 2, "NF4": 4, "K4": 4}
KT = {"INT4_SYM": 1024, "INT4_ASYM": 1024, "INT8_SYM": 512, "INT2_ASYM": 2048, "NF4": 1024, "K4": 1024}


def launch_groups(names):
    """Indices of the step's linears grouped for launch: a linear whose short name (after the last
    '.') reads the same input as the one before it joins that one's group; groups run in order, the
    members of a group on parallel branches."""
    groups = []
    for i, name in enumerate(names):
        if groups and name.split(".")[-1] in SHARES_INPUT_WITH_PREVIOUS:
            groups[-1].append(i)
        else:
            groups.append([i])
    return groups


def alg_bytes(fmt, group, N, K, M):
    """Algorithmic bytes of one linear: codes + metadata + x + y, each moved once."""
    codes = N * K * BITS[fmt] // 8
    if fmt == "K4":
        meta = N * (K // 256) * 16
    else:
        G = K // group
        meta = N * G * 2
        if fmt == "INT4_ASYM":
            meta += N * ((G + 1) // 2)
        elif fmt == "INT2_ASYM":
            meta += N * G * 2
        elif fmt == "NF4":
            meta += 64
    return codes + meta + 2 * M * K + 2 * M * N


def alg_flops(N, K, M):
    """Multiply-adds of one linear counted as two flops each."""
    return 2 * M * N * K


def kernel_source_hash():
    h = hashlib.sha256()
    d = os.path.join(ROOT, "gemm_uq_gb300", "csrc")
    for name in sorted(os.listdir(d)):
        if name in ("uq_gemv.cuh", "uq_common.cuh"):             # the GEMV kernels' own sources
            with open(os.path.join(d, name), "rb") as f:
                h.update(f.read())
    return h.hexdigest()[:16]


def read_traffic(workload, avg_alg_bytes):
    """DRAM bytes per launch, from the committed ncu summary when it was taken on the current kernel
    sources: the captured launch's DRAM/algorithmic byte ratio times this run's average algorithmic
    bytes per launch (traffic scales with the bytes a launch streams)."""
    path = os.path.join(ROOT, "profiles", f"gemv_{workload}.md")
    if not os.path.exists(path):
        return None
    vals = {}
    for line in open(path):
        if ":" in line and line.strip().startswith("- "):
            k, v = line.strip()[2:].split(":", 1)
            vals[k.strip()] = v.strip()
    if vals.get("kernel_source_sha") != kernel_source_hash():
        return None
    try:
        return round(float(vals["dram_over_algorithmic"]) * avg_alg_bytes)
    except (KeyError, ValueError):
        return None


def read_share(workload):
    """Share of the step's device time in the dominant kernel, from the committed ncu launch list."""
    path = os.path.join(ROOT, "profiles", f"launches_{workload}.md")
    if not os.path.exists(path):
        return None
    for line in open(path):
        if line.strip().startswith("- dominant_share:"):
            try:
                return float(line.split(":", 1)[1])
            except ValueError:
                return None
    return None


def dominant_kernel(fmt, group, M, shapes):
    """Name of the kernel template the library dispatches for this workload's linears (uq_gemm's
    automatic routing: the mma.sync GEMM for 9..15 rows of the 4-bit / 2-bit formats and for K4, the
    tensor cores for other blocks of 16..64 rows, the mma.sync GEMVs below: per-warp rings for one
    row of the 4-bit flat formats, the copy-warp ring otherwise)."""
    mma_fmt = fmt in ("INT4_SYM", "INT4_ASYM", "INT2_ASYM", "K4")        # the mma.sync GEMM's formats
    tc_ok = M >= 16 and all(K % KT[fmt] == 0 for _, K in shapes)
    if mma_fmt and M >= 9 and (M <= 15 or fmt == "K4" or not tc_ok):
        mb = min(M, 64)
        return f"gemm_mma_kernel<{fmt},{16 if mb <= 16 else (32 if mb <= 32 else 64)} columns>"
    if tc_ok:
        mpad = (min(M, 64) + 15) // 16 * 16
        return f"tc_kernel<{fmt},{mpad}>"
    gs = 32 if fmt == "K4" else group
    if M == 1 and fmt in ("INT4_SYM", "INT4_ASYM"):
        return f"gemv_warp_kernel<{fmt},GB={gs // 16}>"
    return f"gemv_mma_kernel<{fmt},GB={gs // 16}>"


def kernels_per_call(fmt, group, M, N, K):
    """Kernel launches one uq_gemm call of this shape makes on the current device, as the library
    itself counts them."""
    import gemm_uq_gb300 as uq
    return uq.gemm_kernel_count(M, N, K, group, fmt)


def measured_peaks():
    """(HBM GB/s, bf16 TFLOP/s burst, source) from MEASURED_PEAKS.json, else the fallback figures."""
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        try:
            d = json.load(open(path))
            return float(d["hbm_gbs"]), float(d.get("bf16_tflops", FALLBACK_BF16_TFLOPS)), "measured"
        except Exception:
            pass
    return FALLBACK_HBM_GBS, FALLBACK_BF16_TFLOPS, "fallback"


def roofline_time_s(nbytes, flops, hbm_gbs, tflops):
    """The roofline time: the slower of the bytes at HBM bandwidth and the flops at bf16 dense peak."""
    return max(nbytes / (hbm_gbs * 1e9), flops / (tflops * 1e12))


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 200 ms while the timed region runs."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.f = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=self.f, stderr=subprocess.DEVNULL)
        except (FileNotFoundError, OSError):
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *a):
        if self.proc is not None:
            time.sleep(0.25)
            self.proc.terminate()
            self.proc.wait(timeout=5)

    def summary(self):
        self.f.flush()
        rows = []
        with open(self.f.name) as fh:
            for line in fh:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.unlink(self.f.name)
        if not rows:
            return None
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows)}


def max_over_ranks(values, dist, device):
    """Element-wise maximum of per-rank timings (identity without a process group)."""
    if not dist:
        return list(values)
    import torch
    t = torch.tensor(list(values), device=device, dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(v) for v in t]


# ---------------------------------------------------------------------------------------------
def build_weights(spec, dev, layers=None, seed_base=12345):
    """Quantize and pack every linear of the workload on the GPU; returns per-linear records."""
    import torch
    import gemm_uq_gb300 as uq
    fmt, group = spec["fmt"], spec["group"]
    gen = torch.Generator(device=dev)
    recs = []
    cb = None
    if fmt == "NF4":
        import numpy as np
        cb = torch.from_numpy(np.loadtxt(os.path.join(ROOT, "tests", "golden", "nf4_codebook.txt"),
                                         dtype=np.float64).astype(np.float32)).to(dev)
    idx = 0
    for layer in range(layers or spec["layers"]):
        for name, N, K in spec["linears"]:
            gen.manual_seed(seed_base + idx)
            if spec.get("source") == "gguf:Q4_0":
                # random GGUF Q4_0 blocks (any byte pattern is a valid block) with an fp16 d, repacked
                raw = torch.randint(0, 256, (N, K // 32, 18), generator=gen, device=dev, dtype=torch.int32).to(torch.uint8)
                d = (torch.randn((N, K // 32), generator=gen, device=dev) * spec["sigma"]).half().view(torch.uint8)
                raw[..., 0:2] = d.view(N, K // 32, 2)
                wq, scales = uq.pack_gguf(raw.contiguous(), "Q4_0", N, K)
                del raw, d
                recs.append(dict(name=f"L{layer}.{name}", N=N, K=K, wq=wq, scales=scales, zc=None))
                idx += 1
                continue
            w = torch.randn((N, K), generator=gen, device=dev, dtype=torch.float32) * spec["sigma"]
            if spec["outlier_p"] > 0:
                mask = torch.rand((N, K), generator=gen, device=dev) < spec["outlier_p"]
                w = torch.where(mask, w * 20.0, w)
                del mask
            if fmt == "K4":
                codes, d, dmin, sc, mm = uq.quantize_k4(w)
                scales = uq.pack_kmeta(d, dmin, sc, mm)
                zc = None
                del d, dmin, sc, mm
            else:
                codes, scales, zeros = uq.quantize(w, group, fmt, codebook=cb)
                zc = uq.pack_zeros(zeros) if fmt == "INT4_ASYM" else (zeros if fmt == "INT2_ASYM" else cb)
            del w
            wq = uq.pack_layout(codes, group, fmt)
            del codes
            recs.append(dict(name=f"L{layer}.{name}", N=N, K=K, wq=wq, scales=scales, zc=zc))
            idx += 1
    torch.cuda.synchronize()
    return recs


def gated_bytes(fmt, group, N, K, M):
    """Algorithmic bytes of the gated projection: both weights' codes and metadata, x once, h once."""
    w = alg_bytes(fmt, group, N, K, 0)
    return 2 * w + 2 * M * K + 2 * M * N


def step_ops(recs, gated):
    """The step's ops in launch order: one uq_gemm per linear, except that with `gated` a layer's gate
    linear and the up linear right after it (same shape) form one uq_gemm_gated op."""
    ops = []
    i = 0
    while i < len(recs):
        r = recs[i]
        nxt = recs[i + 1] if i + 1 < len(recs) else None
        if (gated and r["name"].endswith(".gate") and nxt is not None and nxt["name"].endswith(".up")
                and (nxt["N"], nxt["K"]) == (r["N"], r["K"])):
            ops.append(dict(kind="gated", recs=[r, nxt], name=r["name"][:-len("gate")] + "gate_up",
                            N=r["N"], K=r["K"]))
            i += 2
        else:
            ops.append(dict(kind="gemm", recs=[r], name=r["name"], N=r["N"], K=r["K"]))
            i += 1
    return ops


class Step:
    """One pass over every linear of a workload at M rows: x and output buffers, the launch order (ops
    reading the same input on parallel branches), and its CUDA graph.  With `gated`, a layer's gate
    and up linears are one op: uq_gemm_gated, h = silu(x Wg^T) * (x Wu^T)."""

    def __init__(self, recs, fmt, group, M, dev, stream, seed, gated=False, mode="gemm"):
        import torch
        self.recs, self.fmt, self.group, self.M, self.stream = recs, fmt, group, M, stream
        self.mode = mode                          # "gemm" (bf16 x) or "w4a8" (per-row int8 x)
        self.ops = step_ops(recs, gated)
        x_sizes = [M * op["K"] for op in self.ops]
        y_sizes = [M * op["N"] for op in self.ops]
        # x of every op in one device buffer (the end-to-end leg copies it with one memcpy)
        self.xbuf = torch.empty(sum(x_sizes), dtype=torch.bfloat16, device=dev)
        self.ybuf = torch.empty(sum(y_sizes), dtype=torch.bfloat16, device=dev)
        g = torch.Generator(device=dev)
        g.manual_seed(seed)
        self.xbuf.copy_(torch.randn(self.xbuf.numel(), generator=g, device=dev,
                                    dtype=torch.float32).to(torch.bfloat16))
        self.io = []
        ox = oy = 0
        for xs, ys in zip(x_sizes, y_sizes):
            self.io.append((self.xbuf[ox:ox + xs], self.ybuf[oy:oy + ys]))
            ox += xs
            oy += ys
        self.bytes = sum(gated_bytes(fmt, group, op["N"], op["K"], M) if op["kind"] == "gated"
                         else alg_bytes(fmt, group, op["N"], op["K"], M) for op in self.ops)
        self.flops = sum(alg_flops(r["N"], r["K"], M) for r in recs)
        self.groups = launch_groups([op["name"] for op in self.ops])
        width = max(len(gr) for gr in self.groups)
        self.side = [torch.cuda.Stream(device=dev) for _ in range(width - 1)]
        self.graph = None

    def launch(self, i, st):
        import gemm_uq_gb300 as uq
        op = self.ops[i]
        x, y = self.io[i]

        def ptrs(r):
            return (r["wq"].data_ptr(), r["scales"].data_ptr(), r["zc"].data_ptr() if r["zc"] is not None else 0)

        if op["kind"] == "gated":
            uq.gemm_gated_ptrs(x.data_ptr(), ptrs(op["recs"][0]), ptrs(op["recs"][1]), y.data_ptr(), self.M,
                               op["N"], op["K"], self.group, self.fmt, st.cuda_stream)
        else:
            w, sc, zc = ptrs(op["recs"][0])
            f = uq.gemm_w4a8_ptrs if self.mode == "w4a8" else uq.gemm_ptrs
            f(x.data_ptr(), w, sc, zc, y.data_ptr(), self.M, op["N"], op["K"], self.group, self.fmt, st.cuda_stream)

    def issue(self):
        import torch
        for gr in self.groups:
            if len(gr) > 1:
                fork = torch.cuda.Event()
                fork.record(self.stream)
                for j, i in enumerate(gr[1:]):
                    self.side[j].wait_event(fork)
                    self.launch(i, self.side[j])
            self.launch(gr[0], self.stream)
            for j in range(len(gr) - 1):
                join = torch.cuda.Event()
                join.record(self.side[j])
                self.stream.wait_event(join)

    def capture(self):
        import torch
        with torch.cuda.stream(self.stream):
            for _ in range(2):
                self.issue()               # grows the per-stream workspaces outside capture
        torch.cuda.synchronize()
        self.graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(self.graph, stream=self.stream):
            self.issue()
        torch.cuda.synchronize()
        return self

    def replay(self, n):
        import torch
        with torch.cuda.stream(self.stream):
            for _ in range(n):
                self.graph.replay()

    def time(self, warmup, steps):
        """Device time per replay (ms): CUDA events on the launching stream, synchronized on both sides."""
        import torch
        self.replay(warmup)
        torch.cuda.synchronize()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(self.stream)
        self.replay(steps)
        e1.record(self.stream)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / steps

    def launches(self):
        import gemm_uq_gb300 as uq
        n = 0
        for op in self.ops:
            if op["kind"] == "gated":
                n += uq.gemm_gated_kernel_count(self.M, op["N"], op["K"], self.group, self.fmt)
            elif self.mode == "w4a8":
                n += uq.gemm_w4a8_kernel_count(self.M, op["N"], op["K"], self.group, self.fmt)
            else:
                n += kernels_per_call(self.fmt, self.group, self.M, op["N"], op["K"])
        return n


def run_sweep(dev, stream, hbm, tf):
    """The M sweep, the format sweep, the 70B-shaped stack and the gated decode step, each point on
    its own graph."""
    import torch
    out = []
    for wl, layers, ms, gated in [p + (False,) for p in SWEEP] + [p + (True,) for p in SWEEP_GATED]:
        spec = WORKLOADS[wl]
        fmt, group = spec["fmt"], spec["group"]
        recs = build_weights(spec, dev, layers=layers, seed_base=20000)
        shapes = sorted({(r["N"], r["K"]) for r in recs})
        for M in ms:
            mode = spec.get("mode", "gemm")
            st = Step(recs, fmt, group, M, dev, stream, seed=4242 + M, gated=gated, mode=mode).capture()
            probe = st.time(3, 2)
            reps = int(min(200, max(5, 25.0 / max(probe, 1e-3))))
            ms_ = st.time(3, reps)
            t_roof = roofline_time_s(st.bytes, st.flops, hbm, tf)
            out.append({"workload": wl, "fmt": fmt, "group": group, "M": M, "linears": len(recs),
                        "ops": len(st.ops), "gated": gated,
                        "shapes": [f"{n}x{k}" for n, k in shapes],
                        "GB/s": round(st.bytes / (ms_ * 1e-3) / 1e9, 1),
                        "TFLOP/s": round(st.flops / (ms_ * 1e-3) / 1e12, 2),
                        "frac": round(t_roof / (ms_ * 1e-3), 4),
                        "bound": "hbm" if st.bytes / (hbm * 1e9) >= st.flops / (tf * 1e12) else "tensor",
                        "us_per_linear": round(ms_ * 1e3 / len(recs), 2),
                        "kernel": (f"gemv_mma_kernel<{fmt},GB={group // 16},A8>" if mode == "w4a8"
                                   else dominant_kernel(fmt, group, M, shapes)),
                        "launches": st.launches(),
                        "reps": reps})
            del st
        del recs
        torch.cuda.empty_cache()
    out.extend(run_rope_points(dev, stream, hbm))
    return out


def run_rope_points(dev, stream, hbm):
    """The fused RMSNorm + RoPE: a bulk case (8192 rows of 4096, bandwidth) and a decode row (latency)."""
    import torch
    import gemm_uq_gb300 as uq
    out = []
    D, hd, max_pos = 4096, 128, 8192
    table = uq.rope_table(max_pos, hd, 500000.0, device=dev)
    g = torch.Generator(device=dev)
    g.manual_seed(31337)
    gamma = (1.0 + 0.1 * torch.randn(D, generator=g, device=dev)).to(torch.bfloat16)
    for M, copies in ((8192, 4), (1, 64)):
        xs = [torch.randn((M, D), generator=g, device=dev).to(torch.bfloat16) for _ in range(copies)]
        ys = [torch.empty_like(x) for x in xs]
        pos = torch.randint(0, max_pos, (M,), generator=g, device=dev, dtype=torch.int32)
        with torch.cuda.stream(stream):
            for x, y in zip(xs, ys):
                uq.rmsnorm_rope(x, gamma, pos, table, hd, 1e-5, y=y, stream=stream)
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=stream):
            for x, y in zip(xs, ys):
                uq.rmsnorm_rope(x, gamma, pos, table, hd, 1e-5, y=y, stream=stream)
        with torch.cuda.stream(stream):
            for _ in range(3):
                graph.replay()
        torch.cuda.synchronize()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        reps = 20
        e0.record(stream)
        with torch.cuda.stream(stream):
            for _ in range(reps):
                graph.replay()
        e1.record(stream)
        torch.cuda.synchronize()
        t = e0.elapsed_time(e1) * 1e-3 / (reps * copies)
        nbytes = 2 * M * D * 2 + D * 2 + M * 4 + M * (hd // 2) * 8       # x, y, gamma, positions, table rows
        out.append({"workload": "rmsnorm-rope", "M": M, "D": D, "head_dim": hd, "GB/s": round(nbytes / t / 1e9, 1),
                    "frac": round(nbytes / t / 1e9 / hbm, 4), "us_per_call": round(t * 1e6, 2),
                    "kernel": "rmsnorm_rope_kernel", "launches": copies})
        del xs, ys
    return out


def run_uq(args, rank, world, dist):
    import torch
    import gemm_uq_gb300 as uq

    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    spec = dict(WORKLOADS[args.workload])
    fmt, group = spec["fmt"], spec["group"]
    M = args.m if args.m else spec["m"]
    recs = build_weights(spec, dev, layers=args.layers or None)
    stream = torch.cuda.Stream(device=dev)
    # consecutive linears of a decode step read fixed weights: let each launch stream its weights
    # while the previous one drains (uq_set_launch_overlap)
    uq.set_launch_overlap(not args.no_overlap)
    step = Step(recs, fmt, group, M, dev, stream, seed=777 + rank, gated=args.gated,
                mode=spec.get("mode", "gemm")).capture()

    step.replay(args.warmup)
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    with ClockSampler(local) as clk:
        torch.cuda.synchronize()
        if dist:
            dist.barrier()
        t_start.record(stream)
        step.replay(args.steps)
        t_end.record(stream)
        torch.cuda.synchronize()
    if dist:
        dist.barrier()
    ms = t_start.elapsed_time(t_end)
    clocks = clk.summary()

    # end to end through the public API: H2D of every x, the step, D2H of every y, each step
    xh = torch.empty(step.xbuf.numel(), dtype=torch.bfloat16, pin_memory=True)
    yh = torch.empty(step.ybuf.numel(), dtype=torch.bfloat16, pin_memory=True)
    xh.copy_(step.xbuf.cpu())
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)

    def e2e_step():
        step.xbuf.copy_(xh, non_blocking=True)
        step.graph.replay()
        yh.copy_(step.ybuf, non_blocking=True)

    with torch.cuda.stream(stream):
        for _ in range(max(3, args.warmup)):
            e2e_step()
    torch.cuda.synchronize()
    e0.record(stream)
    with torch.cuda.stream(stream):
        for _ in range(args.steps):
            e2e_step()
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = e0.elapsed_time(e1)

    ms, e2e_ms = max_over_ranks([ms, e2e_ms], dist, dev)
    info = dict(bytes=step.bytes, flops=step.flops, linears=len(recs), ops=len(step.ops), launches=step.launches(),
                gated=any(op["kind"] == "gated" for op in step.ops),
                width=len(step.side) + 1, h2d=step.xbuf.numel() * 2, d2h=step.ybuf.numel() * 2,
                shapes=sorted({(r["N"], r["K"]) for r in recs}), layers=len(recs) // len(spec["linears"]))
    sweep = None
    if world == 1 and not args.no_sweep:
        del step, recs
        torch.cuda.empty_cache()
        sweep = run_sweep(dev, stream, *measured_peaks()[:2])
    if rank != 0:
        return
    out = report(args, spec, M, world, ms, e2e_ms, clocks, info, sweep)
    if world == 1 and not args.no_cpu_baseline:
        out["cpu_baseline"] = cpu_baseline(args.workload, M)
    print(json.dumps(out), flush=True)


def report(args, spec, M, world, ms, e2e_ms, clocks, info, sweep):
    """The JSON line of the GPU arm."""
    fmt, group = spec["fmt"], spec["group"]
    hbm, tf, peak_src = measured_peaks()
    step_s = ms * 1e-3 / args.steps
    value = info["bytes"] * world / step_s / 1e9
    achieved = info["bytes"] / step_s / 1e9
    t_roof = roofline_time_s(info["bytes"], info["flops"], hbm, tf)
    share = read_share(args.workload) if M == spec["m"] and not args.layers else None
    traffic = read_traffic(args.workload, info["bytes"] / info["ops"]) if M == spec["m"] else None
    return {
        "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms / args.steps, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None,
        "dtype": f"bf16 x {fmt.lower()} -> fp32 acc",
        "data": "synthetic (seeded N(0,sigma) weights quantized on the GPU; bf16 N(0,1) x)",
        "config": {"workload": args.workload, "description": spec["title"], "fmt": fmt, "group": group, "M": M,
                   "layers": info["layers"], "linears_per_step": info["linears"], "bytes_per_step": info["bytes"],
                   "flops_per_step": info["flops"], "parallelism": f"replicas x{world}",
                   "l2": "no flush: packed weights per step exceed L2 (%.2f GB)" % (info["bytes"] / 1e9),
                   "ops_per_step": info["ops"],
                   "launch": "one CUDA graph per step" + (
                       "; ops reading the same input (q, k, v) on parallel branches" if info["width"] > 1 else "")
                   + ("; each layer's gate and up as one fused uq_gemm_gated op (h = silu(x Wg^T) * (x Wu^T))"
                      if info["gated"] else ""),
                   "launch_overlap": not args.no_overlap},
        "tflops": round(info["flops"] * world / step_s / 1e12, 4),
        "gpu_launches": info["launches"] * args.steps,
        "e2e": {"value": round(info["bytes"] * args.steps * world / (e2e_ms * 1e-3) / 1e9, 2), "unit": "GB/s",
                "h2d_bytes_per_step": info["h2d"], "d2h_bytes_per_step": info["d2h"]},
        # the step is the dominant kernel's launches (plus the small second passes of the split
        # linears); its algorithmic bytes over the step's device time can therefore not exceed what
        # the kernel moves, and the ncu launch list gives the kernel's share of that time
        "roofline": {"bound": "hbm" if info["bytes"] / (hbm * 1e9) >= info["flops"] / (tf * 1e12) else "tensor",
                     "achieved": round(achieved, 1), "peak": hbm, "unit": "GB/s",
                     "frac": round(t_roof / step_s, 4), "traffic": traffic,
                     "peak_source": f"{peak_src} HBM copy bandwidth (burst)",
                     "kernel": dominant_kernel(fmt, group, M, info["shapes"]),
                     "kernel_share_of_step": share,
                     "timing": "algorithmic bytes per step / step device time (CUDA events over the timed region)"},
        "clocks": clocks,
        "sweep": sweep,
    }


# ---------------------------------------------------------------------------------------------
# the oracle legs: cpu_baseline of the GPU arm and the reference arm

def _oracle_sample(spec, M, rows_per_linear):
    """Oracle inputs for a bounded sample: the first rows of one layer's linears (quantized untimed)."""
    from oracle import quant as oquant
    from oracle.nf4 import nf4_codebook
    from synth import activations, normal_weights
    cb = nf4_codebook() if spec["fmt"] == "NF4" else None
    items = []
    for i, (name, N, K) in enumerate(spec["linears"]):
        n = min(N, rows_per_linear)
        w = normal_weights(9000 + i, n, K, spec["sigma"], outlier_p=spec["outlier_p"], outlier_mult=20.0)
        qz = oquant.quantize(w, spec["fmt"], spec["group"], codebook=cb)
        x = activations(9000 + i, M, K)
        items.append((qz, x, alg_bytes(spec["fmt"], spec["group"], n, K, M)))
    return items


def _oracle_pass(items):
    from oracle import gemm as ogemm
    for qz, x, _ in items:
        ogemm.quantized_gemm(x, qz)


def _threads_in_use():
    """Threads the oracle's BLAS calls may use: the thread-count variables if set, else the CPUs this
    process may run on (NumPy's elementwise dequantization itself runs on one thread)."""
    for var in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS"):
        if os.environ.get(var, "").isdigit():
            return int(os.environ[var])
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count()


def oracle_leg(workload, M, target_s, rows_per_linear):
    """Times the oracle (as it stands) on a bounded sample; returns the cpu_baseline fields."""
    spec = WORKLOADS[workload]
    items = _oracle_sample(spec, M, rows_per_linear)
    nbytes = sum(b for _, _, b in items)
    _oracle_pass(items)
    t0 = time.perf_counter()
    passes = 0
    while True:
        _oracle_pass(items)
        passes += 1
        el = time.perf_counter() - t0
        if el >= target_s:
            break
    return {"value": round(nbytes * passes / el / 1e9, 4), "unit": "GB/s", "cores": _threads_in_use(),
            "kind": "oracle",
            "sample": f"first {rows_per_linear} rows of each of the {len(items)} linears of one layer, M={M}, "
                      f"{passes} passes of the float64 dequantize-then-matmul ({el:.1f} s)"}


def cpu_baseline(workload, M, target_s=10.0, rows_per_linear=512):
    """The oracle timed twice in fresh processes (the BLAS thread count is fixed at start-up): on one
    thread and on every core this process may use."""
    legs = {}
    for name, threads in (("single_thread", 1), ("all_cores", None)):
        env = dict(os.environ)
        for var in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
            if threads:
                env[var] = str(threads)
            else:
                env.pop(var, None)
        r = subprocess.run([sys.executable, os.path.abspath(__file__), "--oracle-leg", workload, "--m", str(M),
                            "--oracle-seconds", str(target_s), "--oracle-rows", str(rows_per_linear)],
                           env=env, capture_output=True, text=True, timeout=600)
        if r.returncode != 0:
            legs[name] = {"error": r.stderr.strip().splitlines()[-1:] or ["oracle leg failed"]}
            continue
        legs[name] = json.loads(r.stdout.strip().splitlines()[-1])
    out = dict(legs.get("all_cores", {}))
    out["single_thread"] = legs.get("single_thread")
    out["cpus_on_host"] = os.cpu_count()
    return out


def run_reference(args, rank, world):
    """The oracle as the reference arm: each step is a bounded sample of the same workload."""
    if rank != 0:
        return
    spec = WORKLOADS[args.workload]
    M = args.m if args.m else spec["m"]
    items = _oracle_sample(spec, M, rows_per_linear=256)
    nbytes = sum(b for _, _, b in items)
    for _ in range(args.warmup):
        _oracle_pass(items)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        _oracle_pass(items)
    el = time.perf_counter() - t0
    value = nbytes * args.steps / el / 1e9
    sample = f"first 256 rows of each of the {len(items)} linears of one layer, M={M} (float64 oracle)"
    out = {"impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s", "n_gpus": world,
           "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(el / args.steps * 1e3, 3),
           "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
           "data": "synthetic", "config": {"workload": args.workload, "description": spec["title"],
                                           "fmt": spec["fmt"], "group": spec["group"], "M": M},
           "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": _threads_in_use(),
                            "cpus_on_host": os.cpu_count(), "kind": "oracle", "sample": sample},
           "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(out), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["uq", "reference"], default="uq")
    ap.add_argument("--workload", choices=sorted(WORKLOADS), default="llama8b-int4a-decode")
    ap.add_argument("--m", type=int, default=0, help="override the batch rows M")
    ap.add_argument("--layers", type=int, default=0, help="override the number of layers (profiling runs)")
    ap.add_argument("--no-sweep", action="store_true", help="leave the sweep workloads out of the line")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-overlap", action="store_true", help="launch without programmatic dependent launch")
    ap.add_argument("--gated", action="store_true",
                    help="each layer's gate and up linears as one uq_gemm_gated op instead of two uq_gemm")
    ap.add_argument("--oracle-leg", default=None, help=argparse.SUPPRESS)
    ap.add_argument("--oracle-seconds", type=float, default=10.0, help=argparse.SUPPRESS)
    ap.add_argument("--oracle-rows", type=int, default=512, help=argparse.SUPPRESS)
    args = ap.parse_args()
    if args.oracle_leg:
        spec = WORKLOADS[args.oracle_leg]
        print(json.dumps(oracle_leg(args.oracle_leg, args.m or spec["m"], args.oracle_seconds, args.oracle_rows)))
        return
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if args.impl == "reference":
        run_reference(args, rank, world)
        return
    dist = None
    if world > 1:
        import torch
        import torch.distributed as tdist
        torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", "0")))
        tdist.init_process_group("nccl")
        dist = tdist
    try:
        run_uq(args, rank, world, dist)
    finally:
        if dist:
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
