#!/usr/bin/env python3
"""Benchmark of the fused dequant-GEMV (decode, batch 1) on one GB300 per rank.

Workload (headline): the 3-bit super-block GEMV of an 11008x4096 weight matrix (110-byte / 256-weight
super-blocks, Laplace(0, 0.015) weights, seed 0), fp16 activations ~ N(0, 1), fp32 output. One step = one GEMV
over each of R distinct packed copies of that matrix with R distinct activation vectors (R chosen so the copies
total well over the 129 MB L2, so every step streams its weights from HBM). Metric: effective weight GB/s =
packed bytes (codes + scales + row padding) / time, the definition of the DBHOO-CIM article (pwwt.cn/news/
4452170) §4.4 and of the 2/3/5/6-bit article (lpnh.cn/news/2857666) §1.2; also reported as a fraction of the
measured HBM copy bandwidth.

Extra (rank 0): a 7B-Llama-shaped decode step (32 layers x {q,k,v,o 4096x4096, gate/up 11008x4096,
down 4096x11008}) per super-block format, as tokens/s-equivalent and GB/s.

`--impl reference` times the CPU oracle (the plain C++ implementation the tests check against) on the same
workload, on the host cores.
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

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "fused dequant-GEMV effective weight GB/s & % of GB300 HBM peak; decode tok/s equiv"
N_ROWS, K_COLS = 11008, 4096
WORKLOAD = "3-bit super-block fused dequant-GEMV, W 11008x4096 (Laplace(0,0.015), seed 0), batch-1 fp16 x, fp32 y"
FORMAT_DESC = "Q3S (110 B / 256 weights)"
FALLBACK_HBM, FALLBACK_BF16 = 6800.0, 1900.0
# The decode arithmetic: activations rounded to int16 per 16-element half (step max|x| / 32767), times the unsigned
# integer codes by dp2a into exact int32 sums per half, then fp32 scaling and fp32 accumulation.
DTYPE = "int16 x uint8 (dp2a) -> int32 per 16 activations, fp32 scale and accumulate"

# dram__bytes_read.sum + dram__bytes_write.sum of one headline launch from an ncu capture (the third gemv1_kernel
# launch of `python bench.py --ncu-case gemv --fmt Q3S --N 11008 --K 4096 --copies 12`), valid only for the CUDA
# sources whose digest is recorded here.
TRAFFIC = {"csrc_digest": "7d7320a8adfcbc79", "bytes_per_launch": 19432192}


def csrc_digest() -> str:
    """Digest of the sources the batch-1 decode kernel's code comes from (its own file and the device helpers): a
    traffic figure measured on other sources is not reported."""
    h = hashlib.sha256()
    d = os.path.join(ROOT, "bit_weight_quantized_qpack_gb300", "csrc")
    for f in ("qpack_gemv.cu", "qpack_dev.cuh"):
        with open(os.path.join(d, f), "rb") as fh:
            h.update(f.encode() + fh.read())
    return h.hexdigest()[:16]


def measured_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            m = json.load(f)
        return float(m["hbm_gbs"]), float(m["bf16_tflops"]), "measured"
    except Exception:
        return FALLBACK_HBM, FALLBACK_BF16, "fallback"


class ClockSampler:
    """nvidia-smi clock / throttle sampling while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu_index = gpu_index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu_index), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self._t = threading.Thread(target=self._read, daemon=True)
            self._t.start()
        except Exception:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        sm, smax, reasons, power = [], [], set(), []
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
                power.append(float(parts[3]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax), "reasons": sorted(reasons),
                "samples": len(sm), "power_w_max": max(power) if power else None}


def dist_setup(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def cpu_oracle_gemv_sample(packed_np, x_np, seconds_target=10.0, max_seconds=30.0):
    """Time the oracle's fp64 GEMV over the whole matrix with every host core, repeated ~10-30 s."""
    import oracle
    n = os.cpu_count() or 1
    wbytes = packed_np.nbytes
    reps, t0 = 0, time.perf_counter()
    while True:
        oracle.gemv(oracle.Q3S, N_ROWS, K_COLS, packed_np, None, x_np, nthreads=n)
        reps += 1
        el = time.perf_counter() - t0
        if el >= seconds_target or el * (reps + 1) / reps > max_seconds:
            break
    return {"value": wbytes * reps / el / 1e9, "unit": "GB/s", "cores": n, "kind": "oracle",
            "sample": f"{reps} full 11008x4096 3-bit GEMV(s) ({wbytes} packed bytes each), fp64 oracle, "
                      f"{n} threads, {el:.1f} s"}


def run_reference(args, world, rank):
    """The oracle (CPU) on the same workload: one full 11008x4096 GEMV per step, all host cores."""
    if rank != 0:
        return 0
    import numpy as np
    import oracle
    from bit_weight_quantized_qpack_gb300 import synth
    W = synth.laplace((N_ROWS, K_COLS), 0.015, seed=0)
    packed, _, _ = oracle.quantize_pack(oracle.Q3S, W.numpy())
    x = synth.normal((K_COLS,), 1.0, seed=1).half().numpy().view(np.uint16)
    n = os.cpu_count() or 1
    for _ in range(args.warmup):
        oracle.gemv(oracle.Q3S, N_ROWS, K_COLS, packed, None, x, nthreads=n)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle.gemv(oracle.Q3S, N_ROWS, K_COLS, packed, None, x, nthreads=n)
    el = time.perf_counter() - t0
    v = packed.nbytes * args.steps / el / 1e9
    line = {"impl": "reference", "metric": METRIC, "value": v, "unit": "GB/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": el / args.steps * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": WORKLOAD, "format": FORMAT_DESC, "N": N_ROWS, "K": K_COLS, "batch": 1,
                       "bytes_per_gemv": int(packed.nbytes)},
            "cpu_baseline": {"value": v, "unit": "GB/s", "cores": n, "kind": "oracle",
                             "sample": f"{args.steps} full GEMVs, fp64 oracle, {n} threads"},
            "e2e": {"value": v, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def decode_7b_extra(qp, torch, synth, dev, steps=10):
    """7B-Llama-shaped decode step per super-block format: tokens/s-equivalent = 1 / (sum of GEMV times). Each layer's
    q/k/v (which read the same activations) are one row-concatenated packed matrix, and so are gate/up, so a layer is
    4 products (qkv 12288x4096, o 4096x4096, gate|up 22016x4096, down 4096x11008); quantization is per row group,
    so the packed bytes equal those of the separate matrices. The 7-launch form is timed as well."""
    shapes = [(4096, 4096)] * 4 + [(11008, 4096)] * 2 + [(4096, 11008)]
    groups = [[0, 1, 2], [3], [4, 5], [6]]           # q|k|v, o, gate|up, down
    out = {}
    for name in ("Q2S", "Q3S", "Q5S", "Q6S"):
        fmt = qp.FORMATS[name]
        fused, separate, total = [], [], 0
        for layer in range(32):
            packed = []
            for mi, (N, K) in enumerate(shapes):
                W = synth.laplace((N, K), 0.02, seed=synth.seed_for(3, layer, mi), device=dev)
                p, g = qp.qpack_quantize_pack(fmt, W)
                del W
                packed.append(p)
                separate.append((p, N, K))
                total += qp.layout(fmt, N, K)["weight_bytes"]
            for gidx in groups:
                K = shapes[gidx[0]][1]
                fused.append((torch.cat([packed[i] for i in gidx], 0), sum(shapes[i][0] for i in gidx), K))
        x4 = synth.normal((4096,), 1.0, seed=11, device=dev, dtype=torch.float16)
        x11 = synth.normal((11008,), 1.0, seed=12, device=dev, dtype=torch.float16)
        ys = {N: torch.empty(N, device=dev) for N in (4096, 11008, 12288, 22016)}
        res = {}
        for kind, mats in (("fused", fused), ("separate", separate)):

            def fn(s, mats=mats):
                for p, N, K in mats:
                    qp.qgemv(fmt, p, None, N, K, x4 if K == 4096 else x11, ys[N], stream=s)

            t = _time_graph(torch, fn, dev, reps=steps)
            res[kind] = {"tok_per_s_equiv": 1.0 / t, "GBps": total / t / 1e9, "ms_per_step": t * 1e3,
                         "launches": len(mats)}
        out[name] = {"bytes_per_step": total, **res["fused"], "separate_launches": res["separate"]}
        del fused, separate
        torch.cuda.empty_cache()
    return out


def _time_graph(torch, fn, dev, reps=5, warm=3):
    """Capture fn (a sequence of launches on its own stream) in one CUDA graph; seconds per replay."""
    s = torch.cuda.Stream(device=dev)
    s.wait_stream(torch.cuda.current_stream(dev))     # the inputs were written on the current stream
    with torch.cuda.stream(s):
        fn(s)
        torch.cuda.synchronize(dev)
        gr = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gr, stream=s):
            fn(s)
        for _ in range(warm):
            gr.replay()
        torch.cuda.synchronize(dev)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(s)
        for _ in range(reps):
            gr.replay()
        e1.record(s)
    torch.cuda.synchronize(dev)
    return e0.elapsed_time(e1) / 1e3 / reps


# Integer dot-product peak of the CUDA cores at the maximum SM clock: dp2a (two 16 x 8-bit multiply-adds) issues at
# 60 per clock per SM on this GPU (measured), so 152 SMs x 60 x 2 MACs x 2 ops x 2.07 GHz; the small-batch products
# are bound by it once M multiply-adds per weight outweigh the packed bytes.
DP2A_TOPS = 152 * 60 * 2 * 2 * 2.07e9 / 1e12


def int4_4096_extra(qp, torch, synth, dev, hbm_peak, fmt=None, N=4096, K=4096):
    """INT4 group-32 GEMV on the 4096x4096 matrix with 0.1% outliers (the INT4 workload), batch 1; also used for the
    fp16-scale variant and other shapes."""
    fmt = qp.Q4G32 if fmt is None else fmt
    W = synth.normal_with_outliers((N, K), 0.02, 0.001, 0.1, 0.5, seed=0).to(dev)
    p0, g0 = qp.qpack_quantize_pack(fmt, W)
    del W
    wb = qp.layout(fmt, N, K)["weight_bytes"]
    R = max(8, int(-(-8 * (126 << 20) // wb)))
    P = [p0.clone() for _ in range(R)]
    G = [g0.clone() for _ in range(R)]
    X = synth.normal((R, K), 1.0, seed=1, device=dev, dtype=torch.float16)
    Y = torch.empty((R, N), device=dev)

    def fn(s):
        for i in range(R):
            qp.qgemv(fmt, P[i], G[i], N, K, X[i], Y[i], stream=s)

    t = _time_graph(torch, fn, dev, reps=20) / R
    return {"GBps": wb / t / 1e9, "pct_hbm_peak": wb / t / 1e9 / hbm_peak, "us_per_gemv": t * 1e6,
            "bytes_per_gemv": wb, "copies": R}


def batch1_all_formats_extra(qp, torch, synth, dev, hbm_peak, N=28672, K=8192):
    """Batch-1 fused dequant-GEMV of every format on one 70B-shaped gate/up matrix (28672x8192, Laplace(0, 0.01),
    seed 4), over distinct packed copies totalling at least 4x L2, back to back in one CUDA graph: the per-format
    rate once the per-launch chain is small next to the stream."""
    out = {}
    W = synth.laplace((N, K), 0.01, seed=4, device=dev)
    for name, fmt in qp.FORMATS.items():
        p0, g0 = qp.qpack_quantize_pack(fmt, W)
        wb = qp.layout(fmt, N, K)["weight_bytes"]
        R = max(3, int(-(-4 * (126 << 20) // wb)))
        P = [p0.clone() for _ in range(R)]
        G = [None if g0 is None else g0.clone() for _ in range(R)]
        del p0, g0
        x = synth.normal((K,), 1.0, seed=5, device=dev, dtype=torch.float16)
        Y = torch.empty((R, N), device=dev)

        def fn(s):
            for i in range(R):
                qp.qgemv(fmt, P[i], G[i], N, K, x, Y[i], stream=s)

        t = _time_graph(torch, fn, dev, reps=10) / R
        out[name] = {"GBps": wb / t / 1e9, "pct_hbm_peak": wb / t / 1e9 / hbm_peak, "us_per_gemv": t * 1e6,
                     "bytes_per_gemv": wb, "copies": R}
        del P, G, Y
        torch.cuda.empty_cache()
    del W
    torch.cuda.empty_cache()
    return out


def mixed_7b_extra(qp, torch, synth, dev, steps=10):
    """7B-Llama-shaped decode step with a per-matrix format mix (2/3/5/6-bit article §2.4: the sensitive attention
    projections get 5 or 6 bits, the wide feed-forward matrices 2 or 3): q and k Q5S, v and o Q6S, gate, up and down
    Q3S. Launches per layer: q|k (row-concatenated), v, o, gate|up, down. Same weights and activations as the
    single-format step."""
    shapes = [(4096, 4096)] * 4 + [(11008, 4096)] * 2 + [(4096, 11008)]
    fmts = ["Q5S", "Q5S", "Q6S", "Q6S", "Q3S", "Q3S", "Q3S"]
    groups = [[0, 1], [2], [3], [4, 5], [6]]
    launches, total, weights = [], 0, 0
    for layer in range(32):
        packed = []
        for mi, (N, K) in enumerate(shapes):
            fmt = qp.FORMATS[fmts[mi]]
            W = synth.laplace((N, K), 0.02, seed=synth.seed_for(3, layer, mi), device=dev)
            p, _ = qp.qpack_quantize_pack(fmt, W)
            del W
            packed.append(p)
            total += qp.layout(fmt, N, K)["weight_bytes"]
            weights += N * K
        for gidx in groups:
            K = shapes[gidx[0]][1]
            launches.append((qp.FORMATS[fmts[gidx[0]]], torch.cat([packed[i] for i in gidx], 0),
                             sum(shapes[i][0] for i in gidx), K))
    x4 = synth.normal((4096,), 1.0, seed=11, device=dev, dtype=torch.float16)
    x11 = synth.normal((11008,), 1.0, seed=12, device=dev, dtype=torch.float16)
    ys = {N: torch.empty(N, device=dev) for N in (4096, 8192, 11008, 22016)}

    def fn(s):
        for fmt, p, N, K in launches:
            qp.qgemv(fmt, p, None, N, K, x4 if K == 4096 else x11, ys[N], stream=s)

    t = _time_graph(torch, fn, dev, reps=steps)
    out = {"formats": "q,k Q5S; v,o Q6S; gate,up,down Q3S", "bpw": 8.0 * total / weights,
           "bytes_per_step": total, "tok_per_s_equiv": 1.0 / t, "GBps": total / t / 1e9, "ms_per_step": t * 1e3,
           "launches": len(launches)}
    del launches
    torch.cuda.empty_cache()
    return out


def kv_cache_extra(qp, torch, synth, dev, hbm_peak):
    """8-bit KV cache of the 7B grouped-query model at 8192 tokens (2 x 32 layers x 8 KV heads x 8192 x 128 fp16,
    1.07 GB; 2/3/5/6-bit article §4.1): quantize (fp16 in, int8 + one fp16 scale per 32 out) and dequantize back.
    Both are HBM streams of 2 + 34/32 bytes per element; the cache is far larger than L2."""
    v = synth.normal((2, 32, 8, 8192, 128), 1.0, seed=21, device=dev, dtype=torch.float16)
    n = v.numel()
    q, s = qp.qpack_kv_quantize(v)
    out = qp.qpack_kv_dequant(q, s)
    nbytes = n * 2 + n + (n // 32) * 2
    res = {"elements": n, "bytes_per_call": nbytes}
    for name, fn in (("quantize", lambda st: qp.qpack_kv_quantize(v, q, s, stream=st)),
                     ("dequant", lambda st: qp.qpack_kv_dequant(q, s, out, stream=st))):
        t = _time_graph(torch, fn, dev, reps=10)
        res[name] = {"GBps": nbytes / t / 1e9, "pct_hbm_peak": nbytes / t / 1e9 / hbm_peak, "us": t * 1e6}
    del v, q, s, out
    torch.cuda.empty_cache()
    return res


def small_batch_extra(qp, torch, synth, dev, hbm_peak):
    """Decode products with M = 1..16 activation rows over 80 layers of 70B-shaped MLP weights (gate/up 28672x8192,
    down 8192x28672, Laplace(0, 0.01)), streamed in turn: one pass = 240 products."""
    shapes = [(28672, 8192), (28672, 8192), (8192, 28672)]
    out = {}
    for name in ("Q4G32", "Q5S"):
        fmt = qp.FORMATS[name]
        mats, total, weights = [], 0, 0
        for layer in range(80):
            for mi, (N, K) in enumerate(shapes):
                W = synth.laplace((N, K), 0.01, seed=synth.seed_for(4, layer, mi), device=dev)
                p, g = qp.qpack_quantize_pack(fmt, W)
                del W
                mats.append((p, g, N, K))
                total += qp.layout(fmt, N, K)["weight_bytes"]
                weights += N * K
        res = {}
        for M in (1, 2, 4, 8, 16):
            X = {K: synth.normal((M, K), 1.0, seed=100 + M + K, device=dev, dtype=torch.float16) for K in (8192, 28672)}
            Y = {N: torch.empty((M, N), device=dev) for N in (8192, 28672)}

            def fn(s):
                for p, g, N, K in mats:
                    qp.qgemm_small(fmt, p, g, N, K, X[K], Y[N], stream=s)

            t = _time_graph(torch, fn, dev, reps=3)
            tf = 2.0 * M * weights / t / 1e12
            res[f"M{M}"] = {"GBps": total / t / 1e9, "pct_hbm_peak": total / t / 1e9 / hbm_peak,
                            "TOPs": tf, "pct_dp2a_peak": tf / DP2A_TOPS,
                            "tok_per_s_equiv": M / t, "ms_per_pass": t * 1e3}
        out[name] = {"bytes_per_pass": total, "launches_per_pass": len(mats), **res}
        del mats
        torch.cuda.empty_cache()
    return out


def prefill_extra(qp, torch, synth, dev, bf16_peak, hbm_peak):
    """Prefill GEMM (M = 2048 bf16 tokens) on the tensor cores, and the quantize+pack kernels on the same fp16
    matrices (INT4 14336x4096, 6-bit 4096x14336; Laplace(0, 0.02), seed 7)."""
    out = {"gemm": {}, "quantize_pack": {}}
    M = 2048
    for name, (N, K) in (("Q4G32", (14336, 4096)), ("Q6S", (4096, 14336))):
        fmt = qp.FORMATS[name]
        W = synth.laplace((N, K), 0.02, seed=7, device=dev, dtype=torch.float16)
        p, g = qp.qpack_quantize_pack(fmt, W)
        X = synth.normal((M, K), 1.0, seed=8, device=dev, dtype=torch.bfloat16)
        Y = torch.empty((M, N), device=dev, dtype=torch.bfloat16)

        def fn(s):
            qp.qgemm_prefill(fmt, p, g, N, K, X, Y, stream=s)

        t = _time_graph(torch, fn, dev, reps=10)
        tf = 2.0 * M * N * K / t / 1e12
        out["gemm"][f"{name}_{N}x{K}"] = {"TFLOPs": tf, "pct_bf16_peak": tf / bf16_peak, "us": t * 1e6, "M": M}
        for qn in ("Q4G32", "Q2S", "Q3S", "Q5S", "Q6S"):
            qf = qp.FORMATS[qn]
            pk, gk = qp.alloc_packed(qf, N, K, dev)
            lay = qp.layout(qf, N, K)

            def qfn(s):
                qp.qpack_quantize_pack(qf, W, pk, gk, stream=s)

            tq = _time_graph(torch, qfn, dev, reps=10)
            moved = W.numel() * 2 + lay["weight_bytes"]
            out["quantize_pack"][f"{qn}_{N}x{K}"] = {"GBps": moved / tq / 1e9, "pct_hbm_peak": moved / tq / 1e9 / hbm_peak,
                                                     "us": tq * 1e6}
        del W, p, g, X, Y
        torch.cuda.empty_cache()
    return out


def run_ours(args, world, rank, local):
    import numpy as np
    import torch
    from bit_weight_quantized_qpack_gb300 import _build
    _build.build()
    import bit_weight_quantized_qpack_gb300 as qp
    from bit_weight_quantized_qpack_gb300 import synth

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    pg = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
        pg = dist
    hbm_peak, bf16_peak, peak_src = measured_peaks()

    # decode over resident weights: products may start streaming their weights while the previous kernel ends
    qp.qpack_set_option(qp.OPT_WEIGHT_PREFETCH, 0 if args.no_prefetch else 1)
    fmt = qp.Q3S
    lay = qp.layout(fmt, N_ROWS, K_COLS)
    wbytes = lay["weight_bytes"]
    W = synth.laplace((N_ROWS, K_COLS), 0.015, seed=0, device=dev)
    packed0, _ = qp.qpack_quantize_pack(fmt, W)
    del W
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size or (126 << 20)
    R = args.copies or max(8, int(-(-8 * l2 // wbytes)))              # copies total >= 8x L2
    P = torch.empty((R, N_ROWS, lay["row_stride"]), dtype=torch.uint8, device=dev)
    P.copy_(packed0.unsqueeze(0).expand(R, -1, -1))
    del packed0
    X = synth.normal((R, K_COLS), 1.0, seed=1, device=dev, dtype=torch.float16)
    Y = torch.empty((R, N_ROWS), dtype=torch.float32, device=dev)
    s = torch.cuda.Stream(device=dev)
    s.wait_stream(torch.cuda.current_stream(dev))     # the inputs were written on the current stream

    def step():
        for i in range(R):
            qp.qgemv(fmt, P[i], None, N_ROWS, K_COLS, X[i], Y[i], stream=s)

    with torch.cuda.stream(s):
        step()
        torch.cuda.synchronize(dev)
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=s):
            step()
    torch.cuda.synchronize(dev)
    for _ in range(args.warmup):
        graph.replay()
    torch.cuda.synchronize(dev)
    if pg:
        pg.barrier()
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize(dev)
    with torch.cuda.stream(s):
        e0.record(s)
        for _ in range(args.steps):
            graph.replay()
        e1.record(s)
    torch.cuda.synchronize(dev)
    if pg:
        pg.barrier()
    clk = clocks.stop()
    t_step = e0.elapsed_time(e1) / 1e3 / args.steps
    if pg:
        tt = torch.tensor([t_step], device=dev, dtype=torch.float64)
        pg.all_reduce(tt, op=pg.ReduceOp.MAX)
        t_step = float(tt.item())
    value = world * R * wbytes / t_step / 1e9
    per_launch = t_step / R
    achieved = wbytes / per_launch / 1e9
    faults = qp.qpack_fetch_fault_flags()

    # ---- end to end through the C ABI with host buffers: H2D of the step's activations, the step's qgemv calls
    # (the C entry point called with its arguments prepared once, as a serving loop over resident weights would),
    # D2H of its outputs. Every step's copies are inside the timed region; as a serving loop would, the step's H2D
    # runs on one copy stream and its D2H on another, double-buffered, so they overlap the neighbouring steps'
    # products instead of serialising with them. ----
    import ctypes
    Xh = torch.empty((R, K_COLS), dtype=torch.float16, pin_memory=True)
    Xh.copy_(X.cpu())
    Xb = [X, torch.empty_like(X)]
    Yb = [Y, torch.empty_like(Y)]
    Yh = [torch.empty((R, N_ROWS), dtype=torch.float32, pin_memory=True) for _ in range(2)]
    s_h2d, s_d2h = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    ev_in = [torch.cuda.Event(), torch.cuda.Event()]     # the step's activations landed
    ev_done = [torch.cuda.Event(), torch.cuda.Event()]   # the step's products finished (its activations free again)
    ev_out = [torch.cuda.Event(), torch.cuda.Event()]    # the step's outputs copied out (its output buffer free again)
    c_qgemv = qp.lib().qgemv
    c_args = [[(int(fmt), ctypes.c_void_p(P[i].data_ptr()), None, N_ROWS, K_COLS, ctypes.c_void_p(Xb[b][i].data_ptr()),
                ctypes.c_void_p(Yb[b][i].data_ptr()), ctypes.c_void_p(s.cuda_stream)) for i in range(R)] for b in range(2)]
    for e in ev_done:
        e.record(s)
    for e in ev_out:
        e.record(s_d2h)

    def e2e_step(i):
        b = i & 1
        s_h2d.wait_event(ev_done[b])
        with torch.cuda.stream(s_h2d):
            Xb[b].copy_(Xh, non_blocking=True)
        ev_in[b].record(s_h2d)
        s.wait_event(ev_in[b])
        s.wait_event(ev_out[b])
        for a in c_args[b]:
            rc = c_qgemv(*a)
            if rc != 0:
                raise RuntimeError(f"qgemv failed with status {rc}")
        ev_done[b].record(s)
        s_d2h.wait_event(ev_done[b])
        with torch.cuda.stream(s_d2h):
            Yh[b].copy_(Yb[b], non_blocking=True)
        ev_out[b].record(s_d2h)

    with torch.cuda.stream(s):
        for i in range(args.warmup):
            e2e_step(i)
        torch.cuda.synchronize(dev)
        f0, f1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        f0.record(s)
        s_h2d.wait_stream(s)
        for i in range(args.steps):
            e2e_step(i)
        s.wait_stream(s_d2h)                         # the last step's outputs are on the host
        f1.record(s)
    torch.cuda.synchronize(dev)
    t_e2e = f0.elapsed_time(f1) / 1e3 / args.steps
    if pg:
        tt = torch.tensor([t_e2e], device=dev, dtype=torch.float64)
        pg.all_reduce(tt, op=pg.ReduceOp.MAX)
        t_e2e = float(tt.item())
    e2e = {"value": world * R * wbytes / t_e2e / 1e9, "unit": "GB/s", "h2d_bytes_per_step": int(Xh.nbytes),
           "d2h_bytes_per_step": int(Yh[0].nbytes)}

    cpu = None
    extra = None
    if rank == 0:
        if not args.no_cpu_baseline:
            pk = P[0].cpu().numpy()
            cpu = cpu_oracle_gemv_sample(pk, X[0].cpu().numpy().view(np.uint16))
        if not args.no_extra:
            del P, X, Y
            torch.cuda.empty_cache()
            extra = {"batch1_all_formats_28672x8192": batch1_all_formats_extra(qp, torch, synth, dev, hbm_peak),
                     "decode_7b": decode_7b_extra(qp, torch, synth, dev),
                     "decode_7b_mixed": mixed_7b_extra(qp, torch, synth, dev),
                     "int4_4096": int4_4096_extra(qp, torch, synth, dev, hbm_peak),
                     "int4_fp16_scales": {
                         "4096x4096": int4_4096_extra(qp, torch, synth, dev, hbm_peak, qp.Q4G32H),
                         "28672x8192": int4_4096_extra(qp, torch, synth, dev, hbm_peak, qp.Q4G32H, 28672, 8192)},
                     "int4_group16": {
                         "4096x4096": int4_4096_extra(qp, torch, synth, dev, hbm_peak, qp.Q4G16),
                         "28672x8192": int4_4096_extra(qp, torch, synth, dev, hbm_peak, qp.Q4G16, 28672, 8192)},
                     "int4_asymmetric": {
                         "4096x4096": int4_4096_extra(qp, torch, synth, dev, hbm_peak, qp.Q4G32A),
                         "28672x8192": int4_4096_extra(qp, torch, synth, dev, hbm_peak, qp.Q4G32A, 28672, 8192)},
                     "small_batch_70b_mlp": small_batch_extra(qp, torch, synth, dev, hbm_peak),
                     "prefill_2048": prefill_extra(qp, torch, synth, dev, bf16_peak, hbm_peak),
                     "kv_cache_8bit": kv_cache_extra(qp, torch, synth, dev, hbm_peak)}

    traffic = TRAFFIC["bytes_per_launch"] if TRAFFIC["csrc_digest"] == csrc_digest() else None
    line = {
        "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": t_step * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": DTYPE, "data": "synthetic",
        "config": {"workload": WORKLOAD, "format": FORMAT_DESC, "N": N_ROWS, "K": K_COLS, "batch": 1,
                   "copies_per_step": R, "bytes_per_gemv": wbytes,
                   "l2": f"inputs larger than L2: {R} distinct packed copies ({R * wbytes / 1e9:.2f} GB) per step",
                   "parallelism": "one GPU per rank; row shards need no exchange (weak-scaling replicas)",
                   "weight_prefetch": not args.no_prefetch},
        "pct_hbm_peak": value / world / hbm_peak,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": hbm_peak, "unit": "GB/s",
                     "frac": achieved / hbm_peak, "traffic": traffic, "peak_source": peak_src,
                     "kernel": "gemv1_kernel<Q3S>", "algorithmic_bytes_per_launch": wbytes},
        "cpu_baseline": cpu,
        "e2e": e2e,
        "gpu_launches": args.steps * R,
        "clocks": clk,
        "faults": faults,
    }
    if extra:
        line["extra"] = extra
    if rank == 0:
        print(json.dumps(line), flush=True)
    if pg:
        pg.barrier()
        pg.destroy_process_group()
    return 0


def run_ncu_case(args):
    """A short run sized for an ncu capture (a few launches, a few hundred MB on the device): quantize one
    matrix, replicate it `copies` times (> L2 in total) and run the product on each copy."""
    import torch
    from bit_weight_quantized_qpack_gb300 import _build
    _build.build()
    import bit_weight_quantized_qpack_gb300 as qp
    from bit_weight_quantized_qpack_gb300 import synth
    dev = torch.device("cuda", 0)
    if args.ncu_case == "kv":
        v = synth.normal((args.M, args.N, args.K), 1.0, seed=21, device=dev, dtype=torch.float16)
        q, s = qp.qpack_kv_quantize(v)
        out = qp.qpack_kv_dequant(q, s)
        torch.cuda.synchronize()
        print(json.dumps({"ncu_case": "kv", "elements": v.numel(), "faults": qp.qpack_fetch_fault_flags()}))
        return 0
    fmt = qp.FORMATS[args.fmt]
    N, K = args.N, args.K
    if args.ncu_case == "quant":
        W16 = synth.laplace((N, K), 0.02, seed=7, device=dev).half()
        for _ in range(3):
            qp.qpack_quantize_pack(fmt, W16)
        torch.cuda.synchronize()
        print(json.dumps({"ncu_case": "quant", "fmt": args.fmt, "N": N, "K": K, "faults": qp.qpack_fetch_fault_flags()}))
        return 0
    W = synth.laplace((N, K), 0.02, seed=1, device=dev)
    p0, g0 = qp.qpack_quantize_pack(fmt, W)
    del W
    copies = args.copies or 8
    ps = [p0.clone() for _ in range(copies)]
    gs = [None if g0 is None else g0.clone() for _ in range(copies)]
    if args.ncu_case == "gemv":
        x = synth.normal((K,), 1.0, seed=2, device=dev, dtype=torch.float16)
        y = torch.empty(N, device=dev)
        for i in range(copies):
            qp.qgemv(fmt, ps[i], gs[i], N, K, x, y)
    elif args.ncu_case == "small":
        X = synth.normal((args.M, K), 1.0, seed=2, device=dev, dtype=torch.float16)
        Y = torch.empty((args.M, N), device=dev)
        for i in range(copies):
            qp.qgemm_small(fmt, ps[i], gs[i], N, K, X, Y)
    else:
        X = synth.normal((args.M, K), 1.0, seed=2, device=dev, dtype=torch.bfloat16)
        Y = torch.empty((args.M, N), device=dev, dtype=torch.bfloat16)
        qp.qpack_set_option(qp.OPT_PREFILL_TILE_ROWS, args.prefill_tile_rows)
        for i in range(copies):
            qp.qgemm_prefill(fmt, ps[i], gs[i], N, K, X, Y)
    torch.cuda.synchronize()
    print(json.dumps({"ncu_case": args.ncu_case, "fmt": args.fmt, "N": N, "K": K, "copies": copies,
                      "faults": qp.qpack_fetch_fault_flags()}))
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--copies", type=int, default=0, help="distinct weight copies per step (default: >= 8x L2)")
    ap.add_argument("--no-extra", action="store_true", help="skip the 7B decode-step extra")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-prefetch", action="store_true", help="disable QPACK_OPT_WEIGHT_PREFETCH")
    ap.add_argument("--ncu-case", choices=["gemv", "small", "prefill", "kv", "quant"], default=None,
                    help="short run of one product, sized for an ncu capture")
    ap.add_argument("--fmt", default="Q3S")
    ap.add_argument("--N", type=int, default=N_ROWS)
    ap.add_argument("--K", type=int, default=K_COLS)
    ap.add_argument("--M", type=int, default=8)
    ap.add_argument("--prefill-tile-rows", type=int, default=0, choices=[0, 112, 128, 224, 256],
                    help="--ncu-case prefill: the tiling (0: chosen per launch; 256/224: CTA pairs; 128/112: single CTAs)")
    args = ap.parse_args()
    if args.ncu_case:
        return run_ncu_case(args)
    if args.warmup < 3:
        args.warmup = 3
    world, rank, local = dist_setup(args)
    if args.impl == "reference":
        return run_reference(args, world, rank)
    return run_ours(args, world, rank, local)


if __name__ == "__main__":
    sys.exit(main())
