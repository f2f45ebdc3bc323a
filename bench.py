#!/usr/bin/env python
"""Throughput of fused scaled-dot-product attention forward + backward on GB300.

One step = sdpa_fwd + the three sdpa_bwd phases on one batch of synthetic,
seeded inputs resident in HBM. The default workload is the long-context
causal case: b1 h32 s16384 d128 bf16 (inputs of 537 MB, far larger than L2,
so no flush is needed between steps).

FLOP convention: forward = 4*b*h*s_q*s_kv*(d_qk+d_v)/2, halved for causal;
backward = 2.5x forward; a step = 3.5x forward.

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
       python bench.py --impl reference ...   (the fp64 CPU oracle on a bounded sample)
Prints one JSON line (rank 0).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "SDPA fwd+bwd TFLOP/s (bf16, causal) and % of GB300 dense BF16 tensor peak"
UNIT = "TFLOP/s"
L2_BYTES = 129 * 1000 * 1000  # GB300 L2 (about 126 MiB)

WORKLOADS = {
    "b1h2-s128-d64": dict(B=1, H=2, S_q=128, S_kv=128, D_qk=64, D_v=64, dtype="bf16",
                          causal=False, bias=False, p=0.0, scale=0.125),
    "b4h16-s2048-d128-causal": dict(B=4, H=16, S_q=2048, S_kv=2048, D_qk=128, D_v=128,
                                    dtype="bf16", causal=True, bias=False, p=0.0, scale=None),
    "b2h16-s4096-d192x128-causal-bias": dict(B=2, H=16, S_q=4096, S_kv=4096, D_qk=192, D_v=128,
                                             dtype="bf16", causal=True, bias=True, p=0.0,
                                             scale=None),
    "b8h16-s1024x2048-d64-fp16-dropout0.1": dict(B=8, H=16, S_q=1024, S_kv=2048, D_qk=64, D_v=64,
                                                 dtype="fp16", causal=False, bias=False, p=0.1,
                                                 scale=None),
    # the dropout case's shape without dropout: what the Philox draws cost
    "b8h16-s1024x2048-d64-fp16": dict(B=8, H=16, S_q=1024, S_kv=2048, D_qk=64, D_v=64,
                                      dtype="fp16", causal=False, bias=False, p=0.0, scale=None),
    # the dropout case with its keep bits drawn once per step (sdpa_dropout_mask,
    # timed with the forward) and read by the three kernels
    "b8h16-s1024x2048-d64-fp16-dropout0.1-bits": dict(B=8, H=16, S_q=1024, S_kv=2048, D_qk=64,
                                                      D_v=64, dtype="fp16", causal=False,
                                                      bias=False, p=0.1, scale=None, bits=True),
    "b1h32-s16384-d128-causal": dict(B=1, H=32, S_q=16384, S_kv=16384, D_qk=128, D_v=128,
                                     dtype="bf16", causal=True, bias=False, p=0.0, scale=None),
    # grouped-query attention at the long-context size: 32 query heads on 4 K/V
    # heads (groups of 8)
    "b1h32kv4-s16384-d128-causal": dict(B=1, H=32, H_kv=4, S_q=16384, S_kv=16384, D_qk=128,
                                        D_v=128, dtype="bf16", causal=True, bias=False, p=0.0,
                                        scale=None),
    # multi-query attention (one K/V head) at the long-context size
    "b1h32kv1-s16384-d128-causal": dict(B=1, H=32, H_kv=1, S_q=16384, S_kv=16384, D_qk=128,
                                        D_v=128, dtype="bf16", causal=True, bias=False, p=0.0,
                                        scale=None),
    # a sliding window of 4096 keys back (local attention) at the long-context size
    "b1h32-s16384-d128-window4096": dict(B=1, H=32, S_q=16384, S_kv=16384, D_qk=128, D_v=128,
                                         dtype="bf16", causal=True, window=(4096, 0),
                                         bottom_right=False, bias=False, p=0.0, scale=None),
    # ALiBi (geometric slopes 2^(-8 (h + 1) / H), one per head) on the causal
    # long-context case
    "b1h32-s16384-d128-causal-alibi": dict(B=1, H=32, S_q=16384, S_kv=16384, D_qk=128, D_v=128,
                                           dtype="bf16", causal=True, alibi=True, bias=False,
                                           p=0.0, scale=None),
    # packed variable-length sequences (group mode): 16 sequences of 512..8192
    # tokens (seeded; 74,372 in all), 32 heads, d 128, causal
    "varlen16-h32-d128-causal": dict(lengths=dict(n=16, lo=512, hi=8192, seed=2024), H=32,
                                     D_qk=128, D_v=128, dtype="bf16", causal=True, bias=False,
                                     p=0.0, scale=None),
    # half the heads and half the sequence of the long-context case: the size the
    # full ncu section captures in profiles/ are taken at (inputs 134 MB > L2)
    "b1h16-s8192-d128-causal": dict(B=1, H=16, S_q=8192, S_kv=8192, D_qk=128, D_v=128,
                                    dtype="bf16", causal=True, bias=False, p=0.0, scale=None),
}
DEFAULT_WORKLOAD = "b1h32-s16384-d128-causal"
DROP_SEED, DROP_OFFSET = 0x1234, 0

# Kernel sources whose ncu DRAM counters are recorded in profiles/traffic.json.
KERNEL_SOURCES = {
    "bwd_dkdv": ["scaled_dot_product_06_gb300/csrc/bwd_dkdv_kernel.cuh",
                 "scaled_dot_product_06_gb300/csrc/common.cuh",
                 "scaled_dot_product_06_gb300/csrc/ptx.cuh"],
    "bwd_dq": ["scaled_dot_product_06_gb300/csrc/bwd_dq_kernel.cuh",
               "scaled_dot_product_06_gb300/csrc/common.cuh",
               "scaled_dot_product_06_gb300/csrc/ptx.cuh"],
    "fwd": ["scaled_dot_product_06_gb300/csrc/fwd_kernel.cuh",
            "scaled_dot_product_06_gb300/csrc/common.cuh",
            "scaled_dot_product_06_gb300/csrc/ptx.cuh"],
    "bwd_fused": ["scaled_dot_product_06_gb300/csrc/bwd_fused_kernel.cuh",
                  "scaled_dot_product_06_gb300/csrc/bwd_dkdv_kernel.cuh",
                  "scaled_dot_product_06_gb300/csrc/common.cuh",
                  "scaled_dot_product_06_gb300/csrc/ptx.cuh"],
    "bwd_pre": ["scaled_dot_product_06_gb300/csrc/aux.cu",
                "scaled_dot_product_06_gb300/csrc/common.cuh"],
    "dq_convert": ["scaled_dot_product_06_gb300/csrc/aux.cu",
                   "scaled_dot_product_06_gb300/csrc/common.cuh"],
}


def visible_pairs_per_head(w: dict) -> int:
    """(query, key) pairs a head's mask leaves visible (summed over the
    sequences of a packed workload)."""
    if w.get("lens"):
        return sum(n * (n + 1) // 2 if w["causal"] else n * n for n in w["lens"])
    if w.get("window") is not None:
        return visible_pairs(w["S_q"], w["S_kv"], w["window"], w.get("bottom_right", False))
    if w["causal"]:  # top-left: row i sees min(i + 1, S_kv) keys
        return sum(min(i + 1, w["S_kv"]) for i in range(w["S_q"]))
    return w["S_q"] * w["S_kv"]


def kernel_bytes(w: dict, fused: bool) -> dict:
    """Algorithmic DRAM bytes per launch of each kernel: every operand read
    once and every result written once; the bias read and dBias written once
    per head over the visible pairs (shared by the batch); the row statistics
    8 bytes per query row. The fused kernel's dQ reductions stay in L2; its dQ
    is written by the convert pass, which reads the fp32 accumulator."""
    e = 2
    B = 1 if w.get("lens") else w["B"]
    H, Hkv, Dk, Dv = w["H"], w.get("H_kv", w["H"]), w["D_qk"], w["D_v"]
    rq = H * sum(w["lens"]) if w.get("lens") else B * H * w["S_q"]
    rk = Hkv * sum(w["lens"]) if w.get("lens") else B * Hkv * w["S_kv"]
    q, o, lse, st = rq * Dk * e, rq * Dv * e, rq * 4, rq * 8
    kv = rk * (Dk + Dv) * e
    bias = H * visible_pairs_per_head(w) * 4 if w["bias"] else 0  # read over the visible pairs
    dbias = H * w["S_q"] * w["S_kv"] * 4 if w["bias"] else 0       # written in full (0 where masked)
    # the fp32 dQ accumulator: rows padded to 128 per (b, h), or per head over the packed rows
    acc = (H * ((sum(w["lens"]) + 127) // 128) if w.get("lens") else B * H * ((w["S_q"] + 127) // 128)) \
        * 128 * Dk * 4
    out = {"fwd": q + kv + o + lse + bias, "bwd_pre": 2 * o + lse + st}
    main = q + o + kv + st + kv + bias + dbias  # Q, dO, K, V, stats, Bias in; dK, dV, dBias out
    if fused:
        out["bwd_fused"] = main
        out["dq_convert"] = acc + q
    else:
        out["bwd_dkdv"] = main
        out["bwd_dq"] = q + o + kv + st + q + bias
    return out


def workload_bound(w: dict, fwd_gflop: float, draws: bool) -> str:
    """The roofline that bounds the dominant kernel (the hot-path table's
    bound column): HBM with an fp32 bias (its 4-byte-per-pair Bias and dBias
    dominate the bytes), the integer ALU for a kernel that draws dropout
    numbers (Philox4x32-10, ten rounds per four elements), HBM (latency) for a
    problem too small to fill the GPU, the tensor cores otherwise."""
    if w["bias"]:
        return "hbm"
    if draws:
        return "alu"
    if fwd_gflop < 1.0:
        return "hbm"
    return "tensor"


def resolve(w: dict) -> dict:
    """The workload with its sizes filled in: a packed workload gets its
    sequence lengths ("lens"), B = their number and S_q = S_kv = the longest."""
    if "lengths" not in w:
        return dict(w)
    from scaled_dot_product_06_gb300.inputs import packed_lengths
    lens = packed_lengths(**w["lengths"])
    return dict(w, lens=lens, B=len(lens), S_q=max(lens), S_kv=max(lens))


def visible_pairs(S_q: int, S_kv: int, window, bottom_right: bool) -> int:
    """Number of (query, key) pairs a local window leaves visible."""
    import numpy as np
    left, right = window
    off = S_kv - S_q if bottom_right else 0
    i = np.arange(S_q, dtype=np.int64)
    lo = np.maximum(i + off - left, 0) if left >= 0 else np.zeros_like(i)
    hi = np.minimum(i + off + right, S_kv - 1) if right >= 0 else np.full_like(i, S_kv - 1)
    return int(np.maximum(hi - lo + 1, 0).sum())


def fwd_flops(w: dict) -> float:
    """Forward FLOPs by the convention; a packed workload sums its sequences; a
    windowed one counts its visible pairs, 2 (D_qk + D_v) FLOPs each (the
    convention's causal half, S^2 / 2 pairs, is the same count for a causal
    mask)."""
    if w.get("lens"):
        one = {k: v for k, v in w.items() if k != "lens"}
        return sum(fwd_flops(dict(one, B=1, S_q=n, S_kv=n)) for n in w["lens"])
    if w.get("window") is not None:
        pairs = visible_pairs(w["S_q"], w["S_kv"], w["window"], w.get("bottom_right", False))
        return 2.0 * w["B"] * w["H"] * pairs * (w["D_qk"] + w["D_v"])
    f = 4.0 * w["B"] * w["H"] * w["S_q"] * w["S_kv"] * (w["D_qk"] + w["D_v"]) / 2.0
    return f / 2.0 if w["causal"] else f


def source_sha(kernel: str) -> str:
    h = hashlib.sha256()
    for rel in KERNEL_SOURCES[kernel]:
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def measured_peaks() -> tuple[dict, str]:
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            return json.load(f), "measured"
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}, "fallback"


# ---------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons while running."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.dev = device_index
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.dev), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        time.sleep(0.3)

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
        self.proc.terminate()
        self.proc.wait(timeout=10)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sm.append(float(parts[1]))
                    smax.append(float(parts[2]))
                except ValueError:
                    continue
                for n, v in zip(names, parts[5:9]):
                    if v.lower() == "active":
                        reasons.add(n)
        os.unlink(self.path)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None, "samples": len(sm),
                "reasons": sorted(reasons)}


# ---------------------------------------------------------------- oracle (CPU)
def oracle_sample(w: dict, s_sample: int) -> tuple[float, float]:
    """fp64 oracle fwd+bwd on one head restricted to the first s_sample
    positions of the workload. Returns (seconds, FLOPs by the convention)."""
    import oracle
    from scaled_dot_product_06_gb300.inputs import Shape, make_inputs
    s_q = min(s_sample, w["S_q"])
    s_kv = min(s_sample * w["S_kv"] // w["S_q"], w["S_kv"])
    shp = Shape(1, 1, s_q, s_kv, w["D_qk"], w["D_v"])
    x = make_inputs(shp, w["dtype"], with_bias=w["bias"])
    scale = w["scale"] if w["scale"] is not None else 1.0 / math.sqrt(w["D_qk"])
    pr = oracle.Problem(1, 1, s_q, s_kv, w["D_qk"], w["D_v"], scale, w["causal"], w["p"],
                        DROP_SEED, DROP_OFFSET, window=w.get("window"),
                        bottom_right=w.get("bottom_right", False),
                        alibi_slopes=((2.0 ** (-8.0 / w["H"]),),) if w.get("alibi") else None)
    t0 = time.perf_counter()
    oracle.forward(pr, x["q"], x["k"], x["v"], x["bias"])
    oracle.backward(pr, x["q"], x["k"], x["v"], x["do"], x["bias"])
    dt = time.perf_counter() - t0
    ws = {k: v for k, v in w.items() if k != "lens"}  # one head of one sequence
    return dt, 3.5 * fwd_flops(dict(ws, B=1, H=1, S_q=s_q, S_kv=s_kv))


def cpu_threads() -> int:
    try:
        from threadpoolctl import threadpool_info
        n = [i.get("num_threads", 0) for i in threadpool_info() if i.get("user_api") == "blas"]
        if n:
            return int(max(n))
    except Exception:
        pass
    return os.cpu_count() or 1


def run_reference(args, w, rank):
    """The reference arm: the oracle as it stands, on the host cores."""
    if rank != 0:
        return
    s_sample = args.ref_sample
    for _ in range(args.warmup):
        oracle_sample(w, s_sample)
    secs, flops = 0.0, 0.0
    for _ in range(args.steps):
        dt, f = oracle_sample(w, s_sample)
        secs += dt
        flops += f
    value = flops / secs / 1e12
    sample = (f"one head, first {min(s_sample, w['S_q'])} query positions of {args.workload} "
              f"(fp64 numpy oracle, fwd+bwd, FLOPs by the same convention)")
    out = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT,
           "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
           "ms_per_step": 1e3 * secs / args.steps, "higher_is_better": True, "scaling": "weak",
           "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded normal)",
           "config": {"workload": args.workload, **{k: w[k] for k in ("B", "H", "S_q", "S_kv",
                                                                      "D_qk", "D_v")}},
           "cpu_baseline": {"value": value, "unit": UNIT, "cores": cpu_threads(),
                            "kind": "oracle", "sample": sample},
           "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0,
                   "d2h_bytes_per_step": 0}}
    print(json.dumps(out), flush=True)


# ---------------------------------------------------------------- host placement
def bind_near_gpu(index: int):
    """Run this process on the CPUs the GPU's PCI device reports as local, so
    that the pinned host buffers of the end-to-end measurement (placed on
    first touch) sit on the GPU's own memory node rather than across a socket
    link. Returns the CPU list used, or None when the system does not say."""
    import torch
    try:
        pr = torch.cuda.get_device_properties(index)
        path = (f"/sys/bus/pci/devices/{pr.pci_domain_id:04x}:{pr.pci_bus_id:02x}:"
                f"{pr.pci_device_id:02x}.0/local_cpulist")
        with open(path) as f:
            spec = f.read().strip()
        cpus = set()
        for part in spec.split(","):
            if "-" in part:
                a, b = part.split("-")
                cpus.update(range(int(a), int(b) + 1))
            elif part:
                cpus.add(int(part))
        allowed = cpus & os.sched_getaffinity(0)
        if not allowed:
            return None
        os.sched_setaffinity(0, allowed)
        return spec
    except (OSError, ValueError, AttributeError):
        return None


# ---------------------------------------------------------------- ranks
def max_over_ranks(x: float, world: int, device=None) -> float:
    """Slowest rank's value (all ranks get it); identity for one rank."""
    if world <= 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_tflops(world: int, step_flops: float, ms_per_step: float) -> float:
    """Units all ranks processed / the slowest rank's time: every rank runs
    the same workload (independent replicas, no data-path collective)."""
    return world * step_flops / (ms_per_step * 1e-3) / 1e12


# ---------------------------------------------------------------- GPU arm
def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(WORKLOADS))
    ap.add_argument("--e2e-steps", type=int, default=16)
    ap.add_argument("--cpu-sample", type=int, default=16384,
                    help="query positions of the one-head oracle sample (cpu_baseline); the "
                         "default is a whole head of the long-context workload, ~15 s of CPU")
    ap.add_argument("--ref-sample", type=int, default=4096,
                    help="query positions of the one-head oracle sample per reference step")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-record", action="store_true",
                    help="with dropout, let the backward draw its own keep bits instead of reading "
                         "the record the forward leaves")
    ap.add_argument("--deterministic", action="store_true",
                    help="time the deterministic backward (query-stationary dQ kernel beside the "
                         "dK/dV kernel) instead of the default fused one")
    args = ap.parse_args()
    w = resolve(WORKLOADS[args.workload])

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        run_reference(args, w, rank)
        return

    import torch
    import torch.distributed as dist

    from scaled_dot_product_06_gb300 import (SDPA_BWD_ALL, SDPA_BWD_DKDV, SDPA_BWD_DQ,
                                             SDPA_BWD_PREPROCESS, sdpa_bwd_phases,
                                             sdpa_dropout_mask,
                                             sdpa_bwd_phases_varlen, sdpa_bwd_varlen_workspace_size,
                                             sdpa_bwd_workspace_size, sdpa_device_error, sdpa_fwd,
                                             sdpa_fwd_varlen)
    from scaled_dot_product_06_gb300.inputs import (Shape, make_inputs, make_packed_inputs,
                                                    seqstarts)

    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA device")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    host_cpus = bind_near_gpu(local)
    if world > 1:
        dist.init_process_group("nccl", device_id=dev)

    def barrier():
        if world > 1:
            dist.barrier()

    scale = w["scale"] if w["scale"] is not None else 1.0 / math.sqrt(w["D_qk"])
    kw = dict(scale=scale, is_causal=w["causal"], dropout_p=w["p"], seed=DROP_SEED,
              offset=DROP_OFFSET)
    if w.get("window") is not None or w.get("bottom_right"):
        kw.update(window=w.get("window"), bottom_right=w.get("bottom_right", False))
    mask_words = 0
    if w.get("bits"):
        mask_words = (w["B"] * w["H"] * w["S_q"] * w["S_kv"] + 31) // 32
        kw["dropout_mask"] = torch.empty(mask_words, dtype=torch.int32, device=dev)
    # With dropout (batch mode, s_kv % 32 == 0) the forward records the keep
    # bits it draws and the backward reads them: Philox runs once per step.
    record_words = 0
    if (w["p"] > 0 and not w.get("bits") and "lens" not in w and w["S_kv"] % 32 == 0
            and not args.no_record):
        record_words = (w["B"] * w["H"] * w["S_q"] * w["S_kv"] + 31) // 32
        keep_record = torch.empty(record_words, dtype=torch.int32, device=dev)
    if w.get("alibi"):
        kw["alibi_slopes"] = torch.tensor([2.0 ** (-8.0 * (hh + 1) / w["H"]) for hh in range(w["H"])],
                                          dtype=torch.float32, device=dev)
    packed = "lens" in w
    if packed:
        # [H, total, D] tensors; sequence i owns rows seqstart[i] .. seqstart[i+1]-1
        total = sum(w["lens"])
        x = make_packed_inputs(w["H"], total, total, w["D_qk"], w["D_v"], w["dtype"],
                               w.get("H_kv", 0), seed_base=rank, device=dev)
        x["bias"] = None
        starts = torch.tensor(seqstarts(w["lens"]), dtype=torch.int32, device=dev)
        o = torch.empty(w["H"], total, w["D_v"], dtype=x["q"].dtype, device=dev)
        lse = torch.empty(w["H"], total, dtype=torch.float32, device=dev)
        ws = torch.empty(sdpa_bwd_varlen_workspace_size(w["B"], w["H"], total, w["D_qk"],
                                                        args.deterministic),
                         dtype=torch.uint8, device=dev)
        mx = w["S_q"]

        def fwd_call(D):
            sdpa_fwd_varlen(D["q"], D["k"], D["v"], starts, starts, mx, mx, out=D["o"],
                            lse=D["lse"], **kw)

        def bwd_call(ph, D, stream=None):
            sdpa_bwd_phases_varlen(ph, D["q"], D["k"], D["v"], D["o"], D["do"], D["lse"], starts,
                                   starts, mx, mx, workspace=ws, dq=D["dq"], dk=D["dk"],
                                   dv=D["dv"], stream=stream, deterministic=args.deterministic,
                                   **kw)
    else:
        shp = Shape(w["B"], w["H"], w["S_q"], w["S_kv"], w["D_qk"], w["D_v"], w.get("H_kv", 0))
        x = make_inputs(shp, w["dtype"], with_bias=w["bias"], seed_base=rank, device=dev)
        o = torch.empty(shp.B, shp.H, shp.S_q, shp.D_v, dtype=x["q"].dtype, device=dev)
        lse = torch.empty(shp.B, shp.H, shp.S_q, dtype=torch.float32, device=dev)
        ws = torch.empty(sdpa_bwd_workspace_size(shp.B, shp.H, shp.S_q, shp.S_kv, shp.D_qk,
                                                 shp.D_v, shp.kv_heads,
                                                 deterministic=args.deterministic),
                         dtype=torch.uint8, device=dev)

        rec_fwd = {"dropout_mask_out": keep_record} if record_words else {}
        rec_bwd = {"dropout_mask": keep_record} if record_words else {}

        def fwd_call(D):
            sdpa_fwd(D["q"], D["k"], D["v"], out=D["o"], lse=D["lse"], bias=D["bias"], **kw,
                     **rec_fwd)

        def bwd_call(ph, D, stream=None):
            sdpa_bwd_phases(ph, D["q"], D["k"], D["v"], D["o"], D["do"], D["lse"], workspace=ws,
                            dq=D["dq"], dk=D["dk"], dv=D["dv"], bias=D["bias"], dbias=D["dbias"],
                            stream=stream, deterministic=args.deterministic, **kw, **rec_bwd)
    # The default backward at d_qk <= 128 is the fused one: the preprocess,
    # one key/value-stationary kernel that also accumulates dQ, and the dQ
    # convert pass, one after the other. Otherwise (d_qk = 192,
    # --deterministic) the dK/dV and dQ kernels run concurrently after the
    # preprocess.
    fused = not args.deterministic and w["D_qk"] <= 128
    # With one key tile that every query tile meets (here: s_kv <= 128 under a
    # plain mask, no grouped heads) the fused kernel writes dQ itself: no
    # accumulator, no convert pass (sdpa_bwd decides the same way).
    direct = (fused and not packed and w["S_kv"] <= 128 and w.get("window") is None
              and not w.get("bottom_right") and w.get("H_kv", w["H"]) == w["H"])
    q, k, v, do, bias = x["q"], x["k"], x["v"], x["do"], x["bias"]
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)

    def philox_peak_gblocks(wl):
        """Philox4x32-10 blocks per second (G) of sdpa_dropout_mask over the
        workload's [B, H, S_q, S_kv] elements: the path's ALU roofline."""
        nb = 1 if wl.get("lens") else wl["B"]
        words = (nb * wl["H"] * wl["S_q"] * wl["S_kv"] + 31) // 32
        buf = torch.empty(words, dtype=torch.int32, device=dev)
        best = None
        for _ in range(6):
            a, b2 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(torch.cuda.current_stream())
            sdpa_dropout_mask(nb, wl["H"], wl["S_q"], wl["S_kv"], wl["p"], DROP_SEED, DROP_OFFSET,
                              out=buf)
            b2.record(torch.cuda.current_stream())
            torch.cuda.synchronize()
            t = a.elapsed_time(b2)
            best = t if best is None else min(best, t)
        return nb * wl["H"] * wl["S_q"] * wl["S_kv"] / 4.0 / (best * 1e-3) / 1e9
    dbias = torch.empty_like(bias) if bias is not None else None
    set0 = {"q": q, "k": k, "v": v, "do": do, "bias": bias, "o": o, "lse": lse, "dq": dq,
            "dk": dk, "dv": dv, "dbias": dbias}
    stream = torch.cuda.current_stream()
    # The dK/dV kernel runs on a high-priority side stream, concurrently with
    # the dQ kernel on the main one (both need only the preprocess output), as
    # sdpa_bwd runs them: dQ's CTAs fill the SMs dK/dV's last wave leaves idle.
    side = torch.cuda.Stream(priority=-1)
    names = ["fwd", "bwd_pre", "bwd_dkdv", "bwd_dq"]

    def step(ev=None):
        # ev: fwd start, fwd end = pre start, pre end = dQ start, dQ end,
        # dK/dV start, dK/dV end (the last two on the side stream; fused:
        # all on one stream, dK/dV start = pre end, dK/dV end = dQ start)
        if ev is not None:
            ev[0].record(stream)
        if mask_words:  # the keep bits of this step, drawn once for all three kernels
            sdpa_dropout_mask(w["B"], w["H"], w["S_q"], w["S_kv"], w["p"], DROP_SEED, DROP_OFFSET,
                              out=kw["dropout_mask"])
        fwd_call(set0)
        if ev is not None:
            ev[1].record(stream)
        bwd_call(SDPA_BWD_PREPROCESS, set0)
        if fused:
            if ev is not None:
                ev[2].record(stream)
                ev[4].record(stream)
            bwd_call(SDPA_BWD_DKDV, set0)
            if ev is not None:
                ev[5].record(stream)
            bwd_call(SDPA_BWD_DQ, set0)
            if ev is not None:
                ev[3].record(stream)
            return
        fork = torch.cuda.Event()
        fork.record(stream)
        if ev is not None:
            ev[2].record(stream)
        side.wait_event(fork)
        if ev is not None:
            ev[4].record(side)
        bwd_call(SDPA_BWD_DKDV, set0, stream=side)
        if ev is not None:
            ev[5].record(side)
        bwd_call(SDPA_BWD_DQ, set0)
        if ev is not None:
            ev[3].record(stream)
        join = torch.cuda.Event()
        join.record(side)
        stream.wait_event(join)

    def user_step(D):
        # one step as a user runs it: the forward and the whole backward, one
        # call each (plus this step's keep bits where they are drawn beforehand)
        if mask_words:
            sdpa_dropout_mask(w["B"], w["H"], w["S_q"], w["S_kv"], w["p"], DROP_SEED, DROP_OFFSET,
                              out=kw["dropout_mask"])
        t0 = time.perf_counter()
        fwd_call(D)
        t1 = time.perf_counter()
        bwd_call(SDPA_BWD_ALL, D)
        t2 = time.perf_counter()
        return t1 - t0, t2 - t1

    # Inputs that fit in L2 (the smallest workload) are flushed out of it
    # between timed steps by writing a buffer twice its size; each step is
    # then timed by its own pair of events, so the flush is not counted.
    in_bytes = sum(t.numel() * t.element_size() for t in (q, k, v, do) if t is not None)
    in_bytes += bias.numel() * bias.element_size() if bias is not None else 0
    flush = torch.empty(2 * L2_BYTES, dtype=torch.uint8, device=dev) if in_bytes < L2_BYTES else None

    for _ in range(max(args.warmup, 0)):
        user_step(set0)
        step()
    torch.cuda.synchronize()
    if sdpa_device_error() != 0:
        raise SystemExit("a kernel wait ran out during warm-up")

    # timed region: K user steps, bracketed by a barrier and synchronize
    host_fwd = host_bwd = 0.0
    step_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(args.steps)] if flush is not None else []
    sampler = ClockSampler(local)
    sampler.start()
    barrier()
    torch.cuda.synchronize()
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    t_start.record(stream)
    for s_ in range(args.steps):
        if flush is not None:
            flush.zero_()
            step_ev[s_][0].record(stream)
        hf, hb = user_step(set0)
        host_fwd += hf
        host_bwd += hb
        if flush is not None:
            step_ev[s_][1].record(stream)
    t_end.record(stream)
    torch.cuda.synchronize()
    barrier()
    clocks = sampler.stop()
    if sdpa_device_error() != 0:
        raise SystemExit("a kernel wait ran out during the timed steps")
    if flush is not None:
        total_ms = sum(a.elapsed_time(b) for a, b in step_ev)
    else:
        total_ms = t_start.elapsed_time(t_end)
    host_us = {"sdpa_fwd": host_fwd / args.steps * 1e6, "sdpa_bwd": host_bwd / args.steps * 1e6}

    # per-kernel durations: the same K steps again, issued phase by phase with
    # events between the kernels (on the stream each kernel runs on)
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(6)] for _ in range(args.steps)]
    barrier()
    torch.cuda.synchronize()
    for s_ in range(args.steps):
        if flush is not None:
            flush.zero_()
        step(evs[s_])
    torch.cuda.synchronize()
    barrier()
    if sdpa_device_error() != 0:
        raise SystemExit("a kernel wait ran out during the per-kernel steps")
    per_kernel = {n: 0.0 for n in names}
    spans = {"fwd": (0, 1), "bwd_pre": (1, 2), "bwd_dkdv": (4, 5),
             "bwd_dq": (5, 3) if fused else (2, 3)}
    for e in evs:
        for n, (a, b) in spans.items():
            per_kernel[n] += e[a].elapsed_time(e[b])
    per_kernel = {n: t / args.steps for n, t in per_kernel.items()}
    ms = max_over_ranks(total_ms / args.steps, world, dev)

    # The smallest workload is bound by host time per call: a step issued call
    # by call back to back (no flush, what a loop of calls sees), and the same
    # step captured once in a CUDA graph and replayed.
    latency = None
    if fwd_flops(w) < 1e9:
        n_l = 200
        torch.cuda.synchronize()
        a_ev, b_ev = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a_ev.record(stream)
        for _ in range(n_l):
            user_step(set0)
        b_ev.record(stream)
        torch.cuda.synchronize()
        loop_us = a_ev.elapsed_time(b_ev) / n_l * 1e3
        graph_us = None
        g = torch.cuda.CUDAGraph()
        cap = torch.cuda.Stream()
        cap.wait_stream(stream)
        with torch.cuda.stream(cap):
            user_step(set0)
        stream.wait_stream(cap)
        torch.cuda.synchronize()
        with torch.cuda.graph(g, stream=cap):
            user_step(set0)
        for _ in range(10):
            g.replay()
        torch.cuda.synchronize()
        a_ev.record(stream)
        for _ in range(n_l):
            g.replay()
        b_ev.record(stream)
        torch.cuda.synchronize()
        graph_us = a_ev.elapsed_time(b_ev) / n_l * 1e3
        # host time of each call with the device idle before it (the launch
        # queue empty, so no call waits for room in it)
        hf = hb = 0.0
        for _ in range(n_l):
            torch.cuda.synchronize()
            a_, b_ = user_step(set0)
            hf += a_
            hb += b_
        torch.cuda.synchronize()
        if sdpa_device_error() != 0:
            raise SystemExit("a kernel wait ran out during the latency loops")
        host_us = {"sdpa_fwd": hf / n_l * 1e6, "sdpa_bwd": hb / n_l * 1e6}
        latency = {"device_us_per_step_l2_flushed": ms * 1e3,
                   "api_loop_us_per_step": loop_us,
                   "graph_replay_us_per_step": graph_us,
                   "host_us_per_call": host_us,
                   "method": "api loop: sdpa_fwd + sdpa_bwd called back to back 200 times, no "
                             "flush, events around the loop; graph: the same step captured once "
                             "in a CUDA graph (torch.cuda.graph) and replayed 200 times; host: "
                             "each call timed on the host with the device idle before it"}

    ff = fwd_flops(w)
    step_flops = 3.5 * ff
    value = whole_job_tflops(world, step_flops, ms)
    peaks, peak_kind = measured_peaks()
    peak = float(peaks["bf16_tflops"])
    hbm = float(peaks["hbm_gbs"])
    # display names: the fused backward's main kernel and its convert pass
    if fused:
        per_kernel = {{"bwd_dkdv": "bwd_fused", "bwd_dq": "dq_convert"}.get(n, n): t
                      for n, t in per_kernel.items()}
        if direct:  # the DQ phase launches nothing
            per_kernel.pop("dq_convert")

    # algorithmic FLOPs per launch: the dK/dV kernel forms S^T, dP^T, dV, dK
    # (2x the forward), the fused one dQ as well; the deterministic dQ
    # kernel's algorithmic share is the dQ product alone (its recomputed S and
    # dP are not counted); the preprocess and convert passes are memory
    # traffic only
    dq_share = 2.0 * w["D_qk"] / (w["D_qk"] + w["D_v"]) * 0.5 * ff
    if fused:
        kernel_flops = {"fwd": ff, "bwd_fused": 2.0 * ff + dq_share}
    else:
        kernel_flops = {"fwd": ff, "bwd_dkdv": 2.0 * ff, "bwd_dq": dq_share}
    kbytes = kernel_bytes(w, fused)
    if direct:  # the fused kernel writes dQ; no accumulator
        kbytes["bwd_fused"] += kbytes.pop("dq_convert") - (
            w["B"] * w["H"] * ((w["S_q"] + 127) // 128) * 128 * w["D_qk"] * 4)
    # Philox4x32-10 blocks (four elements each) a kernel draws per launch:
    # every visible element once in the forward and, unless the forward
    # recorded its keep bits for it, once in the main backward kernel(s)
    # (the deterministic dQ kernel draws them again)
    drawn = 0.0
    if w["p"] > 0 and not w.get("bits"):
        drawn = (1 if w.get("lens") else w["B"]) * w["H"] * visible_pairs_per_head(w) / 4.0
    drawers = ("fwd",) if record_words else ("fwd", "bwd_fused", "bwd_dkdv", "bwd_dq")
    kernel_blocks = {n: drawn for n in drawers if n in per_kernel}

    # the roofline of the workload's bound, for its dominant kernel (the
    # deterministic dQ span holds the concurrent dK/dV, so there the choice is
    # among the kernels timed alone)
    dom = max((n for n in per_kernel if fused or n != "bwd_dq"), key=per_kernel.get)
    bound = workload_bound(w, ff / 1e9, bool(kernel_blocks.get(dom)))
    sec = per_kernel[dom] * 1e-3
    traffic = None
    tpath = os.path.join(ROOT, "profiles", "traffic.json")
    if os.path.exists(tpath) and dom in KERNEL_SOURCES:
        with open(tpath) as f:
            tr = json.load(f).get(args.workload, {}).get(dom)
        if tr and tr.get("source_sha") == source_sha(dom):
            traffic = tr.get("bytes_per_launch")
    if bound == "tensor" and dom in kernel_flops:
        achieved = kernel_flops[dom] / sec / 1e12
        roof = {"bound": "tensor", "kernel": dom, "achieved": achieved, "peak": peak,
                "unit": "TFLOP/s", "frac": achieved / peak, "traffic": traffic,
                "peak_source": f"{peak_kind} bf16 dense (burst)"}
    elif bound == "alu" and kernel_blocks.get(dom):
        # peak: the same Philox4x32-10 arithmetic alone at full occupancy,
        # sdpa_dropout_mask over this workload's elements (timed here)
        alu_peak = philox_peak_gblocks(w)
        achieved = kernel_blocks[dom] / sec / 1e9
        roof = {"bound": "alu", "kernel": dom, "achieved": achieved, "peak": alu_peak,
                "unit": "G Philox4x32-10 blocks/s", "frac": achieved / alu_peak,
                "traffic": traffic,
                "peak_source": "measured: sdpa_dropout_mask (the same Philox draws, nothing else) "
                               "over this workload's elements, best of 5"}
    else:
        achieved = kbytes[dom] / sec / 1e9
        roof = {"bound": "hbm", "kernel": dom, "achieved": achieved, "peak": hbm, "unit": "GB/s",
                "frac": achieved / hbm, "traffic": traffic,
                "peak_source": f"{peak_kind} HBM copy",
                "bytes_per_launch": kbytes[dom]}
    if bound != "tensor":
        roof["tensor_frac"] = (kernel_flops.get(dom, 0.0) / sec / 1e12) / peak
    if dom == "bwd_dkdv" and w["bias"]:
        # the deterministic backward zeroes dBias inside its dK/dV phase, on
        # the kernel's stream right before it (so that the pass overlaps the
        # dQ kernel); the events around the phase hold both launches
        roof["span"] = ("the dK/dV phase: the dBias zero pass, then the dK/dV kernel, on one stream; "
                        "achieved and frac are lower bounds for the kernel alone")

    # End to end through the public API (sdpa_fwd + sdpa_bwd, or their packed
    # forms: the calls a user makes) with pinned host buffers: every step uploads its inputs and reads
    # back its results. Two sets of device tensors and two copy streams let the
    # upload of step n+1 and the read-back of step n-1 overlap step n's
    # compute, the way a serving loop would run; each step still moves all its
    # bytes through the host link. A set's inputs are refilled once the step
    # two back has read them (its kernels are done), and its outputs are
    # rewritten once that step's read-back is done, so an upload and a
    # read-back need not follow one another within one step's compute. The
    # first upload and the last read-back are inside the timed region too.
    e2e = None
    if args.e2e_steps > 0:
        in_names = ["q", "k", "v", "do"] + (["bias"] if bias is not None else [])
        out_names = ["o", "lse", "dq", "dk", "dv"] + (["dbias"] if dbias is not None else [])
        set1 = {n: (torch.empty_like(t) if t is not None else None) for n, t in set0.items()}
        sets = [set0, set1]
        hin = {n: set0[n].cpu().pin_memory() for n in in_names}
        hout = {n: torch.empty(set0[n].shape, dtype=set0[n].dtype).pin_memory() for n in out_names}
        h2d = sum(t.numel() * t.element_size() for t in hin.values())
        d2h = sum(t.numel() * t.element_size() for t in hout.values())
        s_in, s_cmp, s_out = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
        n_e = args.e2e_steps
        ev_in = [torch.cuda.Event() for _ in range(n_e)]
        ev_cmp = [torch.cuda.Event() for _ in range(n_e)]
        ev_out = [torch.cuda.Event() for _ in range(n_e)]
        barrier()
        torch.cuda.synchronize()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(s_in)
        for i in range(n_e):
            D = sets[i % 2]
            with torch.cuda.stream(s_in):
                if i >= 2:
                    s_in.wait_event(ev_cmp[i - 2])  # step i-2's kernels have read this set's inputs
                for n in in_names:
                    D[n].copy_(hin[n], non_blocking=True)
                ev_in[i].record(s_in)
            with torch.cuda.stream(s_cmp):
                s_cmp.wait_event(ev_in[i])
                if i >= 2:
                    s_cmp.wait_event(ev_out[i - 2])  # step i-2's results are read back from this set
                if mask_words:
                    sdpa_dropout_mask(w["B"], w["H"], w["S_q"], w["S_kv"], w["p"], DROP_SEED,
                                      DROP_OFFSET, out=kw["dropout_mask"], stream=s_cmp)
                fwd_call(D)
                bwd_call(SDPA_BWD_ALL, D)
                ev_cmp[i].record(s_cmp)
            with torch.cuda.stream(s_out):
                s_out.wait_event(ev_cmp[i])
                for n in out_names:
                    hout[n].copy_(D[n], non_blocking=True)
                ev_out[i].record(s_out)
        e1.record(s_out)
        torch.cuda.synchronize()
        barrier()
        e2e_ms = max_over_ranks(e0.elapsed_time(e1) / n_e, world, dev)
        e2e = {"value": whole_job_tflops(world, step_flops, e2e_ms), "unit": UNIT,
               "ms_per_step": e2e_ms, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
               "steps": n_e,
               "host_cpus": host_cpus,
               "method": ("sdpa_fwd_varlen + sdpa_bwd_varlen" if packed else "sdpa_fwd + sdpa_bwd") +
                         " from pinned host buffers; uploads of step n+1 and "
                         "read-backs of step n-1 overlap step n on two copy streams "
                         "(double-buffered device tensors)"}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        secs, flops = oracle_sample(w, args.cpu_sample)
        cpu = {"value": flops / secs / 1e12, "unit": UNIT, "cores": cpu_threads(),
               "kind": "oracle",
               "sample": (f"one head (of {w['B'] * w['H']}), first {min(args.cpu_sample, w['S_q'])} "
                          f"query positions of the workload, fp64 numpy oracle fwd+bwd "
                          f"({secs:.1f} s)")}

    if rank == 0:
        kt = {n: {"ms": t} for n, t in per_kernel.items()}
        for n, t in per_kernel.items():
            if n in kernel_flops and not (n == "bwd_dq"):
                kt[n]["tflops"] = kernel_flops[n] / (t * 1e-3) / 1e12
            if n in kbytes:
                gbs = kbytes[n] / (t * 1e-3) / 1e9
                kt[n]["gbs"] = gbs
                kt[n]["hbm_frac"] = gbs / hbm
            if kernel_blocks.get(n):
                kt[n]["philox_gblocks_per_s"] = kernel_blocks[n] / (t * 1e-3) / 1e9
        if fused and direct:
            kt["bwd_fused"]["note"] = ("fused key/value-stationary kernel: S^T, dP^T, dV, dK and dQ "
                                       "(one key tile: dQ written directly, no convert pass)")
        elif fused:
            kt["bwd_fused"]["note"] = ("fused key/value-stationary kernel: S^T, dP^T, dV, dK and dQ "
                                       "(fp32 reductions into the workspace accumulator)")
            kt["dq_convert"]["note"] = "dQ = scale * dQacc convert pass"
        else:
            kt["bwd_dq"]["tflops_algorithmic"] = dq_share / (per_kernel["bwd_dq"] * 1e-3) / 1e12
            kt["bwd_dq"]["tflops_executed"] = (dq_share + ff) / (per_kernel["bwd_dq"] * 1e-3) / 1e12
            kt["bwd_dq"]["note"] = ("span from the end of the preprocess to the end of dQ, which "
                                    "runs concurrently with dK/dV (side stream) and fills its "
                                    "last wave; gbs counts its own bytes over that span")
        # dK/dV and dQ overlap: the backward is the step without the forward
        bwd_ms = ms - per_kernel["fwd"]
        out = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": w["dtype"], "data": "synthetic (seeded normal inputs, no dataset)",
            "config": {"workload": args.workload, "B": w["B"], "H": w["H"],
                       "H_kv": w.get("H_kv", w["H"]), "S_q": w["S_q"],
                       "S_kv": w["S_kv"], "D_qk": w["D_qk"], "D_v": w["D_v"],
                       **({"packed_lengths": w["lens"], "total_tokens": sum(w["lens"])}
                          if packed else {}),
                       "causal": w["causal"], "bias": w["bias"], "dropout_p": w["p"],
                       **({"window": list(w["window"]), "bottom_right": w.get("bottom_right", False)}
                          if w.get("window") is not None else {}),
                       **({"alibi": "slopes 2^(-8(h+1)/H)"} if w.get("alibi") else {}),
                       "backward": "fused (dQ by fp32 reductions)" if fused else "deterministic",
                       **({"dropout_bits": "drawn once by the forward, recorded, read by the "
                                           "backward"} if record_words else {}),
                       "l2": ("inputs smaller than L2: a 2x L2 buffer written between timed "
                              "steps, each step timed by its own events"
                              if flush is not None else "inputs larger than L2, no flush"),
                       "parallelism": f"{world} independent replicas" if world > 1 else "1 GPU"},
            "pct_of_peak": 100.0 * value / world / peak,
            "fwd_tflops": ff / (per_kernel["fwd"] * 1e-3) / 1e12,
            "bwd_tflops": 2.5 * ff / (bwd_ms * 1e-3) / 1e12,
            "kernels": kt,
            "roofline": roof, "cpu_baseline": cpu, "e2e": e2e, "clocks": clocks,
            "host_us_per_call": host_us,
            **({"latency_us_per_step": ms * 1e3, "latency": latency} if latency else {}),
            # per step: forward, preprocess, two backward kernels, plus the keep
            # bits' kernel where the step draws them beforehand or the forward
            # draws its record with it (no mask)
            "gpu_launches": ((5 if (mask_words or (record_words and not w["causal"]
                                                   and w.get("window") is None))
                              else 4) - (1 if direct else 0)) * args.steps,
        }
        print(json.dumps(out), flush=True)
    if world > 1:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
