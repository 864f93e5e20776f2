"""Benchmark of the quantized matrix product on GB300.

Headline (one JSON line on stdout): decode qGEMV weight-GB/s on the 2B-class
MLP projections, INT4 group-64 affine codes: a step is one decode pass through
L layers, each layer an up-projection (K=2048 -> N=6144) and a
down-projection (K=6144 -> N=2048) with its own weights and activations.  L
is chosen so that one step's weights exceed the L2 cache several times, so
every timed step reads its codes from HBM (no flush needed).  The other
decode and prefill shapes are measured the same way and reported under
"per_config".

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Under torchrun (N > 1) every rank runs the same per-GPU workload on its own
GPU with no data exchange (weak scaling); the timed region is bracketed by a
barrier and the slowest rank's time is used.

--impl reference times the CPU oracle (plain C, FP64, all host cores) on a
bounded sample of the same workload: the reference arm for this method.
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
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from quantized_weight_gb300 import inputs  # noqa: E402

HEADLINE_UP = "decode_int4_up_k2048_n6144"
HEADLINE_DOWN = "decode_int4_down_k6144_n2048"
WORKLOAD_NAME = "decode_int4_g64_mlp_up_k2048_n6144+down_k6144_n2048"
METRIC = "decode qGEMV weight-GB/s (% of HBM peak)"
NOMINAL_HBM_GBS = 8000.0
TRAFFIC_JSON = os.path.join(ROOT, "profiles", "traffic.json")
HEADLINE_KERNEL = "gemv_tc_kernel (INT4 tensor-core decode product)"


# ---------------------------------------------------------------- algorithmic work

def gemv_bytes(M, N, K, bits, group):
    """Bytes a decode product must move: codes + coefficients + x + y."""
    codes = N * K * bits // 8
    coeffs = N * (K // group) * 2 * (2 if bits == 4 else 1)
    return codes + coeffs + M * K * 4 + M * N * 4


def gemm_flops(M, N, K):
    return 2.0 * M * N * K


# ---------------------------------------------------------------- environment

def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return {"hbm_gbs": d["hbm_gbs"], "bf16_tflops": d["bf16_tflops"],
                "bf16_tflops_sustained": d.get("bf16_tflops_sustained"), "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "source": "fallback"}


class ClockSampler:
    """nvidia-smi clock / throttle-reason samples while the GPU is under load."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,utilization.gpu,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.QUERY}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except (FileNotFoundError, OSError):
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.thread.join(timeout=2)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [t.strip() for t in ln.split(",")]
            if len(f) < 10:
                continue
            try:
                util = float(f[4])
                mhz, mx = float(f[1]), float(f[2])
            except ValueError:
                continue
            if util < 5:
                continue
            sm.append(mhz)
            smax.append(mx)
            for name, v in zip(names, f[6:10]):
                if v.lower() == "active":
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax), "reasons": sorted(reasons),
                "samples": len(sm)}


# ---------------------------------------------------------------- device workloads

def device_inputs(name, seed, torch, qmm):
    w = inputs.WORKLOADS[name]
    d = inputs.make(w.M, w.N, w.K, w.bits, w.group, seed, w.prefill)
    dev = "cuda"
    codes = torch.from_numpy(d["codes"]).to(dev)
    t = {
        "packed": qmm.pack(codes, w.bits),
        "scales": torch.from_numpy(d["scales"].view(np.float16)).to(dev),
        "biases": None if d["biases"] is None else torch.from_numpy(d["biases"].view(np.float16)).to(dev),
        "x": torch.from_numpy(d["x"]).to(dev),
    }
    if w.prefill:
        t["x_bf16"] = torch.from_numpy(d["x_bf16"].view(np.int16)).to(dev).view(torch.bfloat16)
    del codes
    return w, d, t


def replicate(t, copies, torch):
    """`copies` independent device copies (distinct HBM) of one set of inputs."""
    out = [t]
    for _ in range(copies - 1):
        out.append({k: (None if v is None else v.clone()) for k, v in t.items()})
    return out


def l2_bytes(torch):
    try:
        return torch.cuda.get_device_properties(0).L2_cache_size
    except Exception:
        return 126 * 1024 * 1024


class Chain:
    """A list of products launched back to back on one stream; captured in a CUDA graph."""

    def __init__(self, calls, torch):
        self.calls = calls
        self.torch = torch
        self.graph = None
        self.stream = None

    def launch_eager(self):
        for c in self.calls:
            c()

    def capture(self, stream):
        torch = self.torch
        with torch.cuda.stream(stream):
            self.launch_eager()          # first run outside capture (loads the kernels)
        stream.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            self.launch_eager()
        self.graph = g
        self.stream = stream
        return self

    def replay(self):
        # a graph launches on the current stream: make that the timed stream
        with self.torch.cuda.stream(self.stream):
            self.graph.replay()


def time_graph(chain, reps, warmup, torch, stream):
    for _ in range(warmup):
        chain.replay()
    stream.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(reps):
        chain.replay()
    e1.record(stream)
    e1.synchronize()
    return e0.elapsed_time(e1) / 1000.0 / reps      # seconds per replay


def gemv_call(qmm, t, w, y):
    return lambda: qmm.gemv(t["x"], t["packed"], t["scales"], t["biases"], w.N, w.bits, w.group, out=y)


def gemm_call(qmm, t, w, y):
    return lambda: qmm.gemm(t["x_bf16"], t["packed"], t["scales"], t["biases"], w.N, w.bits, w.group, out=y)


def measure_config(name, torch, qmm, stream, pk, reps=20):
    """Per-launch time of one workload with L2-cold weights (copies > L2)."""
    w, d, t = device_inputs(name, 0, torch, qmm)
    if w.prefill:
        per = w.N * w.K * w.bits // 8 + w.M * w.K * 2 + w.N * (w.K // w.group) * (4 if w.bits == 4 else 2)
    else:
        per = gemv_bytes(w.M, w.N, w.K, w.bits, w.group)
    copies = max(2, min(64, -(-4 * l2_bytes(torch) // per)))
    if w.prefill and w.N * w.K * w.bits // 8 > l2_bytes(torch):
        copies = 2
    ts = replicate(t, copies, torch)
    ys = [torch.empty((w.M, w.N), dtype=torch.float32, device="cuda") for _ in range(copies)]
    mk = gemm_call if w.prefill else gemv_call
    chain = Chain([mk(qmm, ts[i], w, ys[i]) for i in range(copies)], torch).capture(stream)
    sec = time_graph(chain, reps, 3, torch, stream) / copies
    out = {"M": w.M, "N": w.N, "K": w.K, "bits": w.bits, "group": w.group, "us_per_launch": sec * 1e6,
           "copies": copies}
    if w.prefill:
        tf = gemm_flops(w.M, w.N, w.K) / sec / 1e12
        out.update({"tflops": tf, "frac_of_measured_bf16": tf / pk["bf16_tflops"]})
    else:
        gbs = gemv_bytes(w.M, w.N, w.K, w.bits, w.group) / sec / 1e9
        out.update({"gbs": gbs, "frac_of_measured_hbm": gbs / pk["hbm_gbs"],
                    "frac_of_8tbs": gbs / NOMINAL_HBM_GBS})
    out["parity_vs_oracle"] = sampled_parity(w, d, ys[0].cpu().numpy())
    del ts, ys, chain
    torch.cuda.empty_cache()
    return out


EXTRA_WORKLOADS = {
    # greedy argmax over the tied output head (no logits written): weight-GB/s
    "head_argmax_int4_m1_k2048_n151936": ("argmax", 1, 151936, 2048),
    # stored-format INT4 quantization of a 2B-class up-projection: bytes read + written per second
    "quantize_int4_g64_k2048_n6144": ("quantize", 0, 6144, 2048),
    # embedding lookup of 256 token ids in the tied INT4 table: bytes read + written per second
    "gather_dequant_int4_t256_k2048_n151936": ("gather", 256, 151936, 2048),
}


def measure_extra(name, torch, qmm, stream, pk, reps=20):
    """Per-launch time of the quantizer, gather and greedy-head entry points
    (inputs in HBM, copies larger than L2 where the inputs are reused)."""
    kind, M, N, K = EXTRA_WORKLOADS[name]
    L2 = l2_bytes(torch)
    if kind == "argmax":
        d = inputs.make(1, N, K, 4, 64, 0)
        t = {"x": torch.from_numpy(d["x"]).cuda(),
             "packed": qmm.pack(torch.from_numpy(d["codes"]).cuda(), 4),
             "scales": torch.from_numpy(d["scales"].view(np.float16)).cuda(),
             "biases": torch.from_numpy(d["biases"].view(np.float16)).cuda()}
        nbytes = gemv_bytes(1, N, K, 4, 64) - 4 * N          # no logits are written
        copies = max(2, -(-4 * L2 // nbytes))
        ts = replicate(t, copies, torch)
        ws = [qmm.argmax_workspace(1, N) for _ in range(copies)]
        res = [None] * copies

        def head(i):
            res[i] = qmm.gemv_argmax(ts[i]["x"], ts[i]["packed"], ts[i]["scales"], ts[i]["biases"], N, 4, 64,
                                     ws[i], idx=res[i][0] if res[i] else None, val=res[i][1] if res[i] else None)
        calls = [(lambda i=i: head(i)) for i in range(copies)]
        for i in range(copies):
            head(i)                              # result tensors exist before capture
    elif kind == "quantize":
        w = torch.randn((N, K), device="cuda", generator=torch.Generator("cuda").manual_seed(0)) * 0.05
        nbytes = N * K * 4 + N * K // 2 + N * (K // 64) * 4
        copies = max(2, -(-4 * L2 // nbytes))
        ws = [w.clone() for _ in range(copies)]
        outs = [(torch.empty((N, K // 8), dtype=torch.int32, device="cuda"),
                 torch.empty((N, K // 64), dtype=torch.float16, device="cuda"),
                 torch.empty((N, K // 64), dtype=torch.float16, device="cuda")) for _ in range(copies)]
        calls = [(lambda i=i: qmm.quantize(ws[i], 64, out=outs[i])) for i in range(copies)]
    else:
        d = inputs.make(1, N, K, 4, 64, 0)
        packed = qmm.pack(torch.from_numpy(d["codes"]).cuda(), 4)
        sc = torch.from_numpy(d["scales"].view(np.float16)).cuda()
        bi = torch.from_numpy(d["biases"].view(np.float16)).cuda()
        ids = torch.from_numpy(np.random.default_rng(0).integers(0, N, M).astype(np.int32)).cuda()
        nbytes = M * (K // 2 + (K // 64) * 4) + M * 4 + M * K * 4
        copies = 8
        outs = [torch.empty((M, K), device="cuda") for _ in range(copies)]
        calls = [(lambda i=i: qmm.gather_dequant(ids, packed, sc, bi, N, K, 4, 64, out=outs[i]))
                 for i in range(copies)]
    chain = Chain(calls, torch).capture(stream)
    sec = time_graph(chain, reps, 3, torch, stream) / copies
    gbs = nbytes / sec / 1e9
    torch.cuda.synchronize()
    if kind == "argmax":
        parity = head_parity(d, N, K, int(res[0][0].item()), float(res[0][1].item()))
    elif kind == "quantize":
        parity = quantize_parity(ws[0].cpu().numpy(), [o.cpu().numpy() for o in outs[0]])
    else:
        parity = gather_parity(d, ids.cpu().numpy(), outs[0].cpu().numpy(), K)
    del chain
    torch.cuda.empty_cache()
    return {"kind": kind, "M": M, "N": N, "K": K, "us_per_launch": sec * 1e6, "bytes_per_launch": nbytes,
            "gbs": gbs, "frac_of_measured_hbm": gbs / pk["hbm_gbs"], "copies": copies,
            "parity_vs_oracle": parity}


def head_parity(d, N, K, idx, val):
    """The greedy head's winner against the oracle's full FP64 logits: the
    winner's logit must be within the float32 accumulation bound of the
    largest one, and its reported value within that bound of its own logit."""
    import oracle
    y = oracle.qmm_f32x(d["x"], oracle.pack(d["codes"], 4), d["scales"], d["biases"], N, K, 4, 64)[0]
    top = int(np.argmax(y))
    # |sum of K float32 products| error bound: K * 2^-23 * sum |x_k w_k| (taken loosely over the winner row)
    w = oracle.dequant(oracle.pack(d["codes"][[idx]], 4), d["scales"][[idx]], d["biases"][[idx]], 1, K, 4, 64)[0]
    bound = K * 2.0 ** -23 * float(np.sum(np.abs(d["x"][0].astype(np.float64) * w)))
    return {"oracle_argmax": top, "idx": idx, "gap_to_max": float(y[top] - y[idx]),
            "val_err": float(abs(val - y[idx])), "bound": bound,
            "ok": bool(y[top] - y[idx] <= 2 * bound and abs(val - y[idx]) <= bound)}


def quantize_parity(w, outs, rows=64):
    """Bit-exact comparison of sampled rows of the stored-format quantizer's
    outputs (packed codes, scales, biases) with the oracle's quantizer."""
    import oracle
    sel = np.random.default_rng(1).choice(w.shape[0], rows, replace=False)
    codes, sc, bi = oracle.quantize_affine4_f32(w[sel], 64)
    packed = oracle.pack(codes, 4)
    same = (np.array_equal(outs[0][sel].view(np.uint32), packed.view(np.uint32))
            and np.array_equal(outs[1][sel].view(np.uint16), sc) and np.array_equal(outs[2][sel].view(np.uint16), bi))
    return {"rows": rows, "bit_exact": bool(same)}


def gather_parity(d, ids, out, K, rows=32):
    """Sampled gathered rows against the oracle's dequantized table rows (bit-exact)."""
    import oracle
    pos = np.random.default_rng(1).choice(len(ids), rows, replace=False)
    sel = ids[pos]
    ref = oracle.dequant(oracle.pack(d["codes"][sel], 4), d["scales"][sel], d["biases"][sel], rows, K, 4, 64)
    same = np.array_equal(out[pos].astype(np.float32).view(np.uint32), ref.astype(np.float32).view(np.uint32))
    return {"rows": rows, "bit_exact": bool(same)}


def sources_sha256(paths):
    """sha256 over the listed repository files, in order."""
    h = hashlib.sha256()
    for rel in paths:
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()


def traffic_from_profile():
    """DRAM bytes per launch of the headline kernel, from the committed ncu
    figures in profiles/traffic.json, or None if the file is missing or a
    source file the kernel is built from changed since the capture."""
    if not os.path.exists(TRAFFIC_JSON):
        return None
    try:
        d = json.load(open(TRAFFIC_JSON))
        rec = d["headline"]
        if sources_sha256(rec["sources"]) != rec["sources_sha256"]:
            return None
        return float(rec["bytes_per_launch"])
    except (OSError, KeyError, ValueError, TypeError):
        return None


# ---------------------------------------------------------------- sampled parity

def sampled_parity(w, d, y, nsample=256, seed=1):
    """Relative L2 error and the largest element error (over the oracle's
    largest |y|) of `nsample` outputs of y (a host float32 array [M, N])
    against the oracle evaluated at those outputs only."""
    import oracle
    rng = np.random.default_rng(seed)
    ms = rng.integers(0, w.M, nsample)
    ns = rng.integers(0, w.N, nsample)
    x = d["x_bf16"] if w.prefill else d["x"]
    sel = np.unique(ns)
    remap = {int(n): i for i, n in enumerate(sel)}
    sub = oracle.pack(d["codes"][sel], w.bits)
    ref = oracle.qmm_sampled(x, sub, d["scales"][sel], None if d["biases"] is None else d["biases"][sel],
                             ms, np.array([remap[int(n)] for n in ns]), len(sel), w.K, w.bits, w.group)
    got = y[ms, ns].astype(np.float64)
    err = got - ref
    return {"samples": int(nsample), "rel_l2": float(np.linalg.norm(err) / np.linalg.norm(ref)),
            "max_err_over_max_ref": float(np.max(np.abs(err)) / np.max(np.abs(ref)))}


# ---------------------------------------------------------------- multi-rank host logic

def slowest_rank_seconds(sec, world, device):
    """The timed region's length on the slowest rank (every rank gets it).
    One rank per GPU, each timing its own replica of the workload; the job
    finishes when the slowest one does."""
    if world <= 1:
        return sec
    import torch
    import torch.distributed as dist
    t = torch.tensor([sec], device=device, dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_gbs(bytes_per_step, steps, world, sec):
    """Whole-job weight-GB/s: the bytes all ranks processed over the slowest
    rank's time (weak scaling: every rank runs the same per-GPU workload)."""
    return bytes_per_step * steps * world / sec / 1e9


# ---------------------------------------------------------------- CPU oracle timing

def oracle_sample(seconds, nthreads=None):
    """The oracle, as it stands, on whole layers of the headline workload until
    `seconds` of CPU time have passed (at least one layer).  Returns
    (bytes processed, elapsed seconds, threads, layers)."""
    import oracle
    oracle.build()
    up, down = inputs.WORKLOADS[HEADLINE_UP], inputs.WORKLOADS[HEADLINE_DOWN]
    mats = []
    for w in (up, down):
        d = inputs.make(w.M, w.N, w.K, w.bits, w.group, 0)
        mats.append((w, d, oracle.pack(d["codes"], w.bits)))
    th = nthreads or max(1, len(os.sched_getaffinity(0)))
    done, layers = 0, 0
    t0 = time.perf_counter()
    while True:
        for w, d, p in mats:
            oracle.qmm_f32x(d["x"], p, d["scales"], d["biases"], w.N, w.K, w.bits, w.group, nthreads=th)
            done += gemv_bytes(w.M, w.N, w.K, w.bits, w.group)
        layers += 1
        el = time.perf_counter() - t0
        if el >= seconds:
            return done, el, th, layers


def run_reference(args, rank, world):
    if rank != 0:
        return
    up, down = inputs.WORKLOADS[HEADLINE_UP], inputs.WORKLOADS[HEADLINE_DOWN]
    per_layer = gemv_bytes(up.M, up.N, up.K, 4, 64) + gemv_bytes(down.M, down.N, down.K, 4, 64)
    import oracle
    oracle.build()
    mats = []
    for w in (up, down):
        d = inputs.make(w.M, w.N, w.K, w.bits, w.group, 0)
        mats.append((w, d, oracle.pack(d["codes"], w.bits)))
    th = max(1, len(os.sched_getaffinity(0)))

    def step():
        for w, d, p in mats:
            oracle.qmm_f32x(d["x"], p, d["scales"], d["biases"], w.N, w.K, w.bits, w.group, nthreads=th)

    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step()
    el = time.perf_counter() - t0
    gbs = per_layer * args.steps / el / 1e9
    sample = (f"{args.steps} steps x one layer (up + down projection, INT4 g64) of the "
              f"{WORKLOAD_NAME} workload on {th} host threads")
    line = {
        "impl": "reference", "metric": METRIC, "value": gbs, "unit": "GB/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": el / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": WORKLOAD_NAME, "layers_per_step": 1, "seed": 0},
        "cpu_baseline": {"value": gbs, "unit": "GB/s", "cores": th, "kind": "oracle", "sample": sample},
        "e2e": {"value": gbs, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def profile_workload(name, launches):
    """Plain launches of one workload on the current stream, nothing timed."""
    import torch
    from quantized_weight_gb300 import build as qbuild
    from quantized_weight_gb300 import qmm
    qbuild.build()
    if name in EXTRA_WORKLOADS and EXTRA_WORKLOADS[name][0] == "argmax":
        _, M, N, K = EXTRA_WORKLOADS[name]
        d = inputs.make(M, N, K, 4, 64, 0)
        t = {"x": torch.from_numpy(d["x"]).cuda(),
             "packed": qmm.pack(torch.from_numpy(d["codes"]).cuda(), 4),
             "scales": torch.from_numpy(d["scales"].view(np.float16)).cuda(),
             "biases": torch.from_numpy(d["biases"].view(np.float16)).cuda()}
        ws = qmm.argmax_workspace(M, N)
        f = lambda: qmm.gemv_argmax(t["x"], t["packed"], t["scales"], t["biases"], N, 4, 64, ws)
    else:
        w, d, t = device_inputs(name, 0, torch, qmm)
        y = torch.empty((w.M, w.N), dtype=torch.float32, device="cuda")
        f = (gemm_call if w.prefill else gemv_call)(qmm, t, w, y)
    for _ in range(launches):
        f()
    qmm.check()
    print(json.dumps({"profiled": name, "launches": launches}), flush=True)


# ---------------------------------------------------------------- main

def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-configs", action="store_true", help="skip the per-config table")
    ap.add_argument("--oracle-seconds", type=float, default=10.0)
    ap.add_argument("--no-clock-load", action="store_true",
                    help="skip the 1 s sustained replay after the timed region (for profiler runs)")
    ap.add_argument("--e2e-steps", type=int, default=50)
    ap.add_argument("--profile-workload", default=None,
                    help="only run LAUNCHES plain launches of one named workload (for profiler captures)")
    ap.add_argument("--launches", type=int, default=5)
    args = ap.parse_args()

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))

    if args.impl == "reference":
        return run_reference(args, rank, world)
    if args.profile_workload:
        return profile_workload(args.profile_workload, args.launches)

    import torch
    import torch.distributed as dist
    from quantized_weight_gb300 import build as qbuild
    from quantized_weight_gb300 import qmm

    qbuild.build()
    torch.cuda.set_device(local)
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    pk = peaks()
    stream = torch.cuda.Stream()

    def barrier():
        if world > 1:
            dist.barrier()

    # ---- headline: L layers of up + down projections, weights > 4x L2
    up_w, up_d, up_t = device_inputs(HEADLINE_UP, 0, torch, qmm)
    dn_w, dn_d, dn_t = device_inputs(HEADLINE_DOWN, 0, torch, qmm)
    layer_bytes = (gemv_bytes(1, up_w.N, up_w.K, 4, 64) + gemv_bytes(1, dn_w.N, dn_w.K, 4, 64))
    layers = max(8, -(-4 * l2_bytes(torch) // layer_bytes))
    ups, dns = replicate(up_t, layers, torch), replicate(dn_t, layers, torch)
    y_up = [torch.empty((1, up_w.N), device="cuda") for _ in range(layers)]
    y_dn = [torch.empty((1, dn_w.N), device="cuda") for _ in range(layers)]
    calls = []
    for i in range(layers):
        calls.append(gemv_call(qmm, ups[i], up_w, y_up[i]))
        calls.append(gemv_call(qmm, dns[i], dn_w, y_dn[i]))
    chain = Chain(calls, torch).capture(stream)
    step_bytes = layers * layer_bytes
    launches_per_step = 2 * layers

    # parity of the timed configuration, on sampled outputs (carried with the number)
    import oracle
    oracle.build()
    y0 = y_up[0].cpu().numpy()[0]
    ns = np.arange(0, up_w.N, 97)
    ref = oracle.qmm_sampled(up_d["x"], oracle.pack(up_d["codes"], 4), up_d["scales"], up_d["biases"],
                             np.zeros_like(ns), ns, up_w.N, up_w.K, 4, 64)
    parity = float(np.linalg.norm(y0[ns] - ref) / np.linalg.norm(ref))
    parity_dn = sampled_parity(dn_w, dn_d, y_dn[0].cpu().numpy())

    sampler = ClockSampler(local)
    sampler.start()
    time.sleep(0.3)
    for _ in range(args.warmup):
        chain.replay()
    stream.synchronize()
    barrier()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.steps):
        chain.replay()
    e1.record(stream)
    e1.synchronize()
    torch.cuda.synchronize()
    barrier()
    sec = e0.elapsed_time(e1) / 1000.0
    # keep the same load running long enough for the clock sampler to see it
    t_end = time.perf_counter() + (0.0 if args.no_clock_load else 1.0)
    while time.perf_counter() < t_end:
        for _ in range(50):
            chain.replay()
        stream.synchronize()
    clocks = sampler.stop()

    sec = slowest_rank_seconds(sec, world, "cuda")
    ms_per_step = sec / args.steps * 1e3
    value = job_gbs(step_bytes, args.steps, world, sec)
    per_launch_s = sec / args.steps / launches_per_step
    achieved = (step_bytes / launches_per_step) / per_launch_s / 1e9

    # ---- end to end through the public API: host activations in, host results out.
    # Every step copies all layers' activations from pinned host memory in one
    # copy per projection, runs the 2L products (qmm.gemv calls captured once in
    # a CUDA graph, as a decode loop runs them) and reads all results back.
    X_up = torch.stack([t["x"][0] for t in ups])          # [L, K_up]
    X_dn = torch.stack([t["x"][0] for t in dns])          # [L, K_dn]
    Y_up = torch.empty((layers, up_w.N), device="cuda")
    Y_dn = torch.empty((layers, dn_w.N), device="cuda")
    X_up_h, X_dn_h = X_up.cpu().pin_memory(), X_dn.cpu().pin_memory()
    Y_up_h = torch.empty(Y_up.shape, dtype=torch.float32).pin_memory()
    Y_dn_h = torch.empty(Y_dn.shape, dtype=torch.float32).pin_memory()
    e2e_calls = []
    for i in range(layers):
        e2e_calls.append(gemv_call(qmm, dict(ups[i], x=X_up[i:i + 1]), up_w, Y_up[i:i + 1]))
        e2e_calls.append(gemv_call(qmm, dict(dns[i], x=X_dn[i:i + 1]), dn_w, Y_dn[i:i + 1]))
    e2e_chain = Chain(e2e_calls, torch).capture(stream)
    h2d = (X_up_h.numel() + X_dn_h.numel()) * 4
    d2h = (Y_up_h.numel() + Y_dn_h.numel()) * 4

    def e2e_step():
        X_up.copy_(X_up_h, non_blocking=True)
        X_dn.copy_(X_dn_h, non_blocking=True)
        e2e_chain.graph.replay()
        Y_up_h.copy_(Y_up, non_blocking=True)
        Y_dn_h.copy_(Y_dn, non_blocking=True)

    e2e_steps = max(3, min(args.steps, args.e2e_steps))
    with torch.cuda.stream(stream):
        for _ in range(3):
            e2e_step()
        stream.synchronize()
        barrier()
        f0, f1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        f0.record(stream)
        for _ in range(e2e_steps):
            e2e_step()
        f1.record(stream)
        f1.synchronize()
        barrier()
    # the results read back are the products of the copied activations
    e2e_ok = bool(torch.equal(Y_up_h[0].cuda(), qmm.gemv(X_up[0:1], ups[0]["packed"], ups[0]["scales"],
                                                         ups[0]["biases"], up_w.N, 4, 64)[0]))
    e2e_sec = slowest_rank_seconds(f0.elapsed_time(f1) / 1000.0, world, "cuda")
    e2e_val = job_gbs(step_bytes, e2e_steps, world, e2e_sec)

    # the same end-to-end step without a graph: every product is its own C-ABI
    # call (qmm_gemv through ctypes, arguments marshalled in advance), so the
    # library's host-side validation and launch run inside the timed region
    L = qmm.lib()
    sh = stream.cuda_stream
    abi_args = []
    for i in range(layers):
        for t, w, X, Y in ((ups[i], up_w, X_up, Y_up), (dns[i], dn_w, X_dn, Y_dn)):
            abi_args.append((X[i:i + 1].data_ptr(), t["packed"].data_ptr(), t["scales"].data_ptr(),
                             t["biases"].data_ptr(), Y[i:i + 1].data_ptr(), 1, w.N, w.K, 4, 64, sh))

    def percall_step():
        X_up.copy_(X_up_h, non_blocking=True)
        X_dn.copy_(X_dn_h, non_blocking=True)
        for a in abi_args:
            rc = L.qmm_gemv(*a)
            if rc != 0:
                raise RuntimeError(f"qmm_gemv returned {rc}")
        Y_up_h.copy_(Y_up, non_blocking=True)
        Y_dn_h.copy_(Y_dn, non_blocking=True)

    with torch.cuda.stream(stream):
        for _ in range(3):
            percall_step()
        stream.synchronize()
        barrier()
        f0.record(stream)
        for _ in range(e2e_steps):
            percall_step()
        f1.record(stream)
        f1.synchronize()
        barrier()
    pc_ok = bool(torch.equal(Y_up_h[0].cuda(), qmm.gemv(X_up[0:1], ups[0]["packed"], ups[0]["scales"],
                                                        ups[0]["biases"], up_w.N, 4, 64)[0]))
    pc_sec = slowest_rank_seconds(f0.elapsed_time(f1) / 1000.0, world, "cuda")
    pc_val = job_gbs(step_bytes, e2e_steps, world, pc_sec)

    del chain, e2e_chain
    torch.cuda.empty_cache()

    per_config = {}
    if not args.no_configs:
        for name in inputs.WORKLOADS:
            try:
                per_config[name] = measure_config(name, torch, qmm, stream, pk)
            except Exception as ex:        # report, do not hide
                per_config[name] = {"error": repr(ex)}
        for name in EXTRA_WORKLOADS:
            try:
                per_config[name] = measure_extra(name, torch, qmm, stream, pk)
            except Exception as ex:
                per_config[name] = {"error": repr(ex)}

    line = {
        "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": WORKLOAD_NAME, "layers_per_step": layers, "bytes_per_step": step_bytes,
                   "launches_per_step": launches_per_step, "seed": 0,
                   "l2": f"inputs larger than L2: {step_bytes / 1e6:.0f} MB of weights per step vs "
                         f"{l2_bytes(torch) / 1e6:.0f} MB L2, each step reads every code from HBM",
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                   "graph": "CUDA graph per step, programmatic dependent launch between products"},
        "frac_of_8tbs": value / world / NOMINAL_HBM_GBS,
        "parity": {"sampled_rel_l2_vs_oracle": parity, "down_projection": parity_dn, "tolerance": 1e-5},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": pk["hbm_gbs"], "unit": "GB/s",
                     "frac": achieved / pk["hbm_gbs"], "traffic": traffic_from_profile(),
                     "kernel": HEADLINE_KERNEL,
                     "peak_source": pk["source"] + " (MEASURED_PEAKS.json hbm_gbs)"},
        "e2e": {"value": e2e_val, "unit": "GB/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "steps": e2e_steps, "results_checked": e2e_ok,
                "path": "pinned host x -> device (one copy per projection), the 2L qmm.gemv calls replayed "
                        "from a CUDA graph, device y -> pinned host (one copy per projection)",
                "per_call": {"value": pc_val, "unit": "GB/s", "ms_per_step": pc_sec / e2e_steps * 1e3,
                             "results_checked": pc_ok,
                             "path": "the same copies, and the 2L products as 2L qmm_gemv C-ABI calls from "
                                     "the host each step (no graph)"}},
        "gpu_launches": launches_per_step * args.steps,
        "clocks": clocks,
        "per_config": per_config,
    }
    if rank == 0 and world == 1:
        nbytes, el, th, nl = oracle_sample(args.oracle_seconds)
        n1, el1, _, nl1 = oracle_sample(args.oracle_seconds, nthreads=1)
        line["cpu_baseline"] = {"value": nbytes / el / 1e9, "unit": "GB/s", "cores": th, "kind": "oracle",
                                "sample": f"{nl} layers (up + down) of {WORKLOAD_NAME}, {el:.1f} s",
                                "single_thread": {"value": n1 / el1 / 1e9, "unit": "GB/s", "cores": 1,
                                                  "sample": f"{nl1} layers (up + down), {el1:.1f} s"}}
    elif rank == 0:
        line["cpu_baseline"] = None
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
