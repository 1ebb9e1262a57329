#!/usr/bin/env python3
"""Benchmark of exact multi-head attention (forward + backward) on GB300.

One step = the whole path over one batch: attn_fwd_with_workspace (O, LSE; at long sequences
V is first rounded to fp16 into its workspace), then the three backward phases
(attn_bwd_preprocess, attn_bwd_main, attn_bwd_dq_convert), all through the C ABI on device-
resident inputs.  Default workload: the long-text sequence, B=2, H=16, N=16384, d_k=128, bf16,
Q and K ~ N(0, 2^2), V and dO ~ N(0, 1), scale 1/sqrt(128).  The metric counts
4*B*H*N^2*d_k flops for the forward and 10*B*H*N^2*d_k for the backward.

Prints ONE JSON line (rank 0).  Under torchrun each rank runs its own batch on its own GPU
(independent problems; no data-path collective), `value` is the total over ranks divided by
the slowest rank's time.

--impl reference times the fp64 CPU oracle on a bounded sample of the same workload (one head,
its first --oracle-tokens tokens), the only other place this script runs the oracle.
"""
from __future__ import annotations

import argparse
import dataclasses
import hashlib
import json
import math
import os
import re
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "attention fwd/bwd TFLOPS (4·BHN²d / 10·BHN²d) and % of GB300 bf16 peak"
UNIT = "TFLOPS"
PROFILE_SUMMARY = os.path.join(ROOT, "profiles", "bwd_main_long_text.md")
KERNEL_SOURCES = [os.path.join(ROOT, "self_attention_gb300", "csrc", f)
                  for f in ("attn_bwd.cu", "common.cuh", "ptx.cuh")]
# the forward kernel's counters, hashed on its own sources
FWD_PROFILE_SUMMARY = os.path.join(ROOT, "profiles", "fwd_long_text.md")
FWD_KERNEL_SOURCES = [os.path.join(ROOT, "self_attention_gb300", "csrc", f)
                      for f in ("attn_fwd.cu", "common.cuh", "ptx.cuh")]
# NVIDIA's dense bf16 tensor figure for one GB300 GPU (no sparsity), a second denominator
# beside the measured cuBLAS peak
DATASHEET_BF16_TFLOPS = 2250.0
L2_BYTES = 129e6   # GB300 L2 capacity
# Peaks used when the measured-peaks file is absent (one earlier GB300 measurement).
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def parse_args(argv=None):
    p = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=60)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--workload", default="long_text")
    p.add_argument("--shape", default=None,
                   help="B,H,N,d override of the workload's sizes (profiling small cases)")
    # the first step's input copy and the last step's output copy overlap no compute; 30 steps
    # keep that fill and drain near 1 % of the end-to-end time
    p.add_argument("--e2e-steps", type=int, default=30)
    p.add_argument("--oracle-tokens", type=int, default=2048,
                   help="tokens of one head the CPU oracle runs on per reference-arm step")
    p.add_argument("--cpu-baseline-tokens", type=int, default=8192,
                   help="tokens of one head the CPU oracle runs on for cpu_baseline (~10-30 s)")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-configs", action="store_true",
                   help="skip the per-workload forward/backward table")
    p.add_argument("--no-parity", action="store_true",
                   help="skip the per-workload forward parity against the oracle")
    return p.parse_args(argv)


def workload(args):
    from self_attention_gb300.inputs import WORKLOADS
    w = WORKLOADS[args.workload]
    if args.shape:
        B, H, N, d = (int(x) for x in args.shape.split(","))
        w = dataclasses.replace(w, name=f"{w.name}_{B}x{H}x{N}x{d}", B=B, H=H, N=N, d=d)
    return w


def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def reduce_over_ranks(local: dict, world: int) -> dict:
    """MAX of every '*_ms' entry and SUM of every other numeric entry over the ranks (a single
    all_reduce of a small tensor per operation; nothing else crosses ranks)."""
    if world == 1:
        return dict(local)
    import torch
    import torch.distributed as dist
    keys = sorted(local)
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    mx = torch.tensor([float(local[k]) if k.endswith("_ms") else 0.0 for k in keys],
                      dtype=torch.float64, device=dev)
    sm = torch.tensor([0.0 if k.endswith("_ms") else float(local[k]) for k in keys],
                      dtype=torch.float64, device=dev)
    dist.all_reduce(mx, op=dist.ReduceOp.MAX)
    dist.all_reduce(sm, op=dist.ReduceOp.SUM)
    return {k: (mx[i] if k.endswith("_ms") else sm[i]).item() for i, k in enumerate(keys)}


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            pk = json.load(f)
        return {k: float(pk[k]) for k in FALLBACK_PEAKS}, "measured"
    except (OSError, KeyError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


def kernel_source_hash(sources=None) -> str:
    h = hashlib.sha256()
    for f in (KERNEL_SOURCES if sources is None else sources):
        with open(f, "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def profiled_traffic(units_per_launch: float, summary=None, sources=None):
    """DRAM bytes per launch of a kernel (by default the backward main kernel) from its
    committed ncu summary, scaled from the profiled case by the units (query x key tile pairs)
    a launch processes; None if the kernel's sources changed since the counters were taken."""
    try:
        text = open(PROFILE_SUMMARY if summary is None else summary).read()
    except OSError:
        return None
    m_hash = re.search(r"kernel_source_sha256:\s*([0-9a-f]+)", text)
    m_bytes = re.search(r"dram_bytes_per_unit:\s*([0-9.eE+]+)", text)
    if not m_hash or not m_bytes or m_hash.group(1) != kernel_source_hash(sources):
        return None
    return float(m_bytes.group(1)) * units_per_launch


class ClockSampler:
    """nvidia-smi clock / throttle-reason samples during the timed region."""
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")
    NAMES = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")

    def __init__(self, gpu_id: str):
        self.file = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100", "-i", gpu_id], stdout=self.file, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        self.proc.terminate()
        self.proc.wait()
        self.file.seek(0)
        sm, mx, reasons = [], [], set()
        for line in self.file.read().splitlines():
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 7:
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
            except ValueError:
                continue
            for name, val in zip(self.NAMES, parts[3:7]):
                if val.lower() == "active":
                    reasons.add(name)
        self.file.close()
        os.unlink(self.file.name)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": sorted(reasons),
                "samples": len(sm)}


def cpu_model() -> str:
    """The host CPU's model name (lscpu), else the machine type."""
    import platform
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.startswith("Model name:"):
                return f"{line.split(':', 1)[1].strip()} ({platform.machine()}, {os.cpu_count()} cores)"
    except (OSError, subprocess.SubprocessError):
        pass
    return f"{platform.machine()} ({os.cpu_count()} cores)"


def oracle_sample(w, tokens: int):
    """One head (b=0, h=0) of the workload, its first `tokens` tokens (same distribution)."""
    from self_attention_gb300.inputs import make_workload_inputs
    s = min(tokens, w.N)
    small = dataclasses.replace(w, B=1, H=1, N=s) if not w.model_dim else w
    inp = make_workload_inputs(small)
    sl = lambda t: t[:1, :1, :s].contiguous()
    return {x: sl(inp[x]) for x in ("q", "k", "v", "do")}, s


def time_oracle(w, tokens: int, repeats: int, outputs: dict | None = None):
    """Wall times of the oracle's forward + backward on the sample; `outputs`, if given, receives
    the sample and the last run's results."""
    import oracle
    sample, s = oracle_sample(w, tokens)
    oracle.build()
    times = []
    for _ in range(repeats):
        t0 = time.perf_counter()
        fwd = oracle.fwd(sample["q"], sample["k"], sample["v"], w.scale)
        bwd = oracle.bwd(sample["q"], sample["k"], sample["v"], sample["do"], w.scale)
        times.append(time.perf_counter() - t0)
    if outputs is not None:
        outputs.update(sample=sample, o=fwd[0], lse=fwd[1], dq=bwd["dq"], dk=bwd["dk"], dv=bwd["dv"])
    flops = 14.0 * s * s * w.d
    cores = int(os.environ.get("OMP_NUM_THREADS", os.cpu_count() or 1))
    desc = (f"oracle fwd+bwd (fp64, N x N materialised) on one head of {w.name}: its first {s} "
            f"tokens, d_k={w.d}; {14 * s * s * w.d:.3g} metric flops per run")
    return times, flops, cores, desc


def error_norms(got: dict, ref: dict) -> dict:
    """GPU results against the oracle's fp64 ones (numpy arrays keyed o, lse, dq, dk, dv): O max
    abs and relative Frobenius error, LSE relative error, the gradients' relative Frobenius
    errors.  The stated bounds are 1e-2, 5e-3, 1e-4 and 1e-2, with the O bound read as the bf16
    rounding floor where that exceeds 1e-2 (|O| >= 2, where one bf16 step is 2^-6 or more), so
    the O error is also given in bf16 steps of the reference value at its largest element."""
    import numpy as np
    rel_fro = lambda x: float(np.linalg.norm(got[x] - ref[x]) / max(np.linalg.norm(ref[x]), 1e-300))
    err = np.abs(got["o"] - ref["o"]).ravel()
    i = int(err.argmax())
    r_i = abs(float(ref["o"].ravel()[i]))
    step = 2.0 ** (math.floor(math.log2(max(r_i, 2.0 ** -126))) - 7)   # bf16: 8 significant bits
    return {"o_max_abs": float(err[i]), "o_ref_at_max": r_i, "o_max_abs_in_bf16_steps": float(err[i]) / step,
            "o_elems_over_1e-2": int((err > 1e-2).sum()), "o_rel_fro": rel_fro("o"),
            "lse_rel": float(np.abs(got["lse"] - ref["lse"]).max() / max(np.abs(ref["lse"]).max(), 1.0)),
            "dq_rel_fro": rel_fro("dq"), "dk_rel_fro": rel_fro("dk"), "dv_rel_fro": rel_fro("dv")}


def sample_parity(sa, w, ref: dict, stream) -> dict:
    """The GPU path (attn_fwd, attn_bwd) on the oracle's sample, against the oracle's results."""
    import torch
    q, k, v, do = (ref["sample"][x].cuda() for x in ("q", "k", "v", "do"))
    o, lse = sa.forward(q, k, v, w.scale, stream)
    dq, dk, dv = sa.backward(q, k, v, o, do, lse, w.scale, stream)
    torch.cuda.synchronize()
    got = {name: t.double().cpu().numpy() for name, t in
           (("o", o), ("lse", lse), ("dq", dq), ("dk", dk), ("dv", dv))}
    return error_norms(got, ref)


def parity_by_config(sa, stream, rows_per_head: int = 256) -> dict:
    """Forward parity on every workload's seeded inputs (the tests' inputs), in the launch
    configuration the workload runs in: the oracle evaluates sampled rows of three heads (every
    row where N <= 576) and the GPU's O and LSE there are compared with them.  Reports O max
    abs error, the elements over the stated 1e-2 with the smallest |O_ref| among them, the
    largest |O_ref|, O relative Frobenius error and LSE relative error on the sample; and the
    error of O before its bf16 rounding (attn_fwd_diagnostic, the same arithmetic), which
    separates the kernel's own error from the output rounding."""
    import numpy as np
    import torch
    import oracle
    from self_attention_gb300.inputs import WORKLOADS, make_workload_inputs
    oracle.build()
    out = {}
    for name, w in WORKLOADS.items():
        inp = make_workload_inputs(w)
        q, k, v = (inp[x].cuda() for x in ("q", "k", "v"))
        o, lse = sa.forward(q, k, v, w.scale, stream)
        _, _, o32 = sa.forward_diagnostic(q, k, v, w.scale, stream)
        torch.cuda.synchronize()
        o, lse = o.double().cpu().numpy(), lse.double().cpu().numpy()
        o32 = o32.double().cpu().numpy()
        del q, k, v
        rng = np.random.default_rng(11)
        err, ref_abs, d2, r2, lse_rel, n, err32 = [], [], 0.0, 0.0, 0.0, 0, 0.0
        for b, h in ((0, 0), (w.B - 1, w.H - 1), (w.B // 2, w.H // 3)):
            rows = (np.arange(w.N) if w.N <= 576 else
                    np.unique(np.concatenate([[0, w.N - 1], rng.integers(0, w.N, rows_per_head)])))
            o_ref, lse_ref = oracle.fwd_rows(inp["q"][b, h], inp["k"][b, h], inp["v"][b, h], rows, w.scale)
            o_ref, lse_ref = np.asarray(o_ref, np.float64), np.asarray(lse_ref, np.float64)
            e = np.abs(o[b, h, rows] - o_ref)
            err32 = max(err32, float(np.abs(o32[b, h, rows] - o_ref).max()))
            err.append(e.ravel())
            ref_abs.append(np.abs(o_ref).ravel())
            d2 += float((e ** 2).sum())
            r2 += float((o_ref ** 2).sum())
            lse_rel = max(lse_rel, float((np.abs(lse[b, h, rows] - lse_ref) /
                                          np.maximum(np.abs(lse_ref), 1.0)).max()))
            n += e.size
        err, ref_abs = np.concatenate(err), np.concatenate(ref_abs)
        over = err > 1e-2
        out[name] = {"elements": n, "o_max_abs": float(err.max()),
                     "o_ref_at_max": float(ref_abs[err.argmax()]),
                     "o_elems_over_1e-2": int(over.sum()),
                     "o_over_1e-2_min_abs_ref": float(ref_abs[over].min()) if over.any() else None,
                     "o_ref_max_abs": float(ref_abs.max()), "o_rel_fro": math.sqrt(d2 / r2),
                     "o_fp32_max_abs": err32, "lse_rel": lse_rel}
    return out


def workload_config(w, world: int) -> dict:
    """The `config` keys both arms report for a workload run on `world` GPUs (one batch each)."""
    return {"workload": w.name, "B": w.B, "H": w.H, "N": w.N, "d_k": w.d, "seq_len": w.N,
            "global_batch": w.B * world, "parallelism": f"independent batches x{world}",
            "qk_std": w.qk_std}


def run_reference(args, world, rank):
    if rank != 0:
        return 0
    w = workload(args)
    for _ in range(args.warmup):
        time_oracle(w, args.oracle_tokens, 1)
    times, flops, cores, desc = time_oracle(w, args.oracle_tokens, args.steps)
    per_step = sum(times) / len(times)
    value = flops / per_step / 1e12
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": per_step * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": workload_config(w, world),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                         "sample": desc, "cpu": cpu_model()},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def time_configs(sa, stream, peaks):
    """Forward and backward (all three phases) of every workload, attention only, on device
    inputs of the workload's shape and distribution.  Warm: back-to-back launches, mean.
    Flushed (the small shapes, whose inputs fit in L2): a 256 MB buffer is written before each
    launch, outside its events; median.  Graph (the small shapes): 20 launches captured in a
    CUDA graph and replayed, mean per launch, without host launch overhead.  GB/s counts the
    algorithmic bytes: forward reads Q, K, V and writes O, LSE; backward reads Q, K, V, O, dO,
    LSE and writes dQ, dK, dV.  fwd_unfused_*: standard attention (attn_fwd_unfused: S and P
    written to and read back from HBM) on the same inputs, warm, with the fused forward's
    speedup over it."""
    import torch
    from self_attention_gb300.inputs import WORKLOADS

    flush = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")
    ev = lambda: torch.cuda.Event(enable_timing=True)
    out = {}
    for name, w in WORKLOADS.items():
        B, H, N, D = w.B, w.H, w.N, w.d
        q = (torch.randn(B, H, N, D, device="cuda") * w.qk_std).bfloat16()
        k = (torch.randn(B, H, N, D, device="cuda") * w.qk_std).bfloat16()
        v, do = torch.randn_like(q), torch.randn_like(q)
        o, dq, dk, dv = (torch.empty_like(q) for _ in range(4))
        lse = torch.empty(B, H, N, device="cuda")
        wsb = sa.attn_bwd_workspace_size(B, H, N, D)
        ws = torch.empty(wsb, dtype=torch.uint8, device="cuda")
        fwsb = sa.attn_fwd_workspace_size(B, H, N, D)
        fws = torch.empty(fwsb, dtype=torch.uint8, device="cuda") if fwsb else None
        fwd = lambda st=stream: sa.attn_fwd_with_workspace(q, k, v, o, lse, fws, fwsb, B, H, N, D, w.scale, st)
        bwd = lambda st=stream: sa.attn_bwd(q, k, v, o, do, lse, dq, dk, dv, ws, wsb, B, H, N, D,
                                            w.scale, st)
        flops = B * H * N * N * D
        small = 2 * 4 * B * H * N * D < 130e6   # forward inputs + outputs fit in the 129 MB L2
        rep = 200 if small else (20 if flops < 1e11 else 5)
        row = {"B": B, "H": H, "N": N, "d_k": D}
        for tag, fn, fl, nbytes in (
                ("fwd", fwd, 4 * flops, B * H * N * D * 2 * 4 + 4 * B * H * N),
                ("bwd", bwd, 10 * flops, B * H * N * D * 2 * 8 + 4 * B * H * N)):
            for _ in range(5):
                fn()
            a, b = ev(), ev()
            a.record(stream)
            for _ in range(rep):
                fn()
            b.record(stream)
            torch.cuda.synchronize()
            us = a.elapsed_time(b) / rep * 1e3
            row[tag + "_us"] = us
            row[tag + "_tflops"] = fl / us / 1e6
            row[tag + "_gbs"] = nbytes / us / 1e3
            if small:
                # the same launch captured in a CUDA graph and replayed back to back: the time
                # without host-side launch overhead (what a captured training step sees)
                gs = torch.cuda.Stream()
                gs.wait_stream(stream)
                with torch.cuda.stream(gs):
                    fn(gs)
                gs.synchronize()
                graph = torch.cuda.CUDAGraph()
                with torch.cuda.graph(graph, stream=gs):
                    for _ in range(20):
                        fn(gs)
                graph.replay()
                torch.cuda.synchronize()
                a, b = ev(), ev()
                a.record(stream)
                for _ in range(10):
                    graph.replay()
                b.record(stream)
                torch.cuda.synchronize()
                row[tag + "_us_graph"] = a.elapsed_time(b) / 200 * 1e3
                del graph
                ts = []
                for _ in range(30):
                    flush.fill_(1)
                    a, b = ev(), ev()
                    a.record(stream)
                    fn()
                    b.record(stream)
                    b.synchronize()
                    ts.append(a.elapsed_time(b) * 1e3)
                us_f = statistics.median(ts)
                row[tag + "_us_flushed"] = us_f
                row[tag + "_gbs_flushed"] = nbytes / us_f / 1e3
                row[tag + "_frac_of_hbm_flushed"] = row[tag + "_gbs_flushed"] / peaks["hbm_gbs"]
            row[tag + "_frac_of_hbm"] = row[tag + "_gbs"] / peaks["hbm_gbs"]
            row[tag + "_frac_of_bf16_peak"] = row[tag + "_tflops"] / peaks["bf16_tflops"]
        # standard attention (S and P through HBM) on the same inputs: the article's comparison
        ubytes = sa.attn_fwd_unfused_workspace_size(B, H, N, D)
        uws = torch.empty(ubytes, dtype=torch.uint8, device="cuda")
        o2, lse2 = torch.empty_like(q), torch.empty_like(lse)
        unf = lambda: sa.attn_fwd_unfused(q, k, v, o2, lse2, uws, ubytes, B, H, N, D, w.scale, stream)
        for _ in range(3):
            unf()
        a, b = ev(), ev()
        a.record(stream)
        for _ in range(rep):
            unf()
        b.record(stream)
        torch.cuda.synchronize()
        us = a.elapsed_time(b) / rep * 1e3
        row["fwd_unfused_us"] = us
        row["fwd_unfused_tflops"] = 4 * flops / us / 1e6
        row["fwd_unfused_workspace_gb"] = ubytes / 1e9
        row["fwd_fused_speedup"] = us / row["fwd_us"]
        del uws, o2, lse2
        if sa.attn_get_device_status() != 0:
            raise RuntimeError(f"device status reported a kernel timeout on {name}")
        row["fwd_v_prepass"] = bool(fwsb)
        out[name] = row
        del q, k, v, do, o, dq, dk, dv, lse, ws, fws
    del flush
    torch.cuda.synchronize()
    return out


def run_ours(args, world, rank, local):
    import torch
    import torch.distributed as dist

    import self_attention_gb300 as sa
    from self_attention_gb300.build import build
    from self_attention_gb300.inputs import make_workload_inputs

    torch.cuda.set_device(local)
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    sa.load_library(build())
    w = workload(args)
    B, H, N, D, scale = w.B, w.H, w.N, w.d, w.scale
    inp = make_workload_inputs(dataclasses.replace(w, seed=w.seed + 7919 * rank))
    host = {x: inp[x].pin_memory() for x in ("q", "k", "v", "do")}
    q, k, v, do = (host[x].cuda() for x in ("q", "k", "v", "do"))
    o, dq, dk, dv = (torch.empty_like(q) for _ in range(4))
    lse = torch.empty((B, H, N), dtype=torch.float32, device="cuda")
    ws_bytes = sa.attn_bwd_workspace_size(B, H, N, D)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
    # the forward's workspace: an fp16 copy of V at long sequences (none below)
    fws_bytes = sa.attn_fwd_workspace_size(B, H, N, D)
    fws = torch.empty(fws_bytes, dtype=torch.uint8, device="cuda") if fws_bytes else None
    stream = torch.cuda.current_stream()

    def step(ev=None):
        if ev:
            ev[0].record(stream)
        sa.attn_fwd_with_workspace(q, k, v, o, lse, fws, fws_bytes, B, H, N, D, scale, stream)
        if ev:
            ev[1].record(stream)
        sa.attn_bwd_preprocess(o, do, lse, ws, ws_bytes, B, H, N, D, stream)
        if ev:
            ev[2].record(stream)
        sa.attn_bwd_main(q, k, v, do, dk, dv, ws, ws_bytes, B, H, N, D, scale, stream)
        if ev:
            ev[3].record(stream)
        sa.attn_bwd_dq_convert(ws, ws_bytes, dq, B, H, N, D, scale, stream)
        if ev:
            ev[4].record(stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    if sa.attn_get_device_status() != 0:
        raise RuntimeError("device status reported a kernel timeout during warm-up")
    # Inputs that fit in L2 would stay there from one step to the next: then a buffer larger
    # than L2 is written before each timed step, outside that step's events, and the step time
    # is the mean of the per-step event intervals.
    in_bytes = sum(t.numel() * t.element_size() for t in (q, k, v, do))
    l2_flush = torch.empty(256 << 20, dtype=torch.uint8, device="cuda") if in_bytes < L2_BYTES else None

    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(5)] for _ in range(args.steps)]
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    props = torch.cuda.get_device_properties(local)
    gpu_id = str(getattr(props, "uuid", local))
    gpu_id = gpu_id if gpu_id.startswith("GPU-") or gpu_id.isdigit() else f"GPU-{gpu_id}"
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    sampler = ClockSampler(gpu_id)
    time.sleep(0.3)
    start.record(stream)
    for i in range(args.steps):
        if l2_flush is not None:
            l2_flush.fill_(i & 0xff)
        step(evs[i])
    stop.record(stream)
    torch.cuda.synchronize()
    clocks = sampler.stop()
    if world > 1:
        dist.barrier()
    if sa.attn_get_device_status() != 0:
        raise RuntimeError("device status reported a kernel timeout in the timed region")

    ms = lambda a, b: a.elapsed_time(b)
    local_res = {
        "step_ms": (ms(start, stop) / args.steps if l2_flush is None
                    else statistics.mean(ms(e[0], e[4]) for e in evs)),
        "fwd_ms": statistics.mean(ms(e[0], e[1]) for e in evs),
        "bwd_ms": statistics.mean(ms(e[1], e[4]) for e in evs),
        "bwd_main_ms": statistics.mean(ms(e[2], e[3]) for e in evs),
        "flops": (4.0 + 10.0) * B * H * N * N * D,
    }

    # The deterministic backward (attn_bwd_deterministic: preprocess, the dK / dV pass and the
    # query-stationary dQ pass, no atomics) on the same inputs, outside the timed region above:
    # warm-up, then CUDA events around each call, with the L2 flush as above where the inputs
    # fit in L2.
    det_iters = max(1, min(10, args.steps))
    sa.attn_bwd_deterministic(q, k, v, o, do, lse, dq, dk, dv, ws, ws_bytes, B, H, N, D, scale, stream)
    det_evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(det_iters)]
    for i in range(det_iters):
        if l2_flush is not None:
            l2_flush.fill_(i & 0xff)
        det_evs[i][0].record(stream)
        sa.attn_bwd_deterministic(q, k, v, o, do, lse, dq, dk, dv, ws, ws_bytes, B, H, N, D, scale, stream)
        det_evs[i][1].record(stream)
    torch.cuda.synchronize()
    if sa.attn_get_device_status() != 0:
        raise RuntimeError("device status reported a kernel timeout in the deterministic backward")
    det_ms = statistics.mean(ms(a, b) for a, b in det_evs)

    # End to end through the C-ABI calls: every step copies its inputs from pinned host memory
    # to the device, runs attn_fwd and attn_bwd, and copies all outputs (O, LSE, dQ, dK, dV)
    # back to pinned host memory, all inside the timed region.  The steps are pipelined the way
    # a training loop feeds a GPU: device buffers are double-buffered and the copies run on
    # their own streams, so step k+1's inputs arrive and step k-1's outputs leave while step k
    # computes.
    out_host = {x: torch.empty(t.shape, dtype=t.dtype, pin_memory=True)
                for x, t in (("o", o), ("lse", lse), ("dq", dq), ("dk", dk), ("dv", dv))}
    dev_in = [{x: torch.empty_like(host[x], device="cuda") for x in host} for _ in range(2)]
    dev_out = [{x: torch.empty_like(t) for x, t in (("o", o), ("lse", lse), ("dq", dq), ("dk", dk),
                                                      ("dv", dv))} for _ in range(2)]
    s_h2d, s_comp, s_d2h = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
    ev = lambda: torch.cuda.Event()
    comp_done = [None, None]    # compute of the step that last used buffer j has finished
    out_copied = [None, None]   # the outputs in buffer j have reached the host

    def e2e_step(k):
        j = k & 1
        di, do_ = dev_in[j], dev_out[j]
        with torch.cuda.stream(s_h2d):
            if comp_done[j] is not None:
                s_h2d.wait_event(comp_done[j])
            for x in host:
                di[x].copy_(host[x], non_blocking=True)
            in_ready = ev()
            in_ready.record(s_h2d)
        s_comp.wait_event(in_ready)
        if out_copied[j] is not None:
            s_comp.wait_event(out_copied[j])
        sa.attn_fwd_with_workspace(di["q"], di["k"], di["v"], do_["o"], do_["lse"], fws, fws_bytes,
                                   B, H, N, D, scale, s_comp)
        sa.attn_bwd(di["q"], di["k"], di["v"], do_["o"], di["do"], do_["lse"], do_["dq"],
                    do_["dk"], do_["dv"], ws, ws_bytes, B, H, N, D, scale, s_comp)
        comp_done[j] = ev()
        comp_done[j].record(s_comp)
        with torch.cuda.stream(s_d2h):
            s_d2h.wait_event(comp_done[j])
            for x in out_host:
                out_host[x].copy_(do_[x], non_blocking=True)
            out_copied[j] = ev()
            out_copied[j].record(s_d2h)

    def join_all():
        for st in (s_h2d, s_comp, s_d2h):
            stream.wait_stream(st)

    for x in (s_h2d, s_comp, s_d2h):
        x.wait_stream(stream)
    e2e_step(0)
    e2e_step(1)
    join_all()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    e0.record(stream)
    for x in (s_h2d, s_comp, s_d2h):
        x.wait_stream(stream)
    for k in range(args.e2e_steps):
        e2e_step(k)
    join_all()
    e1.record(stream)
    torch.cuda.synchronize()
    if sa.attn_get_device_status() != 0:
        raise RuntimeError("device status reported a kernel timeout in the end-to-end loop")
    local_res["e2e_ms"] = e0.elapsed_time(e1) / args.e2e_steps
    h2d = sum(t.numel() * t.element_size() for t in host.values())
    d2h = sum(t.numel() * t.element_size() for t in out_host.values())

    # HBM probe: section 2's vector add over three 512 MiB arrays (12 bytes per element moved)
    nvec = 1 << 27
    va, vb = torch.ones(nvec, device="cuda"), torch.ones(nvec, device="cuda")
    vc = torch.empty_like(va)
    sa.vector_add(va, vb, vc, nvec, stream)
    torch.cuda.synchronize()
    p0, p1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    p0.record(stream)
    for _ in range(10):
        sa.vector_add(va, vb, vc, nvec, stream)
    p1.record(stream)
    torch.cuda.synchronize()
    probe_gbs = 12.0 * nvec / (p0.elapsed_time(p1) / 10 * 1e-3) / 1e9
    del va, vb, vc

    # QKV projection (section 1: Q = X W_Q, ...) on the full ViT-B block shape, fwd and bwd
    from self_attention_gb300.inputs import WORKLOADS as _W
    bw = _W["vit_b_mhsa_block"]
    PB, PN, PD, PH = bw.B, bw.N, bw.model_dim, bw.H
    px = torch.randn(PB, PN, PD, device="cuda").bfloat16()
    pw = [(torch.randn(PD, PD, device="cuda") / math.sqrt(PD)).bfloat16() for _ in range(3)]
    pout = [torch.empty(PB, PH, PN, PD // PH, device="cuda", dtype=torch.bfloat16) for _ in range(3)]
    pdy = [torch.randn(PB, PH, PN, PD // PH, device="cuda").bfloat16() for _ in range(3)]
    pdx = torch.empty_like(px)
    pdw = [torch.empty(PD, PD, device="cuda") for _ in range(3)]
    proj = {}
    for name, fn, fl in (
            ("fwd", lambda: sa.attn_qkv_proj(px, *pw, *pout, PB, PN, PD, PH, PD // PH, stream), 6.0),
            ("bwd", lambda: sa.attn_qkv_proj_bwd(px, *pw, *pdy, pdx, *pdw, PB, PN, PD, PH, PD // PH, stream), 12.0)):
        for _ in range(3):
            fn()
        p0.record(stream)
        for _ in range(20):
            fn()
        p1.record(stream)
        torch.cuda.synchronize()
        proj[name + "_tflops"] = fl * PB * PN * PD * PD / (p0.elapsed_time(p1) / 20 * 1e-3) / 1e12
    del px, pw, pout, pdy, pdx, pdw

    configs = None
    if world == 1 and not args.no_configs:
        configs = time_configs(sa, stream, load_peaks()[0])

    res = reduce_over_ranks(local_res, world)
    if rank != 0:
        dist.destroy_process_group()
        return 0

    peaks, peak_src = load_peaks()
    flops_total = res["flops"]
    value = flops_total / (res["step_ms"] * 1e-3) / 1e12
    per_gpu_fwd = 4.0 * B * H * N * N * D / (local_res["fwd_ms"] * 1e-3) / 1e12
    per_gpu_bwd = 10.0 * B * H * N * N * D / (local_res["bwd_ms"] * 1e-3) / 1e12
    main_flops = 10.0 * B * H * N * N * D
    achieved = main_flops / (local_res["bwd_main_ms"] * 1e-3) / 1e12
    fwd_achieved = 4.0 * B * H * N * N * D / (local_res["fwd_ms"] * 1e-3) / 1e12
    # The timed region lasts well under a second (steps x ms_per_step), so the kernels run at
    # burst clocks: the burst peak applies, not the seconds-long sustained one.
    peak = peaks["bf16_tflops"]
    units = B * H * math.ceil(N / 128) * math.ceil(N / 64)       # (key tile, query tile) pairs
    fwd_units = B * H * math.ceil(N / 256) * math.ceil(N / 128)  # (256-query block, key tile)
    # the committed counters are those of the d_k = 128 kernels; other kernels report none
    traffic = profiled_traffic(units) if D == 128 else None
    fwd_traffic = (profiled_traffic(fwd_units, FWD_PROFILE_SUMMARY, FWD_KERNEL_SOURCES)
                   if D == 128 else None)
    if D == 128:
        main_kernel = "bwd_main_kernel<128>"
    elif 128 < N <= 4096:
        main_kernel = "bwd_main_persist_kernel"
    else:
        main_kernel = "bwd_main_wide_kernel"

    cpu = None
    if world == 1 and not args.no_cpu_baseline:
        ref = {}
        times, oflops, cores, desc = time_oracle(w, args.cpu_baseline_tokens, 1, outputs=ref)
        cpu = {"value": oflops / times[0] / 1e12, "unit": UNIT, "cores": cores, "kind": "oracle",
               "sample": desc + f"; wall {times[0]:.2f} s", "cpu": cpu_model(),
               "gpu_errors_on_sample": sample_parity(sa, w, ref, stream)}
        if not args.no_parity:
            # the same oracle, on sampled rows of every workload, against the GPU forward
            cpu["parity_by_config"] = parity_by_config(sa, stream)

    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": res["step_ms"], "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": workload_config(w, world),
        "l2": (f"no flush: inputs (Q,K,V,dO = {in_bytes / 1e6:.0f} MB) are larger than the "
               f"{L2_BYTES / 1e6:.0f} MB L2" if l2_flush is None else
               f"flushed: inputs (Q,K,V,dO = {in_bytes / 1e6:.0f} MB) fit the "
               f"{L2_BYTES / 1e6:.0f} MB L2, so a 256 MB buffer is written before each "
               "timed step, outside its events"),
        "fwd_tflops": per_gpu_fwd, "bwd_tflops": per_gpu_bwd,
        "fwd_pct_of_bf16_peak": 100.0 * per_gpu_fwd / peaks["bf16_tflops"],
        "bwd_pct_of_bf16_peak": 100.0 * per_gpu_bwd / peaks["bf16_tflops"],
        "fwd_pct_of_datasheet_bf16": 100.0 * per_gpu_fwd / DATASHEET_BF16_TFLOPS,
        "peak_source": (f"{peak_src} (MEASURED_PEAKS.json: cuBLAS bf16 GEMM burst {peaks['bf16_tflops']:.0f} "
                        f"TFLOP/s, copy {peaks['hbm_gbs']:.0f} GB/s)" if peak_src == "measured" else
                        "fallback (no MEASURED_PEAKS.json)") +
                       f"; datasheet dense bf16 {DATASHEET_BF16_TFLOPS:.0f} TFLOP/s",
        "roofline": {"kernel": main_kernel,
                     "bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                     "frac": achieved / peak, "traffic": traffic,
                     "note": f"peak = {peak_src} burst dense bf16 (timed region "
                             f"{args.steps * res['step_ms'] / 1e3:.2f} s); achieved = 10*B*H*N^2*d "
                             "flops per launch / CUDA-event launch time; traffic = DRAM bytes per "
                             "launch from profiles/bwd_main_long_text.md"},
        "roofline_fwd": {"kernel": ("v_to_f16_kernel + " if fws_bytes else "") +
                                   ("fwd_kernel<128, 2>" if D == 128 else "fwd_persistent_kernel<64>"),
                         "bound": "tensor", "achieved": fwd_achieved, "peak": peak, "unit": "TFLOP/s",
                         "frac": fwd_achieved / peak, "traffic": fwd_traffic,
                         "frac_of_datasheet": fwd_achieved / DATASHEET_BF16_TFLOPS,
                         "note": "the kernel the >= 60 %-of-peak target is quoted on; achieved = "
                                 "4*B*H*N^2*d flops per call / CUDA-event time of the whole "
                                 "attn_fwd_with_workspace call (V rounded to fp16, then the "
                                 "forward kernel); traffic = DRAM bytes per call (both kernels) "
                                 "from profiles/fwd_long_text.md"},
        "cpu_baseline": cpu,
        "qkv_proj": {"workload": "vit_b_mhsa_block X [32, 576, 768] x 3 W [768, 768], 12 heads",
                     **proj},
        "deterministic_bwd": {
            "call": "attn_bwd_deterministic (preprocess, dK/dV pass, query-stationary dQ pass; "
                    "no atomics, bitwise reproducible)",
            "ms": det_ms, "tflops": 10.0 * B * H * N * N * D / (det_ms * 1e-3) / 1e12,
            "atomic_bwd_ms": local_res["bwd_ms"], "time_vs_atomic": det_ms / local_res["bwd_ms"],
            "calls": det_iters},
        "configs": configs,
        "hbm_probe": {"kernel": "vector_add (fp32, 3 x 512 MiB)", "gbs": probe_gbs,
                      "frac_of_measured_copy": probe_gbs / peaks["hbm_gbs"]},
        "e2e": {"value": flops_total / (res["e2e_ms"] * 1e-3) / 1e12, "unit": UNIT,
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
        "gpu_launches": (5 if fws_bytes else 4) * args.steps,
        "clocks": clocks,
        "system": {"gpu": torch.cuda.get_device_name(local), "torch": torch.__version__,
                   "cuda": torch.version.cuda, "sm_count": props.multi_processor_count},
    }
    print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()
    return 0


def main(argv=None):
    args = parse_args(argv)
    world, rank, local = dist_env()
    if args.impl == "reference":
        return run_reference(args, world, rank)
    return run_ours(args, world, rank, local)


if __name__ == "__main__":
    sys.exit(main())
