#!/usr/bin/env python
"""Benchmark: exact tiled softmax attention, forward + backward, on GB300.

One step = attn_fwd + attn_bwd (the whole hot path) over one batch of the
headline workload (B=2, H=16, Tq=Tk=8192, d=dv=128, bf16, causal), inputs
resident in HBM. Prints one JSON line (rank 0).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

N > 1 runs one process per GPU under torch.distributed (each rank processes
its own batch: weak scaling); the reported time is the max over ranks.
Started without torch.distributed, --gpus N > 1 launches the N ranks itself
(torch.distributed.run, one node); under it, N must equal WORLD_SIZE.
--impl reference times the CPU float64 oracle on the host cores instead.
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
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "attention TFLOP/s fwd+bwd (bf16, causal, 1 GB300)"
METRIC_FWD = "attention TFLOP/s fwd only (bf16, causal, 1 GB300)"   # --fwd-only
UNIT = "TFLOP/s"
L2_FLUSH_BYTES = 256 << 20
# the sources each profiled kernel is built from (a committed DRAM-traffic
# figure counts only while these hash as they did when it was captured)
KERNEL_SOURCES = {
    "attn_fwd_bf16_kernel": ("fwd_bf16.cu", "ptx.cuh", "common.cuh", "launch.h"),
    "dkdv_kernel": ("bwd_bf16.cu", "bwd_common.cuh", "ptx.cuh", "common.cuh", "launch.h"),
    "dq_kernel": ("bwd_bf16.cu", "bwd_common.cuh", "ptx.cuh", "common.cuh", "launch.h"),
    "attn_fwd_d256_kernel": ("fwd_bf16_d256.cu", "ptx.cuh", "common.cuh", "launch.h"),
    "attn_fwd_d256_pair_kernel": ("fwd_d256_pair.cu", "ptx.cuh", "common.cuh", "launch.h"),
    "dq_pair_kernel": ("dq_pair.cu", "bwd_common.cuh", "ptx.cuh", "common.cuh", "launch.h"),
    # both launches (the dV and the dK kernel) of the phase bench.py times together
    "kv256_kernel": ("bwd_d256.cu", "bwd_common.cuh", "ptx.cuh", "common.cuh", "launch.h"),
    "q256_kernel": ("bwd_d256.cu", "bwd_common.cuh", "ptx.cuh", "common.cuh", "launch.h"),
    "simt::fwd_kernel": ("simt_f32.cu", "simt.h", "common.cuh", "launch.h"),
    "simt::dkdv_kernel": ("simt_f32.cu", "simt.h", "common.cuh", "launch.h"),
    "simt::dq_kernel": ("simt_f32.cu", "simt.h", "common.cuh", "launch.h"),
    # the dK/dV kernel with the dQ share and its reductions (atomic dQ mode)
    "dkdv_kernel@atomic": ("bwd_bf16.cu", "bwd_common.cuh", "ptx.cuh", "common.cuh", "launch.h"),
    "simt::dkdv_kernel@atomic": ("simt_f32.cu", "simt.h", "common.cuh", "launch.h"),
    # the fp32 dK/dV kernel that also writes the key tiles' dQ partials (deterministic, no dQ kernel)
    "simt::dkdv_kernel@dqpart": ("simt_f32.cu", "simt.h", "common.cuh", "launch.h"),
}


# ---------------------------------------------------------------- helpers

def useful_flops_rows(w, rows, fwd_only=False):
    """Useful fwd+bwd FLOPs of the given query rows: 2*(d + dv) per (query,
    key) pair forward and 2*(3d + 2dv) backward (14 d per pair when d = dv);
    the forward's share alone with fwd_only.
    Under the causal mask row i counts i + 1/2 keys, so that all Tq rows of a
    square problem sum to the halved full count (the convention of the GPU
    metric)."""
    import numpy as np
    rows = np.asarray(rows, dtype=np.float64)
    keys = np.minimum(rows + 0.5, w.Tk) if w.causal else np.full(rows.shape, float(w.Tk))
    per_pair = 2.0 * (w.d + w.dv) + (0.0 if fwd_only else 2.0 * (3 * w.d + 2 * w.dv))
    return per_pair * float(keys.sum())


def kernel_source_hash(kernel: str) -> str:
    """Hash of the kernel's sources with comments and blank space removed, so
    that editing a comment does not void a committed measurement. Plain
    declarations of other launch functions (`cudaError_t f(...);`,
    `size_t f(...);`) are dropped too: they declare code in other files and
    cannot change this kernel."""
    import re
    h = hashlib.sha256()
    for f in KERNEL_SOURCES[kernel]:
        with open(os.path.join(ROOT, "exact_tiled_softmax_attn_gb300", "csrc", f), encoding="utf-8") as fh:
            text = fh.read()
        text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
        text = re.sub(r"//[^\n]*", " ", text)
        text = " ".join(text.split())
        text = re.sub(r"(?:cudaError_t|size_t) \w+\([^(){};]*\);", " ", text)
        h.update(" ".join(text.split()).encode())
    return h.hexdigest()[:16]


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            j = json.load(f)
        return {"hbm_gbs": j["hbm_gbs"], "bf16_tflops": j["bf16_tflops"],
                "bf16_tflops_sustained": j.get("bf16_tflops_sustained"),
                "sm_max_mhz": j.get("sm_max_mhz", 2070.0), "source": "measured"}
    except Exception:
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "sm_max_mhz": 2070.0,
                "source": "fallback"}


def load_traffic(kernel: str, workload: str):
    """DRAM bytes per launch of `kernel` on `workload` from the committed ncu
    summary, or None when there is none for that workload or it was taken on
    different kernel sources."""
    p = os.path.join(ROOT, "profiles", "traffic.txt")
    try:
        with open(p) as f:
            for line in f:
                parts = line.split()
                if len(parts) >= 4 and not line.startswith("#") and parts[0] == kernel and parts[1] == workload:
                    ok = kernel in KERNEL_SOURCES and parts[2] == kernel_source_hash(kernel)
                    return float(parts[3]) if ok else None
    except OSError:
        pass
    return None


class ClockSampler:
    """nvidia-smi clock / throttle samples taken while the timed region runs."""
    QUERY = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
             "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
             "clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.idx = gpu_index
        self.proc = None
        self.windows = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.idx), f"--query-gpu={self.QUERY}", "--format=csv,noheader,nounits",
                 "-lms", "50"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None

    def mark(self, t0, t1):
        self.windows.append((t0, t1))

    def stop(self):
        if self.proc is None:
            return {"error": "nvidia-smi unavailable"}
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except Exception:
            self.proc.kill()
            out, _ = self.proc.communicate()
        samples = []
        for line in out.splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 8:
                continue
            try:
                ts = time.mktime(time.strptime(parts[0].split(".")[0], "%Y/%m/%d %H:%M:%S"))
                ts += float("0." + parts[0].split(".")[1]) if "." in parts[0] else 0.0
                samples.append((ts, float(parts[1]), float(parts[2]), parts[4:8]))
            except Exception:
                continue
        inside = [s for s in samples if any(a - 0.05 <= s[0] <= b + 0.05 for a, b in self.windows)]
        use = inside if inside else samples
        if not use:
            return {"error": "no samples"}
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for s in use for n, v in zip(names, s[3]) if v.lower() == "active"})
        return {"sm_mhz": statistics.median(s[1] for s in use), "sm_max_mhz": max(s[2] for s in use),
                "reasons": reasons, "samples": len(use), "in_timed_region": bool(inside)}


def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def rank_seed(w, rank: int) -> int:
    """Seed of a rank's batch: every rank draws its own inputs (weak scaling
    over independent (b, h) problems)."""
    return w.seed + 1000 * rank


def free_port() -> int:
    import socket
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def relaunch(n: int, argv) -> int:
    """Run this script as n ranks on one node (one process per GPU) under
    torch.distributed.run; returns its exit code."""
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", f"--nproc-per-node={n}",
           "--master-addr=127.0.0.1", f"--master-port={free_port()}", os.path.abspath(__file__), *argv]
    return subprocess.call(cmd)


def run_dry(args, w):
    """Print this rank's launch plan (one JSON line per rank) without touching a GPU."""
    world, rank, local = dist_setup()
    print(json.dumps({"dry_run": True, "impl": args.impl, "rank": rank, "world": world, "local_rank": local,
                      "n_gpus": world, "seed": rank_seed(w, rank), "workload": w.name}), flush=True)
    return 0


def reduce_max(value: float) -> float:
    """Max of `value` over all ranks (identity without torch.distributed)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()):
        return value
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([value], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier():
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized():
        dist.barrier()


# ---------------------------------------------------------------- CPU oracle legs

def oracle_sample(w, x, rows, n_heads=1, fwd_only=False):
    """Run the CPU float64 oracle forward + backward (forward alone with
    fwd_only) on the given query rows of the first n_heads heads (in (b, h)
    order); returns seconds."""
    from oracle import attention as ref
    t0 = time.perf_counter()
    for k in range(n_heads):
        b, h = divmod(k, x["Q"].shape[1])
        if fwd_only:
            ref.forward_head(x["Q"][b, h], x["K"][b, h], x["V"][b, h], w.softmax_scale, w.causal, rows=rows)
        else:
            ref.backward_head(x["Q"][b, h], x["K"][b, h], x["V"][b, h], x["dO"][b, h], w.softmax_scale, w.causal,
                              rows=rows)
    return time.perf_counter() - t0


def spread_rows(w, n):
    import numpy as np
    n = max(1, min(n, w.Tq))
    return np.unique(np.linspace(0, w.Tq - 1, n).astype(np.int64))


def cpu_baseline(w, x, target_s=15.0, fwd_only=False):
    """The oracle on a bounded sample of the workload (~10-30 s of CPU work):
    query rows spread over head (0, 0), then, when all its rows take less than
    that, whole heads in (b, h) order."""
    probe = spread_rows(w, 128)
    t = oracle_sample(w, x, probe, fwd_only=fwd_only)
    n = int(min(w.Tq, max(128, 128 * target_s / max(t, 1e-3))))
    rows = spread_rows(w, n)
    t = oracle_sample(w, x, rows, fwd_only=fwd_only)
    n_heads = 1
    if rows.size == w.Tq and t < target_s / 2:
        n_heads = int(min(w.B * w.H, max(1, target_s // max(t, 1e-3))))
        if n_heads > 1:
            t = oracle_sample(w, x, rows, n_heads, fwd_only=fwd_only)
    fl = useful_flops_rows(w, rows, fwd_only) * n_heads
    where = "head (0,0)" if n_heads == 1 else f"each of the first {n_heads} heads"
    what = "fwd" if fwd_only else "fwd+bwd"
    return {"value": fl / t / 1e12, "unit": UNIT, "cores": os.cpu_count(), "kind": "oracle",
            "sample": f"float64 numpy oracle, {what} of {rows.size} query rows spread over {where} of "
                      f"{w.name} (Tk={w.Tk}, d={w.d}); useful FLOPs of those rows / {t:.2f} s"}


def run_reference(args, w):
    world, rank, _ = dist_setup()
    if rank != 0:
        return 0
    from exact_tiled_softmax_attn_gb300.workloads import make_inputs
    x = make_inputs(w.with_(B=1, H=1))
    budget = 150.0 / max(1, args.steps + args.warmup)
    fo = args.fwd_only
    cal = spread_rows(w, 64)
    t = oracle_sample(w, x, cal, fwd_only=fo)
    n = int(min(w.Tq, max(64, 64 * budget / max(t, 1e-3))))
    rows = spread_rows(w, n)
    for _ in range(args.warmup):
        oracle_sample(w, x, rows, fwd_only=fo)
    total = 0.0
    for _ in range(args.steps):
        total += oracle_sample(w, x, rows, fwd_only=fo)
    fl = useful_flops_rows(w, rows, fo) * args.steps
    value = fl / total / 1e12
    sample = (f"float64 numpy oracle, {'fwd' if fo else 'fwd+bwd'} of {rows.size} query rows spread over "
              f"head (0,0) of {w.name} "
              f"per step (useful FLOPs of those rows)")
    line = {"impl": "reference", "metric": METRIC_FWD if fo else METRIC, "value": value, "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": total / args.steps * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": workload_config(w),
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": os.cpu_count(), "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def f32_dq_partials(f32: bool, det: bool, Tk: int, dq_splits: int) -> bool:
    """True where the fp32 deterministic backward runs no dQ kernel: its
    dK/dV kernel writes one dQ partial per 64-key tile (or dQ itself, with one
    key tile), and the library reports one split per key tile. The dQ
    kernel's own key ranges hold at least two key tiles each, so they never
    reach that count."""
    return bool(f32 and det and dq_splits == -(-Tk // 64))


def workload_config(w):
    return {"workload": f"{w.name}: B={w.B} H={w.H} Tq={w.Tq} Tk={w.Tk} d={w.d} dv={w.dv} {w.dtype} "
                        f"{'causal' if w.causal else 'no mask'}, scale={w.softmax_scale:.6g}",
            "B": w.B, "H": w.H, "Tq": w.Tq, "Tk": w.Tk, "d": w.d, "dv": w.dv, "causal": w.causal,
            "l2": "256 MiB written between timed steps (outside the timed region); per-step inputs "
                  f"{w.B * w.H * (w.Tq + w.Tk) * (w.d + w.dv) * (2 if w.dtype == 'bf16' else 4) / 1e6:.0f} MB"}


# ---------------------------------------------------------------- GPU leg

def run_ours(args, w):
    import torch
    import torch.distributed as dist

    import exact_tiled_softmax_attn_gb300 as pkg
    from exact_tiled_softmax_attn_gb300.workloads import make_inputs

    world, rank, local = dist_setup()
    if local >= torch.cuda.device_count():
        raise SystemExit(f"rank {rank}: local rank {local} but {torch.cuda.device_count()} visible GPU(s)")
    if world > 1:
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    else:
        torch.cuda.set_device(0)
    dev = torch.device("cuda", torch.cuda.current_device())
    pkg.load_library()
    code = pkg.ATTN_BF16 if w.dtype == "bf16" else pkg.ATTN_F32
    B, H, Tq, Tk, d, dv = w.B, w.H, w.Tq, w.Tk, w.d, w.dv
    det = int(args.dq_mode == "deterministic")
    f32 = w.dtype == "f32"
    es = 2 if w.dtype == "bf16" else 4   # bytes per input element

    host = make_inputs(w.with_(seed=rank_seed(w, rank)))
    x = {k: v.to(dev) for k, v in host.items()}
    o = torch.empty(B, H, Tq, dv, dtype=w.torch_dtype, device=dev)
    lse = torch.empty(B, H, Tq, dtype=torch.float32, device=dev)
    dq, dk, dvv = torch.empty_like(x["Q"]), torch.empty_like(x["K"]), torch.empty_like(x["V"])
    ws_bytes = pkg.attn_bwd_workspace_size(B, H, Tq, Tk, d, dv, code, det)
    dq_splits = pkg.attn_bwd_dq_splits(B, H, Tq, Tk, d, dv, code, det)
    ws = torch.empty(max(ws_bytes, 256), dtype=torch.uint8, device=dev)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()
    sc = w.softmax_scale

    # forward: attn_fwd, or the split-KV forward (key ranges as separate work
    # units, then the merge kernel). --splitkv N takes the split-KV forward
    # with N splits (0: the library's automatic count) and --splitkv -1 takes
    # attn_fwd; by default the split-KV forward runs where the automatic count
    # is above 1 (few query tiles against many keys) and attn_fwd elsewhere.
    splitkv = args.splitkv
    if splitkv is None:
        splitkv = 0 if pkg.attn_fwd_splitkv_splits(B, H, Tq, Tk, d, dv, code, 0) > 1 else -1
    n_splits = 1
    if splitkv >= 0:
        n_splits = pkg.attn_fwd_splitkv_splits(B, H, Tq, Tk, d, dv, code, splitkv)
        sk_bytes = pkg.attn_fwd_splitkv_workspace_size(B, H, Tq, Tk, d, dv, code, splitkv)
        sk_ws = torch.empty(max(sk_bytes, 256), dtype=torch.uint8, device=dev)

    def fwd_call(xi, oi, li, st):
        if splitkv < 0:
            pkg.attn_fwd(xi["Q"], xi["K"], xi["V"], oi, li, B, H, Tq, Tk, d, dv, sc, w.causal, code, st)
        else:
            pkg.attn_fwd_splitkv(xi["Q"], xi["K"], xi["V"], oi, li, B, H, Tq, Tk, d, dv, sc, w.causal, code,
                                 splitkv, sk_ws, sk_ws.numel(), st)

    def fwd():
        fwd_call(x, o, lse, stream)

    def bwd_phase(ph):
        pkg.attn_bwd_phase(x["Q"], x["K"], x["V"], o, lse, x["dO"], dq, dk, dvv, B, H, Tq, Tk, d, dv, sc,
                           w.causal, code, det, ws, ws.numel(), ph, stream)

    # backward launch groups in order: preprocess, dQ kernel (deterministic,
    # or any bf16 rows wider than 128 columns; for bf16 it also forms D), dK/dV kernel,
    # dQ conversion or split-dQ reduction; none with --fwd-only. A group that
    # launches nothing for this configuration (the library's own rule, as in
    # attn_bwd_phase) is not called, so that no event interval of the timed
    # step is an empty one.
    f32_fused = f32_dq_partials(f32, bool(det), Tk, dq_splits)
    launches = {1: f32 or (not det and w.d <= 128), 5: (bool(det) and not f32_fused) or w.d > 128, 6: bool(det), 4: True,
                3: (not f32 and w.d <= 128 and (not det or dq_splits > 1)) or (f32 and bool(det) and dq_splits > 1)}
    phases = () if args.fwd_only else tuple(ph for ph in (1, 6 if args.dq_pairs else 5, 4, 3) if launches[ph])
    slot = {1: 1, 5: 2, 6: 2, 4: 3, 3: 4}   # per-step interval of each group: fwd, pre, q, kv, conv

    def step(ev=None):
        if ev is not None:
            ev[0].record(stream)
        fwd()
        if ev is not None:
            ev[1].record(stream)
        for i, ph in enumerate(phases):
            bwd_phase(ph)
            if ev is not None:
                ev[2 + i].record(stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    assert pkg.attn_device_status(stream) == pkg.ATTN_OK

    clocks = ClockSampler(torch.cuda.current_device()) if rank == 0 else None
    if clocks:
        clocks.start()
        time.sleep(0.3)
    events = [[torch.cuda.Event(enable_timing=True) for _ in range(2 + len(phases))] for _ in range(args.steps)]
    barrier()
    torch.cuda.synchronize()
    t_wall0 = time.time()
    for i in range(args.steps):
        flush.zero_()                  # evict L2 between steps (not timed)
        step(events[i])
    torch.cuda.synchronize()
    t_wall1 = time.time()
    barrier()
    if clocks:
        clocks.mark(t_wall0, t_wall1)
    per = []                           # ms per step: fwd, pre, q, kv, conv (0 for a group not called)
    for e in events:
        row = [e[0].elapsed_time(e[1]), 0.0, 0.0, 0.0, 0.0]
        for i, ph in enumerate(phases):
            row[slot[ph]] = e[1 + i].elapsed_time(e[2 + i])
        per.append(row)
    step_ms = [sum(p) for p in per]
    total_ms = reduce_max(sum(step_ms))
    fwd_ms, pre_ms, q_ms, kv_ms, conv_ms = (statistics.mean(p[j] for p in per) for j in range(5))
    main_ms = kv_ms + q_ms
    bwd_ms = pre_ms + main_ms + conv_ms
    F, Bf = w.fwd_flop(), (0.0 if args.fwd_only else w.bwd_flop())
    value = world * args.steps * (F + Bf) / (total_ms * 1e-3) / 1e12
    assert pkg.attn_device_status(stream) == pkg.ATTN_OK

    # ---- end to end through the public API, host buffers in and out. Every
    # step copies its four inputs from pinned host memory and reads all five
    # results back. Two device buffer sets let step i+1's host-to-device copy
    # and step i-1's device-to-host copy run on copy streams of their own
    # while step i's kernels run (inputs > L2, so no flush between steps).
    outs = (("O", o), ("LSE", lse)) if args.fwd_only else \
        (("O", o), ("LSE", lse), ("dQ", dq), ("dK", dk), ("dV", dvv))
    if args.fwd_only:                  # the forward's inputs and results only
        host = {k: v for k, v in host.items() if k != "dO"}
        x = {k: v for k, v in x.items() if k != "dO"}
    pinned = {k: v.pin_memory() for k, v in host.items()}
    dev_in = [x, {k: torch.empty_like(v) for k, v in x.items()}]
    dev_out = [dict(outs), {n: torch.empty_like(t) for n, t in outs}]
    host_out = [{n: torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for n, t in outs} for _ in range(2)]
    h2d = sum(t.numel() * t.element_size() for t in pinned.values())
    d2h = sum(t.numel() * t.element_size() for t in host_out[0].values())
    s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()

    def e2e_run(n):
        in_ready = [torch.cuda.Event() for _ in range(2)]
        comp_done = [torch.cuda.Event() for _ in range(2)]
        out_done = [torch.cuda.Event() for _ in range(2)]
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        t0.record(stream)
        s_in.wait_stream(stream)
        s_out.wait_stream(stream)
        for i in range(n):
            b = i % 2
            xi, oi = dev_in[b], dev_out[b]
            with torch.cuda.stream(s_in):
                if i >= 2:
                    s_in.wait_event(comp_done[b])       # step i-2 no longer reads these inputs
                for k in xi:
                    xi[k].copy_(pinned[k], non_blocking=True)
                in_ready[b].record(s_in)
            stream.wait_event(in_ready[b])
            if i >= 2:
                stream.wait_event(out_done[b])          # step i-2's results have left the device
            fwd_call(xi, oi["O"], oi["LSE"], stream)
            if not args.fwd_only:
                pkg.attn_bwd(xi["Q"], xi["K"], xi["V"], oi["O"], oi["LSE"], xi["dO"], oi["dQ"], oi["dK"], oi["dV"],
                         B, H, Tq, Tk, d, dv, sc, w.causal, code, det, ws, ws.numel(), stream)
            comp_done[b].record(stream)
            with torch.cuda.stream(s_out):
                s_out.wait_event(comp_done[b])
                for n_ in host_out[b]:
                    host_out[b][n_].copy_(oi[n_], non_blocking=True)
                out_done[b].record(s_out)
        stream.wait_stream(s_in)
        stream.wait_stream(s_out)
        t1.record(stream)
        torch.cuda.synchronize()
        return t0.elapsed_time(t1)

    # as many steps as the timed region, so that the pipeline's fill (the first
    # step's inputs) and drain (the last step's results) weigh as little
    e2e_steps = max(2, args.steps)
    e2e_run(2)                                   # warms the copy engines and streams
    # three runs of e2e_steps steps; their median, so that one stall of the
    # host (page cache, another process) does not stand for the pipeline
    e2e_runs = [e2e_run(e2e_steps) for _ in range(3)]
    e2e_total = reduce_max(statistics.median(e2e_runs))
    e2e_value = world * e2e_steps * (F + Bf) / (e2e_total * 1e-3) / 1e12
    link = copy_link(dev_in[0], pinned, dev_out[0], host_out[0], s_in, s_out, h2d, d2h)
    # a step can take no less than the longer of its kernels and its copies
    link["bound_value"] = world * (F + Bf) / (max(total_ms / args.steps, link["concurrent_ms"]) * 1e-3) / 1e12
    if clocks:
        clk = clocks.stop()
    if world > 1:
        dist.destroy_process_group()
    if rank != 0:
        return 0

    peaks = load_peaks()
    peak = peaks["bf16_tflops"]
    # Algorithmic FLOP per kernel: a product of depth d (S, dQ, dK) costs md,
    # one of depth dv (PV, dP, dV) mv. The forward does S and PV; the dK/dV
    # kernel S, dP, dV, dK (and, atomic mode, dQ); the deterministic dQ
    # kernel's own product is dQ (it recomputes S and dP, which is counted
    # under "executed").
    md, mv = w.pair_flop() * w.d, w.pair_flop() * w.dv
    if f32:
        # the CUDA-core path: FP32 FMA throughput (its scores are formed beyond fp32 precision)
        props = torch.cuda.get_device_properties(dev)
        peak = props.multi_processor_count * 128 * 2 * peaks.get("sm_max_mhz", 2070.0) * 1e6 / 1e12
    tag = "simt::" if f32 else ""
    if n_splits > 1:
        fwd_name = f"fwd split-KV, {n_splits} splits ({'simt::fwd_kernel' if f32 else 'attn_fwd_bf16_kernel'} + merge)"
    else:
        fwd_name = "fwd (simt::fwd_kernel)" if f32 else \
            ("fwd (attn_fwd_d256_pair_kernel)" if w.dv > 64 else "fwd (attn_fwd_d256_kernel)") if w.d > 128 else \
            "fwd (attn_fwd_bf16_kernel)"
    kernels = {fwd_name: {"ms": fwd_ms, "flop": F}}
    if args.fwd_only:
        pass
    elif w.d > 128:
        # rows of 256 columns: a dV kernel (S^T, dV) and a dK kernel (S^T, dP^T, dK), then a dQ kernel
        kernels["bwd dV + dK (kv256_kernel)"] = {"ms": kv_ms, "flop": 2 * md + 2 * mv,
                                                 "executed_flop": 3 * md + 2 * mv, "launches": 2}
        kernels["bwd dQ (q256_kernel)"] = {"ms": q_ms, "flop": md, "executed_flop": 2 * md + mv}
    elif f32_fused:
        kernels["bwd dK/dV + dQ partials (simt::dkdv_kernel)"] = {"ms": kv_ms, "flop": 3 * md + 2 * mv}
    elif det:
        kernels[f"bwd dK/dV ({tag}dkdv_kernel)"] = {"ms": kv_ms, "flop": 2 * md + 2 * mv}
        kernels[f"bwd dQ ({tag}{'dq_pair_kernel' if args.dq_pairs else 'dq_kernel'})"] = \
            {"ms": q_ms, "flop": md, "executed_flop": 2 * md + mv}
    else:
        kernels[f"bwd dK/dV + dQ atomics ({tag}dkdv_kernel)"] = {"ms": kv_ms, "flop": 3 * md + 2 * mv}
    for k, v in kernels.items():
        v["tflops"] = v["flop"] / (v["ms"] * 1e-3) / 1e12
        v["frac_of_peak"] = v["tflops"] / peak
        if "executed_flop" in v:
            v["executed_tflops"] = v["executed_flop"] / (v["ms"] * 1e-3) / 1e12
    if not args.fwd_only:
        kernels["bwd main (all main kernels)"] = {"ms": main_ms, "tflops": Bf / (main_ms * 1e-3) / 1e12}
        kernels["bwd main (all main kernels)"]["frac_of_peak"] = \
            kernels["bwd main (all main kernels)"]["tflops"] / peak
        if launches[1]:
            # reads O, dO, LSE; writes D and -LSE*log2(e) (padded rows); zeroes the fp32 dQ
            # accumulator in atomic mode (bf16 rows of up to 128 columns, deterministic:
            # the dQ kernel forms D itself and this group launches nothing)
            gbs = B * H * Tq * (2 * dv * es + 4 + 8 + (0 if (det or w.d > 128) else d * 4)) / (pre_ms * 1e-3) / 1e9
            kernels["bwd preprocess"] = {"ms": pre_ms, "gbs": gbs, "frac_of_hbm": gbs / peaks["hbm_gbs"]}
        if launches[3]:
            # atomic: fp32 accumulator -> bf16; deterministic with split dQ: the partials' sum -> dQ
            # (bf16, or fp32 for the fp32 path)
            kernels["dQ convert"] = {"ms": conv_ms, "gbs": B * H * Tq * d * (4 * (1 if not det else dq_splits) +
                                                                           (4 if f32 else 2)) / (conv_ms * 1e-3) / 1e9}
    # the dominant kernel: the longest of the single kernels
    dom = max((k for k, v in kernels.items() if "flop" in v), key=lambda k: kernels[k]["ms"])
    achieved = kernels[dom]["tflops"]
    # (atomic dQ mode, and the fp32 dK/dV kernel with dQ partials: lines of their own)
    dom_kernel = dom.split("(")[-1].rstrip(")")
    suffix = "" if "dkdv" not in dom_kernel else "@atomic" if not det else "@dqpart" if f32_fused else ""
    traffic = load_traffic(dom_kernel + suffix, args.workload)
    cfg = workload_config(w)
    cfg.update({"pass": "forward only" if args.fwd_only else "forward + backward",
                "dq_mode": None if args.fwd_only else ("deterministic" if det else "atomic"),
                "fwd_splits": n_splits, "dq_splits": None if args.fwd_only else dq_splits,
                "dq_on_cta_pairs": bool(args.dq_pairs),
                "fwd_tflops": F / (fwd_ms * 1e-3) / 1e12,
                "bwd_tflops": None if args.fwd_only else Bf / (bwd_ms * 1e-3) / 1e12,
                "fwd_bwd_frac_of_peak": (F + Bf) / ((fwd_ms + bwd_ms) * 1e-3) / 1e12 / peak,
                # the same against the measured power-capped (seconds-long) bf16 rate
                "fwd_bwd_frac_of_sustained_peak": None if f32 or not peaks.get("bf16_tflops_sustained") else
                (F + Bf) / ((fwd_ms + bwd_ms) * 1e-3) / 1e12 / peaks["bf16_tflops_sustained"],
                "peak_source": f"derived FP32 FMA {peak:.1f}" if f32 else f"{peaks['source']} bf16_tflops {peak}",
                "kernels": kernels})
    line = {
        "metric": METRIC_FWD if args.fwd_only else METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": total_ms / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32" if f32 else "bf16", "data": "synthetic",
        "config": cfg,
        "roofline": {"bound": "alu" if f32 else "tensor", "kernel": dom, "achieved": achieved, "peak": peak,
                     "unit": UNIT, "frac": achieved / peak, "traffic": traffic,
                     "peak_note": "FP32 FMA peak derived as SMs x 128 lanes x 2 FLOP x max SM clock"
                     if f32 else f"{peaks['source']} dense bf16 burst (cuBLAS 8192^3)"},
        "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "steps": e2e_steps, "runs_ms": [round(t, 4) for t in e2e_runs],
                "statistic": "median of the three runs (max over ranks)",
                "pipeline": "two buffer sets; step i+1 host-to-device and step i-1 device-to-host copies "
                            "overlap step i's kernels on separate streams",
                "link": link},
        # bf16: fwd (+ split-KV merge), dQ (+ split reduction), dK/dV | fwd (+ merge), preprocess,
        # dK/dV, convert; fp32: fwd, preprocess, dK/dV, dQ | fwd, preprocess, dK/dV
        "gpu_launches": args.steps * ((1 + (1 if n_splits > 1 else 0)) if args.fwd_only else
                                      (4 if det and not f32_fused else 3) + (1 if n_splits > 1 else 0) +
                                      (1 if det and dq_splits > 1 else 0) if f32 else
                                      # d = 256: forward, dQ (it forms D), dV, dK kernels
                                      (4 + (1 if n_splits > 1 else 0)) if w.d > 128 else
                                      ((3 if det else 4) + (1 if n_splits > 1 else 0) +
                                       (1 if det and dq_splits > 1 else 0))),
        "clocks": clk,
    }
    if world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(w, host, fwd_only=args.fwd_only)
    print(json.dumps(line), flush=True)
    return 0


def copy_link(dev_in, pinned, dev_out, host_out, s_in, s_out, h2d, d2h, reps=3):
    """One step's copies alone (outside every timed region): host-to-device,
    device-to-host, and both at once, each on its own stream as in the
    end-to-end pipeline. Returns GB/s per direction and the concurrent time."""
    import torch

    def run(do_in, do_out):
        ev = []
        for _ in range(reps):
            t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            t0.record(torch.cuda.current_stream())
            s_in.wait_stream(torch.cuda.current_stream())
            s_out.wait_stream(torch.cuda.current_stream())
            if do_in:
                with torch.cuda.stream(s_in):
                    for k in dev_in:
                        dev_in[k].copy_(pinned[k], non_blocking=True)
            if do_out:
                with torch.cuda.stream(s_out):
                    for n in host_out:
                        host_out[n].copy_(dev_out[n], non_blocking=True)
            torch.cuda.current_stream().wait_stream(s_in)
            torch.cuda.current_stream().wait_stream(s_out)
            t1.record(torch.cuda.current_stream())
            ev.append((t0, t1))
        torch.cuda.synchronize()
        return statistics.median(a.elapsed_time(b) for a, b in ev)
    t_in, t_out, t_both = run(True, False), run(False, True), run(True, True)
    return {"h2d_gbs": h2d / (t_in * 1e-3) / 1e9, "d2h_gbs": d2h / (t_out * 1e-3) / 1e9,
            "concurrent_ms": t_both, "note": "one step's copies alone on this box; bound_value: the metric at "
            "max(kernel time, concurrent copy time) per step"}


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[1])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="c3")
    ap.add_argument("--dq-mode", choices=["deterministic", "atomic"], default="deterministic",
                    help="dQ in a separate fixed-order pass (default) or by fp32 atomics inside the dK/dV kernel")
    ap.add_argument("--dq-pairs", action="store_true",
                    help="time the dQ pass on CTA pairs (attn_bwd_phase phase 6; bf16, d = 128, deterministic)")
    ap.add_argument("--splitkv", type=int, default=None,
                    help="forward through attn_fwd_splitkv with this many key splits (0 = automatic) or, with -1, "
                         "through attn_fwd; default: attn_fwd_splitkv where the automatic count is above 1")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--fwd-only", action="store_true",
                    help="time the forward alone (its FLOPs only)")
    ap.add_argument("--dry-run", action="store_true",
                    help="print each rank's launch plan (rank, world, device, input seed) and exit")
    argv = sys.argv[1:] if argv is None else list(argv)
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.gpus < 1:
        ap.error("--gpus must be >= 1")
    # --gpus N: one rank per GPU. Launched without torch.distributed, N > 1
    # starts the N ranks itself; launched under it, N must be its world size.
    if "WORLD_SIZE" not in os.environ:
        if args.gpus > 1:
            return relaunch(args.gpus, argv)
    elif int(os.environ["WORLD_SIZE"]) != args.gpus:
        ap.error(f"--gpus {args.gpus} but WORLD_SIZE={os.environ['WORLD_SIZE']}")
    from exact_tiled_softmax_attn_gb300.workloads import WORKLOADS
    w = WORKLOADS[args.workload]
    if args.dry_run:
        return run_dry(args, w)
    if args.impl == "reference":
        return run_reference(args, w)
    return run_ours(args, w)


if __name__ == "__main__":
    sys.exit(main())
