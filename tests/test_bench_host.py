"""Host-side logic of bench.py (no GPU): the cross-rank max reduction that the
multi-GPU run uses, on 2 gloo ranks; the launch of one rank per GPU by
--gpus N (ranks, devices and input seeds, through --dry-run); the reference
arm under several ranks; and the FLOP accounting."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench
from exact_tiled_softmax_attn_gb300.workloads import WORKLOADS


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        got = bench.reduce_max(10.0 * (rank + 1))
        bench.barrier()
        q.put((rank, got))
    finally:
        dist.destroy_process_group()


def test_reduce_max_over_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    res = dict(q.get(timeout=5) for _ in range(2))
    assert res == {0: 20.0, 1: 20.0}


def test_reduce_max_without_process_group_is_identity():
    assert bench.reduce_max(3.5) == 3.5


@pytest.mark.parametrize("name", sorted(WORKLOADS))
def test_row_flops_sum_to_the_workload_count(name):
    w = WORKLOADS[name]
    one_head = (w.fwd_flop() + w.bwd_flop()) / (w.B * w.H)
    assert np.isclose(bench.useful_flops_rows(w, np.arange(w.Tq)), one_head, rtol=1e-12)
    fwd_head = w.fwd_flop() / (w.B * w.H)
    assert np.isclose(bench.useful_flops_rows(w, np.arange(w.Tq), fwd_only=True), fwd_head, rtol=1e-12)


def test_spread_rows_are_sorted_unique_and_in_range():
    w = WORKLOADS["c3"]
    r = bench.spread_rows(w, 1000)
    assert r[0] == 0 and r[-1] == w.Tq - 1 and np.all(np.diff(r) > 0)


def test_oracle_legs_forward_only_on_a_small_workload():
    from exact_tiled_softmax_attn_gb300.workloads import make_inputs
    w = WORKLOADS["c1_causal"]
    x = make_inputs(w)
    rows = bench.spread_rows(w, 16)
    assert bench.oracle_sample(w, x, rows, fwd_only=True) >= 0.0
    cb = bench.cpu_baseline(w, x, target_s=0.05, fwd_only=True)
    assert cb["kind"] == "oracle" and cb["value"] > 0 and cb["sample"].startswith("float64 numpy oracle, fwd of")


@pytest.mark.parametrize("fwd_only", [False, True])
def test_reference_arm_prints_one_json_line(fwd_only):
    import json
    import subprocess
    import sys
    cmd = [sys.executable, os.path.join(bench.ROOT, "bench.py"), "--impl", "reference", "--workload", "c1",
           "--steps", "3", "--warmup", "3"] + (["--fwd-only"] if fwd_only else [])
    r = subprocess.run(cmd, capture_output=True, text=True, timeout=600, env={**os.environ, "CUDA_VISIBLE_DEVICES": ""})
    assert r.returncode == 0, r.stderr[-2000:]
    line = json.loads(r.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["value"] > 0 and line["steps"] == 3
    assert line["metric"] == (bench.METRIC_FWD if fwd_only else bench.METRIC)
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["cpu_baseline"]["kind"] == "oracle"


def test_reference_arm_under_torchrun_prints_once():
    """N > 1: rank 0 alone runs the reference arm and prints its line; the
    other rank exits 0 without work."""
    import json
    import subprocess
    import sys
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node=2",
           "--master-addr=127.0.0.1", f"--master-port={_free_port()}", os.path.join(bench.ROOT, "bench.py"),
           "--impl", "reference", "--workload", "c1", "--gpus", "2", "--steps", "3", "--warmup", "3"]
    r = subprocess.run(cmd, capture_output=True, text=True, timeout=600,
                       env={**os.environ, "CUDA_VISIBLE_DEVICES": "", "OMP_NUM_THREADS": "1"})
    assert r.returncode == 0, r.stderr[-3000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    line = json.loads(lines[0])
    assert line["impl"] == "reference" and line["n_gpus"] == 2 and line["value"] > 0


def _json_lines(out):
    import json
    return [json.loads(ln) for ln in out.splitlines() if ln.startswith("{")]


def test_gpus_flag_without_torchrun_starts_one_rank_per_gpu():
    """bench.py --gpus 2 started plainly launches two ranks itself, each with
    its own input seed (seed + 1000 * rank) and the world size in n_gpus."""
    import subprocess
    import sys
    w = WORKLOADS["c3"]
    cmd = [sys.executable, os.path.join(bench.ROOT, "bench.py"), "--gpus", "2", "--dry-run", "--workload", "c3"]
    env = {k: v for k, v in os.environ.items() if k not in ("WORLD_SIZE", "RANK", "LOCAL_RANK")}
    r = subprocess.run(cmd, capture_output=True, text=True, timeout=300, env={**env, "CUDA_VISIBLE_DEVICES": ""})
    assert r.returncode == 0, r.stderr[-3000:]
    lines = sorted(_json_lines(r.stdout), key=lambda j: j["rank"])
    assert [j["rank"] for j in lines] == [0, 1]
    assert all(j["world"] == 2 and j["n_gpus"] == 2 and j["dry_run"] for j in lines)
    assert [j["local_rank"] for j in lines] == [0, 1]
    assert [j["seed"] for j in lines] == [w.seed, w.seed + 1000]


def test_reference_arm_with_gpus_flag_alone_reports_the_world_size():
    import subprocess
    import sys
    cmd = [sys.executable, os.path.join(bench.ROOT, "bench.py"), "--impl", "reference", "--workload", "c1",
           "--gpus", "2", "--steps", "3", "--warmup", "3"]
    env = {k: v for k, v in os.environ.items() if k not in ("WORLD_SIZE", "RANK", "LOCAL_RANK")}
    r = subprocess.run(cmd, capture_output=True, text=True, timeout=600,
                       env={**env, "CUDA_VISIBLE_DEVICES": "", "OMP_NUM_THREADS": "1"})
    assert r.returncode == 0, r.stderr[-3000:]
    lines = _json_lines(r.stdout)
    assert len(lines) == 1 and lines[0]["n_gpus"] == 2 and lines[0]["impl"] == "reference"


def test_gpus_flag_must_match_the_launcher_world_size():
    import subprocess
    import sys
    cmd = [sys.executable, os.path.join(bench.ROOT, "bench.py"), "--gpus", "2", "--dry-run"]
    r = subprocess.run(cmd, capture_output=True, text=True, timeout=120,
                       env={**os.environ, "WORLD_SIZE": "1", "RANK": "0", "LOCAL_RANK": "0"})
    assert r.returncode != 0 and "WORLD_SIZE" in r.stderr


def test_rank_seeds_are_distinct():
    w = WORKLOADS["c3"]
    assert len({bench.rank_seed(w, r) for r in range(8)}) == 8 and bench.rank_seed(w, 0) == w.seed


def test_traffic_entries_name_a_kernel_a_workload_and_a_summary():
    # profiles/traffic.txt: kernel, workload, source hash, DRAM bytes per launch,
    # summary file; bench.py reports a figure only for the line's own workload
    # and only while the kernel's sources still hash the same
    path = os.path.join(bench.ROOT, "profiles", "traffic.txt")
    rows = [ln.split() for ln in open(path) if ln.strip() and not ln.startswith("#")]
    assert rows
    seen = set()
    for kernel, workload, h, nbytes, summary in rows:
        assert kernel in bench.KERNEL_SOURCES, kernel
        assert workload in WORKLOADS, workload
        assert (kernel, workload) not in seen
        seen.add((kernel, workload))
        assert len(h) == 16 and float(nbytes) > 0
        assert os.path.isfile(os.path.join(bench.ROOT, summary)), summary
    k, wl, h, nbytes, _ = rows[0]
    expect = float(nbytes) if h == bench.kernel_source_hash(k) else None
    assert bench.load_traffic(k, wl) == expect
    other = next(n for n in WORKLOADS if (k, n) not in seen)
    assert bench.load_traffic(k, other) is None


def test_bench_functions_use_only_bound_names():
    """Every name a bench.py function reads is bound in that function (an
    argument, an assignment, a local import, a nested def) or at module level:
    torch is imported inside the functions that need it, so a helper that
    forgets its own import would fail only on the GPU machine."""
    import ast
    import builtins

    src = open(os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "bench.py")).read()
    tree = ast.parse(src)
    module = set(dir(builtins)) | {"__file__", "__name__"}
    for node in tree.body:
        if isinstance(node, (ast.Import, ast.ImportFrom)):
            module |= {(a.asname or a.name).split(".")[0] for a in node.names}
        elif isinstance(node, (ast.FunctionDef, ast.ClassDef)):
            module.add(node.name)
        elif isinstance(node, (ast.Assign, ast.AnnAssign)):
            for t in (node.targets if isinstance(node, ast.Assign) else [node.target]):
                module |= {n.id for n in ast.walk(t) if isinstance(n, ast.Name)}
    for fn in (n for n in tree.body if isinstance(n, ast.FunctionDef)):
        bound = set()
        for n in ast.walk(fn):
            if isinstance(n, (ast.Import, ast.ImportFrom)):
                bound |= {(a.asname or a.name).split(".")[0] for a in n.names}
            elif isinstance(n, ast.Name) and isinstance(n.ctx, ast.Store):
                bound.add(n.id)
            elif isinstance(n, ast.arg):
                bound.add(n.arg)
            elif isinstance(n, ast.FunctionDef):
                bound.add(n.name)
        used = {n.id for n in ast.walk(fn) if isinstance(n, ast.Name) and isinstance(n.ctx, ast.Load)}
        assert not (used - bound - module), f"{fn.name} reads unbound names {sorted(used - bound - module)}"


@pytest.mark.parametrize("name", ["c1", "c1_causal", "c4", "c4_scale1", "s1f"])
def test_f32_dq_partials_matches_the_library_rule(name):
    """bench.py's reading of the library's split count (one split per
    64-key tile means the dK/dV kernel writes the dQ partials and no dQ
    kernel runs) agrees with the rule the library states: at most 1 GiB of
    partials, one fp32 [B,H,Tq,d] array per key tile."""
    from exact_tiled_softmax_attn_gb300 import binding as Bn
    from exact_tiled_softmax_attn_gb300 import build as build_mod
    build_mod.build()   # host-side calls only: no device is touched
    w = WORKLOADS[name]
    for det in (0, 1):
        S = Bn.attn_bwd_dq_splits(w.B, w.H, w.Tq, w.Tk, w.d, w.dv, Bn.ATTN_F32, det)
        n_kt = -(-w.Tk // 64)
        want = bool(det) and (n_kt == 1 or n_kt * w.B * w.H * w.Tq * w.d * 4 <= 2 ** 30)
        assert bench.f32_dq_partials(True, bool(det), w.Tk, S) == want
    # above the cap the dQ kernel's ranges hold at least two key tiles each
    S = Bn.attn_bwd_dq_splits(1, 8, 512, 65536, 128, 128, Bn.ATTN_F32, 1)
    assert S > 1 and not bench.f32_dq_partials(True, True, 65536, S)
