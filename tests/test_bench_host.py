"""CPU tier: host-side logic of bench.py — algorithmic bytes, buffer-set
sizing, the reference (oracle) arm, and the multi-rank reduction used when
bench.py runs one replica per GPU (two gloo ranks on the CPU)."""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch
import torch.multiprocessing as mp

import bench
from rmsnorm_fwd_bwd_02_gb300 import workloads as W

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_algorithmic_bytes_of_the_workloads():
    # Qwen3-8B: fwd reads x and w, writes y and rstd; bwd reads x, dy, w and
    # writes dx and dw (rstd read and workspace not counted)
    assert bench.step_bytes(W.WORKLOADS["qwen3-8b-train"]) == (537010176, 805330944)
    assert bench.step_bytes(W.WORKLOADS["qwen3-qknorm"]) == (270532864, 402653952)
    # residual: x, r in and h, y out; dy, h, dh in and dx out
    assert bench.step_bytes(W.WORKLOADS["residual-14b"]) == (671164416, 671119360)
    # decode, one token: x, w in; y, rstd out
    assert bench.step_bytes(W.WORKLOADS["decode-m1"]) == (3 * 1792 + 4, 0)


def test_buffer_sets_defeat_l2():
    for name, wl in W.WORKLOADS.items():
        n = bench.buffer_sets(wl)
        x_bytes = wl.M * wl.H * wl.elem_bytes
        if wl.N:      # the projection weight rotates: > 2 x L2 of weights
            assert 3 <= n <= 128
            assert n * wl.N * wl.H * wl.elem_bytes >= 2 * bench.L2_BYTES
            continue
        assert 3 <= n <= 64
        if bench.streams_from_hbm(wl):
            assert n == 3 and x_bytes > 100e6
        else:
            assert n * x_bytes >= min(2 * bench.L2_BYTES, 64 * x_bytes)
    assert bench.streams_from_hbm(W.WORKLOADS["qwen3-8b-train"].with_rows(16384))


def test_whole_job_value():
    assert bench.whole_job_gbs(1e9, 1, 1.0) == pytest.approx(1000.0)
    assert bench.whole_job_gbs(1e9, 4, 2.0) == pytest.approx(2000.0)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, q):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    local = 1.0 + 2.5 * rank                  # this replica's step time, ms
    q.put((rank, bench.reduce_max(local, dist)))
    dist.barrier()
    dist.destroy_process_group()


def test_reduce_max_over_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    got = dict(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert got == {0: 3.5, 1: 3.5}


def test_reference_arm_prints_one_json_line():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl",
                        "reference", "--steps", "3", "--warmup", "3", "--workload",
                        "tiny-fp32"], capture_output=True, text=True, timeout=600,
                       cwd=ROOT)
    assert r.returncode == 0, r.stderr
    lines = [l for l in r.stdout.splitlines() if l.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for k in ("impl", "metric", "value", "unit", "n_gpus", "steps", "warmup",
              "ms_per_step", "higher_is_better", "config", "cpu_baseline", "e2e"):
        assert k in d
    assert d["impl"] == "reference" and d["metric"] == bench.METRIC
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["value"] > 0


def test_gemv_step_bytes():
    """Fused norm + projection: x, r, w and A read, out and h written."""
    wl = W.WORKLOADS["decode-qkv-m1"]
    f, b = bench.step_bytes(wl)
    assert b == 0
    assert f == (2 * 896 + 896 + 2048 * 896) * 2 + (2048 + 896) * 2


def test_per_call_stats_nearest_rank():
    # 1..20 us: median 10.5, p95 by nearest rank = the 19th value
    s = bench.call_stats([1e-3 * i for i in range(1, 21)])
    assert s["n"] == 20 and s["median"] == pytest.approx(10.5)
    assert s["p95"] == pytest.approx(19.0) and s["mean"] == pytest.approx(10.5)
    assert bench.call_stats([2e-3])["p95"] == pytest.approx(2.0)


def test_threaded_oracle_timing_covers_every_row():
    """The all-cores CPU baseline cuts the rows into contiguous chunks, one per
    thread; with more threads than rows it uses one thread per row."""
    wl = W.WORKLOADS["tiny-fp32"]
    inp = W.make_inputs(wl)
    assert bench.time_oracle(wl, inp, 5, threads=8) > 0
    assert bench.time_oracle(wl, inp, 64, threads=3) > 0
    assert bench.host_cores() >= 1


def test_launch_counts_and_step_calls():
    """gpu_launches counts this library's kernels per step: forward, backward
    and dw reduce for training; the double backward's kernel and dw reduce;
    one fused projection kernel for decode."""
    assert bench.launches_per_step(W.WORKLOADS["qwen3-8b-train"]) == 3
    assert bench.has_bwd_call(W.WORKLOADS["qwen3-8b-train"])
    bwd2 = W.WORKLOADS["qwen3-8b-train-bwd2"]
    assert bench.launches_per_step(bwd2) == 2 and not bench.has_bwd_call(bwd2)
    gemv = W.WORKLOADS["decode-qkv-m1"]
    assert bench.launches_per_step(gemv) == 1 and not bench.has_bwd_call(gemv)
    assert bench.step_name(bwd2) == "double backward"


def test_every_kernel_source_is_in_a_traffic_source_set():
    """Each source under csrc/ belongs to the source set of some workload,
    so a change to it invalidates the DRAM traffic recorded for the
    workloads whose kernels it builds; the norm kernels' set is in every
    other set."""
    d = os.path.join(ROOT, "rmsnorm_fwd_bwd_02_gb300", "csrc")
    files = {f for f in os.listdir(d) if f.endswith((".cu", ".cuh", ".h"))}
    named = set().union(*bench.KERNEL_SOURCES.values())
    assert files == named
    norm = set(bench.KERNEL_SOURCES["norm"])
    assert all(norm <= set(v) for v in bench.KERNEL_SOURCES.values())
    assert {bench.source_set(wl) for wl in W.WORKLOADS.values()} == set(bench.KERNEL_SOURCES)
