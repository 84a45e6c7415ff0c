#!/usr/bin/env python3
"""Benchmark: Qwen3-style RMSNorm forward + backward on GB300.

One step = one pass of the hot path over one batch: rmsnorm_fwd then
rmsnorm_bwd (dx plus the two-stage dw) on the Qwen3-8B training shape
(M = 8 x 4096 = 32768 rows, H = 4096, bf16, fp32 rstd and dw), the shape the
throughput metric is quoted on. Other workloads (--workload) are for
investigation; their correctness is covered by the tests.

Prints ONE JSON line (rank 0). value = algorithmic HBM bytes of all ranks'
steps / max-over-ranks time, in GB/s; rows/s and the roofline fraction ride
along. Inputs stay resident in HBM during the timed region and exceed L2
(each x or dy tensor is 268 MB; three buffer sets rotate). The e2e leg goes
through the same C ABI with pinned host buffers and the host<->device copies
inside its timed region. The cpu_baseline leg times the fp64 CPU oracle on a
bounded sample of rows on this host.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                  [--workload NAME] [--no-e2e] [--no-cpu-baseline]
"""
import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from rmsnorm_fwd_bwd_02_gb300 import workloads as W  # noqa: E402

METRIC = "RMSNorm fwd/bwd achieved HBM GB/s and % of GB300 roofline; rows/s"
DEFAULT_WORKLOAD = "qwen3-8b-train"
NOMINAL_HBM_GBS = 8000.0
FALLBACK_HBM_GBS = 6800.0


# ----------------------------------------------------------------- bytes
def step_bytes(wl):
    """Algorithmic (minimal) HBM bytes of one step, split by call: every
    input read once, every output written once; the saved rstd read by the
    backward and the dw workspace are not counted (rstd can be recomputed
    from x; the workspace is overhead)."""
    es = wl.elem_bytes
    MH, H, M = wl.M * wl.H, wl.H, wl.M
    if wl.N:
        # norm fused with the projection: x (r), w and A in; out (and h) out
        ins = MH * es * (2 if wl.residual else 1) + H * es + wl.N * H * es
        outs = M * wl.N * es + (MH * es if wl.residual else 0)
        return ins + outs, 0
    if wl.double_backward:
        # dy, x, gx, w, gw (fp32), rstd in; ddy, dx2 and dw2 (fp32) out
        return 3 * MH * es + H * es + 4 * H + 4 * M + 2 * MH * es + 4 * H, 0
    if wl.residual:
        fwd = 4 * MH * es + H * es + 4 * M          # x, r in; h, y out; rstd
        bwd = 4 * MH * es + H * es + 4 * H          # dy, h, dh in; dx out; dw
    else:
        fwd = 2 * MH * es + H * es + 4 * M          # x in; y out; rstd
        bwd = 3 * MH * es + H * es + 4 * H          # dy, x in; dx out; dw
    if not wl.backward:
        bwd = 0
    return fwd, bwd


def read_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


L2_BYTES = 129 * 2 ** 20


def streams_from_hbm(wl):
    """True when one step's row tensors exceed the L2 cache, so each step
    streams from HBM."""
    fwd_b, bwd_b = step_bytes(wl)
    return fwd_b + bwd_b > L2_BYTES


def buffer_sets(wl):
    """Rotating buffer sets: three when a step's tensors exceed L2 (each step
    then streams from HBM; three sets keep any leftovers of the previous
    step out of reach), else enough to cycle through twice the L2 size
    (decode-sized steps stay launch-bound)."""
    if streams_from_hbm(wl):
        return 3
    if wl.N:         # the projection weight dominates: rotate copies of it
        a_bytes = wl.N * wl.H * wl.elem_bytes
        return int(min(128, max(3, -(-2 * L2_BYTES // a_bytes))))
    x_bytes = wl.M * wl.H * wl.elem_bytes
    return int(min(64, max(3, -(-2 * L2_BYTES // max(x_bytes, 1)))))


def has_bwd_call(wl):
    """Whether a step makes a separate backward call after the forward one
    (the double backward and the fused projection are one call each)."""
    return wl.backward and not wl.double_backward and not wl.N


def launches_per_step(wl):
    """Kernels of this library launched by one step: the fused projection
    one; the double backward its kernel and the dw reduce; forward +
    backward three (forward, backward, dw reduce); forward only one."""
    if wl.N:
        return 1
    if wl.double_backward:
        return 2
    return 3 if wl.backward else 1


def step_name(wl):
    if wl.double_backward:
        return "double backward"
    return "fwd+bwd" if wl.backward else "fwd"


def base_config(wl):
    c = {"workload": wl.name, "M": wl.M, "H": wl.H, "eps": wl.eps,
         "dtype": str(wl.dtype).replace("torch.", ""),
         "step": "fwd+bwd" if wl.backward else "fwd"}
    if wl.ld:
        c["row_stride"] = wl.ld
    if wl.N:
        c["N"] = wl.N
        c["step"] = ("residual add + " if wl.residual else "") + \
            "RMSNorm + projection GEMV (one call)"
    if wl.double_backward:
        c["step"] = "double backward (rmsnorm_bwd_bwd: ddy, dx2, dw2)"
    return c


def reduce_max(value, dist):
    """Max of a float over all ranks (replicas time independently; the job
    takes as long as its slowest rank). NCCL reduces on the GPU, gloo on the
    CPU."""
    if dist is None:
        return float(value)
    on_gpu = dist.get_backend() == "nccl"
    t = torch.tensor([float(value)], dtype=torch.float64,
                     device=torch.device("cuda", torch.cuda.current_device())
                     if on_gpu else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_gbs(bytes_per_step, world, ms_per_step):
    """GB/s of all ranks' steps over the max-over-ranks step time."""
    return bytes_per_step * world / (ms_per_step * 1e-3) / 1e9


# ---------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons, in a background
    process, so the ones inside the timed region can be reported."""
    FIELDS = ("timestamp,uuid,clocks.sm,clocks.max.sm,power.draw,"
              "clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, uuid):
        self.uuid = uuid
        self.rows = []
        self.proc = None
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.rows.append((time.time(), [c.strip() for c in line.split(",")]))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.thread.join(timeout=5)

    def summary(self, t0, t1):
        if self.proc is None:
            return None
        mine = [r for t, r in self.rows if len(r) >= 10 and
                (self.uuid is None or r[1] == self.uuid)]
        inside = [r for t, r in self.rows if t0 - 0.05 <= t <= t1 + 0.15 and len(r) >= 10
                  and (self.uuid is None or r[1] == self.uuid)]
        use = inside or mine[-3:]
        if not use:
            return None

        def num(s):
            try:
                return float(s)
            except ValueError:
                return None
        sm = [num(r[2]) for r in use if num(r[2]) is not None]
        mx = [num(r[3]) for r in use if num(r[3]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown",
                 "sw_power_cap"]
        reasons = sorted({names[i] for r in use for i in range(4)
                          if r[6 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "samples": len(use), "samples_inside_timed_region": len(inside)}


# ---------------------------------------------------------------- oracle leg
def host_cpu_model():
    """The host CPU's model name (lscpu), else the machine architecture."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.strip().lower().startswith("model name:"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    import platform
    return platform.machine()


def host_cores():
    """Host threads this process may run on."""
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def _oracle_pass(orc, wl, sub):
    """One pass of the workload's calls on the oracle over the rows in `sub`."""
    if wl.N:
        orc.rmsnorm_gemv(sub["x"], sub["w"], sub["A"], wl.eps,
                         r=sub["r"] if wl.residual else None)
    elif wl.double_backward:
        orc.bwd_bwd(sub["dy"], sub["x"], sub["w"], sub["gx"], sub["gw"], wl.eps)
    elif wl.residual:
        h, _, _ = orc.residual_fwd(sub["x"], sub["r"], sub["w"], wl.eps)
        if wl.backward:
            orc.residual_bwd(sub["dy"], sub["dh"], h, sub["w"], wl.eps)
    else:
        orc.fwd(sub["x"], sub["w"], wl.eps)
        if wl.backward:
            orc.bwd(sub["dy"], sub["x"], sub["w"], wl.eps)


def time_oracle(wl, inp, rows, reps=1, threads=1):
    """Wall seconds for the fp64 CPU oracle, as it stands, to run the
    workload's calls on `rows` rows. With threads > 1 the rows are cut into
    that many contiguous chunks, one per thread (the oracle's ctypes calls
    release the GIL, so the chunks run in parallel); the per-chunk dw rows
    are not summed afterwards (threads x H adds, negligible)."""
    import oracle
    orc = oracle.get()
    threads = max(1, min(threads, rows))
    if wl.N:                        # one decode batch: not cut
        threads = 1
    cuts = [rows * i // threads for i in range(threads + 1)]
    subs = [{k: (v[a:b].contiguous() if v.dim() == 2 and k != "A" else v)
             for k, v in inp.items()} for a, b in zip(cuts, cuts[1:])]
    if threads == 1:
        t0 = time.perf_counter()
        for _ in range(reps):
            _oracle_pass(orc, wl, subs[0])
        return (time.perf_counter() - t0) / reps
    from concurrent.futures import ThreadPoolExecutor
    with ThreadPoolExecutor(max_workers=threads) as pool:
        t0 = time.perf_counter()
        for _ in range(reps):
            list(pool.map(lambda sub: _oracle_pass(orc, wl, sub), subs))
        return (time.perf_counter() - t0) / reps


def cpu_baseline(wl, inp, budget_s=8.0):
    """The oracle on bounded samples of the workload's rows, scaled to GB/s
    of the same algorithmic bytes per row: once on every host core (about
    2 x budget_s of CPU work in all) and once on one thread (budget_s)."""
    probe = min(wl.M, 64)
    t_row = time_oracle(wl, inp, probe) / probe
    rows = int(max(1, min(wl.M, budget_s / max(t_row, 1e-9))))
    secs = time_oracle(wl, inp, rows)
    fwd_b, bwd_b = step_bytes(wl.with_rows(rows))
    single = (fwd_b + bwd_b) / secs / 1e9
    cores = host_cores()
    rows_mt = int(max(1, min(wl.M, 2 * budget_s / max(t_row, 1e-9))))
    secs_mt = time_oracle(wl, inp, rows_mt, threads=cores)
    used = 1 if wl.N else max(1, min(cores, rows_mt))
    fwd_b, bwd_b = step_bytes(wl.with_rows(rows_mt))
    what = step_name(wl)
    return {"value": round((fwd_b + bwd_b) / secs_mt / 1e9, 4), "unit": "GB/s",
            "cores": used, "kind": "oracle",
            "sample": f"{rows_mt} of {wl.M} rows of {wl.name} (H={wl.H}), {what}, "
                      f"fp64 oracle on {used} threads (contiguous row chunks), "
                      f"{secs_mt:.2f} s; single thread: {rows} rows, {secs:.2f} s",
            "rows_per_s": round(rows_mt / secs_mt, 2),
            "single_thread_value": round(single, 4),
            "cpu_model": host_cpu_model()}


def run_reference(args, wl):
    """The oracle arm: the same metric on bounded CPU samples per step, the
    oracle as it stands run on every host core (contiguous row chunks)."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    cores = host_cores()
    inp = W.make_inputs(wl.with_rows(min(wl.M, 4096)))
    M_in = inp["x"].shape[0]
    probe = min(16, M_in)
    t_row = time_oracle(wl, inp, probe) / probe
    threads = 1 if wl.N else cores
    per_step = int(max(1, min(M_in, threads * 60.0 / max(args.steps + args.warmup, 1)
                                    / t_row)))
    used = 1 if wl.N else max(1, min(cores, per_step))
    for _ in range(args.warmup):
        time_oracle(wl, inp, per_step, threads=threads)
    times = [time_oracle(wl, inp, per_step, threads=threads) for _ in range(args.steps)]
    total = sum(times)
    fwd_b, bwd_b = step_bytes(wl.with_rows(per_step))
    value = (fwd_b + bwd_b) * args.steps / total / 1e9
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 4),
        "unit": "GB/s", "n_gpus": args.gpus, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(1e3 * total / args.steps, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f64", "data": "synthetic",
        "config": base_config(wl),
        "rows_per_s": round(per_step * args.steps / total, 2),
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": used,
                         "kind": "oracle", "cpu_model": host_cpu_model(),
                         "sample": f"{per_step} rows of {wl.name} per step "
                                   f"({step_name(wl)}), "
                                   f"fp64 oracle on {used} threads"},
        "e2e": {"value": round(value, 4), "unit": "GB/s",
                "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# ---------------------------------------------------------------- GPU leg
class Calls:
    """Device buffers for one step and the C-ABI calls of the step. The
    ctypes arguments are marshalled once (bind), so a timed step costs the
    host two or three foreign calls and nothing else."""

    def __init__(self, rn, wl, src, dev, ws, w):
        self.rn, self.wl = rn, wl
        if wl.ld:        # every [M, H] tensor a column window of an [M, ld] buffer
            place = lambda t: W.in_strided(t, wl.ld, 0.0)  # noqa: E731
        else:
            place = lambda t: t  # noqa: E731
        e = lambda: place(torch.empty(wl.M, wl.H, device=dev, dtype=wl.dtype))  # noqa: E731
        self.x = place(src["x"].to(dev))
        self.dy = place(src["dy"].to(dev)) if wl.backward else None
        self.r = place(src["r"].to(dev)) if wl.residual else None
        self.dh = place(src["dh"].to(dev)) if wl.residual else None
        self.y, self.h = e(), (e() if wl.residual else None)
        self.dx = e() if wl.backward else None
        self.rstd = torch.empty(wl.M, device=dev)
        self.dw = torch.empty(wl.H, device=dev)
        self.ws = ws
        self.w = w
        if wl.N:         # one copy of the projection weight per buffer set
            self.A = src["A"].to(dev)
            self.out = torch.empty(wl.M, wl.N, device=dev, dtype=wl.dtype)
        if wl.double_backward:
            self.gx = src["gx"].to(dev)
            self.gw = src["gw"].to(dev)
            self.ddy, self.dx2 = e(), e()
            self.dw2 = torch.empty(wl.H, device=dev)
            rn.rmsnorm_fwd(self.x, self.w, rstd=self.rstd, eps=wl.eps)   # the saved rstd
        self.bind(torch.cuda.current_stream())

    def bind(self, stream):
        """Marshal the C-ABI arguments for launches on `stream`."""
        lib, wl = self.rn.lib(), self.wl
        P = lambda t: None if t is None else t.data_ptr()  # noqa: E731
        code = self.rn.DTYPES[wl.dtype]
        s = stream.cuda_stream
        ws_bytes = self.ws.numel()
        if wl.double_backward:
            self._f = (lib.rmsnorm_bwd_bwd,
                       (P(self.dy), P(self.x), P(self.w), P(self.rstd), P(self.gx),
                        P(self.gw), P(self.ddy), P(self.dx2), P(self.dw2), P(self.ws),
                        ws_bytes, wl.M, wl.H, wl.eps, code, s))
            self._b = None
            return
        if wl.N:
            # decode: the weights are static while the step runs
            self._f = (lib.rmsnorm_gemv_fwd,
                       (P(self.x), P(self.r), P(self.w), P(self.A), P(self.out),
                        P(self.h), None, None, wl.M, wl.H, wl.N, wl.eps, code,
                        self.rn.GEMV_STATIC_WEIGHTS, s))
            self._b = None
            return
        if wl.ld:
            ld = wl.ld
            self._f = (lib.rmsnorm_fwd_strided,
                       (P(self.x), ld, P(self.r), ld, P(self.w), P(self.y), ld,
                        P(self.h), ld, P(self.rstd), wl.M, wl.H, wl.eps, code, s))
            self._b = (lib.rmsnorm_bwd_strided,
                       (P(self.dy), ld, P(self.dh), ld,
                        P(self.h if wl.residual else self.x), ld, P(self.w),
                        P(self.rstd), P(self.dx), ld, P(self.dw), P(self.ws),
                        ws_bytes, wl.M, wl.H, wl.eps, code, 0, s))
        elif wl.residual:
            self._f = (lib.rmsnorm_residual_fwd,
                       (P(self.x), P(self.r), P(self.w), P(self.h), P(self.y),
                        P(self.rstd), wl.M, wl.H, wl.eps, code, s))
            self._b = (lib.rmsnorm_residual_bwd,
                       (P(self.dy), P(self.dh), P(self.h), P(self.w), P(self.rstd),
                        P(self.dx), P(self.dw), P(self.ws), ws_bytes, wl.M, wl.H,
                        wl.eps, code, s))
        else:
            self._f = (lib.rmsnorm_fwd,
                       (P(self.x), P(self.w), P(self.y), P(self.rstd), wl.M, wl.H,
                        wl.eps, code, s))
            self._b = (lib.rmsnorm_bwd,
                       (P(self.dy), P(self.x), P(self.w), P(self.rstd), P(self.dx),
                        P(self.dw), P(self.ws), ws_bytes, wl.M, wl.H, wl.eps, code, s))
        if not wl.backward:
            self._b = None

    def _call(self, fa):
        st = fa[0](*fa[1])
        if st != 0:
            raise self.rn.RmsNormError(st, fa[0].__name__)

    def fwd(self):
        self._call(self._f)

    def bwd(self):
        if self._b is not None:
            self._call(self._b)


def gpu_uuid():
    try:
        u = torch.cuda.get_device_properties(torch.cuda.current_device()).uuid
        s = str(u)
        return s if s.startswith("GPU-") else "GPU-" + s
    except Exception:
        return None


PER_CALL_N = 200   # calls per direction in the per-call statistics


def time_back_to_back(stream, fns, n):
    """Mean ms per call of n consecutive calls fns[i % len(fns)]() on
    `stream`, with events at the two ends only, so consecutive launches keep
    their programmatic-dependent-launch overlap (as a caller runs them)."""
    for f in fns:                      # warm: every buffer set once
        f()
    s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    s.record(stream)
    for i in range(n):
        fns[i % len(fns)]()
    e.record(stream)
    torch.cuda.synchronize()
    return s.elapsed_time(e) / n


def time_each(stream, fns, n):
    """Per-call ms of n calls, each between its own pair of events on
    `stream`. An event between two launches stops the second from starting
    while the first drains, so these are isolated-call times, a little
    slower than back-to-back calls."""
    for f in fns:
        f()
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(n + 1)]
    ev[0].record(stream)
    for i in range(n):
        fns[i % len(fns)]()
        ev[i + 1].record(stream)
    torch.cuda.synchronize()
    return [ev[i].elapsed_time(ev[i + 1]) for i in range(n)]


def build_sets(rn, wl, dev):
    """Rotating device buffer sets for the workload (see buffer_sets), with
    their C-ABI calls bound to the current stream."""
    src = W.make_inputs(wl)
    w = src["w"].to(dev)
    ws = torch.empty(max(16, rn.bwd_workspace_bytes(wl.M, wl.H, wl.dtype)),
                     device=dev, dtype=torch.uint8)
    sets = [Calls(rn, wl, src, dev, ws, w) for _ in range(buffer_sets(wl))]
    if wl.N:
        # decode: the activations (x, r and the outputs) are one small set
        # that stays in L2, as the previous kernel's output would; only the
        # projection weights rotate, so each call streams its weight from HBM
        for c in sets[1:]:
            c.x, c.r, c.h, c.out = sets[0].x, sets[0].r, sets[0].h, sets[0].out
            c.bind(torch.cuda.current_stream())
    return src, sets


def uses_graph(wl):
    """Decode-sized steps are a few microseconds of GPU work, less than the
    host needs to issue them one by one; they are timed the way a decoder
    runs them, replayed from a CUDA graph of consecutive calls."""
    fwd_b, bwd_b = step_bytes(wl)
    return fwd_b + bwd_b < 64 * 2 ** 20


def capture_graphs(sets, counts, fwd=True, bwd=True):
    """CUDA graphs of consecutive steps over the rotating sets, one per count
    in `counts`, captured on a side stream (the sets are bound back to the
    current stream afterwards)."""
    gstream = torch.cuda.Stream()
    gstream.wait_stream(torch.cuda.current_stream())
    for c in sets:
        c.bind(gstream)
    with torch.cuda.stream(gstream):
        for c in sets:                    # warm the library's caches
            if fwd:
                c.fwd()
            if bwd:
                c.bwd()
    torch.cuda.synchronize()
    graphs = []
    for n in counts:
        gr = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gr, stream=gstream):
            for i in range(n):
                if fwd:
                    sets[i % len(sets)].fwd()
                if bwd:
                    sets[i % len(sets)].bwd()
        graphs.append((n, gr))
    for c in sets:
        c.bind(torch.cuda.current_stream())
    return graphs


def time_graph(stream, graph, n_per, reps):
    """ms per step of a graph of n_per consecutive steps, replayed reps times."""
    graph.replay()
    torch.cuda.synchronize()
    s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    s.record(stream)
    for _ in range(reps):
        graph.replay()
    e.record(stream)
    torch.cuda.synchronize()
    return s.elapsed_time(e) / (reps * n_per)


def direction_times(wl, sets, stream):
    """Per-direction times: the mean of PER_CALL_N back-to-back calls (the
    roofline's figure) and PER_CALL_N isolated calls (median, P95). Graph
    workloads: the mean per call of graph-replayed forward-only and
    backward-only runs of 64 calls."""
    out = {}
    dirs = [("fwd", [c.fwd for c in sets])]
    if has_bwd_call(wl):
        dirs.append(("bwd", [c.bwd for c in sets]))
    if uses_graph(wl):
        for name, _ in dirs:
            (n, gr), = capture_graphs(sets, [64], fwd=name == "fwd", bwd=name == "bwd")
            out[name] = {"back_to_back_ms": time_graph(stream, gr, n, max(4, PER_CALL_N // n)),
                         "n": 64 * max(4, PER_CALL_N // n), "each_ms": None}
        return out
    for name, fns in dirs:
        b2b = time_back_to_back(stream, fns, PER_CALL_N)
        each = time_each(stream, fns, PER_CALL_N)
        out[name] = {"back_to_back_ms": b2b, "n": PER_CALL_N, "each_ms": each}
    return out


# The method's workloads, reported together by the default run: the
# training shapes (fwd + bwd), the decode split-row norms (fwd) and the tiny
# fp32 reference case.
SUITE = ("qwen3-8b-train", "qwen3-qknorm", "residual-14b", "decode-m1", "decode-m8",
         "decode-m64", "tiny-fp32")


def measure_suite(rn, dev, args, headline):
    """Figures for each workload of SUITE in the same run: the headline
    workload's from the main measurement, the others measured here on their
    own rotating buffers. Streamed workloads: max(steps, 20) forward +
    backward steps back to back between two events, and per direction the
    mean of PER_CALL_N back-to-back calls. Decode-sized workloads: CUDA-graph
    replay of 64 consecutive steps, microseconds per step (their inputs are
    L2-resident, so they are latency-bound and a bandwidth fraction says
    little about them)."""
    peak, peak_kind = read_peaks()
    stream = torch.cuda.current_stream()
    out = {}
    for name in SUITE:
        wl = W.WORKLOADS[name]
        fwd_b, bwd_b = step_bytes(wl)
        graph = uses_graph(wl)
        if name == headline["workload"]:
            step_ms, fwd_ms, bwd_ms = (headline["ms_per_step"], headline["fwd_ms"],
                                       headline["bwd_ms"])
        else:
            src, sets = build_sets(rn, wl, dev)
            if graph:
                (n, gr), = capture_graphs(sets, [64])
                step_ms = time_graph(stream, gr, n, 50)
            else:
                step_ms = time_back_to_back(
                    stream, [lambda c=c: (c.fwd(), c.bwd()) for c in sets],
                    max(args.steps, 20))
            dt = direction_times(wl, sets, stream)
            fwd_ms = dt["fwd"]["back_to_back_ms"]
            bwd_ms = dt["bwd"]["back_to_back_ms"] if "bwd" in dt else 0.0
            del sets, src
            torch.cuda.empty_cache()
        gbs = (fwd_b + bwd_b) / (step_ms * 1e-3) / 1e9
        e = {"M": wl.M, "H": wl.H, "dtype": str(wl.dtype).replace("torch.", ""),
             "step": step_name(wl) + (" (dh_out given)" if wl.residual and wl.backward else ""),
             "us_per_step": round(1e3 * step_ms, 3), "GB_per_s": round(gbs, 1),
             "rows_per_s": round(wl.M / (step_ms * 1e-3), 1),
             "frac_of_measured_hbm": round(gbs / peak, 4),
             "frac_of_nominal_8TBs": round(gbs / NOMINAL_HBM_GBS, 4),
             "step_bytes": fwd_b + bwd_b,
             "timing": ("CUDA-graph replay of 64 consecutive steps, L2-resident "
                        "inputs (latency-bound)" if graph else
                        "steps back to back over rotating buffer sets larger than L2")}
        for d, b, ms in (("fwd", fwd_b, fwd_ms), ("bwd", bwd_b, bwd_ms)):
            if b and ms:
                g = b / (ms * 1e-3) / 1e9
                e[d] = {"us": round(1e3 * ms, 3), "GB_per_s": round(g, 1),
                        "frac_of_measured_hbm": round(g / peak, 4), "bytes": b}
        out[name] = e
    out["peak_gbs"] = peak
    out["peak_kind"] = peak_kind
    return out


# The fused projection (rmsnorm_gemv_fwd) against the same work unfused, per
# call: the two decode projections of a 896-feature model at 1 to 64 rows
# and of a 4096-feature model at 16 to 64 rows.
PROJECTIONS = (("decode-qkv-m1", (1, 16, 32, 48, 64)), ("decode-gateup-m1", (1, 16, 32, 48, 64)),
               ("decode-8b-qkv-m16", (16, 32, 48, 64)),
               ("decode-8b-gateup-m16", (16, 32, 48, 64)))
GEMV_KERNELS = {5: "rms_gemv", 6: "rms_gemv_tma", 7: "rms_gemv_umma", 8: "rms_gemv_tc"}


def measure_projections(rn, dev, args):
    """Microseconds per call of rmsnorm_gemv_fwd and of the unfused pair
    (this library's norm, then torch.matmul on cuBLAS) for each shape of
    PROJECTIONS: both replayed from CUDA graphs of consecutive calls, the
    weights rotating through more than twice L2, the activations L2-resident."""
    stream = torch.cuda.current_stream()
    out = {}
    for name, rows in PROJECTIONS:
        for M in rows:
            wl = W.WORKLOADS[name].with_rows(M)
            src, sets = build_sets(rn, wl, dev)
            (n, gr), = capture_graphs(sets, [64])
            sets[0].fwd()
            path = rn.last_path()
            fused = 1e3 * time_graph(stream, gr, n, 20)
            unf = time_unfused_gemv(rn, wl, sets, 64 * 20)["us_per_step"]
            out[f"{M}x{wl.H}->{wl.N}"] = {
                "M": M, "H": wl.H, "N": wl.N, "residual": bool(wl.residual),
                "fused_us": round(fused, 3), "unfused_us": round(unf, 3),
                "fused_over_unfused": round(fused / unf, 3),
                "kernel": GEMV_KERNELS.get(path, str(path))}
            del gr, sets, src
            torch.cuda.empty_cache()
    out["timing"] = ("CUDA-graph replay of 64 consecutive calls, weights rotating "
                     "through more than twice L2; unfused = rmsnorm_residual_fwd + "
                     "torch.matmul (cuBLAS)")
    return out


def run_ours(args, wl):
    from rmsnorm_fwd_bwd_02_gb300 import rmsnorm as rn
    rn.lib()
    if args.path_override:
        rn.set_path_override(args.path_override)
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    stream = torch.cuda.current_stream()

    src, sets = build_sets(rn, wl, dev)
    ws = sets[0].ws
    n_sets = len(sets)
    x_bytes = wl.M * wl.H * wl.elem_bytes
    fwd_b, bwd_b = step_bytes(wl)

    def barrier():
        if dist is not None:
            dist.barrier()
        torch.cuda.synchronize()

    use_graph = uses_graph(wl)
    graphs = []
    if use_graph:
        per = min(args.steps, 64)
        graphs = capture_graphs(sets, sorted({per, args.steps % per} - {0}, reverse=True))

    # warm-up: W steps
    path_f = path_b = 0
    for i in range(args.warmup):
        c = sets[i % n_sets]
        c.fwd()
        path_f = rn.last_path()
        c.bwd()
        path_b = rn.last_path()
    for n, gr in graphs:
        gr.replay()
    barrier()

    sampler = ClockSampler(gpu_uuid()) if rank == 0 else None
    if sampler:
        sampler.start()
        time.sleep(0.3)
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    barrier()
    t_wall0 = time.time()
    start.record(stream)
    if use_graph:
        big_n, big = graphs[0]
        for _ in range(args.steps // big_n):
            big.replay()
        for n, gr in graphs[1:]:
            gr.replay()
    else:
        # the steps run back to back, as a caller runs them (no event in
        # between); the per-call figures come from separate loops below
        for i in range(args.steps):
            c = sets[i % n_sets]
            c.fwd()
            c.bwd()
    end.record(stream)
    barrier()
    t_wall1 = time.time()
    clocks = None
    if sampler:
        time.sleep(0.2)
        sampler.stop()
        clocks = sampler.summary(t_wall0, t_wall1)

    total_ms = reduce_max(start.elapsed_time(end), dist)
    ms_step = total_ms / args.steps

    # per-direction figures, outside the value's timed region
    dt = direction_times(wl, sets, stream)
    fwd_avg = dt["fwd"]["back_to_back_ms"]
    bwd_avg = dt["bwd"]["back_to_back_ms"] if "bwd" in dt else 0.0

    unfused = time_unfused_gemv(rn, wl, sets, args.steps) if wl.N else None

    # ---- e2e: host buffers, copies inside the timed region
    e2e = None
    if not args.no_e2e:
        e2e = (run_e2e_gemv(rn, wl, src, sets, args, dist) if wl.N else
               run_e2e_bwd2(rn, wl, src, sets[0], args, dist) if wl.double_backward else
               run_e2e(rn, wl, src, dev, ws, args, dist))

    suite = None
    if not args.no_workloads and world == 1 and wl.name == DEFAULT_WORKLOAD \
            and not args.path_override:
        del sets
        torch.cuda.empty_cache()
        suite = measure_suite(rn, dev, args, {"workload": wl.name, "ms_per_step": ms_step,
                                              "fwd_ms": fwd_avg, "bwd_ms": bwd_avg})
        suite["projections"] = measure_projections(rn, dev, args)

    if rank != 0:
        if dist is not None:
            dist.destroy_process_group()
        return 0

    peak, peak_kind = read_peaks()
    value = whole_job_gbs(fwd_b + bwd_b, world, ms_step)
    dom_is_bwd = has_bwd_call(wl) and bwd_b >= fwd_b
    dom_bytes, dom_ms = (bwd_b, bwd_avg) if dom_is_bwd else (fwd_b, fwd_avg)
    achieved = dom_bytes / (dom_ms * 1e-3) / 1e9
    # recorded for the automatic kernels only
    traffic = None if args.path_override else load_traffic(wl, "bwd" if dom_is_bwd else "fwd")
    def roof(b, ms, kernel):
        a = b / (ms * 1e-3) / 1e9
        return {"kernel": kernel, "bound": "hbm", "achieved": round(a, 1),
                "peak": peak, "unit": "GB/s", "frac": round(a / peak, 4),
                "peak_kind": peak_kind, "bytes_per_launch": b,
                "avg_ms": round(ms, 5),
                "frac_of_nominal_8TBs": round(a / NOMINAL_HBM_GBS, 4)}

    fam = {1: "rows", 2: "split", 3: "rows, scalar", 4: "stream", 5: "gemv", 6: "gemv_tma"}
    fwd_api = "rmsnorm_bwd_bwd" if wl.double_backward else \
        "rmsnorm_gemv_fwd" if wl.N else "rmsnorm_fwd_strided" if wl.ld else (
            "rmsnorm_residual_fwd" if wl.residual else "rmsnorm_fwd")
    bwd_api = "rmsnorm_bwd_strided" if wl.ld else (
        "rmsnorm_residual_bwd" if wl.residual else "rmsnorm_bwd")
    fwd_kernel = fwd_api + (
        {6: " (rms_gemv_tma)", 7: " (rms_gemv_umma)", 8: " (rms_gemv_tc)"}.get(
            path_f, " (rms_gemv)") if wl.N else
        f" (rms_bwd2_{fam.get(path_f, 'rows').split(',')[0]} + dw_reduce)"
        if wl.double_backward else
        f" (rms_fwd_{fam.get(path_f, 'rows').split(',')[0]})")
    bwd_kernel = bwd_api + \
        f" (rms_bwd_{fam.get(path_b, 'rows').split(',')[0]} + dw_reduce)"
    roofline = roof(dom_bytes, dom_ms, bwd_kernel if dom_is_bwd else fwd_kernel)
    roofline["achieved"] = round(achieved, 1)
    roofline["traffic"] = traffic
    line = {
        "metric": METRIC, "value": round(value, 1), "unit": "GB/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(ms_step, 5), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None,
        "dtype": {torch.bfloat16: "bf16", torch.float16: "f16"}.get(wl.dtype, "f32"),
        "data": "synthetic",
        "config": dict(base_config(wl), **{
            "l2": (f"inputs larger than L2: {n_sets} rotating buffer sets, "
                   f"{x_bytes / 1e6:.0f} MB per row tensor"
                   if streams_from_hbm(wl) else
                   f"{n_sets} rotating copies of the {wl.N}x{wl.H} projection "
                   f"weight ({n_sets * wl.N * wl.H * wl.elem_bytes / 1e6:.0f} MB, "
                   f"more than twice L2: every call reads its weight from HBM); "
                   f"one set of activations, L2-resident as a decode step's are"
                   if wl.N else
                   f"{n_sets} rotating buffer sets of {x_bytes / 1e6:.3f} MB per "
                   f"row tensor (L2-resident; launch-bound)"),
            "parallelism": "replicas" if world > 1 else "single"},
            **({"path_override": args.path_override} if args.path_override else {})),
        "rows_per_s": round(wl.M * world / (ms_step * 1e-3), 1),
        "pct_of_measured_hbm": round(100 * value / world / peak, 2),
        "pct_of_nominal_8TBs": round(100 * value / world / NOMINAL_HBM_GBS, 2),
        "step_bytes": {"fwd": fwd_b, "bwd": bwd_b},
        "roofline": roofline,
        "roofline_fwd": roof(fwd_b, fwd_avg, fwd_kernel),
        "gpu_launches": args.steps * launches_per_step(wl),
        "timing": ("CUDA-graph replay of consecutive calls (decode-sized step); "
                   "per direction, graph replays of 64 calls of that direction"
                   if use_graph else
                   f"value from events around all {args.steps} steps run back to back "
                   f"on the launching stream; per direction afterwards, "
                   f"{PER_CALL_N} back-to-back calls between two events (roofline) "
                   f"and {PER_CALL_N} calls each between its own events (per_call_us)"),
        "clocks": clocks,
        "e2e": e2e,
        "cpu_baseline": None,
    }
    if has_bwd_call(wl):
        line["roofline_bwd"] = roof(bwd_b, bwd_avg, bwd_kernel)
    line["per_call_us"] = {}
    for name, d in dt.items():
        st = call_stats(d["each_ms"]) if d["each_ms"] else {"n": d["n"]}
        st["back_to_back_mean"] = round(1e3 * d["back_to_back_ms"], 3)
        st["back_to_back_n"] = d["n"]
        line["per_call_us"][name] = st
    if suite is not None:
        line["workloads"] = suite
    if wl.N:
        line["unfused"] = unfused
    if not args.no_cpu_baseline and world == 1:
        line["cpu_baseline"] = cpu_baseline(wl, src)
    print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()
    return 0


def call_stats(ms):
    """Mean, median and 95th percentile (nearest rank) of per-call times in
    microseconds, over calls each timed between its own events."""
    us = sorted(1e3 * m for m in ms)
    p95 = us[min(len(us) - 1, max(0, -(-95 * len(us) // 100) - 1))]
    return {"n": len(us), "mean": round(statistics.mean(us), 3),
            "median": round(statistics.median(us), 3), "p95": round(p95, 3)}


def time_unfused_gemv(rn, wl, sets, steps):
    """Microseconds per call of the same work unfused: this library's norm
    (rmsnorm_residual_fwd or rmsnorm_fwd, writing y) followed by a cuBLAS
    product (torch.matmul) of y with A^T, replayed from a CUDA graph over
    the same rotating buffers. Context for the fused call, not part of the
    product."""
    # one set of activations (L2-resident), as for the fused call
    y1 = torch.empty(wl.M, wl.H, device=sets[0].x.device, dtype=wl.dtype)
    o1 = torch.empty(wl.M, wl.N, device=sets[0].x.device, dtype=wl.dtype)
    ys, outs = [y1] * len(sets), [o1] * len(sets)
    gs = torch.cuda.Stream()
    gs.wait_stream(torch.cuda.current_stream())

    def call(i):
        c, y = sets[i % len(sets)], ys[i % len(sets)]
        if wl.residual:
            rn.rmsnorm_residual_fwd(c.x, c.r, c.w, h=c.h, y=y, eps=wl.eps, stream=gs)
        else:
            rn.rmsnorm_fwd(c.x, c.w, y=y, want_rstd=False, eps=wl.eps, stream=gs)
        torch.matmul(y, c.A.t(), out=outs[i % len(sets)])

    with torch.cuda.stream(gs):
        for i in range(len(sets)):
            call(i)
    torch.cuda.synchronize()
    per = min(steps, 64)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=gs):
        for i in range(per):
            call(i)
    g.replay()
    torch.cuda.synchronize()
    reps = max(1, steps // per)
    s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    s.record()
    for _ in range(reps):
        g.replay()
    e.record()
    torch.cuda.synchronize()
    return {"us_per_step": round(1e3 * s.elapsed_time(e) / (reps * per), 3),
            "calls": ("rmsnorm_residual_fwd" if wl.residual else "rmsnorm_fwd") +
                     " + torch.matmul (cuBLAS), CUDA-graph replay"}


def run_e2e_bwd2(rn, wl, src, c, args, dist):
    """The double backward through the binding with host tensors: every step
    copies dy, x, gx, w and gw from pinned host memory, runs
    rmsnorm_bwd_bwd (with the saved rstd already on the device, as a
    training step has it) and copies ddy, dx2 and dw2 back, on one stream."""
    keys = ("dy", "x", "gx", "w", "gw")
    pin = {k: src[k].pin_memory() for k in keys}
    dev_in = {"dy": c.dy, "x": c.x, "gx": c.gx, "w": c.w, "gw": c.gw}
    outs = {"ddy": c.ddy, "dx2": c.dx2, "dw2": c.dw2}
    host = {k: torch.empty(v.shape, dtype=v.dtype, pin_memory=True) for k, v in outs.items()}
    main = torch.cuda.current_stream()

    def step():
        for k in keys:
            dev_in[k].copy_(pin[k], non_blocking=True)
        rn.rmsnorm_bwd_bwd(c.dy, c.x, c.w, c.rstd, c.gx, c.gw, ddy=c.ddy, dx2=c.dx2,
                           dw2=c.dw2, workspace=c.ws, eps=wl.eps, stream=main)
        for k, v in outs.items():
            host[k].copy_(v, non_blocking=True)

    steps = max(1, min(args.steps, 50))
    for _ in range(3):
        step()
    torch.cuda.synchronize()
    if dist is not None:
        dist.barrier()
    s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    s.record(main)
    for _ in range(steps):
        step()
    e.record(main)
    torch.cuda.synchronize()
    ms = reduce_max(s.elapsed_time(e) / steps, dist)
    world = dist.get_world_size() if dist is not None else 1
    fwd_b, _ = step_bytes(wl)
    return {"value": round(whole_job_gbs(fwd_b, world, ms), 1), "unit": "GB/s",
            "h2d_bytes_per_step": sum(v.numel() * v.element_size() for v in pin.values()),
            "d2h_bytes_per_step": sum(v.numel() * v.element_size() for v in host.values()),
            "ms_per_step": round(ms, 4), "steps": steps,
            "pipeline": "one stream: copies in, double backward, copies out"}


def run_e2e_gemv(rn, wl, src, sets, args, dist):
    """The fused norm + projection through the binding with host
    activations: every step copies x and r from pinned host memory, runs
    rmsnorm_gemv_fwd and copies out and h back, all inside the timed region
    on one stream (a decode step's shape of work). The weights w and A stay
    resident, as a model's do; the calls rotate over the benchmark's copies
    of A, so each reads its weight from HBM."""
    M, H, N = wl.M, wl.H, wl.N
    pin = {k: src[k].pin_memory() for k in ("x", "r") if k in src}
    host_out = torch.empty(M, N, dtype=wl.dtype, pin_memory=True)
    host_h = torch.empty(M, H, dtype=wl.dtype, pin_memory=True) if wl.residual else None
    main = torch.cuda.current_stream()

    def step(i):
        c = sets[i % len(sets)]
        c.x.copy_(pin["x"], non_blocking=True)
        if wl.residual:
            c.r.copy_(pin["r"], non_blocking=True)
        rn.rmsnorm_gemv_fwd(c.x, c.w, c.A, r=c.r, out=c.out, h=c.h, eps=wl.eps,
                            static_weights=True, stream=main)
        host_out.copy_(c.out, non_blocking=True)
        if wl.residual:
            host_h.copy_(c.h, non_blocking=True)

    steps = max(1, min(args.steps, 2000))
    for i in range(max(3, min(args.warmup, 20))):
        step(i)
    torch.cuda.synchronize()
    if dist is not None:
        dist.barrier()
    s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    s.record(main)
    for i in range(steps):
        step(i)
    e.record(main)
    torch.cuda.synchronize()
    ms = reduce_max(s.elapsed_time(e) / steps, dist)
    world = dist.get_world_size() if dist is not None else 1
    fwd_b, _ = step_bytes(wl)
    h2d = sum(v.numel() * v.element_size() for v in pin.values())
    d2h = host_out.numel() * host_out.element_size() + \
        (host_h.numel() * host_h.element_size() if host_h is not None else 0)
    return {"value": round(whole_job_gbs(fwd_b, world, ms), 1), "unit": "GB/s",
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "ms_per_step": round(ms, 5), "steps": steps,
            "pipeline": "one stream: copy x, r in; fused call; copy out, h back "
                        "(weights resident)"}


def run_e2e(rn, wl, src, dev, ws, args, dist):
    """The same metric through the C ABI with pinned host inputs and outputs:
    every step copies its inputs host->device (x, dy, w and, for the
    residual variant, r and dh) and every result back (y, rstd, dx, dw, and
    h), inside the timed region. The rows go through in chunks on three
    streams — copies in, forward + backward, copies out — so the two link
    directions and the kernels overlap; dw accumulates over the chunks
    (rmsnorm_bwd_ex). Two device buffer sets alternate between steps, with
    events keeping a set's buffers from being overwritten while in use."""
    M, H = wl.M, wl.H
    chunks = max(1, min(8, M // 1024))
    bounds = [M * c // chunks for c in range(chunks + 1)]
    pin = {k: v.pin_memory() for k, v in src.items()}
    in_keys = ["x", "w"] + (["dy"] if wl.backward else []) + \
        (["r", "dh"] if wl.residual else [])
    out_keys = ["y", "rstd"] + (["dx", "dw"] if wl.backward else []) + \
        (["h"] if wl.residual else [])
    shapes = {"w": (H,), "rstd": (M,), "dw": (H,)}
    dtypes = {"rstd": torch.float32, "dw": torch.float32}

    def dev_set():
        d = {k: torch.empty(shapes.get(k, (M, H)), device=dev,
                            dtype=dtypes.get(k, wl.dtype))
             for k in set(in_keys) | set(out_keys)}
        if wl.ld:        # row tensors as column windows of [M, ld] buffers
            d = {k: (W.in_strided(v, wl.ld, 0.0) if k not in shapes else v)
                 for k, v in d.items()}
        return d
    sets = [dev_set(), dev_set()]
    host_out = {k: torch.empty(shapes.get(k, (M, H)), dtype=dtypes.get(k, wl.dtype),
                               pin_memory=True) for k in out_keys}
    s_in, s_c, s_out = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
    ev = lambda: torch.cuda.Event()  # noqa: E731
    ev_in = [[ev() for _ in range(chunks)] for _ in sets]
    ev_c = [[ev() for _ in range(chunks)] for _ in sets]
    ev_out = [[ev() for _ in range(chunks)] for _ in sets]
    used = [False, False]


    def step(i):
        si = i % 2
        d = sets[si]
        for c in range(chunks):
            a, b = bounds[c], bounds[c + 1]
            with torch.cuda.stream(s_in):
                if c == 0 and used[si]:
                    # the previous step on this set has finished computing
                    s_in.wait_event(ev_c[si][chunks - 1])
                for k in in_keys:
                    if k == "w":
                        if c == 0:
                            d["w"].copy_(pin["w"], non_blocking=True)
                        continue
                    d[k][a:b].copy_(pin[k][a:b], non_blocking=True)
                ev_in[si][c].record(s_in)
            with torch.cuda.stream(s_c):
                s_c.wait_event(ev_in[si][c])
                if c == 0 and used[si]:
                    # ... and its results have been copied out
                    s_c.wait_event(ev_out[si][chunks - 1])
                if wl.ld:
                    rn.rmsnorm_fwd_strided(
                        d["x"][a:b], d["w"], y=d["y"][a:b],
                        r=d["r"][a:b] if wl.residual else None,
                        h=d["h"][a:b] if wl.residual else None,
                        rstd=d["rstd"][a:b], eps=wl.eps, stream=s_c)
                elif wl.residual:
                    rn.rmsnorm_residual_fwd(d["x"][a:b], d["r"][a:b], d["w"],
                                            h=d["h"][a:b], y=d["y"][a:b],
                                            rstd=d["rstd"][a:b], eps=wl.eps, stream=s_c)
                else:
                    rn.rmsnorm_fwd(d["x"][a:b], d["w"], y=d["y"][a:b],
                                   rstd=d["rstd"][a:b], eps=wl.eps, stream=s_c)
                if wl.backward:
                    xin = d["h"] if wl.residual else d["x"]
                    bwd = rn.rmsnorm_bwd_strided if wl.ld else rn.rmsnorm_bwd_ex
                    bwd(d["dy"][a:b], xin[a:b], d["w"], d["rstd"][a:b],
                        dh_out=d["dh"][a:b] if wl.residual else None,
                        dx=d["dx"][a:b], dw=d["dw"], workspace=ws,
                        eps=wl.eps, accumulate_dw=c > 0, stream=s_c)
                ev_c[si][c].record(s_c)
            with torch.cuda.stream(s_out):
                s_out.wait_event(ev_c[si][c])
                for k in out_keys:
                    if k == "dw":
                        continue
                    host_out[k][a:b].copy_(d[k][a:b], non_blocking=True)
                if c == chunks - 1 and "dw" in out_keys:
                    host_out["dw"].copy_(d["dw"], non_blocking=True)
                ev_out[si][c].record(s_out)
        used[si] = True

    h2d = sum(pin[k].numel() * pin[k].element_size() for k in in_keys)
    d2h = sum(v.numel() * v.element_size() for v in host_out.values())
    main = torch.cuda.current_stream()
    steps = max(1, min(args.steps, 200))
    for i in range(max(2, min(args.warmup, 5))):
        step(i)
    torch.cuda.synchronize()
    if dist is not None:
        dist.barrier()
    s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    s.record(main)
    for st in (s_in, s_c, s_out):
        st.wait_event(s)
    for i in range(steps):
        step(i)
    for st in (s_in, s_c, s_out):
        main.wait_stream(st)
    e.record(main)
    torch.cuda.synchronize()
    ms = reduce_max(s.elapsed_time(e) / steps, dist)
    world = dist.get_world_size() if dist is not None else 1
    fwd_b, bwd_b = step_bytes(wl)
    return {"value": round(whole_job_gbs(fwd_b + bwd_b, world, ms), 1),
            "unit": "GB/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "ms_per_step": round(ms, 4), "steps": steps,
            "rows_per_s": round(wl.M * world / (ms * 1e-3), 1),
            "pipeline": f"{chunks} row chunks on 3 streams (copy in / compute / copy out)"}


# The sources a workload's kernels are built from, their dispatch in api.cu
# included: the streamed and row-wise norm kernels and dw_reduce for the
# training shapes; plus the split-row forward for decode-sized batches (at
# most 64 rows), the double backward, or the projection kernels.
_NORM_SOURCES = ("api.cu", "common.cuh", "context.h", "params.h", "registry.h", "reduce.cuh",
                 "rows.cuh", "rows_bf16_generic.cu", "rows_bf16_shaped.cu",
                 "rows_f16_generic.cu", "rows_f16_shaped.cu", "rows_f32.cu", "stream.cuh",
                 "stream_small.cuh", "stream.cu", "stream_f16.cu")
KERNEL_SOURCES = {
    "norm": _NORM_SOURCES,
    "decode": _NORM_SOURCES + ("split.cuh", "split.cu"),
    "bwd2": _NORM_SOURCES + ("bwd2.cuh", "bwd2.cu"),
    "gemv": _NORM_SOURCES + ("split.cuh", "gemv.cuh", "gemv.cu", "gemv_tma.cuh",
                             "gemv_umma.cuh", "gemv_umma.cu", "gemv_tc.cuh", "gemv_tc.cu"),
}


def source_set(wl):
    if wl.N:
        return "gemv"
    if wl.double_backward:
        return "bwd2"
    return "decode" if wl.M <= 64 else "norm"


def kernel_src_hash(wl):
    """Hash of the sources the workload's kernels are built from (the
    kernels, their headers and the dispatch that picks them): the DRAM
    traffic recorded for it in profiles/traffic.json holds only while they
    are unchanged."""
    import hashlib
    h = hashlib.sha256()
    d = os.path.join(ROOT, "rmsnorm_fwd_bwd_02_gb300", "csrc")
    for f in sorted(KERNEL_SOURCES[source_set(wl)]):
        h.update(f.encode())
        with open(os.path.join(d, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def load_traffic(wl, which):
    """DRAM bytes per launch of the dominant call, from the committed ncu
    summary, when one exists for this workload and the kernels' sources are
    unchanged since it was taken; else None."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(p) as f:
            d = json.load(f)
        e = d.get(wl.name, {}).get(which)
        if not e or e.get("src") != kernel_src_hash(wl):
            return None
        return int(e["bytes"])
    except (OSError, ValueError, KeyError):
        return None


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(W.WORKLOADS))
    ap.add_argument("--rows", type=int, default=0,
                    help="run the workload with this many rows (profiling a "
                         "smaller case); the default is the workload's own M")
    ap.add_argument("--path-override", type=int, default=0,
                    help="profiling aid: force a kernel family through the "
                         "library's path override (rmsnorm_set_path_override; "
                         "e.g. 1 the register-fed projection, 7 the tcgen05 "
                         "one); the line then records it under config")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-workloads", action="store_true",
                    help="skip the other workloads' figures (the 'workloads' key "
                         "of the default run)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    wl = W.WORKLOADS[args.workload]
    if args.rows:
        wl = wl.with_rows(args.rows)
    if args.impl == "reference":
        return run_reference(args, wl)
    return run_ours(args, wl)


if __name__ == "__main__":
    sys.exit(main())
