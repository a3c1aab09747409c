"""Benchmark: fused residual add + RMSNorm throughput (GB/s) and fraction of
the HBM roofline on GB300, plus the other operations of the path.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--no-ops] [--workload prefill|...]

One step = the fused add+RMSNorm forward, in place, over the LLM-prefill
batch at rows = 16384 for each hidden size in {4096, 5120, 8192} (three
launches, one per size; every launch's working set is 0.5-1.1 GB, far above
the 129 MB L2, so no flush is needed between steps).  Algorithmic bytes per
launch = 8 * hidden * rows + 2 * hidden (read x and residual, write both,
read the weight once); `value` = those bytes over the timed steps divided by
the device time (CUDA events on the launching stream, max over ranks).

The JSON line also carries: `roofline` for the dominant launch (hidden 8192)
against the measured HBM copy bandwidth; `e2e` through the C ABI with
pinned host buffers (host->device copy of x and residual, the call, and the
device->host copy of both results, every step); `cpu_baseline` (the fp64
oracle on the host cores, a bounded sample); `clocks` sampled with
nvidia-smi during the timed region; and `ops`, per-operation GB/s and
roofline fractions for every fused size, RMSNorm forward, LayerNorm forward /
backward and the small-batch sweep (launches captured back to back in a CUDA
graph over enough input sets that each replay touches twice the L2 size).

`--impl reference` times the oracle instead (the reference arm of this
path), on a bounded sample of the same workload.

Multi-GPU: the path has no exchange step, so N ranks run N replicas (weak
scaling) and `value` sums the bytes of all ranks over the slowest rank's time.
"""
from __future__ import annotations

import argparse
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

import torch  # noqa: E402

import workloads  # noqa: E402

METRIC = "fused add+RMSNorm GB/s and % of HBM roofline (bf16, hidden 4096–8192)"
UNIT = "GB/s"
ROWS = 16384
HIDDENS = (4096, 5120, 8192)
EPS = 1e-5
DOMINANT_HIDDEN = 8192
FALLBACK_HBM_GBS = 6800.0
E2E_CHUNKS = 2
E2E_ROUNDS = 9      # end-to-end timing rounds (pipeline, then bare link, each round)


# ---------------------------------------------------------------- byte accounting

def fused_bytes(rows, hidden):
    return 8 * hidden * rows + 2 * hidden


def rms_bytes(rows, hidden):
    return 4 * hidden * rows + 2 * hidden


def ln_fwd_bytes(rows, hidden):
    return (4 * hidden + 8) * rows + 4 * hidden


def ln_bwd_bytes(rows, hidden):
    return (6 * hidden + 8) * rows + 10 * hidden


def rms_bwd_bytes(rows, hidden):
    # read x, dy; write dx; read w once; write dw (fp32) once
    return 6 * hidden * rows + 6 * hidden


def fused_bwd_bytes(rows, hidden):
    # read s, dy, dres; write dx; read w once; write dw (fp32) once
    return 8 * hidden * rows + 6 * hidden


def outer_fwd_bytes(rows, hidden):
    # read x once, write y; gamma, beta in; mean, rstd (fp32) out
    return 4 * hidden * rows + 12 * hidden


def outer_bwd_bytes(rows, hidden):
    # read x, dy once, write dx; mean, rstd, gamma in; dgamma, dbeta out
    return 6 * hidden * rows + 26 * hidden


# ---------------------------------------------------------------- environment helpers

def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def max_over_ranks(ms, dist, device):
    """The slowest rank's time (every rank gets it); `dist` None = one rank."""
    if dist is None:
        return ms
    t = torch.tensor([ms], device=device, dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_gbs(world, step_bytes, steps, ms):
    """Whole-job throughput: the bytes every rank moved over the slowest
    rank's time (weak scaling: each rank runs its own replica)."""
    return world * step_bytes * steps / (ms * 1e-3) / 1e9


def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


class ClockSampler:
    """nvidia-smi clocks and throttle reasons, sampled while running."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []
        self._t = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return self
        self._t = threading.Thread(target=self._read, daemon=True)
        self._t.start()
        t0 = time.time()
        while not self.lines and time.time() - t0 < 5:
            time.sleep(0.02)
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def mark(self):
        return time.time()

    def stop(self, t_begin, t_end):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        rows = [l for (t, l) in self.lines if t_begin - 0.15 <= t <= t_end + 0.15] or \
            [l for (_, l) in self.lines[-3:]]
        sm, smax, reasons, power = [], [], set(), []
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for l in rows:
            parts = [p.strip() for p in l.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
                power.append(float(parts[3]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "power_w_max": max(power) if power else None,
                "samples": len(sm),
                "reasons": sorted(reasons)}


# ---------------------------------------------------------------- the oracle arm

def host_cores():
    """Cores this process may run on (its affinity mask)."""
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:  # pragma: no cover
        return os.cpu_count() or 1


def oracle_sample(budget_s: float, rows_per_hidden: int = 1024, threads: int = 1):
    """Time the fp64 oracle on a bounded sample of the workload: the first
    `rows_per_hidden` rows of each hidden size, repeated until `budget_s`
    seconds have passed.  With threads > 1 the rows are cut into `threads`
    contiguous slices and each host thread runs the unchanged oracle
    functions on its own slices (ctypes releases the interpreter lock while
    the C code runs).  Returns (GB/s under the same byte accounting,
    description, threads, seconds, passes)."""
    import concurrent.futures as cf
    import oracle
    oracle.build()
    inputs = [workloads.fused_inputs(rows_per_hidden, h, residual_scale=4.0) for h in HIDDENS]
    cuts = [rows_per_hidden * k // threads for k in range(threads + 1)]
    slices = [[(x[cuts[k]:cuts[k + 1]], r[cuts[k]:cuts[k + 1]], w) for (x, r, w) in inputs]
              for k in range(threads)]

    def work(part):
        for (x, r, w) in part:
            if x.shape[0] == 0:
                continue
            s, y, _ = oracle.fused_add_rmsnorm(x, r, w, EPS)
            oracle.to_bf16(s)
            oracle.to_bf16(y)

    pass_bytes = sum(fused_bytes(rows_per_hidden, h) for h in HIDDENS)
    nbytes = 0
    reps = 0
    with cf.ThreadPoolExecutor(max_workers=threads) as ex:
        t0 = time.perf_counter()
        while True:
            list(ex.map(work, slices))
            nbytes += pass_bytes
            reps += 1
            el = time.perf_counter() - t0
            if el >= budget_s:
                break
    gbs = nbytes / el / 1e9
    kind = "single thread" if threads == 1 else f"{threads} host threads (row slices)"
    desc = (f"fp64 C oracle, {kind}, {reps} pass(es) over the first {rows_per_hidden} rows "
            f"of each hidden in {list(HIDDENS)} ({el:.1f} s)")
    return gbs, desc, threads, el, reps


def run_reference(args):
    world, rank, local = dist_env()
    if rank != 0:
        return 0
    steps, warmup = args.steps, max(args.warmup, 0)
    import oracle
    oracle.build()
    # size the per-step sample so that all steps take about --ref-seconds
    probe = [workloads.fused_inputs(64, h, residual_scale=4.0) for h in HIDDENS]
    t0 = time.perf_counter()
    for (x, r, w) in probe:
        s, y, _ = oracle.fused_add_rmsnorm(x, r, w, EPS)
        oracle.to_bf16(s)
        oracle.to_bf16(y)
    per_row = (time.perf_counter() - t0) / 64
    rows_s = int(max(1, min(1024, args.ref_seconds / (max(steps + warmup, 1) * per_row))))
    inputs = [workloads.fused_inputs(rows_s, h, residual_scale=4.0) for h in HIDDENS]

    def step():
        for (x, r, w) in inputs:
            s, y, _ = oracle.fused_add_rmsnorm(x, r, w, EPS)
            oracle.to_bf16(s)
            oracle.to_bf16(y)
    for _ in range(warmup):
        step()
    t0 = time.perf_counter()
    for _ in range(steps):
        step()
    el = time.perf_counter() - t0
    nbytes = steps * sum(fused_bytes(rows_s, h) for h in HIDDENS)
    v = nbytes / el / 1e9
    line = {
        "impl": "reference", "metric": METRIC, "value": round(v, 4), "unit": UNIT,
        "n_gpus": 1, "steps": steps, "warmup": warmup,
        "ms_per_step": round(el / steps * 1e3, 3), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded, torch CPU generator)",
        "config": {"workload": f"fused add+RMSNorm LLM prefill, bounded sample: first {rows_s} rows "
                               f"of each hidden in {list(HIDDENS)} (full batch is {ROWS} rows)",
                   "rows_sampled": rows_s, "hidden": list(HIDDENS), "eps": EPS},
        "cpu_baseline": {"value": round(v, 4), "unit": UNIT, "cores": 1, "kind": "oracle",
                         "sample": f"first {rows_s} rows of each hidden, {steps} steps"},
        "e2e": {"value": round(v, 4), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# ---------------------------------------------------------------- GPU arm

def _ev():
    return torch.cuda.Event(enable_timing=True)


def graph_time_ms(launch, n, stream, replays=5):
    """Mean device time per launch: `n` launches captured back to back in
    one CUDA graph (launch(i, stream_handle) enqueues launch i), the graph
    replayed `replays` times between CUDA events; median of the replays.
    Timing many launches at once keeps the event timer's granularity (4 us
    on the GB300 machines) and host launch latency out of the result."""
    sh = stream.cuda_stream
    launch(0, sh)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        for i in range(n):
            launch(i, sh)
    ts = []
    with torch.cuda.stream(stream):
        g.replay()
        stream.synchronize()
        for _ in range(replays):
            a, b = _ev(), _ev()
            a.record(stream)
            g.replay()
            b.record(stream)
            b.synchronize()
            ts.append(a.elapsed_time(b) / n)
    del g
    return statistics.median(ts)


def op_case(nf, op, rows, hidden, eps, l2_bytes, dev="cuda"):
    """Inputs for timing `op` at (rows, hidden) on L2-cold data: enough
    independent input sets that the launches of one graph replay touch at
    least twice the L2 size.  Returns (launch(i, stream), sets, bytes)."""
    lib = nf.lib()
    if op == "fused_add_rmsnorm":
        foot, nbytes = 4 * hidden * rows, fused_bytes(rows, hidden)
    elif op == "rmsnorm_fwd":
        foot, nbytes = 4 * hidden * rows, rms_bytes(rows, hidden)
    elif op == "layernorm_fwd":
        foot, nbytes = (4 * hidden + 8) * rows, ln_fwd_bytes(rows, hidden)
    elif op == "rmsnorm_bwd":
        foot, nbytes = 6 * hidden * rows, rms_bwd_bytes(rows, hidden)
    elif op == "fused_add_rmsnorm_bwd":
        foot, nbytes = 8 * hidden * rows, fused_bwd_bytes(rows, hidden)
    elif op == "outer_norm_fwd":
        foot, nbytes = 4 * hidden * rows, outer_fwd_bytes(rows, hidden)
    elif op == "outer_norm_bwd":
        foot, nbytes = 6 * hidden * rows, outer_bwd_bytes(rows, hidden)
    elif op == "floor_copy":
        # a plain copy of the fused op's activation bytes at (rows, hidden)
        foot, nbytes = 8 * hidden * rows, 8 * hidden * rows
    elif op == "floor_empty":
        foot, nbytes = 1 << 30, 0
    else:
        foot, nbytes = (6 * hidden + 8) * rows, ln_bwd_bytes(rows, hidden)
    sets = max(1, min(16384, -(-2 * l2_bytes // foot)))
    tot = sets * rows
    a2 = rows * hidden * 2  # bytes per set of one bf16 activation
    # forward calls take a workspace only on the split family (rows longer
    # than a cluster holds); sized for every family by the library
    fwd_ws = None
    if op in ("fused_add_rmsnorm", "rmsnorm_fwd", "layernorm_fwd"):
        fwd_ws = torch.empty(max(nf.nf_workspace_size(nf.OPS[op], rows, hidden), 16),
                             dtype=torch.uint8, device=dev)
        fwp, fwn = fwd_ws.data_ptr(), fwd_ws.numel()
    if op == "floor_empty":
        keep = ()
        fn = lambda i, sh: lib.nf_selftest_floor(0, None, None, 0, sh)  # noqa: E731
    elif op == "floor_copy":
        cb = 4 * hidden * rows  # bytes read (= bytes written) per launch
        src = torch.empty(sets * cb, dtype=torch.uint8, device=dev)
        dst = torch.empty_like(src)
        ps, pd = src.data_ptr(), dst.data_ptr()
        keep = (src, dst)
        fn = lambda i, sh: lib.nf_selftest_floor(1, pd + (i % sets) * cb, ps + (i % sets) * cb,  # noqa: E731
                                                  cb, sh)
    elif op == "fused_add_rmsnorm":
        x, r, w = workloads.fused_inputs(tot, hidden, residual_scale=4.0, device=dev)
        px, pr, pw = x.data_ptr(), r.data_ptr(), w.data_ptr()
        keep = (x, r, w)
        fn = lambda i, sh: lib.nf_fused_add_rmsnorm_ws(px + (i % sets) * a2, pr + (i % sets) * a2, pw,  # noqa: E731
                                                        rows, hidden, eps, fwp, fwn, sh)
    elif op == "rmsnorm_fwd":
        x, w = workloads.rms_inputs(tot, hidden, device=dev)
        y = torch.empty_like(x)
        px, py, pw = x.data_ptr(), y.data_ptr(), w.data_ptr()
        keep = (x, y, w)
        fn = lambda i, sh: lib.nf_rmsnorm_fwd_ws(py + (i % sets) * a2, px + (i % sets) * a2, pw,  # noqa: E731
                                                  rows, hidden, eps, fwp, fwn, sh)
    elif op == "layernorm_fwd":
        x, g, b = workloads.layernorm_fwd_inputs(tot, hidden, device=dev)
        y = torch.empty_like(x)
        m = torch.empty(tot, device=dev)
        rs = torch.empty(tot, device=dev)
        px, py, pg, pb, pm, pr = (t.data_ptr() for t in (x, y, g, b, m, rs))
        keep = (x, y, g, b, m, rs)
        fn = lambda i, sh: lib.nf_layernorm_fwd_ws(py + (i % sets) * a2, pm + (i % sets) * rows * 4,  # noqa: E731
                                                    pr + (i % sets) * rows * 4, px + (i % sets) * a2,
                                                    pg, pb, rows, hidden, eps, fwp, fwn, sh)
    elif op == "rmsnorm_bwd":
        x, dy, w = workloads.rms_bwd_inputs(tot, hidden, device=dev)
        dx = torch.empty_like(x)
        nws = max(nf.nf_rmsnorm_bwd_workspace_size(rows, hidden), 16)
        ws = torch.empty(nws, dtype=torch.uint8, device=dev)
        dw = torch.empty(hidden, device=dev)
        px, pdy, pw, pdx, pws, pdw = (t.data_ptr() for t in (x, dy, w, dx, ws, dw))
        keep = (x, dy, w, dx, ws, dw)
        fn = lambda i, sh: lib.nf_rmsnorm_bwd(pdx + (i % sets) * a2, pdw, pdy + (i % sets) * a2,  # noqa: E731
                                               px + (i % sets) * a2, pw, rows, hidden, eps, pws, nws, sh)
    elif op == "fused_add_rmsnorm_bwd":
        sres, w, dy, dres = workloads.fused_bwd_inputs(tot, hidden, device=dev)
        dx = torch.empty_like(sres)
        nws = max(nf.nf_rmsnorm_bwd_workspace_size(rows, hidden), 16)
        ws = torch.empty(nws, dtype=torch.uint8, device=dev)
        dw = torch.empty(hidden, device=dev)
        ps, pw, pdy, pdr, pdx, pws, pdw = (t.data_ptr() for t in (sres, w, dy, dres, dx, ws, dw))
        keep = (sres, w, dy, dres, dx, ws, dw)
        fn = lambda i, sh: lib.nf_fused_add_rmsnorm_bwd(  # noqa: E731
            pdx + (i % sets) * a2, pdw, pdy + (i % sets) * a2, pdr + (i % sets) * a2,
            ps + (i % sets) * a2, pw, rows, hidden, eps, pws, nws, sh)
    elif op == "outer_norm_fwd":
        # one [rows, hidden] problem per set; per-column statistics are per set
        x, _, g, b = workloads.outer_inputs(tot, hidden, device=dev)
        y = torch.empty_like(x)
        m = torch.empty(hidden, device=dev)
        rs = torch.empty(hidden, device=dev)
        nws = max(nf.nf_outer_norm_workspace_size(rows, hidden), 16)
        ws = torch.empty(nws, dtype=torch.uint8, device=dev)
        px, py, pg, pb, pm, pr, pws = (t.data_ptr() for t in (x, y, g, b, m, rs, ws))
        keep = (x, y, g, b, m, rs, ws)
        fn = lambda i, sh: lib.nf_outer_norm_fwd(py + (i % sets) * a2, pm, pr, px + (i % sets) * a2,  # noqa: E731
                                                  pg, pb, rows, hidden, eps, pws, nws, sh)
    elif op == "outer_norm_bwd":
        x, dy, g, b = workloads.outer_inputs(tot, hidden, device=dev)
        _, m, rs = nf.outer_norm_fwd(x[:rows], g, b, eps)
        dx = torch.empty_like(x)
        nws = max(nf.nf_outer_norm_workspace_size(rows, hidden), 16)
        ws = torch.empty(nws, dtype=torch.uint8, device=dev)
        dg = torch.empty(hidden, device=dev)
        db = torch.empty(hidden, device=dev)
        px, pdy, pg, pm, pr, pdx, pws, pdg, pdb = (t.data_ptr() for t in (x, dy, g, m, rs, dx, ws, dg, db))
        keep = (x, dy, g, m, rs, dx, ws, dg, db)
        fn = lambda i, sh: lib.nf_outer_norm_bwd(pdx + (i % sets) * a2, pdg, pdb, pdy + (i % sets) * a2,  # noqa: E731
                                                  px + (i % sets) * a2, pm, pr, pg, rows, hidden, pws,
                                                  nws, sh)
    else:
        x, dy, g = workloads.layernorm_bwd_inputs(tot, hidden, device=dev)
        _, m, rs = nf.layernorm_fwd(x, g, torch.zeros_like(g), eps)
        dx = torch.empty_like(x)
        nws = max(nf.nf_layernorm_bwd_workspace_size(rows, hidden), 16)
        ws = torch.empty(nws, dtype=torch.uint8, device=dev)
        dg = torch.empty(hidden, device=dev)
        db = torch.empty(hidden, device=dev)
        px, pdy, pg, pm, pr, pdx, pws, pdg, pdb = (t.data_ptr() for t in (x, dy, g, m, rs, dx, ws, dg, db))
        keep = (x, dy, g, m, rs, dx, ws, dg, db)
        fn = lambda i, sh: lib.nf_layernorm_bwd(pdx + (i % sets) * a2, pdg, pdb, pdy + (i % sets) * a2,  # noqa: E731
                                                 px + (i % sets) * a2, pm + (i % sets) * rows * 4,
                                                 pr + (i % sets) * rows * 4, pg, rows, hidden, pws, nws, sh)

    keep = keep + (fwd_ws,)

    def launch(i, sh, _keep=keep):
        st = fn(i, sh)
        if st != 0:
            raise RuntimeError(f"{op} {rows}x{hidden}: status {st}")
    return launch, sets, nbytes


def time_op(nf, op, rows, hidden, eps, l2_bytes, stream, min_launches=20, path=None):
    """Graph-timed device time of `op` at (rows, hidden); with `path` the
    kernel family is forced while the launches are captured (the inputs are
    prepared under the automatic choice)."""
    launch, sets, nbytes = op_case(nf, op, rows, hidden, eps, l2_bytes)
    n = max(sets, min_launches)
    if path is None:
        ms = graph_time_ms(launch, n, stream)
    else:
        with nf.forced_path(path):
            ms = graph_time_ms(launch, n, stream)
    del launch
    torch.cuda.empty_cache()
    return ms, nbytes


def ops_suite(nf, peak, stream, l2_bytes):
    """Per-operation device time at every workload size: launches captured
    back to back in a CUDA graph over L2-cold input sets (section 9 of the
    design notes).  Keys are "op ROWSxHIDDEN", with " [path]" when a kernel
    family is forced instead of the library's own choice."""
    out = {}

    def entry(op, rows, h, eps, path=None):
        ms, nbytes = time_op(nf, op, rows, h, eps, l2_bytes, stream, path=path)
        gbs = nbytes / (ms * 1e-3) / 1e9
        if op.startswith("floor"):
            used = "probe"
        elif op.startswith("outer"):
            used = "outer"
        elif path is not None:
            used = path
        else:
            plan_op = "rmsnorm_bwd" if op == "fused_add_rmsnorm_bwd" else op
            used = nf.nf_plan_query(plan_op, rows, h)["path"]
        key = f"{op} {rows}x{h}" + (f" [{path}]" if path else "")
        out[key] = {"gbs": round(gbs, 1), "frac": round(gbs / peak, 4), "us": round(ms * 1e3, 3),
                    "path": used}

    # the launch floor beside the small-batch rows: an empty dependent launch
    # and a plain copy of the fused op's activation bytes, same harness
    entry("floor_empty", 1, 8, 0.0)
    for h in (4096, 8192):
        for rows in (1, 8, 128):
            entry("floor_copy", rows, h, 0.0)
    for h in (4096, 8192):
        for rows in (1, 2, 4, 8, 16, 32, 128):
            entry("fused_add_rmsnorm", rows, h, 1e-6)
        # both families on the small-batch sweep (the automatic choice
        # follows these numbers)
        for rows in (1, 2, 4, 8, 32, 128):
            entry("fused_add_rmsnorm", rows, h, 1e-6, path="reg")
            entry("fused_add_rmsnorm", rows, h, 1e-6, path="cluster")
    for rows in (4096, 16384, 65536):
        for h in (2048, 4096, 5120, 8192):
            entry("fused_add_rmsnorm", rows, h, EPS)
    for h in (4096, 8192):
        entry("rmsnorm_fwd", ROWS, h, EPS)
    for h in (1024, 4096, 12288):
        entry("layernorm_fwd", ROWS, h, EPS)
    for h in (1024, 2048, 4096, 8192):
        entry("layernorm_bwd", ROWS, h, EPS)
    for h in (1024, 2048, 4096, 8192):
        entry("rmsnorm_bwd", ROWS, h, EPS)
    for h in (1024, 2048, 4096, 5120, 8192, 12288):
        entry("fused_add_rmsnorm_bwd", ROWS, h, EPS)
    for rows, h in ((16384, 1024), (16384, 4096), (65536, 1024), (4096, 8192)):
        entry("outer_norm_fwd", rows, h, EPS)
        entry("outer_norm_bwd", rows, h, EPS)
    # rows longer than a cluster holds: the automatic choice (the grid
    # family where the rows fit on chip, the split family for the RMSNorm
    # backward), and the other of the two forced
    for op in ("rmsnorm_fwd", "layernorm_fwd", "fused_add_rmsnorm", "layernorm_bwd", "rmsnorm_bwd",
               "fused_add_rmsnorm_bwd"):
        entry(op, 4, 1 << 22, EPS)
        plan_op = "rmsnorm_bwd" if op == "fused_add_rmsnorm_bwd" else op
        auto = nf.nf_plan_query(plan_op, 4, 1 << 22)["path"]
        entry(op, 4, 1 << 22, EPS, path="split" if auto == "grid" else "grid")
    # hidden sizes with no compiled kernel: the runtime-hidden family
    for h in (3072, 6144):
        for op in ("fused_add_rmsnorm", "layernorm_fwd", "layernorm_bwd", "rmsnorm_bwd"):
            entry(op, ROWS, h, EPS)
    return out


def run_gpu(args):
    import row_normalization_inner_gb300 as nf
    from row_normalization_inner_gb300 import build as nf_build

    world, rank, local = dist_env()
    torch.cuda.set_device(local)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    nf_build.build()
    nf.lib()

    peak, peak_kind = measured_peaks()
    stream = torch.cuda.Stream()
    dev = "cuda"

    # inputs resident in HBM: one (x, residual, weight) set per hidden size
    sets = [workloads.fused_inputs(ROWS, h, seed=rank, residual_scale=4.0, device=dev) for h in HIDDENS]
    step_bytes = sum(fused_bytes(ROWS, h) for h in HIDDENS)
    dom = HIDDENS.index(DOMINANT_HIDDEN)
    torch.cuda.synchronize()

    def step(evs=None):
        for i, ((x, r, w), h) in enumerate(zip(sets, HIDDENS)):
            if evs is not None and i == dom:
                evs[0].record(stream)
            nf.fused_add_rmsnorm(x, r, w, EPS, stream=stream)
            if evs is not None and i == dom:
                evs[1].record(stream)

    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            step()
    torch.cuda.synchronize()

    sampler = ClockSampler(local).start() if rank == 0 else None
    dom_events = [(_ev(), _ev()) for _ in range(args.steps)]
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    t_begin = time.time()
    start, end = _ev(), _ev()
    start.record(stream)
    for k in range(args.steps):
        step(dom_events[k])
    end.record(stream)
    end.synchronize()
    torch.cuda.synchronize()
    t_end = time.time()
    if dist is not None:
        dist.barrier()
    ms_total = start.elapsed_time(end)
    dom_ms = [a.elapsed_time(b) for a, b in dom_events]
    ms_total = max_over_ranks(ms_total, dist, dev)
    clocks = sampler.stop(t_begin, t_end) if sampler else None

    value = whole_job_gbs(world, step_bytes, args.steps, ms_total)
    dom_avg_ms = sum(dom_ms) / len(dom_ms)
    dom_bytes = fused_bytes(ROWS, DOMINANT_HIDDEN)
    achieved = dom_bytes / (dom_avg_ms * 1e-3) / 1e9
    dom_path = nf.nf_plan_query("fused_add_rmsnorm", ROWS, DOMINANT_HIDDEN)["path"]
    traffic = _profiled_traffic("fused_add_rmsnorm", dom_path, ROWS, DOMINANT_HIDDEN)

    # end to end through the C ABI with pinned host buffers: every step copies
    # x and residual in from pinned host memory, runs the call and copies both
    # results back.  Rows are independent, so each hidden size's batch is cut
    # into E2E_CHUNKS row chunks, and three streams take one role each:
    # host->device copies, kernels, device->host copies, chained per chunk by
    # events.  A chunk's next host->device copy waits for its previous
    # device->host copy, so a buffer is never overwritten while it is read.
    e2e = None
    if not args.no_e2e:
        hosts = [(x.cpu().pin_memory(), r.cpu().pin_memory()) for (x, r, _) in sets]
        outs = [(torch.empty_like(hx).pin_memory(), torch.empty_like(hr).pin_memory()) for hx, hr in hosts]
        h2d = sum(hx.numel() * 2 + hr.numel() * 2 for hx, hr in hosts)
        d2h = h2d
        streams = [torch.cuda.Stream() for _ in range(3)]
        s_in, s_k, s_out = streams
        work = []
        cr = ROWS // E2E_CHUNKS
        for (hx, hr), (ox, orr), (x, r, w) in zip(hosts, outs, sets):
            for c in range(E2E_CHUNKS):
                sl = slice(c * cr, (c + 1) * cr)
                work.append((hx[sl], hr[sl], ox[sl], orr[sl], x[sl], r[sl], w))
        ev_in = [torch.cuda.Event() for _ in work]
        ev_k = [torch.cuda.Event() for _ in work]
        ev_out = [torch.cuda.Event() for _ in work]

        def e2e_step():
            for k, (hx, hr, ox, orr, x, r, w) in enumerate(work):
                with torch.cuda.stream(s_in):
                    s_in.wait_event(ev_out[k])
                    x.copy_(hx, non_blocking=True)
                    r.copy_(hr, non_blocking=True)
                    ev_in[k].record(s_in)
                s_k.wait_event(ev_in[k])
                nf.fused_add_rmsnorm(x, r, w, EPS, stream=s_k)
                ev_k[k].record(s_k)
                with torch.cuda.stream(s_out):
                    s_out.wait_event(ev_k[k])
                    ox.copy_(x, non_blocking=True)
                    orr.copy_(r, non_blocking=True)
                    ev_out[k].record(s_out)

        # the host link's capacity for the same bytes: every host->device copy
        # on one stream while every device->host copy runs on another (from a
        # separate device buffer), no kernel and no dependency between them
        link_src = torch.empty(max(t.numel() for t in (w_[2] for w_ in work)), dtype=torch.bfloat16,
                               device=dev)

        def link_step():
            with torch.cuda.stream(streams[0]):
                for (hx, hr, ox, orr, x, r, w) in work:
                    x.copy_(hx, non_blocking=True)
                    r.copy_(hr, non_blocking=True)
            with torch.cuda.stream(streams[1]):
                for (hx, hr, ox, orr, x, r, w) in work:
                    ox.copy_(link_src[:ox.numel()].view_as(ox), non_blocking=True)
                    orr.copy_(link_src[:orr.numel()].view_as(orr), non_blocking=True)

        def timed(nsteps, step=e2e_step):
            a, b = _ev(), _ev()
            a.record(stream)
            for s in streams:
                s.wait_event(a)
            for _ in range(nsteps):
                step()
            for s in streams:
                ev = _ev()
                ev.record(s)
                stream.wait_event(ev)
            b.record(stream)
            b.synchronize()
            return a.elapsed_time(b)

        # nine rounds, each timing the pipeline and then the bare link on the
        # same bytes; the median round of each is reported (the host link is
        # shared with the rest of the machine: in one run three of five
        # pipeline rounds and one of five link rounds fell from about 335 to
        # about 250 GB/s)
        e2e_steps = max(3, min(args.steps // 40, 25))
        timed(1)
        torch.cuda.synchronize()
        if dist is not None:
            dist.barrier()
        e_round, c_round = [], []
        for r in range(E2E_ROUNDS):
            e_round.append(max_over_ranks(timed(e2e_steps), dist, dev))
            if r == 0:
                # check once that the round trip really returned the device
                # results (before the link timing overwrites both ends)
                torch.cuda.synchronize()
                assert torch.equal(outs[-1][0][-1], sets[-1][0][-1].cpu())
            c_round.append(max_over_ranks(timed(e2e_steps, step=link_step), dist, dev))
        e_ms, c_ms = statistics.median(e_round), statistics.median(c_round)
        e2e_value = whole_job_gbs(world, step_bytes, e2e_steps, e_ms)
        ceiling = whole_job_gbs(world, step_bytes, e2e_steps, c_ms)
        e2e = {"value": round(e2e_value, 2), "unit": UNIT,
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": e2e_steps,
               "ms_per_step": round(e_ms / e2e_steps, 3),
               "pipeline": f"{E2E_CHUNKS} row chunks per hidden size; host->device, kernel and "
                           "device->host streams chained by events",
               "rounds_gbs": [round(whole_job_gbs(world, step_bytes, e2e_steps, m), 1) for m in e_round],
               "link_gbs": round(ceiling, 2),
               "link_rounds_gbs": [round(whole_job_gbs(world, step_bytes, e2e_steps, m), 1)
                                   for m in c_round],
               "frac_of_link": round(e2e_value / ceiling, 4) if ceiling > 0 else None,
               "link": "the same host<->device bytes copied with no kernel, the two directions "
                       "on two streams at once"}
        del hosts, outs, work

    ops = None
    if rank == 0 and not args.no_ops:
        del sets
        torch.cuda.empty_cache()
        ops = ops_suite(nf, peak, stream, torch.cuda.get_device_properties(local).L2_cache_size)

    cpu = None
    if rank == 0 and not args.no_cpu:
        ncores = host_cores()
        v1, desc1, _, _, _ = oracle_sample(args.cpu_seconds)
        vn, descn, used, _, _ = oracle_sample(args.cpu_seconds, threads=ncores)
        cpu = {"value": round(vn, 4), "unit": UNIT, "cores": used, "kind": "oracle", "sample": descn,
               "single_thread": {"value": round(v1, 4), "cores": 1, "sample": desc1},
               "affinity_cores": ncores}

    if rank == 0:
        line = {
            "metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(ms_total / args.steps, 4), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f32", "storage_dtype": "bf16",
            "data": "synthetic (seeded torch generator on the device; x ~ N(0,1), residual ~ 4 N(0,1), "
                    "weight ~ N(1,0.1))",
            "config": {"workload": f"fused add+RMSNorm forward in place, LLM prefill rows={ROWS}, "
                                   f"hidden in {list(HIDDENS)} (one launch per hidden per step)",
                       "rows": ROWS, "hidden": list(HIDDENS), "eps": EPS,
                       "l2": "inputs larger than L2 (0.54-1.07 GB per launch vs 129 MB L2); no flush",
                       "parallelism": f"replicas x{world}",
                       "path": nf.nf_plan_query("fused_add_rmsnorm", ROWS, DOMINANT_HIDDEN)["path"]},
            "rows_per_s": round(world * ROWS * len(HIDDENS) * args.steps / (ms_total * 1e-3), 1),
            "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                         "frac": round(achieved / peak, 4), "traffic": traffic,
                         "kernel": f"fused_add_rmsnorm ({dom_path} path) hidden={DOMINANT_HIDDEN} rows={ROWS}",
                         "peak_source": f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs, burst copy)"
                         if peak_kind == "measured" else "fallback 6.8 TB/s",
                         "frac_of_nominal_8tbs": round(achieved / 8000.0, 4)},
            "gpu_launches": args.steps * len(HIDDENS),
            "e2e": e2e, "cpu_baseline": cpu, "clocks": clocks, "ops": ops,
        }
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.barrier()
        dist.destroy_process_group()
    return 0


def _source_hash(sources, span=None):
    """sha256 over the given files; for a file with a `[kernel-span NAME]`
    marker pair and span == NAME, only the text between the markers (so
    edits to other kernels of the same file do not invalidate it)."""
    import hashlib
    h = hashlib.sha256()
    for fn in sources:
        with open(os.path.join(ROOT, fn), "r") as fh:
            text = fh.read()
        if span:
            b, e = f"// [kernel-span {span}]", f"// [end kernel-span {span}]"
            if b in text and e in text:
                text = text[text.index(b):text.index(e) + len(e)]
        h.update(text.encode())
    return h.hexdigest()


def _profiled_traffic(op, path, rows, hidden):
    """DRAM bytes per launch from the committed ncu summary, if it was taken
    on the kernel source that is built now; else None."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(p) as f:
            d = json.load(f)
        ent = d[f"{op} {path} {rows}x{hidden}"]
        if _source_hash(ent["sources"], ent.get("span")) != ent["sha256"]:
            return None
        return ent["dram_bytes_per_launch"]
    except Exception:
        return None


def run_profile_case(spec: str, reps: int):
    """Run `reps` launches of one operation at one size and exit: the small,
    self-contained command the ncu captures use.  spec = OP:ROWSxHIDDEN with
    OP in fused_add_rmsnorm, rmsnorm_fwd, layernorm_fwd, layernorm_bwd,
    rmsnorm_bwd, fused_add_rmsnorm_bwd, outer_norm_fwd, outer_norm_bwd; an
    optional @FAMILY suffix (e.g. @split) forces that kernel family for the
    timed calls (inputs are prepared under the automatic choice)."""
    import row_normalization_inner_gb300 as nf
    from row_normalization_inner_gb300 import build as nf_build
    nf_build.build()
    spec, _, family = spec.partition("@")
    op, shape = spec.split(":")
    rows, hidden = (int(v) for v in shape.split("x"))
    dev = "cuda"
    if op == "fused_add_rmsnorm":
        x, r, w = workloads.fused_inputs(rows, hidden, residual_scale=4.0, device=dev)
        fn = lambda: nf.fused_add_rmsnorm(x, r, w, EPS)  # noqa: E731
    elif op == "rmsnorm_fwd":
        x, w = workloads.rms_inputs(rows, hidden, device=dev)
        y = torch.empty_like(x)
        fn = lambda: nf.rmsnorm_fwd(x, w, EPS, out=y)  # noqa: E731
    elif op == "layernorm_fwd":
        x, g, b = workloads.layernorm_fwd_inputs(rows, hidden, device=dev)
        y = torch.empty_like(x)
        fn = lambda: nf.layernorm_fwd(x, g, b, EPS, out=y)  # noqa: E731
    elif op == "layernorm_bwd":
        x, dy, g = workloads.layernorm_bwd_inputs(rows, hidden, device=dev)
        _, mean, rstd = nf.layernorm_fwd(x, g, torch.zeros_like(g), EPS)
        ws = torch.empty(max(nf.nf_layernorm_bwd_workspace_size(rows, hidden), 16),
                         dtype=torch.uint8, device=dev)
        dx = torch.empty_like(x)
        fn = lambda: nf.layernorm_bwd(dy, x, mean, rstd, g, workspace=ws, out=dx)  # noqa: E731
    elif op == "rmsnorm_bwd":
        x, dy, w = workloads.rms_bwd_inputs(rows, hidden, device=dev)
        ws = torch.empty(max(nf.nf_rmsnorm_bwd_workspace_size(rows, hidden), 16),
                         dtype=torch.uint8, device=dev)
        dx = torch.empty_like(x)
        fn = lambda: nf.rmsnorm_bwd(dy, x, w, EPS, workspace=ws, out=dx)  # noqa: E731
    elif op == "fused_add_rmsnorm_bwd":
        s_, w, dy, dres = workloads.fused_bwd_inputs(rows, hidden, device=dev)
        ws = torch.empty(max(nf.nf_rmsnorm_bwd_workspace_size(rows, hidden), 16),
                         dtype=torch.uint8, device=dev)
        dx = torch.empty_like(s_)
        fn = lambda: nf.fused_add_rmsnorm_bwd(dy, s_, w, dres, EPS, workspace=ws, out=dx)  # noqa: E731
    elif op in ("outer_norm_fwd", "outer_norm_bwd"):
        x, dy, g, b = workloads.outer_inputs(rows, hidden, device=dev)
        ws = torch.empty(max(nf.nf_outer_norm_workspace_size(rows, hidden), 16),
                         dtype=torch.uint8, device=dev)
        y = torch.empty_like(x)
        _, mean, rstd = nf.outer_norm_fwd(x, g, b, EPS, workspace=ws, out=y)
        if op == "outer_norm_fwd":
            fn = lambda: nf.outer_norm_fwd(x, g, b, EPS, workspace=ws, out=y)  # noqa: E731
        else:
            fn = lambda: nf.outer_norm_bwd(dy, x, mean, rstd, g, workspace=ws, out=y)  # noqa: E731
    else:
        raise SystemExit(f"unknown op {op}")
    nf.set_path(family or "auto")
    try:
        for _ in range(reps):
            fn()
        torch.cuda.synchronize()
        plan = "outer" if op.startswith("outer") else nf.nf_plan_query(
            "rmsnorm_bwd" if op == "fused_add_rmsnorm_bwd" else op, rows, hidden)
    finally:
        nf.set_path("auto")
    print(f"profile case {spec}{'@' + family if family else ''}: {reps} call(s), plan {plan}")
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--no-ops", action="store_true", help="skip the per-operation suite")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--ref-seconds", type=float, default=60.0,
                    help="reference arm: about this many seconds of timed oracle steps in all")
    ap.add_argument("--profile-case", default=None, help="OP:ROWSxHIDDEN, run --reps launches and exit")
    ap.add_argument("--reps", type=int, default=3)
    args = ap.parse_args()
    if args.warmup < 3 and args.impl == "ours":
        print("warning: fewer than 3 warm-up steps", file=sys.stderr)
    if args.profile_case:
        return run_profile_case(args.profile_case, args.reps)
    if args.impl == "reference":
        return run_reference(args)
    return run_gpu(args)


if __name__ == "__main__":
    sys.exit(main())
