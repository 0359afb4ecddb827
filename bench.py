#!/usr/bin/env python
"""Benchmark of the lattice weight-quantization hot path on GB300.

One step = the whole path over one Llama-3-8B decoder layer (q, k, v, o,
gate, up, down; bf16 N(0, 0.02^2) weights, seeds 1000..1006):
  quantize every matrix to E8 codes (tile 256, beta 0.25; signs, RHT, scale,
  nearest point, int8 codes + fp32 scales), then the decode GEMV y = W^ x from
  the codes at batch 1, 4 and 16 (x ~ N(0, 1) bf16) over every matrix, one
  call per group of matrices that share an activation (q+k+v, o, gate+up,
  down).
The step is captured once as a CUDA graph and replayed; the timed region is
exactly K replays between barriers and device synchronisations.

value  = algorithmic bytes of the step / step time (GB/s, whole job over all ranks)
e2e    = the same bytes / time of a step that also copies the layer's weights
         and activations from pinned host memory and reads codes, scales and
         y back to the host (copies in, kernels and copies out pipelined on
         three streams, row piece by row piece, one CUDA graph per step)
parts  = quantize GB/s, GEMV GB/s per batch, the Rice format of the same codes
         (bits per weight, encode GB/s, GEMV-from-stream GB/s per batch) and
         the prefill GEMM TFLOP/s on the Llama-3-70B MLP shapes
roofline = the quantize kernel (largest share of the step) against the measured
         HBM copy bandwidth

--impl reference times the float64 CPU oracle on the same metric over a bounded
row sample of the same layer (rank 0 only).

Other workloads (--workload), each printed as one JSON line of the same form:
  stack  32 such layers with 0.1 % x20 outliers (seeds 2000 + 7 layer + index,
         drawn on the device), all resident in HBM; one step = quantize all 224
         matrices, then the GEMV at batch 1 and 8 over all of them in layer
         order, captured as one CUDA graph.
  kv     one decode step of attention over a Llama-3-8B KV cache (32 layers,
         8 kv heads, 32 query heads, head_dim 128) quantized to E8 codes
         (tile = head_dim, beta 0.25), at 4 K, 32 K and 128 K cached tokens,
         computed from the codes; GB/s of cache bytes (codes + scales) read.
  sweep  gate- and down-shaped matrices (seeds 3000 / 3001) over every lattice,
         beta in {0.125, 0.25, 0.5} and tile in {128, 256, 512, 1024, 2048}:
         relative MSE, normalised second moment, code entropy, quantize GB/s
         and batch-1 GEMV GB/s per run; then the scale that meets 3, 4 and 5
         bits per weight of the Rice stream for every lattice, with its SNR.
"""
from __future__ import annotations

import argparse
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

TILE, BETA, LATTICE = 256, 0.25, "e8"
BATCHES = (1, 4, 16)
FALLBACK_HBM_GBS, FALLBACK_BF16_TFLOPS = 6800.0, 1900.0
METRIC = "quantize GB/s + lattice-GEMV GB/s (frac of HBM peak); prefill GEMM TFLOPS"


def layer_shapes():
    from synthetic import LLAMA3_8B_LAYER
    return [(n, r, c, 1000 + i) for i, (n, r, c) in enumerate(LLAMA3_8B_LAYER)]


def quantize_bytes(rows, cols, in_bytes=2):
    return rows * cols * (in_bytes + 1 + 4.0 / TILE) + cols


# Matrices of a layer that share one activation; each group is one GEMV call
# (q, k and v read the attention input, gate and up the MLP input).
LAYER_GROUPS = (("q", "k", "v"), ("o",), ("gate", "up"), ("down",))


def gemv_bytes(rows, cols, b, x_bytes=2):
    return rows * cols * (1 + 4.0 / TILE) + cols + b * cols * x_bytes + b * rows * 4


def group_gemv_bytes(rows_list, cols, b, x_bytes=2):
    """One call over matrices sharing x: codes, scales, signs and y of each, x once."""
    return sum(r * cols * (1 + 4.0 / TILE) + cols + b * r * 4 for r in rows_list) + b * cols * x_bytes


def layer_groups(shapes):
    """Index lists of `shapes` per activation group."""
    pos = {n: i for i, (n, _, _, _) in enumerate(shapes)}
    return [[pos[n] for n in grp] for grp in LAYER_GROUPS]


def step_bytes(shapes, frac_rows=1.0):
    q = g = 0.0
    per_b = {}
    rows = [max(1, int(r * frac_rows)) for _, r, _, _ in shapes]
    for (_, r, c, _), rr in zip(shapes, rows):
        q += quantize_bytes(rr, c)
    for b in BATCHES:
        per_b[b] = sum(group_gemv_bytes([rows[i] for i in grp], shapes[grp[0]][2], b)
                       for grp in layer_groups(shapes))
        g += per_b[b]
    return q, per_b, q + g


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        try:
            return json.load(open(p)), "measured"
        except Exception:
            pass
    return None, "fallback"


def hbm_peak(kind="burst"):
    peaks, src = measured_peaks()
    if peaks:
        for key in (("hbm_gbs_" + kind), "hbm_gbs", "hbm_gbs_burst", "hbm_gbs_sustained"):
            v = peaks.get(key)
            if isinstance(v, (int, float)) and v > 0:
                return float(v), "of measured"
            if isinstance(v, dict):
                for kk in ("gbs", "value", kind):
                    if isinstance(v.get(kk), (int, float)):
                        return float(v[kk]), "of measured"
    return FALLBACK_HBM_GBS, "of fallback"


def bf16_peak(kind="burst"):
    peaks, _ = measured_peaks()
    if peaks:
        for key in ("bf16_tflops" if kind == "burst" else "bf16_tflops_sustained", "bf16_tflops"):
            v = peaks.get(key)
            if isinstance(v, (int, float)) and v > 0:
                return float(v), "of measured"
    return FALLBACK_BF16_TFLOPS, "of fallback"


# ---------------------------------------------------------------- clocks
class ClockSampler:
    """Samples nvidia-smi clocks and throttle reasons while the timed region runs."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index):
        self.dev = device_index
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(prefix="lq_clocks_", suffix=".csv")
            os.close(fd)
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.dev}", f"--query-gpu={self.QUERY}", "--format=csv,noheader,nounits",
                 "-lms", "200", "-f", self.path], stdout=subprocess.DEVNULL, stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        try:
            for line in open(self.path):
                f = [x.strip() for x in line.split(",")]
                if len(f) < 9:
                    continue
                try:
                    sm.append(float(f[1]))
                    mx.append(float(f[2]))
                except ValueError:
                    continue
                for n, v in zip(names, f[5:9]):
                    if v.lower().startswith("active"):
                        reasons.add(n)
            os.unlink(self.path)
        except Exception:
            return None
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


# ---------------------------------------------------------------- CPU oracle leg
def cpu_oracle_sample(frac_rows: float, repeats: int = 1) -> dict:
    """Time the float64 oracle on the first frac_rows of every layer matrix."""
    import numpy as np
    import oracle as O
    from synthetic import gaussian_matrix, gaussian_vectors
    shapes = layer_shapes()
    mats, xs = [], {}
    for n, r, c, seed in shapes:
        rr = max(1, int(r * frac_rows))
        mats.append((n, gaussian_matrix(rr, c, 0.02, seed, dtype="bf16"), c, seed))
    for b in BATCHES:
        for c in sorted({c for _, _, c, _ in shapes}):
            xs[(b, c)] = gaussian_vectors(b, c, 5000 + b, dtype="bf16")
    times = []
    for _ in range(repeats):
        t0 = time.perf_counter()
        for n, W, c, seed in mats:
            d = O.splitmix64_signs(seed, c)
            q = O.quantize(W, LATTICE, TILE, d, BETA)
            for b in BATCHES:
                O.gemv(q.codes, q.scales, d, TILE, LATTICE, xs[(b, c)])
        times.append(time.perf_counter() - t0)
    _, _, total = step_bytes(shapes, frac_rows)
    return {"seconds": times, "bytes": total}


def _oracle_worker(wid, nproc, frac_rows, barrier, q):
    """One row block of every sampled layer matrix (spawned process, one BLAS thread)."""
    import numpy as np
    import oracle as O
    from synthetic import gaussian_matrix, gaussian_vectors
    shapes = layer_shapes()
    work = []
    for n, r, c, seed in shapes:
        rr = max(1, int(r * frac_rows))
        lo, hi = rr * wid // nproc, rr * (wid + 1) // nproc
        W = gaussian_matrix(rr, c, 0.02, seed, dtype="bf16")[lo:hi].copy()
        work.append((W, c, seed, {b: gaussian_vectors(b, c, 5000 + b, dtype="bf16") for b in BATCHES}))
    barrier.wait()
    t0 = time.perf_counter()
    for W, c, seed, xs in work:
        if W.shape[0] == 0:
            continue
        d = O.splitmix64_signs(seed, c)
        qz = O.quantize(W, LATTICE, TILE, d, BETA)
        for b in BATCHES:
            O.gemv(qz.codes, qz.scales, d, TILE, LATTICE, xs[b])
    q.put(time.perf_counter() - t0)


def cpu_oracle_all_cores(frac_rows: float, nproc: int) -> dict:
    """The oracle over row blocks on nproc spawned processes; wall time of the compute."""
    import multiprocessing as mp
    ctx = mp.get_context("spawn")
    barrier = ctx.Barrier(nproc + 1)
    q = ctx.Queue()
    procs = [ctx.Process(target=_oracle_worker, args=(w, nproc, frac_rows, barrier, q)) for w in range(nproc)]
    for p in procs:
        p.start()
    barrier.wait()
    t0 = time.perf_counter()
    per = [q.get() for _ in procs]
    wall = time.perf_counter() - t0
    for p in procs:
        p.join()
    _, _, total = step_bytes(layer_shapes(), frac_rows)
    return {"seconds": wall, "bytes": total, "worker_seconds_max": max(per)}


def run_cpu_baseline_all_cores(frac_rows: float) -> dict:
    nproc = os.cpu_count() or 1
    env = dict(os.environ, OMP_NUM_THREADS="1", OPENBLAS_NUM_THREADS="1", MKL_NUM_THREADS="1")
    code = ("import json,sys; sys.path.insert(0, %r); import bench; "
            "print(json.dumps(bench.cpu_oracle_all_cores(%r, %d)))" % (ROOT, frac_rows, nproc))
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, env=env, cwd=ROOT)
    if r.returncode != 0:
        raise RuntimeError("CPU oracle (all cores) failed:\n" + r.stderr[-2000:])
    out = json.loads(r.stdout.strip().splitlines()[-1])
    out["cores"] = nproc
    return out


def run_cpu_baseline(frac_rows: float, repeats: int) -> dict:
    env = dict(os.environ, OMP_NUM_THREADS="1", OPENBLAS_NUM_THREADS="1", MKL_NUM_THREADS="1")
    code = ("import json,sys; sys.path.insert(0, %r); import bench; "
            "print(json.dumps(bench.cpu_oracle_sample(%r, %d)))" % (ROOT, frac_rows, repeats))
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, env=env, cwd=ROOT)
    if r.returncode != 0:
        raise RuntimeError("CPU oracle leg failed:\n" + r.stderr[-2000:])
    return json.loads(r.stdout.strip().splitlines()[-1])


# ---------------------------------------------------------------- distributed
def dist_setup(args):
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if ws > 1:
        import torch.distributed as dist
        backend = os.environ.get("LQ_DIST_BACKEND", "nccl")
        dist.init_process_group(backend=backend)
    return ws, rank, local


def barrier(ws):
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(ws, value, device):
    if ws == 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ---------------------------------------------------------------- reference arm
def reference_arm(args, ws, rank):
    if rank != 0:
        return
    for k in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
        os.environ[k] = "1"      # the oracle runs on one host core
    shapes = layer_shapes()
    frac = args.reference_frac
    for _ in range(args.warmup):
        cpu_oracle_sample(frac, 1)
    t0 = time.perf_counter()
    res = cpu_oracle_sample(frac, args.steps)
    total = time.perf_counter() - t0
    step_s = statistics.mean(res["seconds"])
    value = res["bytes"] / step_s / 1e9
    sample = (f"first {frac:.4g} of the rows of each Llama-3-8B layer matrix per step "
              f"(quantize + GEMV b=1,4,16), float64 NumPy oracle")
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 6),
        "unit": "GB/s", "n_gpus": 0, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(step_s * 1e3, 3), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": "llama3-8b-layer e8 tile256 beta0.25 quantize+gemv(b=1,4,16)",
                   "sample_rows_fraction": frac},
        "cpu_baseline": {"value": round(value, 6), "unit": "GB/s", "cores": 1, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": round(value, 6), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "wall_s": round(total, 3),
    }
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------- GPU arm
def gpu_arm(args, ws, rank, local):
    import numpy as np
    import torch

    from lattice_vq_weight_gb300 import build as _build
    _build.build()
    import lattice_vq_weight_gb300 as L
    from synthetic import bf16_bits_to_f32, f32_to_bf16_bits, gaussian_matrix, gaussian_vectors  # noqa

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    shapes = layer_shapes()

    # ---- inputs: host (pinned) copies for the end-to-end leg, device copies for the kernel leg
    host_w, dev_w = [], []
    for n, r, c, seed in shapes:
        w = gaussian_matrix(r, c, 0.02, seed, dtype="bf16")
        hw = torch.from_numpy(f32_to_bf16_bits(w).view(np.int16)).view(torch.bfloat16).pin_memory()
        host_w.append(hw)
        dev_w.append(hw.to(dev, non_blocking=False))
    host_x = {}
    dev_x = {}
    for b in BATCHES:
        for c in sorted({c for _, _, c, _ in shapes}):
            x = gaussian_vectors(b, c, 5000 + b, dtype="bf16")
            hx = torch.from_numpy(f32_to_bf16_bits(x).view(np.int16)).view(torch.bfloat16).pin_memory()
            host_x[(b, c)] = hx
            dev_x[(b, c)] = hx.to(dev)
    codes = [torch.empty((r, c), dtype=torch.int8, device=dev) for _, r, c, _ in shapes]
    scales = [torch.empty((r, c // TILE), dtype=torch.float32, device=dev) for _, r, c, _ in shapes]
    signs = [torch.empty((c,), dtype=torch.int8, device=dev) for _, _, c, _ in shapes]
    ys = {(b, i): torch.empty((b, r), dtype=torch.float32, device=dev)
          for b in BATCHES for i, (_, r, _, _) in enumerate(shapes)}
    groups = layer_groups(shapes)
    ws_bytes = max(L.lq_gemv_grouped_workspace_size(len(grp), b, shapes[grp[0]][2], TILE)
                   for b in BATCHES for grp in groups)
    work = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    stream = torch.cuda.Stream(device=dev)

    def quantize_all():
        # the layer's seven matrices in one grouped call (one launch pair)
        L.lq_quantize_grouped(LATTICE, dev_w, TILE, [seed for _, _, _, seed in shapes], BETA, codes, scales,
                              signs, status)

    def gemv_all(b):
        for grp in groups:
            x = dev_x[(b, shapes[grp[0]][2])]
            if len(grp) == 1:
                i = grp[0]
                L.lq_gemv(LATTICE, codes[i], scales[i], signs[i], TILE, x, ys[(b, i)], work, status)
            else:
                L.lq_gemv_grouped(LATTICE, [codes[i] for i in grp], [scales[i] for i in grp],
                                  [signs[i] for i in grp], TILE, x, [ys[(b, i)] for i in grp], work, status)

    def step():
        quantize_all()
        for b in BATCHES:
            gemv_all(b)

    launches_per_step = 2 + 2 * len(groups) * len(BATCHES)

    with torch.cuda.stream(stream):
        for _ in range(max(1, args.warmup)):
            step()
    torch.cuda.synchronize(dev)
    if int(status.item()) != 0:
        raise RuntimeError(f"device status {int(status.item())} after warm-up")

    def capture(fn):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            fn()
        return g

    g_step = capture(step)
    g_quant = capture(quantize_all)
    g_gemv = {b: capture(lambda b=b: gemv_all(b)) for b in BATCHES}
    for _ in range(args.warmup):
        g_step.replay()
    torch.cuda.synchronize(dev)

    def time_graph(g, reps):
        with torch.cuda.stream(stream):
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for _ in range(reps):
                g.replay()
            e1.record(stream)
        e1.synchronize()
        return e0.elapsed_time(e1) / reps

    # ---- timed region: exactly K steps
    clocks = ClockSampler(torch.cuda.current_device() if local is None else local)
    clocks.start()
    barrier(ws)
    torch.cuda.synchronize(dev)
    with torch.cuda.stream(stream):
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(args.steps):
            g_step.replay()
        e1.record(stream)
    torch.cuda.synchronize(dev)
    barrier(ws)
    clk = clocks.stop()
    ms_step_local = e0.elapsed_time(e1) / args.steps
    ms_step = max_over_ranks(ws, ms_step_local, dev)
    qb, gb_per_b, total_bytes = step_bytes(shapes)
    value = total_bytes * ws / (ms_step * 1e-3) / 1e9

    # ---- per-part timings (quantize kernel = roofline kernel; GEMV per batch)
    reps = max(3, args.steps)
    ms_quant = time_graph(g_quant, reps)
    ms_gemv = {b: time_graph(g_gemv[b], reps) for b in BATCHES}
    quant_gbs = qb / (ms_quant * 1e-3) / 1e9
    parts = {"quantize_gbs": round(quant_gbs, 1)}
    for b in BATCHES:
        parts[f"gemv_b{b}_gbs"] = round(gb_per_b[b] / (ms_gemv[b] * 1e-3) / 1e9, 1)
    parts["quantize_ms"] = round(ms_quant, 4)
    parts.update({f"gemv_b{b}_ms": round(ms_gemv[b], 4) for b in BATCHES})

    # ---- end-to-end through the public API with host buffers
    h_codes = [torch.empty(cd.shape, dtype=torch.int8).pin_memory() for cd in codes]
    h_scales = [torch.empty(s.shape, dtype=torch.float32).pin_memory() for s in scales]
    h_ys = {k: torch.empty(v.shape, dtype=torch.float32).pin_memory() for k, v in ys.items()}
    h2d = sum(w.numel() * 2 for w in host_w) + sum(x.numel() * 2 for x in host_x.values())
    d2h = sum(c.numel() for c in codes) + sum(s.numel() * 4 for s in scales) + sum(v.numel() * 4 for v in ys.values())

    # One step end to end, pipelined over three streams and captured as one graph:
    # s_in copies x and the weights in (row piece by row piece), `stream`
    # quantizes each piece as soon as it has landed and then runs the GEMVs,
    # s_out copies each piece's codes and scales out as soon as they are
    # written, then y.  The host link (about 0.2 TB/s each way here) bounds it.
    s_in = torch.cuda.Stream(device=dev)
    s_out = torch.cuda.Stream(device=dev)

    # row pieces of about 16 MB of bf16 weights, so that copies in, quantize and
    # copies out overlap with a short head and tail
    def pieces(r, c):
        step = max(1, (8 << 20) // c)
        return [(r0, min(r, r0 + step)) for r0 in range(0, r, step)]

    def e2e_body():
        start = torch.cuda.Event()
        start.record(stream)
        s_in.wait_event(start)
        s_out.wait_event(start)
        work_items = []          # (matrix, r0, r1, event after its copy in)
        with torch.cuda.stream(s_in):
            for k in host_x:
                dev_x[k].copy_(host_x[k], non_blocking=True)
            for i, (n, r, c, seed) in enumerate(shapes):
                for r0, r1 in pieces(r, c):
                    dev_w[i][r0:r1].copy_(host_w[i][r0:r1], non_blocking=True)
                    ev = torch.cuda.Event()
                    ev.record(s_in)
                    work_items.append((i, r0, r1, ev))
        done_q = []
        with torch.cuda.stream(stream):
            for i, r0, r1, ev_in in work_items:
                stream.wait_event(ev_in)
                seed = shapes[i][3]
                L.lq_quantize(LATTICE, dev_w[i][r0:r1], TILE, seed, BETA, codes[i][r0:r1], scales[i][r0:r1],
                              signs[i], status)
                ev = torch.cuda.Event()
                ev.record(stream)
                done_q.append((i, r0, r1, ev))
        with torch.cuda.stream(s_out):
            for i, r0, r1, ev in done_q:
                s_out.wait_event(ev)
                h_codes[i][r0:r1].copy_(codes[i][r0:r1], non_blocking=True)
                h_scales[i][r0:r1].copy_(scales[i][r0:r1], non_blocking=True)
        for b in BATCHES:
            with torch.cuda.stream(stream):
                gemv_all(b)
                ev = torch.cuda.Event()
                ev.record(stream)
            with torch.cuda.stream(s_out):
                s_out.wait_event(ev)
                for i in range(len(shapes)):
                    h_ys[(b, i)].copy_(ys[(b, i)], non_blocking=True)
        done = torch.cuda.Event()
        done.record(s_out)
        stream.wait_event(done)

    with torch.cuda.stream(stream):
        e2e_body()
    torch.cuda.synchronize(dev)
    g_e2e = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g_e2e, stream=stream):
        e2e_body()
    g_e2e.replay()
    torch.cuda.synchronize(dev)
    barrier(ws)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        g_e2e.replay()
    torch.cuda.synchronize(dev)
    barrier(ws)
    e2e_ms = max_over_ranks(ws, (time.perf_counter() - t0) * 1e3 / args.steps, dev)
    e2e_val = total_bytes * ws / (e2e_ms * 1e-3) / 1e9
    if int(status.item()) != 0:
        raise RuntimeError(f"device status {int(status.item())} after the timed region")

    # ---- Rice format of the same codes: encode, and the GEMV from the stream
    rice = rice_part(L, torch, dev, stream, shapes, codes, scales, signs, dev_x, reps=max(3, min(args.steps, 10)))

    # ---- per-row bf16 scale format (the int8 layout): quantize and GEMV of the same layer
    rowfmt = rowscale_part(L, torch, dev, stream, shapes, dev_w, dev_x, reps=max(3, min(args.steps, 10)))

    # ---- prefill GEMM (Llama-3-70B MLP shapes), when the library provides it
    gemm = None
    if not args.no_gemm:
        gemm = gemm_part(L, torch, dev, stream, reps=max(3, min(args.steps, 10)))

    peak, peak_src = hbm_peak("burst")
    roof_achieved = quant_gbs
    traffic = None
    tpath = os.path.join(ROOT, "profiles", "traffic.json")
    if os.path.exists(tpath):
        try:
            traffic = json.load(open(tpath)).get("quantize_layer_bytes")
        except Exception:
            traffic = None

    line = {
        "metric": METRIC, "value": round(value, 1), "unit": "GB/s",
        "n_gpus": ws, "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_step, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16->int8 (fp32 compute)",
        "data": "synthetic",
        "config": {"workload": "llama3-8b-layer e8 tile256 beta0.25 quantize+gemv(b=1,4,16)",
                   "matrices": [f"{n} {r}x{c}" for n, r, c, _ in shapes], "lattice": LATTICE, "tile": TILE,
                   "beta": BETA, "batches": list(BATCHES), "parallelism": f"replicas{ws}",
                   "l2": "inputs larger than L2 (436 MB bf16 weights, 218 MB codes per step); no flush",
                   "graph": "step captured as one CUDA graph",
                   "quantize": "the seven matrices in one grouped call (one launch pair)",
                   "gemv_groups": "q+k+v, o, gate+up, down (one call each, activation shared in a group)"},
        "gpu_launches": launches_per_step * args.steps,
        "parts": parts,
        "e2e": {"value": round(e2e_val, 1), "unit": "GB/s", "h2d_bytes_per_step": int(h2d),
                "d2h_bytes_per_step": int(d2h), "ms_per_step": round(e2e_ms, 3)},
        "roofline": {"kernel": "quantize_kernel (one grouped launch over the 7 matrices of the layer)", "bound": "hbm",
                     "achieved": round(roof_achieved, 1), "peak": peak, "unit": "GB/s",
                     "frac": round(roof_achieved / peak, 4), "peak_source": peak_src,
                     "traffic": traffic},
        "clocks": clk,
    }
    line["parts"].update(rice)
    line["parts"].update(rowfmt)
    if gemm is not None:
        line["parts"].update(gemm)

    if rank == 0 and not args.no_cpu_baseline:
        try:
            cb = run_cpu_baseline(args.cpu_frac, 1)
            secs = cb["seconds"][0]
            line["cpu_baseline"] = {
                "value": round(cb["bytes"] / secs / 1e9, 6), "unit": "GB/s", "cores": 1, "kind": "oracle",
                "sample": (f"first {args.cpu_frac:.4g} of the rows of each layer matrix, quantize + GEMV "
                           f"b=1,4,16, float64 NumPy, 1 thread, {secs:.1f} s")}
        except Exception as exc:  # reported, not fatal for the GPU number
            line["cpu_baseline"] = {"value": None, "error": str(exc)[-300:]}
        try:
            ac = run_cpu_baseline_all_cores(args.cpu_frac)
            line["cpu_baseline"]["all_cores"] = {
                "value": round(ac["bytes"] / ac["seconds"] / 1e9, 6), "unit": "GB/s", "cores": ac["cores"],
                "kind": "oracle", "sample": (f"same sample split into {ac['cores']} row blocks on "
                                             f"{ac['cores']} spawned processes (1 BLAS thread each), "
                                             f"{ac['seconds']:.1f} s wall")}
        except Exception as exc:
            line["cpu_baseline"]["all_cores"] = {"value": None, "error": str(exc)[-300:]}
    if rank == 0:
        print(json.dumps(line), flush=True)


def _graph_ms(torch, g, stream, reps):
    with torch.cuda.stream(stream):
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(reps):
            g.replay()
        e1.record(stream)
    e1.synchronize()
    return e0.elapsed_time(e1) / reps


def stack_arm(args, ws, rank, local):
    """32 Llama-3-8B layers resident in HBM: quantize all, then GEMV b = 1 and 8."""
    import torch

    from lattice_vq_weight_gb300 import build as _build
    _build.build()
    import lattice_vq_weight_gb300 as L
    from synthetic import LLAMA3_8B_LAYER, stack_seed, torch_gaussian_matrix

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    n_layers, batches = 32, (1, 8)
    mats = []          # (layer, name, rows, cols, seed)
    for layer in range(n_layers):
        for i, (n, r, c) in enumerate(LLAMA3_8B_LAYER):
            mats.append((layer, n, r, c, stack_seed(layer, i)))
    W = [torch_gaussian_matrix(r, c, 0.02, seed, device=dev, outlier_frac=0.001) for _, _, r, c, seed in mats]
    codes = [torch.empty((r, c), dtype=torch.int8, device=dev) for _, _, r, c, _ in mats]
    scales = [torch.empty((r, c // TILE), dtype=torch.float32, device=dev) for _, _, r, c, _ in mats]
    signs = [torch.empty((c,), dtype=torch.int8, device=dev) for _, _, _, c, _ in mats]
    cols_set = sorted({c for _, _, _, c, _ in mats})
    xs = {(b, c): torch.randn((b, c), device=dev, generator=torch.Generator(device=dev).manual_seed(6000 + b)
                              ).to(torch.bfloat16) for b in batches for c in cols_set}
    ys = {(b, k): torch.empty((b, r), dtype=torch.float32, device=dev)
          for b in batches for k, (_, _, r, _, _) in enumerate(mats)}
    # activation groups of every layer (matrix indices into mats), in layer order
    shapes7 = [(n, r, c, 0) for n, r, c in LLAMA3_8B_LAYER]
    groups = [[7 * layer + i for i in grp] for layer in range(n_layers) for grp in layer_groups(shapes7)]
    work = torch.empty(max(L.lq_gemv_grouped_workspace_size(len(grp), b, mats[grp[0]][3], TILE)
                           for b in batches for grp in groups), dtype=torch.uint8, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    stream = torch.cuda.Stream(device=dev)

    def quantize_all():
        # one grouped call (one launch pair) per layer
        for k0 in range(0, len(mats), 7):
            L.lq_quantize_grouped(LATTICE, W[k0:k0 + 7], TILE, [m[4] for m in mats[k0:k0 + 7]], BETA,
                                  codes[k0:k0 + 7], scales[k0:k0 + 7], signs[k0:k0 + 7], status)

    def gemv_all(b):
        for grp in groups:
            x = xs[(b, mats[grp[0]][3])]
            if len(grp) == 1:
                k = grp[0]
                L.lq_gemv(LATTICE, codes[k], scales[k], signs[k], TILE, x, ys[(b, k)], work, status)
            else:
                L.lq_gemv_grouped(LATTICE, [codes[k] for k in grp], [scales[k] for k in grp],
                                  [signs[k] for k in grp], TILE, x, [ys[(b, k)] for k in grp], work, status)

    def step():
        quantize_all()
        for b in batches:
            gemv_all(b)

    with torch.cuda.stream(stream):
        for _ in range(max(1, args.warmup)):
            step()
    torch.cuda.synchronize(dev)
    if int(status.item()) != 0:
        raise RuntimeError(f"device status {int(status.item())} after warm-up")
    graphs = {}
    for name, fn in (("step", step), ("quantize", quantize_all), ("gemv1", lambda: gemv_all(1)),
                     ("gemv8", lambda: gemv_all(8))):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            fn()
        graphs[name] = g
    for _ in range(args.warmup):
        graphs["step"].replay()
    torch.cuda.synchronize(dev)

    clocks = ClockSampler(local)
    clocks.start()
    barrier(ws)
    torch.cuda.synchronize(dev)
    ms_step = _graph_ms(torch, graphs["step"], stream, args.steps)
    torch.cuda.synchronize(dev)
    barrier(ws)
    clk = clocks.stop()
    ms_step = max_over_ranks(ws, ms_step, dev)
    qb = sum(quantize_bytes(r, c) for _, _, r, c, _ in mats)
    gb = {b: sum(group_gemv_bytes([mats[k][2] for k in grp], mats[grp[0]][3], b) for grp in groups)
          for b in batches}
    total = qb + sum(gb.values())
    reps = max(3, min(args.steps, 10))
    ms_q = _graph_ms(torch, graphs["quantize"], stream, reps)
    ms_g = {b: _graph_ms(torch, graphs[f"gemv{b}"], stream, reps) for b in batches}
    if int(status.item()) != 0:
        raise RuntimeError(f"device status {int(status.item())} after the timed region")
    peak, src = hbm_peak("sustained")
    qgbs = qb / (ms_q * 1e-3) / 1e9
    line = {
        "metric": METRIC, "value": round(total * ws / (ms_step * 1e-3) / 1e9, 1), "unit": "GB/s",
        "n_gpus": ws, "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_step, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16->int8 (fp32 compute)",
        "data": "synthetic",
        "config": {"workload": "llama3-8b 32-layer stack e8 tile256 beta0.25 quantize+gemv(b=1,8)",
                   "matrices": len(mats), "weights_bytes": int(sum(w.numel() * 2 for w in W)),
                   "codes_bytes": int(sum(cd.numel() for cd in codes)), "outliers": "0.1% x20",
                   "parallelism": f"replicas{ws}", "l2": "inputs far larger than L2; no flush",
                   "graph": f"one CUDA graph of {2 * n_layers + 2 * len(groups) * len(batches)} launches",
                   "quantize": "one grouped call (one launch pair) per layer",
                   "gemv_groups": "q+k+v, o, gate+up, down per layer (one call each)"},
        "gpu_launches": (2 * n_layers + 2 * len(groups) * len(batches)) * args.steps,
        "parts": {"quantize_gbs": round(qgbs, 1), "quantize_ms": round(ms_q, 3),
                  **{f"gemv_b{b}_gbs": round(gb[b] / (ms_g[b] * 1e-3) / 1e9, 1) for b in batches},
                  **{f"gemv_b{b}_ms": round(ms_g[b], 3) for b in batches}},
        "roofline": {"kernel": "quantize_kernel (224 matrices, one grouped launch per layer)", "bound": "hbm", "achieved": round(qgbs, 1),
                     "peak": peak, "unit": "GB/s", "frac": round(qgbs / peak, 4), "peak_source": src,
                     "traffic": None},
        "clocks": clk,
    }
    if rank == 0:
        print(json.dumps(line), flush=True)


# covolume and textbook normalised second moment of each lattice at its native scale
_LATTICE_GEOM = {"e8": (8, 1.0), "d4": (4, 2.0), "a2": (2, 3 ** 0.5 / 2), "z1": (1, 1.0)}


def sweep_arm(args, ws, rank, local):
    """Lattice x beta x tile sweep on gate- and down-shaped bf16 matrices."""
    import math

    import torch

    from lattice_vq_weight_gb300 import build as _build
    _build.build()
    import lattice_vq_weight_gb300 as L
    from synthetic import LLAMA3_8B_LAYER, torch_gaussian_matrix

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    stream = torch.cuda.Stream(device=dev)
    shapes = {n: (r, c) for n, r, c in LLAMA3_8B_LAYER if n in ("gate", "down")}
    seeds = {"gate": 3000, "down": 3001}
    runs = []
    reps = max(3, min(args.steps, 10))
    for name, (r, c) in shapes.items():
        W = torch_gaussian_matrix(r, c, 0.02, seeds[name], device=dev)
        Wf = W.double()
        w2 = float((Wf * Wf).sum())
        x = torch.randn((1, c), device=dev, generator=torch.Generator(device=dev).manual_seed(6100)).to(torch.bfloat16)
        for lat in ("e8", "d4", "a2", "z1"):
            n, vol = _LATTICE_GEOM[lat]
            for beta in (0.125, 0.25, 0.5):
                for tile in (128, 256, 512, 1024, 2048):
                    codes = torch.empty((r, c), dtype=torch.int8, device=dev)
                    sc = torch.empty((r, c // tile), dtype=torch.float32, device=dev)
                    sg = torch.empty((c,), dtype=torch.int8, device=dev)
                    y = torch.empty((1, r), dtype=torch.float32, device=dev)
                    wk = torch.empty(L.lq_gemv_workspace_size(1, c, tile), dtype=torch.uint8, device=dev)
                    st = torch.zeros(1, dtype=torch.int32, device=dev)
                    with torch.cuda.stream(stream):
                        L.lq_quantize(lat, W, tile, seeds[name], beta, codes, sc, sg, st)
                        L.lq_gemv(lat, codes, sc, sg, tile, x, y, wk, st)
                    torch.cuda.synchronize(dev)
                    gq = torch.cuda.CUDAGraph()
                    with torch.cuda.graph(gq, stream=stream):
                        for _ in range(4):
                            L.lq_quantize(lat, W, tile, seeds[name], beta, codes, sc, sg, st)
                    gg = torch.cuda.CUDAGraph()
                    with torch.cuda.graph(gg, stream=stream):
                        for _ in range(4):
                            L.lq_gemv(lat, codes, sc, sg, tile, x, y, wk, st)
                    gq.replay(); gg.replay()
                    torch.cuda.synchronize(dev)
                    ms_q = _graph_ms(torch, gq, stream, reps) / 4
                    ms_g = _graph_ms(torch, gg, stream, reps) / 4
                    What = L.dequantize(codes, sc, sg, lattice=lat, tile=tile, dtype=torch.float32)
                    err = (What.double() - Wf)
                    # per-dimension distortion in lattice units: the rotation is orthonormal,
                    # so |w - w^|^2 over a tile equals |w~ - s p|^2 = s^2 |y - p|^2
                    tile_err = (err * err).view(r, c // tile, tile).sum(-1)
                    s2 = sc.double() ** 2
                    nz = s2 > 0
                    d_per_dim = float((tile_err[nz] / s2[nz]).sum()) / (int(nz.sum()) * tile)
                    G = d_per_dim / vol ** (2.0 / n)
                    hist = torch.bincount((codes.view(-1).to(torch.int32) + 128), minlength=256).double()
                    pr = hist[hist > 0] / hist.sum()
                    ent = float(-(pr * pr.log2()).sum())
                    runs.append({"shape": name, "lattice": lat, "beta": beta, "tile": tile,
                                 "rel_mse": float((err * err).sum()) / w2, "G": round(G, 6),
                                 "code_entropy_bits": round(ent, 4), "status": int(st.item()),
                                 "quantize_gbs": round(quantize_bytes_t(r, c, tile) / (ms_q * 1e-3) / 1e9, 1),
                                 "gemv_b1_gbs": round(gemv_bytes_t(r, c, 1, tile) / (ms_g * 1e-3) / 1e9, 1)})
                    del codes, sc, sg, y, wk, What, err, gq, gg
        del W, Wf
    # rate -> scale calibration (bisection of beta for a target Rice rate) per lattice
    calib = []
    Wc = torch_gaussian_matrix(1024, 4096, 1.0, 3002, device=dev)
    for lat in ("e8", "d4", "a2", "z1"):
        wsc = torch.empty(L.lq_calibrate_workspace_size(lat, 1024, 4096, TILE), dtype=torch.uint8, device=dev)
        for target in (3.0, 4.0, 5.0):
            t0 = time.perf_counter()
            beta, bps, snr = L.lq_calibrate_bps(lat, TILE, target, Wc, 0, wsc)
            calib.append({"lattice": lat, "target_bps": target, "beta": round(beta, 6), "bps": round(bps, 4),
                          "snr_db": round(snr, 3), "closed_form_beta_at_snr": round(L.lq_beta_for_snr(lat, snr), 6),
                          "ms": round((time.perf_counter() - t0) * 1e3, 2)})
        del wsc
    e8 = [x for x in runs if x["lattice"] == "e8" and x["tile"] == TILE and x["beta"] == BETA]
    best_q = max(x["quantize_gbs"] for x in runs)
    line = {
        "metric": METRIC, "value": round(statistics.mean(x["quantize_gbs"] for x in e8), 1), "unit": "GB/s",
        "n_gpus": ws, "steps": reps, "warmup": args.warmup, "ms_per_step": None, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16->int8 (fp32 compute)", "data": "synthetic",
        "config": {"workload": "lattice sweep: gate 14336x4096 and down 4096x14336 bf16, "
                               "{e8,d4,a2,z1} x beta {0.125,0.25,0.5} x tile {128..2048}",
                   "value_is": "mean quantize GB/s of the e8 tile-256 beta-0.25 runs",
                   "best_quantize_gbs": best_q},
        "textbook_G": {"e8": 929 / 12960, "d4": 0.076603, "a2": 5 / (36 * math.sqrt(3)), "z1": 1 / 12},
        "runs": runs,
        "calibration": {"sample": "1024 x 4096 N(0, 1) fp32 (seed 3002), tile 256; 25 quantize + Rice encode "
                                  "probes per target", "results": calib},
    }
    if rank == 0:
        print(json.dumps(line), flush=True)


def kv_arm(args, ws, rank, local):
    """Decode attention over a quantized 32-layer Llama-3-8B KV cache."""
    import torch

    from lattice_vq_weight_gb300 import build as _build
    _build.build()
    import lattice_vq_weight_gb300 as L
    from synthetic import torch_gaussian_matrix

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    stream = torch.cuda.Stream(device=dev)
    layers, kvh, qh, d = 32, 8, 32, 128
    results = {}
    reps = max(3, min(args.steps, 10))
    # float32 norms at every context; fp16 norms (the pages' cache layout) at 32 K
    # and the subtractive dither (fp16 norms, dither regenerated on chip) at 32 K
    # and the Rice-coded cache (fp16 norms, decoded on chip) at 32 K
    for tokens, fmt, dith, rice in ((4096, "tile_f32", False, False), (32768, "tile_f32", False, False),
                                    (32768, "tile_f16", False, False), (32768, "tile_f16", True, False),
                                    (32768, "tile_f16", False, True), (131072, "tile_f32", False, False)):
        caches = []
        for layer in range(layers):
            pair = []
            for which in range(2):
                X = torch_gaussian_matrix(tokens, kvh * d, 1.0, 7000 + 2 * layer + which, device=dev)
                if dith:
                    pair.append(L.quantize_dithered(X, lattice="e8", tile=d, seed=7100 + 2 * layer + which,
                                                    dither_seed=7300 + 2 * layer + which, beta=BETA,
                                                    scale_format=fmt))
                else:
                    pair.append(L.quantize_ex(X, lattice="e8", tile=d, seed=7100 + 2 * layer + which, beta=BETA,
                                              scale_format=fmt))
                del X
            caches.append(pair)
        stream_bytes = 0
        if rice:
            rcaches = []
            for pair in caches:
                rp = []
                for (c, sc, sg) in pair:
                    nb = L.lq_rice_stream_bound("e8", tokens, kvh * d, d)
                    words = torch.empty(nb // 4, dtype=torch.int32, device=dev)
                    offs = torch.empty((tokens, kvh), dtype=torch.int32, device=dev)
                    tot = torch.empty(1, dtype=torch.int64, device=dev)
                    rws = torch.empty(L.lq_rice_workspace_size(tokens, kvh * d, d), dtype=torch.uint8, device=dev)
                    L.lq_rice_encode("e8", c, d, words, offs, tot, rws)
                    torch.cuda.synchronize(dev)
                    nw = (int(tot.item()) + 31) // 32 + 4
                    stream_bytes += int(tot.item()) / 8.0
                    rp.append((words[:nw].clone(), offs, sc, sg))
                    del words, rws
                rcaches.append(rp)
            caches = rcaches
        q = [torch.randn((qh, d), device=dev, generator=torch.Generator(device=dev).manual_seed(7200 + i)
                         ).to(torch.bfloat16) for i in range(layers)]
        out = [torch.empty((qh, d), dtype=torch.float32, device=dev) for _ in range(layers)]
        wsz = torch.empty(L.lq_attention_workspace_size(tokens, kvh, qh, d), dtype=torch.uint8, device=dev)

        def step():
            if rice:
                for i, ((kw, ko, ks, kd), (vw, vo, vs, vd)) in enumerate(caches):
                    L.lq_attention_decode_rice("e8", kw, ko, ks, kd, vw, vo, vs, vd, fmt, q[i], out[i], wsz)
                return
            for i, ((kc, ks, kd), (vc, vs, vd)) in enumerate(caches):
                if dith:
                    L.lq_attention_decode_dithered("e8", kc, ks, kd, 7300 + 2 * i, vc, vs, vd, 7301 + 2 * i, fmt,
                                                   q[i], out[i], wsz)
                else:
                    L.lq_attention_decode_ex("e8", kc, ks, kd, vc, vs, vd, fmt, q[i], out[i], wsz)

        torch.cuda.synchronize(dev)
        with torch.cuda.stream(stream):
            step()
        torch.cuda.synchronize(dev)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            step()
        g.replay()
        torch.cuda.synchronize(dev)
        ms = _graph_ms(torch, g, stream, reps)
        sbytes = 2 if fmt == "tile_f16" else 4
        cache_bytes = layers * 2 * tokens * kvh * (d + sbytes)
        if rice:   # stream + 32-bit segment offsets + norms
            cache_bytes = int(stream_bytes + layers * 2 * tokens * kvh * (4 + sbytes))
        key = (f"ctx{tokens}" + ("_fp16_norms" if fmt == "tile_f16" else "") + ("_dithered" if dith else "")
               + ("_rice" if rice else ""))
        results[key] = {"ms_per_step": round(ms, 4), "cache_gbs": round(cache_bytes / (ms * 1e-3) / 1e9, 1),
                        "cache_bytes": cache_bytes,
                        "compression_vs_bf16": round(layers * 2 * tokens * kvh * d * 2 / cache_bytes, 3)}
        del caches, q, out, wsz, g
        torch.cuda.empty_cache()
    peak, src = hbm_peak("burst")
    best = max(r["cache_gbs"] for r in results.values())
    line = {
        "metric": METRIC, "value": results["ctx32768"]["cache_gbs"], "unit": "GB/s",
        "n_gpus": ws, "steps": reps, "warmup": args.warmup, "ms_per_step": results["ctx32768"]["ms_per_step"],
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "int8 codes (fp32 compute)",
        "data": "synthetic",
        "config": {"workload": "llama3-8b decode attention over an E8-quantized KV cache (32 layers, 8 kv heads, "
                               "32 q heads, head_dim 128), one graph of 96 launches per step",
                   "value_is": "cache GB/s at 32 768 tokens (float32 norms)", "beta": BETA, "tile": 128},
        "gpu_launches": layers * 3 * reps,
        "contexts": results,
        "roofline": {"kernel": "attn_partial_kernel + attn_combine_kernel", "bound": "hbm", "achieved": best,
                     "peak": peak, "unit": "GB/s", "frac": round(best / peak, 4), "peak_source": src,
                     "traffic": None},
    }
    if rank == 0:
        print(json.dumps(line), flush=True)


def quantize_bytes_t(rows, cols, tile, in_bytes=2):
    return rows * cols * (in_bytes + 1 + 4.0 / tile) + cols


def gemv_bytes_t(rows, cols, b, tile, x_bytes=2):
    return rows * cols * (1 + 4.0 / tile) + cols + b * cols * x_bytes + b * rows * 4


def rice_part(L, torch, dev, stream, shapes, codes, scales, signs, dev_x, reps):
    """Rice stream of the layer's codes: bits per weight, encode GB/s (codes in,
    stream + offsets out) and GEMV-from-stream GB/s per batch (stream, offsets,
    scales, signs, x in; y out)."""
    enc = []
    for i, (n, r, c, seed) in enumerate(shapes):
        nbytes = L.lq_rice_stream_bound(LATTICE, r, c, TILE)
        enc.append((torch.empty(nbytes // 4, dtype=torch.int32, device=dev),
                    torch.empty((r, c // TILE), dtype=torch.int32, device=dev),
                    torch.empty(1, dtype=torch.int64, device=dev),
                    torch.empty(L.lq_rice_workspace_size(r, c, TILE), dtype=torch.uint8, device=dev)))
    status = torch.zeros(1, dtype=torch.int32, device=dev)

    def encode_all():
        for i in range(len(shapes)):
            words, offs, tot, ws = enc[i]
            L.lq_rice_encode(LATTICE, codes[i], TILE, words, offs, tot, ws, status)

    with torch.cuda.stream(stream):
        encode_all()
    torch.cuda.synchronize(dev)
    bits = [int(e[2].item()) for e in enc]
    ys = {(b, i): torch.empty((b, r), dtype=torch.float32, device=dev)
          for b in BATCHES for i, (_, r, _, _) in enumerate(shapes)}
    work = torch.empty(max(L.lq_gemv_workspace_size(b, c, TILE) for b in BATCHES for _, _, c, _ in shapes),
                       dtype=torch.uint8, device=dev)

    def gemv_all(b):
        for i, (n, r, c, seed) in enumerate(shapes):
            words, offs, _, _ = enc[i]
            L.lq_gemv_rice(LATTICE, words, offs, scales[i], signs[i], TILE, dev_x[(b, c)], ys[(b, i)], work, status)

    def graph_of(fn):
        with torch.cuda.stream(stream):
            fn()
        torch.cuda.synchronize(dev)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            fn()
        return g

    out = {}
    weights = sum(r * c for _, r, c, _ in shapes)
    stream_bytes = sum(bits) / 8.0
    offs_bytes = sum(4 * r * (c // TILE) for _, r, c, _ in shapes)
    g_enc = graph_of(encode_all)
    ms = _graph_ms(torch, g_enc, stream, reps)
    out["rice_bits_per_weight"] = round(sum(bits) / weights, 4)
    out["rice_encode_gbs"] = round((weights + stream_bytes + offs_bytes) / (ms * 1e-3) / 1e9, 1)
    for b in BATCHES:
        g = graph_of(lambda b=b: gemv_all(b))
        ms = _graph_ms(torch, g, stream, reps)
        nbytes = stream_bytes + sum(4 * r * (c // TILE) * 2 + c + b * c * 2 + b * r * 4 for _, r, c, _ in shapes)
        out[f"rice_gemv_b{b}_gbs"] = round(nbytes / (ms * 1e-3) / 1e9, 1)
        out[f"rice_gemv_b{b}_ms"] = round(ms, 4)
    torch.cuda.synchronize(dev)
    if int(status.item()) != 0:
        raise RuntimeError(f"device status {int(status.item())} in the Rice part")
    return out


def rowscale_part(L, torch, dev, stream, shapes, dev_w, dev_x, reps):
    """The layer with one bf16 scale per row (lq_quantize_ex / lq_gemv_ex): quantize
    GB/s (W in, codes + row scales out; W is read twice, the second time in L2-sized
    row blocks) and GEMV GB/s per batch (codes, row scales, signs, x in; y out)."""
    fmt = "row_bf16"
    codes = [torch.empty((r, c), dtype=torch.int8, device=dev) for _, r, c, _ in shapes]
    scales = [L.scales_tensor(r, c, TILE, fmt, dev) for _, r, c, _ in shapes]
    signs = [torch.empty((c,), dtype=torch.int8, device=dev) for _, _, c, _ in shapes]
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    ys = {(b, i): torch.empty((b, r), dtype=torch.float32, device=dev)
          for b in BATCHES for i, (_, r, _, _) in enumerate(shapes)}
    work = torch.empty(max(L.lq_gemv_workspace_size(b, c, TILE) for b in BATCHES for _, _, c, _ in shapes),
                       dtype=torch.uint8, device=dev)

    def quant_all():
        for i, (n, r, c, seed) in enumerate(shapes):
            L.lq_quantize_ex(LATTICE, dev_w[i], TILE, seed, BETA, fmt, codes[i], scales[i], signs[i], status)

    def gemv_all(b):
        for i, (n, r, c, seed) in enumerate(shapes):
            L.lq_gemv_ex(LATTICE, codes[i], scales[i], fmt, signs[i], TILE, dev_x[(b, c)], ys[(b, i)], work, status)

    def graph_of(fn):
        with torch.cuda.stream(stream):
            fn()
        torch.cuda.synchronize(dev)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            fn()
        return g

    out = {}
    ms = _graph_ms(torch, graph_of(quant_all), stream, reps)
    qbytes = sum(r * c * 3 + 2 * r + c for _, r, c, _ in shapes)
    out["rowbf16_quantize_gbs"] = round(qbytes / (ms * 1e-3) / 1e9, 1)
    for b in BATCHES:
        ms = _graph_ms(torch, graph_of(lambda b=b: gemv_all(b)), stream, reps)
        nbytes = sum(r * c + 2 * r + c + b * c * 2 + b * r * 4 for _, r, c, _ in shapes)
        out[f"rowbf16_gemv_b{b}_gbs"] = round(nbytes / (ms * 1e-3) / 1e9, 1)
    torch.cuda.synchronize(dev)
    if int(status.item()) != 0:
        raise RuntimeError(f"device status {int(status.item())} in the row-scale part")
    return out


def gemm_part(L, torch, dev, stream, reps):
    """Prefill GEMM TFLOP/s on Llama-3-70B MLP shapes (E8 codes, X bf16 M x K)."""
    from synthetic import LLAMA3_70B_MLP
    out = {}
    for name, N, K in LLAMA3_70B_MLP:
        W = (torch.randn((N, K), device=dev, generator=torch.Generator(device=dev).manual_seed(4000))
             * 0.015).to(torch.bfloat16)
        codes, scales, signs = L.quantize(W, lattice="e8", tile=TILE, seed=4000, beta=BETA)
        del W
        for M in (256, 2048):
            X = torch.randn((M, K), device=dev, generator=torch.Generator(device=dev).manual_seed(4100 + M)
                            ).to(torch.bfloat16)
            Y = torch.empty((M, N), dtype=torch.float32, device=dev)
            wsz = torch.empty(L.lq_gemm_workspace_size(M, N, K), dtype=torch.uint8, device=dev)
            torch.cuda.synchronize(dev)      # inputs were written on the default stream
            try:
                with torch.cuda.stream(stream):
                    L.lq_gemm("e8", codes, scales, signs, TILE, X, Y, wsz)
            except L.LQError as e:
                if e.status == L.LQ_ERR_UNSUPPORTED:
                    return None
                raise
            torch.cuda.synchronize(dev)
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                L.lq_gemm("e8", codes, scales, signs, TILE, X, Y, wsz)
            for _ in range(2):
                g.replay()
            torch.cuda.synchronize(dev)
            with torch.cuda.stream(stream):
                e0 = torch.cuda.Event(enable_timing=True)
                e1 = torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                for _ in range(reps):
                    g.replay()
                e1.record(stream)
            e1.synchronize()
            ms = e0.elapsed_time(e1) / reps
            out[f"gemm_{name}_M{M}_tflops"] = round(2.0 * M * N * K / (ms * 1e-3) / 1e12, 1)
            out[f"gemm_{name}_M{M}_ms"] = round(ms, 4)
        del codes, scales, signs
    pk, src = bf16_peak("burst")
    best = max(v for k, v in out.items() if k.endswith("_tflops"))
    out["gemm_peak_tflops"] = pk
    out["gemm_best_frac"] = round(best / pk, 4)
    out["gemm_peak_source"] = src
    return out


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=("lq", "reference"), default="lq")
    ap.add_argument("--no-gemm", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-frac", type=float, default=0.75)
    ap.add_argument("--reference-frac", type=float, default=1.0 / 64)
    ap.add_argument("--workload", choices=("layer", "stack", "sweep", "kv"), default="layer")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        args.warmup = 3
    ws, rank, local = dist_setup(args)
    try:
        if args.impl == "reference":
            reference_arm(args, ws, rank)
        elif args.workload == "stack":
            stack_arm(args, ws, rank, local)
        elif args.workload == "sweep":
            sweep_arm(args, ws, rank, local)
        elif args.workload == "kv":
            kv_arm(args, ws, rank, local)
        else:
            gpu_arm(args, ws, rank, local)
    finally:
        if ws > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
