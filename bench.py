#!/usr/bin/env python3
"""Benchmark of the fused packed-weight decode step (and the prefill qmm).

One step = one Llama-3.2-1B-shaped decode step, M = 1, 8-bit codes, group 64,
f16 activations/scales/biases: 16 layers x (q, k, v, o, gate, up, down) + the
lm_head (N = 128256), each linear a fused dequantise-into-matvec whose input is
an earlier linear's output: 65 launches (q/k/v and gate/up fused) overlapped
with programmatic dependent launch, captured in one CUDA graph.  1.31 GB of packed weights stream
per step, ten times the L2, so no flush is needed between steps.  The headline
value is tokens/s-equivalent = steps / second.

Also measured in the same run (reported beside the headline):
  * each qmv launch's own duration (CUDA events around it on its stream)
    -> achieved HBM GB/s against the measured copy bandwidth (roofline);
  * the same step as one persistent chain launch (qlin_qmv_chain);
  * the tensor-core qmm at M = 2048 on the prefill shapes (8192x2048,
    2048x8192, 2048x2048; 4- and 8-bit; f16; 1% outlier rows), L2 flushed
    between timed launches -> TFLOP/s against the dense bf16 peak;
  * end to end: per step the input copied from pinned host memory, the graph
    replayed, the logits read back to pinned host memory;
  * the CPU oracle on a bounded row sample of the same step, one core.

--impl reference times the CPU oracle alone, as the reference arm.
Multi-GPU: replicas only (the decode step does not shard here); under torchrun
every rank runs its own replica and rank 0 reports the aggregate.
"""

from __future__ import annotations

import argparse
import ctypes
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

METRIC = "M=1 qmv achieved HBM GB/s (% of peak); qmm TFLOP/s at M=2048; tokens/s eq"
UNIT = "tokens/s-eq"
WORKLOAD = ("llama-3.2-1b-shaped decode step: 16 x (q 2048x2048, k 512x2048, v 512x2048, "
            "o 2048x2048, gate 8192x2048, up 8192x2048, down 2048x8192) + lm_head "
            "128256x2048; M=1; 8-bit codes, group 64; f16 activations/scales/biases; "
            "q/k/v and gate/up stored fused (65 dependent launches); each launch's input is an "
            "earlier launch's output; launches overlapped with programmatic dependent launch; "
            "one CUDA graph")
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


# ------------------------------------------------------------------- helpers
def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        out = {k: float(d[k]) for k in ("hbm_gbs", "bf16_tflops") if k in d}
        out["bf16_tflops_sustained"] = float(d.get("bf16_tflops_sustained",
                                                   out.get("bf16_tflops", 0)))
        if "hbm_gbs" in out and "bf16_tflops" in out:
            out["source"] = "measured"
            return out
    except (OSError, ValueError, KeyError):
        pass
    return dict(FALLBACK_PEAKS, source="fallback")


# sources of qmv_kernel: a recorded traffic figure is used only while they are
# byte-identical to the ones the capture was taken with
QMV_SOURCES = ("qmv.cu", "qmv_core.cuh", "device_common.cuh", "sm100_ptx.cuh")


def sources_sha256(sources) -> str:
    """SHA-256 over the named kernel sources, concatenated in order."""
    h = hashlib.sha256()
    for name in sources:
        with open(os.path.join(ROOT, "int8_qmv_qmm_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()


def profile_traffic(profile_name: str, sources):
    """DRAM bytes per launch recorded by an ncu capture under profiles/, or
    None when absent or when the kernel's sources changed since the capture."""
    prof = os.path.join(ROOT, "profiles", profile_name)
    try:
        fields = {}
        with open(prof) as f:
            for line in f:
                if ":" in line and line.strip().startswith(("traffic_bytes_per_launch",
                                                            "source_sha256")):
                    k, v = line.split(":", 1)
                    fields[k.strip()] = v.strip()
        if fields.get("source_sha256") != sources_sha256(sources):
            return None
        return float(fields["traffic_bytes_per_launch"])
    except (OSError, KeyError, ValueError):
        return None


class ClockSampler:
    """Samples SM clock / throttle reasons through NVML (ctypes) in a thread;
    falls back to an `nvidia-smi -lms` subprocess.  Reads settings only."""

    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown",
               0x2: "applications_clocks_setting", 0x1: "gpu_idle"}

    def __init__(self, pci_bus_id: str | None, index: int = 0):
        self.samples, self.reasons_mask, self.max_mhz = [], 0, None
        self._stop = threading.Event()
        self._nvml = None
        self._handle = None
        self._proc = None
        try:
            nv = ctypes.CDLL("libnvidia-ml.so.1")
            if nv.nvmlInit_v2() != 0:
                raise OSError("nvmlInit failed")
            h = ctypes.c_void_p()
            ok = False
            if pci_bus_id:
                ok = nv.nvmlDeviceGetHandleByPciBusId_v2(pci_bus_id.encode(),
                                                         ctypes.byref(h)) == 0
            if not ok and nv.nvmlDeviceGetHandleByIndex_v2(index, ctypes.byref(h)) != 0:
                raise OSError("no NVML handle")
            self._nvml, self._handle = nv, h
            mx = ctypes.c_uint()
            if nv.nvmlDeviceGetMaxClockInfo(h, 1, ctypes.byref(mx)) == 0:
                self.max_mhz = mx.value
        except OSError:
            self._nvml = None

    def _loop(self):
        nv, h = self._nvml, self._handle
        clk, rs = ctypes.c_uint(), ctypes.c_ulonglong()
        get_reasons = getattr(nv, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            getattr(nv, "nvmlDeviceGetCurrentClocksThrottleReasons")
        while not self._stop.is_set():
            if nv.nvmlDeviceGetClockInfo(h, 1, ctypes.byref(clk)) == 0:
                self.samples.append(clk.value)
            if get_reasons(h, ctypes.byref(rs)) == 0:
                self.reasons_mask |= rs.value
            time.sleep(0.002)

    def __enter__(self):
        if self._nvml is not None:
            self._thread = threading.Thread(target=self._loop, daemon=True)
            self._thread.start()
        else:
            try:
                self._proc = subprocess.Popen(
                    ["nvidia-smi", "--query-gpu=clocks.sm,clocks.max.sm,"
                     "clocks_event_reasons.active", "--format=csv,noheader,nounits",
                     "-lms", "50", "-i", "0"], stdout=subprocess.PIPE, text=True)
            except OSError:
                self._proc = None
        return self

    def __exit__(self, *exc):
        if self._nvml is not None:
            self._stop.set()
            self._thread.join()
        elif self._proc is not None:
            self._proc.terminate()
            out, _ = self._proc.communicate()
            for line in out.splitlines():
                parts = [p.strip() for p in line.split(",")]
                try:
                    self.samples.append(int(parts[0]))
                    self.max_mhz = int(parts[1])
                    self.reasons_mask |= int(parts[2], 16)
                except (ValueError, IndexError):
                    pass

    def summary(self):
        reasons = [name for bit, name in self.REASONS.items()
                   if self.reasons_mask & bit and name != "gpu_idle"]
        return {"sm_mhz": statistics.median(self.samples) if self.samples else None,
                "sm_max_mhz": self.max_mhz, "samples": len(self.samples),
                "reasons": reasons}


def dist_setup(n_gpus: int):
    import torch
    world = int(os.environ.get("WORLD_SIZE", "1"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        dist.init_process_group(backend=backend)
        rank = dist.get_rank()
        local = int(os.environ.get("LOCAL_RANK", rank))
        return dist, rank, world, local
    return None, 0, 1, 0


def max_over_ranks(dist, value: float, device):
    if dist is None:
        return value
    import torch
    t = torch.tensor([value], dtype=torch.float64,
                     device=device if dist.get_backend() == "nccl" else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def replica_throughput(world: int, steps: int, t_max: float) -> float:
    """Whole-job steps per second: every rank ran `steps` independent steps;
    the job took as long as its slowest rank."""
    return world * steps / t_max


def barrier(dist):
    if dist is not None:
        dist.barrier()


# ---------------------------------------------------------- CPU oracle leg
# The oracle's per-token work for the decode step (unpack, exact dequant in
# float64, float64 matmul) on the host cores.  The rows of every linear are
# cut into the generator's 1024-row blocks, dealt to N worker processes
# (spawned, one BLAS thread each) so that each holds about the same number of
# weights; a step sends every worker "go" and ends when the last one is done.
# Generating and quantising the weights (load-time work) is not timed.

def _step_shapes():
    from int8_qmv_qmm_gb300 import synthetic as S
    shapes = [(n, k) for _ in range(S.LLAMA_1B_LAYERS) for (_, n, k) in S.LLAMA_1B_LINEARS]
    shapes.append(S.LLAMA_1B_LM_HEAD[1:])
    return shapes


def oracle_partition(n_workers: int, block: int = 1024):
    """Work units (linear index, N, K, first row, end row) per worker:
    row blocks, largest first, each to the least-loaded worker."""
    units = []
    for idx, (n, k) in enumerate(_step_shapes()):
        for r0 in range(0, n, block):
            units.append((idx, n, k, r0, min(n, r0 + block)))
    units.sort(key=lambda u: -(u[4] - u[3]) * u[2])
    load = [0] * n_workers
    parts = [[] for _ in range(n_workers)]
    for u in units:
        w = min(range(n_workers), key=lambda i: load[i])
        parts[w].append(u)
        load[w] += (u[4] - u[3]) * u[2]
    return parts


def _oracle_worker(conn, units, stride):
    """Worker process: prepares its rows (every `stride`-th row of each unit),
    then, per message `skip` (0 ends), runs one pass of the per-token work over
    every `skip`-th prepared unit and sends back (seconds, weights done)."""
    import numpy as np

    from int8_qmv_qmm_gb300 import synthetic as S
    from oracle import qlin_oracle as O
    prepared = []
    for idx, n, k, r0, r1 in units:
        rows = np.arange(r0, r1)
        rows = rows[rows % stride == 0]
        if rows.size == 0:
            continue
        w = S.weights_f32(S.weight_seed(2, idx), n, k, rows=rows, threads=1)
        codes, scale, bias = O.quantize_affine(w, 8, 64, "f16")
        x = S.activations(S.weight_seed(2, idx), 1, k, "f16").float().numpy()
        prepared.append((O.pack(codes, 8), scale, bias, x, k, rows.size))
    conn.send(True)
    while True:
        skip = conn.recv()
        if not skip:
            break
        t0 = time.perf_counter()
        done = 0
        for words, scale, bias, x, k, nrows in prepared[::skip]:
            codes = O.unpack(words, 8, k)
            w_hat = O.dequant_exact(codes, scale, bias, 64)
            O.matmul_ref(x, w_hat)
            done += nrows * k
        conn.send((time.perf_counter() - t0, done))
    conn.close()


def oracle_steps_child(n_workers: int, stride: int, warmup: int, steps: int,
                       budget_s: int) -> dict:
    """Runs in a child process without a GPU: starts the workers, runs one
    whole pass over the prepared rows as the first warm-up, and, if whole
    passes would not fit `warmup - 1 + steps` times into `budget_s` seconds,
    makes each further pass cover every `skip`-th row block only.  Returns the
    timed passes and the share of the step's weights each covered."""
    import math
    import multiprocessing as mp
    ctx = mp.get_context("spawn")
    parts = oracle_partition(n_workers)
    procs, conns = [], []
    for part in parts:
        a, b = ctx.Pipe()
        pr = ctx.Process(target=_oracle_worker, args=(b, part, stride), daemon=True)
        pr.start()
        procs.append(pr)
        conns.append(a)
    for c in conns:
        c.recv()

    def one_pass(skip):
        t0 = time.perf_counter()
        for c in conns:
            c.send(skip)
        done = sum(c.recv()[1] for c in conns)
        return time.perf_counter() - t0, done

    skip = 1
    t_first, _ = one_pass(1)
    if t_first * (max(warmup - 1, 0) + steps) > budget_s:
        skip = math.ceil(t_first * (max(warmup - 1, 0) + steps) / budget_s)
    for _ in range(max(warmup - 1, 0)):
        one_pass(skip)
    times, done = [], 0
    for _ in range(steps):
        t, done = one_pass(skip)
        times.append(t)
    for c in conns:
        c.send(0)
    for pr in procs:
        pr.join(timeout=60)
    total = sum(n * k for n, k in _step_shapes())
    return {"times": times, "fraction": done / total, "workers": n_workers, "skip": skip,
            "row_stride": stride, "first_pass_s": t_first}


def host_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def run_oracle(n_workers: int, stride: int, warmup: int, steps: int, budget_s: int) -> dict:
    env = dict(os.environ, OMP_NUM_THREADS="1", OPENBLAS_NUM_THREADS="1",
               MKL_NUM_THREADS="1", CUDA_VISIBLE_DEVICES="")
    r = subprocess.run([sys.executable, os.path.abspath(__file__), "--oracle-child",
                        str(n_workers), str(stride), str(warmup), str(steps), str(budget_s)],
                       env=env, stdout=subprocess.PIPE, stderr=subprocess.PIPE, text=True,
                       timeout=3600)
    if r.returncode != 0:
        raise RuntimeError(f"oracle child failed: {r.stderr[-2000:]}")
    res = json.loads(r.stdout.strip().splitlines()[-1])
    frac, times = res["fraction"], res["times"]
    per_pass = sum(times) / len(times)
    if frac >= 0.999999:
        what = "whole decode steps (all 113 linears, every output row)"
    else:
        what = (f"{frac * 100:.2f}% of the decode step's weights per pass (every "
                f"{res['row_stride']}th row, every {res['skip']}th block of 1024 rows; a whole "
                f"step took {res['first_pass_s']:.2f} s); tokens/s-eq extrapolated from that share")
    return {"value": frac / per_pass, "fraction": frac, "times": times, "s_per_pass": per_pass,
            "extrapolated": frac < 0.999999,
            "sample": (f"{what}: unpack + exact dequant + f64 matmul, rows dealt to "
                       f"{n_workers} worker process(es) with one BLAS thread each, "
                       f"{len(times)} timed pass(es) of {per_pass:.2f} s")}


def run_oracle_baseline() -> dict:
    """cpu_baseline: two whole decode steps on every host core, and beside it
    one core on every 16th row (extrapolated)."""
    cores = host_cores()
    r = run_oracle(cores, 1, 1, 2, budget_s=30)
    one = run_oracle(1, 16, 1, 1, budget_s=10)
    return {"value": r["value"], "unit": UNIT, "cores": cores, "kind": "oracle",
            "sample": r["sample"],
            "one_core": {"value": one["value"], "unit": UNIT, "cores": 1,
                         "sample": one["sample"]}}


# ------------------------------------------------------------- GPU legs
def flush_l2(buf):
    """Write a buffer larger than L2, then read half of it back: L2 ends up
    holding clean lines, so the write-back of the flush's dirty lines does not
    land inside the next timed launch."""
    buf.add_(1.0)
    buf[: buf.numel() // 2].sum()


def l2_bytes(device) -> int:
    import torch
    return int(getattr(torch.cuda.get_device_properties(device), "L2_cache_size", 0)) or 132 << 20


def rotation_sets(bytes_per_set: int, device) -> int:
    """Distinct input sets whose total is 2.5x the L2 size (at least 3)."""
    return max(3, -(-int(2.5 * l2_bytes(device)) // max(1, bytes_per_set)))


def time_rotating(launch, sets: int, device, reps: int = 5) -> float:
    """Mean GPU seconds per launch of launch(i), i = 0 .. sets-1, each on its
    own inputs and outputs (together larger than L2, so no launch finds its
    operands there), run back to back in one CUDA graph replayed `reps`
    times between two CUDA events on the launching stream."""
    import torch
    stream = torch.cuda.current_stream(device)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for i in range(sets):
            launch(i)
    for _ in range(2):
        g.replay()
    torch.cuda.synchronize(device)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(reps):
        g.replay()
    e1.record(stream)
    torch.cuda.synchronize(device)
    del g
    return e0.elapsed_time(e1) * 1e-3 / (reps * sets)


def _replicas(t, sets):
    return [t] + [t.clone() for _ in range(sets - 1)]


def time_qmm(q, device, peaks):
    """Tensor-core qmm on the prefill shapes (M = 512 and 2048): launches back
    to back over rotating copies of the operands (2.5x the L2 size in all),
    in one CUDA graph; and, as a diagnostic, the median of single launches
    with L2 flushed before each."""
    import torch

    from int8_qmv_qmm_gb300 import synthetic as S
    flush = torch.empty(512 * 1024 * 1024 // 4, dtype=torch.float32, device=device)
    rows = []
    cases = [(m, b, nk) for m in (2048, 512) for b in (4, 8)
             for nk in ((8192, 2048), (2048, 8192), (2048, 2048))]
    for m, bits, (n, k) in cases:
        w = torch.from_numpy(S.weights_f32(S.weight_seed(4, n + k + bits), n, k)).to(device)
        wq, sc, bi = q.quantize_affine(w, bits, sdtype=torch.float16)
        del w
        x = S.activations(4, m, k, "f16", outlier_frac=0.01).to(device)
        y = torch.empty((m, n), dtype=torch.float16, device=device)
        per_set = (x.numel() + y.numel() + 2 * sc.numel()) * 2 + wq.numel() * 4
        sets = rotation_sets(per_set, device)
        xs, wqs, scs, bis, ys = (_replicas(t, sets) for t in (x, wq, sc, bi, y))
        t = time_rotating(lambda i: q.qmm(xs[i], wqs[i], scs[i], bis[i], bits, out=ys[i]),
                          sets, device)
        # the same launches as programmatic dependent launches (qlin_qmm_ex), as
        # a chain of prefill linears would issue them: each kernel's set-up
        # overlaps the previous one's tail
        t_pdl = time_rotating(lambda i: q.qmm(xs[i], wqs[i], scs[i], bis[i], bits, out=ys[i],
                                              overlap_previous=i > 0), sets, device)
        del xs, wqs, scs, bis, ys
        t_iso = time_flushed(lambda: q.qmm(x, wq, sc, bi, bits, out=y), device, flush, reps=30)
        flops = 2.0 * m * n * k
        rows.append({"m": m, "n": n, "k": k, "bits": bits, "us": t * 1e6,
                     "tflops": flops / t / 1e12, "rotating_sets": sets,
                     "overlapped_us": t_pdl * 1e6, "overlapped_tflops": flops / t_pdl / 1e12,
                     "isolated_flushed_us": t_iso * 1e6})
    del flush
    torch.cuda.empty_cache()
    best = max(r["tflops"] for r in rows)
    mean = statistics.mean(r["tflops"] for r in rows)
    worst = min(r["tflops"] for r in rows)
    return {
        "tflops_mean": mean, "tflops_best": best, "tflops_worst": worst, "cases": rows,
        "timing": "us = GPU time per launch, launches back to back over rotating operand "
                  "copies (2.5x L2) in one CUDA graph (the roofline uses these); overlapped_us "
                  "= the same as programmatic dependent launches (qlin_qmm_ex), as a chain "
                  "of prefill linears issues them; isolated_flushed_us = median of single "
                  "launches after an L2 flush (event overhead included)",
        "overlapped_tflops_mean": statistics.mean(r["overlapped_tflops"] for r in rows),
        "roofline": {"bound": "tensor", "achieved": mean, "peak": peaks["bf16_tflops"],
                     "unit": "TFLOP/s", "frac": mean / peaks["bf16_tflops"],
                     "frac_worst": worst / peaks["bf16_tflops"],
                     "traffic": None,
                     "note": f"f16 MMA; peak = dense bf16 burst ({peaks['source']}), "
                             "f16/bf16 nominal ratio 1"},
    }


# the batched-decode sweep's token counts: the workload's 1, 2, 4, 8, 16, 32 and
# the counts around qmv's 4-token tiles
SWEEP_M = (1, 2, 3, 4, 5, 6, 8, 12, 16, 32)


def crossover_sweep(q, device):
    """qmv vs qmm on the batched-decode sweep (M = 1..32, 4-bit, bf16 as the
    workload has it, and f16; also M = 3, 5, 6, 12 around qmv's 4-token
    tiles), each timed back to back over rotating operand
    copies (2.5x the L2 size); per dtype the crossover is the smallest M from
    which qmm is at least as fast on every shape, next to the library's
    choice."""
    import torch

    from int8_qmv_qmm_gb300 import synthetic as S
    out = {}
    for dt, tdt in (("bf16", torch.bfloat16), ("f16", torch.float16)):
        table = []
        for (n, k) in ((8192, 2048), (2048, 8192)):
            w = torch.from_numpy(S.weights_f32(S.weight_seed(3, n), n, k)).to(device)
            wq, sc, bi = q.quantize_affine(w, 4, sdtype=tdt)
            del w
            sets = rotation_sets(wq.numel() * 4 + 2 * sc.numel() * 2, device)
            wqs, scs, bis = (_replicas(t, sets) for t in (wq, sc, bi))
            for m in SWEEP_M:
                x = S.activations(3, m, k, dt).to(device)
                y = torch.empty((m, n), dtype=tdt, device=device)
                row = {"n": n, "k": k, "m": m}
                for name in ("qmv", "qmm"):
                    fn = getattr(q, name)
                    t = time_rotating(lambda i: fn(x, wqs[i], scs[i], bis[i], 4, out=y), sets,
                                      device)
                    row[name + "_us"] = t * 1e6
                row["packed_gbs_qmv"] = (wq.numel() * 4 + 2 * sc.numel() * 2) / row["qmv_us"] / 1e3
                row["library_picks"] = "qmm" if m >= q.crossover_m(n, k, 4, tdt) else "qmv"
                table.append(row)
            del wqs, scs, bis
        cross = None
        for m in SWEEP_M:
            if all(r["qmm_us"] <= r["qmv_us"] for r in table if r["m"] == m):
                cross = m
                break
        out[dt] = {"crossover_m": cross, "table": table,
                   "timing": "back to back over rotating weight copies (2.5x L2), one graph"}
    return out


def time_flushed(fn, device, flush, reps: int = 100, warm: int = 10):
    """Median GPU time of fn() (one or more launches on the current stream),
    L2 flushed before each timed repetition, host enqueue hidden behind a GPU
    sleep."""
    import torch
    stream = torch.cuda.current_stream(device)
    for _ in range(warm):
        fn()
    ts = []
    for _ in range(reps):
        flush_l2(flush)
        torch.cuda._sleep(100000)
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        fn()
        e1.record(stream)
        e1.synchronize()
        ts.append(e0.elapsed_time(e1) * 1e-3)
    return statistics.median(ts)


def small_workloads(q, device, peaks):
    """The two M = 1 workloads below the L2 size, each timed over rotating
    copies of its weights (2.5x the L2 size, back to back in one CUDA graph)
    and, as a diagnostic, as single launches after an L2 flush (median; event
    overhead included): the single 300 x 512 qmv (4-bit) and one
    Llama-3.2-1B decoder layer's seven linears (4-bit).  The layer is timed as
    the decode step runs it (q/k/v and gate/up fused, 4 overlapped launches;
    rotating = 8 distinct layers chained in one graph, time per layer) and as
    seven separate launches."""
    import torch

    from int8_qmv_qmm_gb300 import synthetic as S
    from int8_qmv_qmm_gb300.decode_step import DecodeStep
    flush = torch.empty(512 * 1024 * 1024 // 4, dtype=torch.float32, device=device)
    hbm = peaks["hbm_gbs"]

    def rec(t, t_iso, b, **extra):
        return dict(extra, us=t * 1e6, algorithmic_bytes=b, gbs=b / t / 1e9,
                    frac=b / t / 1e9 / hbm, isolated_flushed_us=t_iso * 1e6)

    out = {"timing": "us: back to back over rotating weight copies (2.5x L2) in one CUDA "
                     "graph; isolated_flushed_us: median single launch after an L2 flush"}
    # single qmv: M = 1, K = 512, N = 300 (N not a multiple of 4)
    w = torch.from_numpy(S.weights_f32(0, 300, 512)).to(device)
    wq, sc, bi = q.quantize_affine(w, 4, sdtype=torch.float16)
    x = S.activations(0, 1, 512, "f16").to(device)
    y = torch.empty((1, 300), dtype=torch.float16, device=device)
    b = wq.numel() * 4 + 2 * sc.numel() * 2 + (512 + 300) * 2
    sets = rotation_sets(b, device)
    wqs, scs, bis = (_replicas(t, sets) for t in (wq, sc, bi))
    t = time_rotating(lambda i: q.qmv(x, wqs[i], scs[i], bis[i], 4, out=y), sets, device)
    del wqs, scs, bis
    t_iso = time_flushed(lambda: q.qmv(x, wq, sc, bi, 4, out=y), device, flush)
    out["single_qmv_300x512_4bit"] = rec(t, t_iso, b, rotating_sets=sets)
    # one decoder layer, 4-bit, as the decode step runs it: 8 distinct layers
    # chained (rotating), and one layer alone (flushed)
    chained = DecodeStep(device, bits=4, dtype=torch.float16, seed=1, layers=8, lm_head=False)
    chained.x0.copy_(S.activations(1, 1, 2048, "f16").to(device))
    chained.capture()
    for _ in range(2):
        chained.replay()
    torch.cuda.synchronize(device)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(20):
        chained.replay()
    e1.record()
    torch.cuda.synchronize(device)
    t8 = e0.elapsed_time(e1) * 1e-3 / 20 / 8
    b = sum(chained.algorithmic_bytes()) / 8
    del chained
    layer = DecodeStep(device, bits=4, dtype=torch.float16, seed=1, layers=1, lm_head=False)
    layer.x0.copy_(S.activations(1, 1, 2048, "f16").to(device))
    layer.capture()
    t_iso = time_flushed(layer.replay, device, flush)
    res = {"fused_4_launches_graph": rec(t8, t_iso, b, rotating="8 distinct layers chained")}
    per = {}
    for i, (name, n, k) in enumerate(S.LLAMA_1B_LINEARS):
        _, _, _, _, lwq, lsc, lbi, wseed = layer.linear_rows(i)
        lwq, lsc, lbi = lwq.contiguous(), lsc.contiguous(), lbi.contiguous()
        xx = S.activations(wseed, 1, k, "f16").to(device)
        yy = torch.empty((1, n), dtype=torch.float16, device=device)
        b = lwq.numel() * 4 + 2 * lsc.numel() * 2 + (k + n) * 2
        sets = rotation_sets(b, device)
        wqs, scs, bis = (_replicas(tt, sets) for tt in (lwq, lsc, lbi))
        t = time_rotating(lambda j: q.qmv(xx, wqs[j], scs[j], bis[j], 4, out=yy), sets, device)
        del wqs, scs, bis
        t_iso = time_flushed(lambda: q.qmv(xx, lwq, lsc, lbi, 4, out=yy), device, flush)
        per[name] = rec(t, t_iso, b, n=n, k=k, rotating_sets=sets)
    res["separate_launches"] = per
    out["decoder_layer_4bit"] = res
    del layer, flush
    torch.cuda.empty_cache()
    return out


def per_launch_durations(step, device, reps: int = 3):
    """Diagnostic: each launch of the step alone, bracketed by CUDA events on
    its stream.  A GPU
    sleep is queued first so that the host enqueues every launch and event
    before the GPU reaches them: the events then time the kernels back to back
    (as in the graph), not the host's launch latency.  The launches here are
    plain stream-ordered ones (no overlap), so each duration is the kernel's
    own."""
    import torch
    stream = torch.cuda.current_stream(device)
    n = step.n_launches
    sums = [0.0] * n
    saved = step.overlap
    step.overlap = False
    for _ in range(reps):
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(n)]

        def hook(i, when):
            ev[i][0 if when == "before" else 1].record(stream)

        torch.cuda._sleep(int(2e7))  # ~10 ms at 2 GHz, longer than enqueuing the step
        step.launch_all(per_launch_hook=hook)
        torch.cuda.synchronize(device)
        for i in range(n):
            sums[i] += ev[i][0].elapsed_time(ev[i][1]) * 1e-3
    step.overlap = saved
    return [s / reps for s in sums]


def per_shape_summary(step, durs, alg):
    """Mean duration and GB/s of the launches of each fused shape."""
    out = {}
    for u, d, b in zip(step.units, durs, alg):
        e = out.setdefault(u["name"], {"n": u["N"], "k": u["K"], "launches": 0, "us": 0.0,
                                       "bytes": 0})
        e["launches"] += 1
        e["us"] += d * 1e6
        e["bytes"] += b
    for e in out.values():
        e["gbs"] = e["bytes"] / (e["us"] * 1e-6) / 1e9
        e["us"] /= e["launches"]
        del e["bytes"]
    return out


def time_eager(fn, device, reps: int = 5):
    """Mean GPU duration of fn() (one or more launches on the current stream),
    events recorded after a GPU sleep so that host enqueue time is excluded."""
    import torch
    stream = torch.cuda.current_stream(device)
    tot = 0.0
    for _ in range(reps):
        torch.cuda._sleep(int(2e7))
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        fn()
        e1.record(stream)
        e1.synchronize()
        tot += e0.elapsed_time(e1) * 1e-3
    return tot / reps


def time_graph_steps(step, steps, device, dist=None):
    import torch
    stream = torch.cuda.current_stream(device)
    barrier(dist)
    torch.cuda.synchronize(device)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(steps):
        step.replay()
    e1.record(stream)
    torch.cuda.synchronize(device)
    barrier(dist)
    return e0.elapsed_time(e1) * 1e-3


def qmm_chain_timing(q, device, m: int = 512, layers: int = 4, reps: int = 50):
    """A prefill-like chain of dependent qmm launches (o 2048x2048, gate
    8192x2048, down 2048x8192 per layer, 4-bit, M tokens; each output is the
    next input), in one CUDA graph, plain and with QLIN_OVERLAP_PREVIOUS.
    The weights (about 40 MB) stay in L2 across replays: this measures the
    launch overlap, not HBM."""
    import torch

    from int8_qmv_qmm_gb300 import synthetic as S
    dims = [(2048, 2048), (8192, 2048), (2048, 8192)] * layers
    ws = []
    for i, (n, k) in enumerate(dims):
        w = torch.from_numpy(S.weights_f32(S.weight_seed(9, i), n, k)).to(device)
        ws.append(q.quantize_affine(w, 4, sdtype=torch.float16))
        del w
    x0 = (S.activations(9, m, 2048, "f16") * 0.05).to(device)
    outs = [torch.empty((m, n), dtype=torch.float16, device=device) for n, _ in dims]
    res = {"links": len(dims), "m": m, "note": "L2-warm; 4-bit; o, gate, down per layer"}
    for overlap in (False, True):
        def run():
            x = x0
            for i, (wq, sc, bi) in enumerate(ws):
                x = q.qmm(x, wq, sc, bi, 4, out=outs[i], overlap_previous=overlap and i > 0)
        run()
        torch.cuda.synchronize(device)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            run()
        for _ in range(3):
            g.replay()
        torch.cuda.synchronize(device)
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        torch.cuda._sleep(20_000_000)
        e0.record()
        for _ in range(reps):
            g.replay()
        e1.record()
        torch.cuda.synchronize(device)
        us = e0.elapsed_time(e1) * 1e3 / reps
        flops = sum(2.0 * m * n * k for n, k in dims)
        res["overlap_us" if overlap else "plain_us"] = us
        res["overlap_tflops" if overlap else "plain_tflops"] = flops / us / 1e6
        del g
    return res


def dense_f16_step(step, device, steps: int):
    """The same decode step with every weight resident as dense f16 (built
    once with qlin_dequant, outside the timed region) and each linear run as
    torch.matmul (cuBLAS): the unfused f16 path the packed kernels replace.
    Same chaining, one CUDA graph, same number of replays."""
    import torch

    from int8_qmv_qmm_gb300.decode_step import DenseF16Step
    dense = DenseF16Step(step)
    dense.capture()
    for _ in range(3):
        dense.replay()
    torch.cuda.synchronize(device)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    torch.cuda._sleep(20_000_000)
    e0.record()
    for _ in range(steps):
        dense.replay()
    e1.record()
    torch.cuda.synchronize(device)
    t = e0.elapsed_time(e1) * 1e-3 / steps
    dense_bytes = dense.weight_bytes()
    del dense
    torch.cuda.empty_cache()
    return {"tokens_per_s": 1.0 / t, "ms_per_step": t * 1e3, "weight_bytes": dense_bytes,
            "gbs": dense_bytes / t / 1e9, "how": "dense f16 weights, torch.matmul (cuBLAS), "
            "one CUDA graph of the same 65 chained linears"}


def bench_ours(args):
    import torch

    import int8_qmv_qmm_gb300 as q
    from int8_qmv_qmm_gb300 import build_lib
    from int8_qmv_qmm_gb300.decode_step import DecodeStep

    dist, rank, world, local = dist_setup(args.gpus)
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    if rank == 0 or dist is None:
        build_lib.build()
    barrier(dist)
    q.lib()
    peaks = load_peaks()

    step = DecodeStep(device, bits=8, dtype=torch.float16, seed=2, mode="launches")
    x_host = torch.randn((1, 2048), generator=torch.Generator().manual_seed(0)).to(
        torch.float16).pin_memory()
    step.x0.copy_(x_host)
    step.capture()
    stream = torch.cuda.current_stream(device)
    for _ in range(args.warmup):
        step.replay()
    torch.cuda.synchronize(device)

    props = torch.cuda.get_device_properties(device)
    pci = None
    if hasattr(props, "pci_bus_id"):
        pci = "%08x:%02x:%02x.0" % (getattr(props, "pci_domain_id", 0), props.pci_bus_id,
                                    props.pci_device_id)
    # ---- timed region: exactly `steps` graph replays (65 overlapped launches each)
    sampler = ClockSampler(pci)
    with sampler:
        t_local = time_graph_steps(step, args.steps, device, dist)
    t = max_over_ranks(dist, t_local, device)
    per_step = t / args.steps
    value = replica_throughput(world, args.steps, t)

    # ---- the dominant kernel (qmv): its launches are the whole graph, so its
    # average launch duration over the timed region is per_step / launches
    alg_list = step.algorithmic_bytes()
    alg = sum(alg_list)
    achieved = alg / per_step / 1e9
    # diagnostic: each launch alone (no overlap), CUDA events around it
    durs = per_launch_durations(step, device)
    top = max(range(step.n_launches), key=lambda i: durs[i])

    # ---- the same step as one persistent chain launch (qlin_qmv_chain), for comparison
    step.mode = "chain"
    step.capture()
    for _ in range(3):
        step.replay()
    t_c = time_graph_steps(step, args.steps, device)
    chain_s = time_eager(step.launch_chain, device)
    step.mode = "launches"
    step.capture()

    # ---- the unfused comparator: the same step on dense f16 weights (cuBLAS)
    dense = dense_f16_step(step, device, args.steps)

    # ---- end to end through the public API with host buffers
    logits_host = torch.empty((1, step.logits.shape[1]), dtype=torch.float16).pin_memory()
    torch.cuda.synchronize(device)
    barrier(dist)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step.x0.copy_(x_host, non_blocking=True)
        step.replay()
        logits_host.copy_(step.logits, non_blocking=True)
        stream.synchronize()
    t_e2e = max_over_ranks(dist, time.perf_counter() - t0, device)
    e2e_value = world * args.steps / t_e2e

    small = small_workloads(q, device, peaks)
    qmm_res = None if args.no_qmm else time_qmm(q, device, peaks)
    qmm_chain = None if args.no_qmm else qmm_chain_timing(q, device)
    cross = None if args.no_qmm else crossover_sweep(q, device)
    status = q.device_status()

    if rank != 0:
        return
    cpu = None if args.no_cpu_baseline else run_oracle_baseline()
    clocks = sampler.summary()
    bytes_step = step.packed_bytes()
    traffic = profile_traffic("qmv_decode_step.txt", QMV_SOURCES)
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": per_step * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f32", "data": "synthetic",
        "config": {"workload": WORKLOAD, "weights": "u8 codes, affine g64, f16 scale/bias",
                   "activations": "f16", "accumulate": "f32",
                   "packed_bytes_per_step": bytes_step,
                   "l2": "inputs larger than L2 (packed weights per step = %.0f MB)"
                         % (bytes_step / 1e6),
                   "parallelism": "replicas" if world > 1 else "single GPU"},
        "qmv_step_gbs": bytes_step / per_step / 1e9,
        "qmv_step_frac_of_peak": bytes_step / per_step / 1e9 / peaks["hbm_gbs"],
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"],
                     "unit": "GB/s", "frac": achieved / peaks["hbm_gbs"], "traffic": traffic,
                     "kernel": "qmv_kernel: the %d launches of a step, which make up the whole "
                               "timed graph; average launch = ms_per_step / %d"
                               % (step.n_launches, step.n_launches),
                     "algorithmic_bytes_per_launch": alg / step.n_launches,
                     "mean_launch_us": per_step / step.n_launches * 1e6,
                     "peak_source": peaks["source"]},
        "isolated_launches": {"note": "diagnostic: each launch of the step alone, no overlap "
                                      "with its neighbours, CUDA events around it",
                              "sum_us": sum(durs) * 1e6,
                              "per_shape": per_shape_summary(step, durs, alg_list),
                              "largest_launch": {"name": step.units[top]["name"],
                                                 "us": durs[top] * 1e6,
                                                 "gbs": alg_list[top] / durs[top] / 1e9}},
        "small_workloads": small,
        "chain_mode": {"tokens_per_s": world * args.steps / t_c,
                       "kernel_us": chain_s * 1e6,
                       "kernel_gbs": alg / chain_s / 1e9},
        "dense_f16_step": dense,
        "dense_f16_tokens_per_s": dense["tokens_per_s"],
        "packed_speedup_vs_dense_f16": value / world / dense["tokens_per_s"],
        "qmm": qmm_res,
        "qmm_chain": qmm_chain,
        "crossover": cross,
        "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": x_host.numel() * 2,
                "d2h_bytes_per_step": logits_host.numel() * 2},
        "gpu_launches": args.steps * step.n_launches,
        "cpu_baseline": cpu,
        "clocks": clocks,
        "device_status": status,
    }
    print(json.dumps(line), flush=True)


def bench_reference(args):
    """The reference arm: the CPU oracle as it stands, on every host core,
    each step one whole decode step of the same workload (all 113 linears,
    every output row)."""
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if world > 1 and rank != 0:
        return
    cores = host_cores()
    r = run_oracle(cores, 1, max(1, args.warmup), args.steps, budget_s=150)
    value = r["value"]
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": r["s_per_pass"] * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": {"workload": WORKLOAD},
        "cpu_baseline": {"kind": "oracle", "cores": cores, "sample": r["sample"],
                         "value": value, "unit": UNIT},
        "sample_fraction": r["fraction"], "value_extrapolated": r["extrapolated"],
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def profile_case(which: str, launches: int = 3):
    """A small fixed case for ncu: `launches` back-to-back launches of one
    kernel on one workload shape (no timing, no oracle).
      qmv: the lm_head of the decode step (M=1, 128256x2048, 8-bit, f16),
           279 MB of packed weights (above the L2 size);
      qmv_qkv / qmv_o / qmv_gate_up / qmv_down: the step's other launch shapes
           (ncu flushes L2 before each captured launch);
      qmm: M=2048, N=8192, K=2048, 4-bit, f16 (the largest prefill case);
      qmm_split: M=512, N=2048, K=8192, 4-bit (K split over 4-CTA clusters)."""
    import torch

    import int8_qmv_qmm_gb300 as q
    from int8_qmv_qmm_gb300 import build_lib
    from int8_qmv_qmm_gb300 import synthetic as S
    build_lib.build()
    dev = torch.device("cuda", 0)
    cases = {"qmv": (1, 128256, 2048, 8, q.qmv), "qmv_qkv": (1, 3072, 2048, 8, q.qmv),
             "qmv_o": (1, 2048, 2048, 8, q.qmv),
             "qmv_gate_up": (1, 16384, 2048, 8, q.qmv), "qmv_down": (1, 2048, 8192, 8, q.qmv),
             "qmm": (2048, 8192, 2048, 4, q.qmm), "qmm8": (2048, 8192, 2048, 8, q.qmm),
             "qmm_sq": (2048, 2048, 2048, 8, q.qmm),
             "qmm_split": (512, 2048, 8192, 4, q.qmm)}
    m, n, k, bits, fn = cases[which]
    w = torch.from_numpy(S.weights_f32(7, n, k)).to(dev)
    wq, sc, bi = q.quantize_affine(w, bits, sdtype=torch.float16)
    del w
    x = S.activations(7, m, k, "f16").to(dev)
    y = torch.empty((m, n), dtype=torch.float16, device=dev)
    for _ in range(launches):
        fn(x, wq, sc, bi, bits, out=y)
    torch.cuda.synchronize()
    print(json.dumps({"profile_case": which, "m": m, "n": n, "k": k, "bits": bits,
                      "launches": launches, "status": q.device_status()}))


def main():
    if len(sys.argv) >= 2 and sys.argv[1] == "--oracle-child":
        print(json.dumps(oracle_steps_child(*(int(v) for v in sys.argv[2:7]))), flush=True)
        return
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-qmm", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--profile", choices=["qmv", "qmv_qkv", "qmv_o", "qmv_gate_up", "qmv_down", "qmm",
                                          "qmm8", "qmm_sq", "qmm_split"],
                    help="run a small fixed case for ncu instead of the benchmark")
    args = ap.parse_args()
    if args.profile:
        profile_case(args.profile)
        return
    if args.warmup < 3 and args.impl == "ours":
        ap.error("--warmup must be >= 3")
    if args.impl == "reference":
        bench_reference(args)
    else:
        bench_ours(args)


if __name__ == "__main__":
    main()
