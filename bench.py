"""Benchmark of the CSA2 decode step (one JSON line on rank 0).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference] [--config 1]

A step is one pass of the whole hot path over one batch: append of the new
token (main KV FP4, indexer key FP8, one FP8 window row per layer), the Full
layer's indexer (scan, pool of 2,048 blocks, top-512), Reindex layers, Reuse
layers, and every layer's sparse attention.  The headline workload is the
decode batch of 32 sequences at 65,536 tokens (one Full + three Reuse layers).
The same run also times, under their own keys: the single Full layer at 4,096
tokens ("cfg0"), the 1M-token 20-layer batch of 4 ("ctx_1m"), the ragged batch
of 64 sessions through the 20-layer pattern ("ragged_b64"), draft verification
("verify") and the chunked-query workload ("chunked").  Each decode line gives
the scan's fraction of the HBM roofline on 68 B per cached position and the
step's fraction on the step's algorithmic bytes, plus a per-call breakdown
(append, Full select, Reindex select, attention).  Inputs are seeded synthetic
data; caches stay resident in HBM.

Multi-GPU: sequences are independent, so each rank runs its own batch (weak
scaling, no collective on the data path); value = all ranks' query-steps over
the slowest rank's time.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "decode query-steps/s and achieved HBM GB/s (% of roofline) at 64K and 1M ctx"
SCAN_BYTES_PER_POS = 68          # algorithmic bytes per cached position: 64 FP8 key bytes + a 4-byte scale
SCAN_SCORE_STORE = 4             # the scan's own per-position score store (scratch, reported apart)
SCAN_SAMPLE_EVERY = 10           # the timed graph times the scan on one step in this many

# DRAM bytes (dram__bytes_read.sum + dram__bytes_write.sum) of one scan launch, from one ncu
# capture of the decode batch, valid only while the scan's sources are the ones captured: the
# digest covers them, and any change reports the traffic as null.
SCAN_NCU_TRAFFIC = {"decode_b32_ctx65536_full+3reuse": 142743808 + 5939200}
SCAN_NCU_SOURCES = ("sparse_attention_fp4_02_b300/csrc/indexer.cu", "sparse_attention_fp4_02_b300/csrc/common.cuh",
                    "sparse_attention_fp4_02_b300/csrc/tcgen05.cuh")
SCAN_NCU_DIGEST = "ea28df0a1d0319d4b3aa4b6446d84560e480f45cb6d2f3b6ebe86e79df77c1eb"


def scan_traffic(workload: str):
    import hashlib
    h = hashlib.sha256()
    for f in SCAN_NCU_SOURCES:
        with open(os.path.join(ROOT, f), "rb") as fh:
            h.update(fh.read())
    return SCAN_NCU_TRAFFIC.get(workload) if h.hexdigest() == SCAN_NCU_DIGEST else None


NOMINAL_HBM_GBS = 8000.0         # HBM3e nominal, reported beside the measured copy bandwidth
FALLBACK_BF16_TFLOPS = 1800.0
FALLBACK_HBM_GBS = 6400.0


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return FALLBACK_HBM_GBS, "fallback"


def peaks_tensor():
    """Dense f16/bf16 tensor peak in TFLOP/s (f16 runs at the bf16 rate): the measured cuBLAS
    burst figure, for a kernel timed on its own."""
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["bf16_tflops"]), "measured"
    return FALLBACK_BF16_TFLOPS, "fallback"


# ------------------------------------------------------------------ clocks

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.path = tempfile.mktemp(suffix=".csv")
        self.proc = None
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                                          "-i", str(gpu_index), "-lms", "50"], stdout=self.f,
                                         stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.f.close()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return {"samples": 0}
        def num(x):
            try:
                return float(x)
            except ValueError:
                return float("nan")
        sm = [num(r[1]) for r in rows]
        mx = [num(r[2]) for r in rows]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": reasons,
                "samples": len(rows), "power_w_max": max(num(r[3]) for r in rows),
                "window": "warm-up and timed steps"}


# ------------------------------------------------------------------ distributed plumbing

def dist_setup(n_gpus: int):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    return world, rank, local


def max_over_ranks(x: float, world: int) -> float:
    """The largest of every rank's x (the slowest rank's time)."""
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def aggregate_rate(units_per_rank: int, world: int, ms_max: float) -> float:
    """Whole-job throughput: the units all ranks processed over the slowest rank's time."""
    return units_per_rank * world / (ms_max / 1e3)


def barrier(world: int):
    import torch
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    if torch.cuda.is_available():
        torch.cuda.synchronize()


# ------------------------------------------------------------------ our arm

def kernels_per_step(wl) -> int:
    from synth.workloads import REINDEX
    n_re = sum(1 for m in wl.schedule if m == REINDEX)
    n_blocks = -(-int(wl.lengths.max()) // wl.block)
    full = 3 if n_blocks <= 16384 else 4            # clear, scan, [collect,] finalize
    if wl.drafts > 1:                               # every indexer layer also runs the verify rows' selection
        n_re += 1
    return 1 + full + 3 * n_re + wl.n_layers        # append, Full select, Reindex (clear, score, select), attention


def measure_workload(cfg, steps: int, warmup: int, world: int, graph_steps: int = 100, breakdown: bool = True):
    """Device time of whole decode steps (CUDA graph of up to graph_steps steps, replayed), the
    scan's own launch time from events recorded inside the graph on its stream, the same step
    end to end with host copies, and optionally a per-call breakdown."""
    import torch
    from sparse_attention_fp4_02_b300.runner import DecodeRunner, StepPipeline
    from synth.workloads import config

    wl = config(cfg) if isinstance(cfg, int) else cfg
    r = DecodeRunner(wl)
    r.build_cache()
    G = max(1, min(graph_steps, steps))
    R = max(1, steps // G)
    steps = R * G
    # events around the scan on every SCAN_SAMPLE_EVERY-th step of the timed graph: an event
    # between the workspace clear and the scan turns their programmatic overlap into a full
    # dependency, so timing every scan would slow every step it samples
    n_ev = (G + SCAN_SAMPLE_EVERY - 1) // SCAN_SAMPLE_EVERY
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n_ev)]
    for a, b in ev:          # torch creates the CUDA event on first record; the library needs the handle
        a.record()
        b.record()
    # one graph holding G steps; the sampled steps record events around the scan kernel
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        r.step()
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    r.check_device_errors()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for i in range(G):
            r.step(prof=ev[i // SCAN_SAMPLE_EVERY] if i % SCAN_SAMPLE_EVERY == 0 else None)
    for _ in range(max(1, math.ceil(warmup / G))):
        g.replay()
    barrier(world)
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0.record()
    for _ in range(R):
        g.replay()
    t1.record()
    barrier(world)
    ms = t0.elapsed_time(t1)
    scan_ms = float(np.mean([a.elapsed_time(b) for a, b in ev]))
    r.check_device_errors()
    ms = max_over_ranks(ms, world)

    # end to end through the public API with host buffers: every step copies its inputs in from
    # pinned host memory and its outputs back, on copy streams that overlap the neighbouring
    # steps' compute (runner.StepPipeline: two alternating sets of step buffers)
    pin = lambda a: torch.from_numpy(np.ascontiguousarray(a)).pin_memory()
    h_in = {"kv_new": pin(r.h_kv_new.view(np.int16)), "ik_new": pin(r.h_ik_new.view(np.int16)),
            "swa_new": pin(r.h_swa_new.view(np.int16)), "q": pin(r.h_q.view(np.int16))}
    for l in r.idx_layers:
        h_in[f"qidx{l}"] = pin(r.h_qidx[l].view(np.int16))
        h_in[f"w{l}"] = pin(r.h_w[l])
    if r.D > 1:                  # the Full layer's own copy of each session's last row
        for l in r.full_layers:
            h_in[f"qidx_last{l}"] = pin(r.h_qidx[l][r.D - 1::r.D].view(np.int16))
            h_in[f"w_last{l}"] = pin(r.h_w[l][r.D - 1::r.D])
    h_out = {"out": torch.empty(r.out.shape, dtype=torch.float32).pin_memory(),
             "lse": torch.empty(r.lse.shape, dtype=torch.float32).pin_memory()}
    h2d = sum(h.numel() * h.element_size() for h in h_in.values())
    d2h = sum(h.numel() * h.element_size() for h in h_out.values())
    n_e2e = min(steps, 2000)
    pipe = StepPipeline(r)

    pipe.begin()
    for _ in range(3):
        pipe.step(h_in, h_out)
    pipe.end()
    barrier(world)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    pipe.begin()
    for _ in range(n_e2e):
        pipe.step(h_in, h_out)
    pipe.end()
    e1.record()
    barrier(world)
    e2e_ms = max_over_ranks(e0.elapsed_time(e1), world)
    r.check_device_errors()
    # the same copies on the compute stream, one step after another: a single batch whose
    # next inputs depend on its own last outputs cannot overlap them
    dev0 = pipe.sets[0]

    def serial_step():
        for name, h in h_in.items():
            d = dev0[name]
            (d.view(torch.int16) if d.dtype == torch.bfloat16 else d).copy_(h, non_blocking=True)
        pipe.graphs[0].replay()
        for name, h in h_out.items():
            h.copy_(dev0[name], non_blocking=True)

    for _ in range(3):
        serial_step()
    barrier(world)
    e0.record()
    for _ in range(n_e2e):
        serial_step()
    e1.record()
    barrier(world)
    serial_ms = max_over_ranks(e0.elapsed_time(e1), world)
    r.check_device_errors()

    parts = r.step_bytes()
    res = {
        "wl": wl, "steps": steps, "ms": ms, "ms_per_step": ms / steps, "value": aggregate_rate(r.T * steps, world, ms),
        "scan_ms": scan_ms, "positions": int(wl.lengths.sum()),
        "scan_bytes": SCAN_BYTES_PER_POS * int(wl.lengths.sum()),
        "step_bytes": parts, "step_bytes_total": int(sum(parts.values())),
        "e2e": {"value": aggregate_rate(r.T * n_e2e, world, e2e_ms), "unit": "query-steps/s",
                "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h), "steps": n_e2e,
                "overlap": "two alternating step-buffer sets (two independent batches in flight)",
                "serial": aggregate_rate(r.T * n_e2e, world, serial_ms)},
        "launches": kernels_per_step(wl) * steps,
        "rows_per_step": r.T,
    }
    del g, pipe
    if breakdown:
        res["breakdown_us"] = measure_breakdown(r)
    del r
    torch.cuda.empty_cache()
    return res


def measure_breakdown(r, reps: int = 20) -> dict:
    """Mean device time per step of each C-ABI call, from events recorded after every call
    inside one captured graph of ``reps`` steps (the events serialise consecutive kernels,
    so the parts add up to a little more than the step)."""
    import torch
    marks = []

    def mark(name):
        e = torch.cuda.Event(enable_timing=True, external=True)
        e.record()
        marks.append((name, e))

    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        r.step()
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    with torch.cuda.graph(g):
        mark("start")
        for _ in range(reps):
            r.step(mark=mark)
    g.replay()
    g.replay()
    torch.cuda.synchronize()
    r.check_device_errors()
    out: dict = {}
    for (_, a), (name, b) in zip(marks[:-1], marks[1:]):
        out[name] = out.get(name, 0.0) + a.elapsed_time(b) * 1e3 / reps
    return {k: round(v, 2) for k, v in out.items()}


def measure_chunked(iters: int = 20, warmup: int = 3):
    """The chunked-query workload (4,096 query rows, 64 heads, 262,144-token cache): the
    chunked-query indexer's call (every row's Full selection), then one sparse_attn_decode
    call per iteration over its top-k lists, device-timed; attention inputs (229 MB) exceed L2."""
    import torch
    from sparse_attention_fp4_02_b300.runner import ChunkedRunner
    from synth.workloads import config

    r = ChunkedRunner(config(3))
    torch.cuda.synchronize()
    r.check_device_errors()
    # the chunked-query indexer (produces the attention's top-k lists)
    n_sel = 3
    r.select()
    torch.cuda.synchronize()
    s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    s0.record()
    for _ in range(n_sel):
        r.select()
    s1.record()
    torch.cuda.synchronize()
    r.check_device_errors()
    sel_ms = s0.elapsed_time(s1) / n_sel
    for _ in range(warmup):
        r.step()
    torch.cuda.synchronize()
    r.check_device_errors()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0.record()
    for _ in range(iters):
        r.step()
    t1.record()
    torch.cuda.synchronize()
    r.check_device_errors()
    us = t0.elapsed_time(t1) / iters * 1e3
    nbytes = r.bytes()
    res = {"workload": r.wl.name, "us_per_call": us, "tflops": r.flops() / (us * 1e-6) / 1e12,
           "gbs": nbytes / (us * 1e-6) / 1e9, "flops_per_call": r.flops(), "bytes_per_call": nbytes,
           "bytes_rule": "unique bytes: distinct gathered rows and window rows once, indices, q, o, lse",
           "iters": iters, "indices": "chunked-query indexer",
           "indexer": {"ms_per_call": sel_ms, "rows": r.wl.n_query, "row_positions": r.positions,
                       "tflops": r.select_flops() / (sel_ms * 1e-3) / 1e12, "iters": n_sel}}
    del r
    torch.cuda.empty_cache()
    return res


def host_cores() -> int:
    return len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else (os.cpu_count() or 1)


def blas_threads() -> int:
    """Threads the oracle's numpy/BLAS calls use on this host."""
    try:
        from threadpoolctl import threadpool_info
        return max([i.get("num_threads", 1) for i in threadpool_info()] + [1])
    except ImportError:
        for var in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS"):
            if os.environ.get(var, "").isdigit():
                return int(os.environ[var])
        return host_cores()


def oracle_step(wl, states, i):
    """One whole decode step of the oracle for sequence i mod len(states): the append of the
    step's new token, then every layer's selection and attention."""
    from oracle import pipeline
    b = i % len(states)
    pipeline.append_token(states[b]["new"])
    pipeline.step(wl, b, states[b])


def cpu_worker(cfg: int, budget_s: float):
    """Runs in a child process whose BLAS libraries were started with one thread: times the
    oracle's whole decode steps single-threaded, then with one worker thread per host core;
    prints one JSON object."""
    from concurrent.futures import ThreadPoolExecutor
    from oracle import pipeline
    from synth.workloads import config

    wl = config(cfg)
    n_prep = max(1, min(wl.B, 4))
    states = [pipeline.prepare(wl, b) for b in range(n_prep)]
    cores = host_cores()
    n, t0 = 0, time.perf_counter()
    while n < n_prep or time.perf_counter() - t0 < budget_s / 2:
        oracle_step(wl, states, n)
        n += 1
    single_s = time.perf_counter() - t0
    single = n / single_s
    per = max(1, math.ceil(single * budget_s / 2))          # steps per worker (~budget/2 at full scaling)
    with ThreadPoolExecutor(cores) as ex:
        t0 = time.perf_counter()
        list(ex.map(lambda w: [oracle_step(wl, states, w + j * cores) for j in range(per)], range(cores)))
        multi_s = time.perf_counter() - t0
    multi = cores * per / multi_s
    print(json.dumps({"value": multi, "unit": "query-steps/s", "cores": cores, "kind": "oracle",
                      "single_thread": {"value": single, "cores": 1, "steps": n, "seconds": round(single_s, 2)},
                      "all_cores": {"value": multi, "cores": cores, "steps": cores * per,
                                    "seconds": round(multi_s, 2)},
                      "sample": f"whole decode steps (append + every layer) of {n_prep} of the {wl.B} sequences of "
                                f"{wl.name}, cycled; single-threaded ({n} steps, {single_s:.1f} s) and {cores} "
                                f"worker threads with one BLAS thread each ({cores * per} steps, {multi_s:.1f} s); "
                                f"cache preparation excluded"}), flush=True)


def cpu_baseline(cfg: int, budget_s: float = 10.0):
    """The oracle as it stands on this host's cores, in a child process (one BLAS thread per
    worker thread, set before its libraries start)."""
    env = dict(os.environ)
    for var in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS", "BLIS_NUM_THREADS"):
        env[var] = "1"
    env["CUDA_VISIBLE_DEVICES"] = ""
    r = subprocess.run([sys.executable, os.path.abspath(__file__), "--cpu-worker", "--config", str(cfg),
                        "--cpu-budget", str(budget_s)], capture_output=True, text=True, env=env, cwd=ROOT)
    if r.returncode != 0:
        return {"value": None, "unit": "query-steps/s", "kind": "oracle", "error": r.stderr[-400:]}
    return json.loads(r.stdout.strip().splitlines()[-1])


def workload_line(res, peak):
    """The per-workload summary: rate, step time, the scan's and the step's roofline fractions."""
    wl = res["wl"]
    a = res["scan_bytes"] / (res["scan_ms"] / 1e3) / 1e9
    step_gbs = res["step_bytes_total"] / (res["ms_per_step"] / 1e3) / 1e9
    return {"workload": wl.name, "value": res["value"], "unit": "query-steps/s",
            "steps_per_s": 1e3 / res["ms_per_step"], "rows_per_step": res["rows_per_step"],
            "ms_per_step": res["ms_per_step"], "us_per_step": res["ms_per_step"] * 1e3, "steps": res["steps"],
            "scan_us": res["scan_ms"] * 1e3, "scan_gbs": a, "scan_frac": a / peak, "scan_frac_nominal": a / NOMINAL_HBM_GBS,
            "step_bytes": res["step_bytes"], "step_gbs": step_gbs, "step_frac": step_gbs / peak,
            "step_frac_nominal": step_gbs / NOMINAL_HBM_GBS,
            "e2e": res["e2e"]["value"], "e2e_serial": res["e2e"]["serial"],
            "h2d_bytes_per_step": res["e2e"]["h2d_bytes_per_step"],
            "d2h_bytes_per_step": res["e2e"]["d2h_bytes_per_step"], "gpu_launches": res["launches"],
            "breakdown_us": res.get("breakdown_us")}


def run_ours(args, world, rank, local):
    peak, peak_kind = peaks()
    clock = ClockSampler(local)
    res = measure_workload(args.config, args.steps, args.warmup, world)
    extra = {}
    if not args.only_headline:
        if args.config != 0:
            extra["cfg0"] = measure_workload(0, args.steps, args.warmup, world)
        if args.config != 2:
            extra["ctx_1m"] = measure_workload(2, max(1, args.steps // 2), args.warmup, world)
        if args.config != 4:
            extra["ragged_b64"] = measure_workload(4, max(1, args.steps // 2), args.warmup, world)
        from synth.workloads import verify_workload
        extra["verify"] = measure_workload(verify_workload(), max(1, args.steps // 2), args.warmup, world,
                                           breakdown=False)
        extra["chunked"] = measure_chunked()
    clocks = clock.stop()
    if rank != 0:
        return
    wl = res["wl"]
    achieved = res["scan_bytes"] / (res["scan_ms"] / 1e3) / 1e9
    head = workload_line(res, peak)
    line = {
        "metric": METRIC, "value": res["value"], "unit": "query-steps/s", "n_gpus": world,
        "steps": res["steps"], "warmup": args.warmup, "ms_per_step": res["ms_per_step"],
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "fp4-e2m1/fp8-e4m3 storage; f16 mma, f32 accumulate",
        "data": "synthetic (seeded N(0,1) bf16 KV with 1% x8 outlier channels, U(0,1) head weights)",
        "config": {"workload": wl.name, "batch": wl.B, "ctx": int(wl.lengths[0]), "layers": wl.schedule,
                   "topk": wl.topk, "pool_blocks": wl.n_keep, "block": wl.block, "window": wl.window,
                   "heads": wl.H, "l2": "inputs larger than L2 (the scan streams "
                                       f"{res['scan_bytes'] / 1e6:.1f} MB of keys per step)",
                   "parallelism": f"replicas x{world} (one batch per GPU)"},
        "roofline": {"bound": "hbm", "kernel": "indexer scan", "achieved": achieved, "peak": peak,
                     "unit": "GB/s", "frac": achieved / peak, "peak_source": peak_kind,
                     "frac_nominal": achieved / NOMINAL_HBM_GBS,
                     "bytes_per_unit": SCAN_BYTES_PER_POS, "units": res["positions"],
                     "algorithmic_bytes": res["scan_bytes"],
                     "traffic": scan_traffic(wl.name),
                     "traffic_extra": SCAN_SCORE_STORE * res["positions"],
                     "scan_us": res["scan_ms"] * 1e3,
                     "step_bytes": head["step_bytes"], "step_frac": head["step_frac"],
                     "step_frac_nominal": head["step_frac_nominal"]},
        "e2e": {k: v for k, v in res["e2e"].items() if k != "steps"},
        "gpu_launches": res["launches"],
        "breakdown_us": res.get("breakdown_us"),
        "clocks": clocks,
    }
    if "kv_append_fp4" in (res.get("breakdown_us") or {}):
        line["append_us"] = res["breakdown_us"]["kv_append_fp4"]
    for key in ("cfg0", "ctx_1m", "ragged_b64", "verify"):
        if key in extra:
            line[key] = workload_line(extra[key], peak)
    if "verify" in line:
        line["verify"]["unit"] = "verified-rows/s"
    if "ragged_b64" in line:
        line["ragged_b64"]["batch_steps_per_s"] = line["ragged_b64"]["steps_per_s"]
    if "chunked" in extra:
        resq = extra["chunked"]
        tpeak = peaks_tensor()
        line["chunked"] = dict(resq, bound="tensor", peak_tflops=tpeak[0], peak_source=tpeak[1],
                               tensor_frac=resq["tflops"] / tpeak[0])
    if not args.no_cpu:
        line["cpu_baseline"] = cpu_baseline(args.config)
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------ reference arm (the CPU oracle)

def run_reference(args, world, rank):
    if rank != 0:
        return
    from oracle import pipeline
    from synth.workloads import config

    wl = config(args.config)
    # each step: one sequence's whole decode step, append included (a bounded sample of the batch)
    n_prep = max(1, min(wl.B, 4))
    states = [pipeline.prepare(wl, b) for b in range(n_prep)]
    for i in range(args.warmup):
        oracle_step(wl, states, i)
    t = time.perf_counter()
    for i in range(args.steps):
        oracle_step(wl, states, i)
    dt = time.perf_counter() - t
    value = args.steps / dt
    cores = blas_threads()
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "query-steps/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded)",
        "config": {"workload": wl.name, "batch": wl.B, "ctx": int(wl.lengths[0]), "layers": wl.schedule},
        "cpu_baseline": {"value": value, "unit": "query-steps/s", "cores": cores, "kind": "oracle",
                         "sample": f"each step is one sequence of {wl.name} (of {wl.B}) through the append and "
                                   f"every layer"},
        "e2e": {"value": value, "unit": "query-steps/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=50)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--config", type=int, default=1, choices=[0, 1, 2, 4])
    ap.add_argument("--only-headline", action="store_true",
                    help="time only the --config workload (skip config 0, 1M, ragged, verify, chunked)")
    ap.add_argument("--no-cpu", action="store_true", help="skip the CPU oracle baseline")
    ap.add_argument("--cpu-worker", action="store_true", help=argparse.SUPPRESS)
    ap.add_argument("--cpu-budget", type=float, default=10.0, help=argparse.SUPPRESS)
    args = ap.parse_args()
    if args.cpu_worker:
        cpu_worker(args.config, args.cpu_budget)
        return
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    if args.impl == "reference":
        world = int(os.environ.get("WORLD_SIZE", "1"))
        rank = int(os.environ.get("RANK", "0"))
        run_reference(args, world, rank)
        return
    world, rank, local = dist_setup(args.gpus)
    run_ours(args, world, rank, local)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
