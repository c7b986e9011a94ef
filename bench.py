"""Benchmark of the 2:4 sparse multiply-accumulate hot path on GB300.

One step = one pass of the whole path over one batch of synthetic input:
    sp24_compress_meta (compression and the metadata image in one pass, mask mode)
    ->  sp24_mma (D = A_sp B + C)
(--pass separate: sp24_compress -> sp24_meta_prepare -> sp24_mma; --pass index:
sp24_compress -> sp24_mma_index.)  The K timed steps are independent: they run either
with their compressions and products on two streams, so that step i+1's compression
overlaps step i's product, or back to back on one stream with the product overlapping the
compression's tail; by default the faster of the two in an untimed probe (--schedule).
Default workload: the largest single-GPU configuration, FP8 E4M3 M = N = K = 8192, keep
mask drawn per group from the six two-of-four patterns, A, B ~ N(0,1) scaled per tensor to
the format's range, no C, f32 output (--config bf16-4096 and the others stay selectable).
The metric is dense-equivalent TFLOP/s (TOP/s for integers) = 2 M N K / step time.
Timing: the K steps are recorded once (a CUDA graph); the graph is replayed R times, each
replay bracketed by CUDA events, R chosen so that the timed region lasts at least
--min-seconds (2 s by default), and the step time is the median replay time / K.

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--config NAME] [--impl reference]
Prints ONE JSON line (rank 0).  For N > 1 it runs under torch.distributed.run, one rank
per GPU, each rank an independent problem (weak scaling, no collective on the data path).
"""
from __future__ import annotations

import argparse
import csv
import hashlib
import io
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

import inputs  # noqa: E402

METRIC = "2:4 sparse GEMM dense-equiv TFLOPS/TOPS and % of GB300 sparse tensor peak"
L2_BYTES = 129 * 1024 * 1024
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
# NVIDIA's nominal dense peaks, used only for their ratios: fp8 / bf16 = 4.5 / 2.25 = 2,
# and 2:4 sparse executes twice the dense-equivalent rate of dense.
FP8_OVER_BF16 = 2.0
SPARSE_OVER_DENSE = 2.0

CONFIGS = {
    # name: (generator, ta, mode, out dtype, description)
    "bf16-4096": (lambda: inputs.bf16_square(), "bf16", "mask", torch.float32,
           "bf16 M=N=K=4096, random 2:4 mask, C f32, D f32"),
    "fixed-f16-64x128": (lambda: inputs.fixed_pattern_case(), "f16", "mask", torch.float32,
           "f16 64x64x128, fixed positions-0-and-2 pattern, integers in [-4,4], C f32"),
    "e4m3-8192": (lambda: inputs.fp8_square("e4m3"), "e4m3", "mask", torch.float32,
                "fp8 E4M3 M=N=K=8192, random 2:4 mask, no C, D f32"),
    "e5m2-8192": (lambda: inputs.fp8_square("e5m2"), "e5m2", "mask", torch.float32,
                "fp8 E5M2 M=N=K=8192, random 2:4 mask, no C, D f32"),
    "s8-8192": (lambda: inputs.int8_square("s8"), "s8", "mask", torch.int32,
              "int8 s8 x s8 M=N=K=8192, random 2:4 mask, C s32, D s32 (exact)"),
    "u8s8-8192": (lambda: inputs.int8_square("u8"), "u8", "mask", torch.int32,
              "int8 u8 x s8 M=N=K=8192, random 2:4 mask, C s32, D s32 (exact)"),
    "llm-n16": (lambda: inputs.llm_layer(16), "bf16", "magnitude", torch.bfloat16,
              "LLM layer W 14336x4096 bf16 magnitude-pruned, X 4096x16, D bf16"),
    "llm-n128": (lambda: inputs.llm_layer(128), "bf16", "magnitude", torch.bfloat16,
               "LLM layer W 14336x4096 bf16 magnitude-pruned, X 4096x128, D bf16"),
    "llm-n2048": (lambda: inputs.llm_layer(2048), "bf16", "magnitude", torch.bfloat16,
                "LLM layer W 14336x4096 bf16 magnitude-pruned, X 4096x2048, D bf16"),
}


def log(*a):
    print(*a, file=sys.stderr, flush=True)


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return p, "measured"
    except (OSError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


# the sources each kernel is built from (its ncu summary is stale once they change)
SPMMA_SOURCES = ("spmma.cu", "sp24_device.cuh", "sp24_internal.h")
COMPRESS_SOURCES = ("compress.cu", "sp24_device.cuh", "sp24_internal.h")


def source_hash(sources=SPMMA_SOURCES) -> str:
    h = hashlib.sha256()
    cs = os.path.join(ROOT, "structured_sparse_matrix_gb300", "csrc")
    for name in sources:
        with open(os.path.join(cs, name), "rb") as f:
            h.update(name.encode() + f.read())
    return h.hexdigest()[:16]


def profile_traffic(config: str, kernel: str = "spmma"):
    """DRAM bytes per launch of a kernel ("spmma" or "compress_meta") from the committed
    ncu summary of this workload, or None when no summary exists or the kernel's sources
    changed since it was taken."""
    path = os.path.join(ROOT, "profiles", f"{kernel}_{config}.txt")
    sources = SPMMA_SOURCES if kernel == "spmma" else COMPRESS_SOURCES
    try:
        fields = {}
        with open(path) as f:
            for line in f:
                if ":" in line:
                    k, v = line.split(":", 1)
                    fields[k.strip()] = v.strip()
        if fields.get("source_hash") != source_hash(sources):
            return None
        return float(fields["dram_bytes_per_launch"])
    except (OSError, KeyError, ValueError):
        return None


class ClockSampler:
    """nvidia-smi clocks and throttle reasons, sampled every 100 ms while running."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        time.sleep(0.25)
        self.text = ""
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.text, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                self.text, _ = self.proc.communicate()

    def summary(self):
        rows = [r for r in csv.reader(io.StringIO(self.text or "")) if len(r) >= 9]
        if not rows:
            return None
        sm = [float(r[1]) for r in rows if r[1].strip().replace(".", "").isdigit()]
        smax = [float(r[2]) for r in rows if r[2].strip().replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for r in rows for n, v in zip(names, r[5:9])
                          if v.strip() == "Active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None, "reasons": reasons,
                "samples": len(rows)}


def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    elif torch.cuda.is_available():
        torch.cuda.set_device(0)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int) -> float:
    if world == 1:
        return x
    import torch.distributed as dist
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ------------------------------------------------------------------ CPU oracle legs

def oracle_sample(c: dict, mode: str, budget_s: float):
    """Time the oracle (as it stands) on a bounded row sample of the workload: its
    compression of those rows plus its product.  Returns (flops/s, rows, seconds,
    threads)."""
    import oracle
    M, N, K, ta, tb = c["M"], c["N"], c["K"], c["ta"], c["tb"]
    Ab = inputs.bits(c["A"])
    Bb = inputs.bits(c["B"])
    mask = c["mask"].numpy() if (mode == "mask" and c["mask"] is not None) else None
    C = None if c["C"] is None else c["C"].numpy()

    def run(rows):
        t0 = time.perf_counter()
        sub = np.ascontiguousarray(Ab[:rows])
        v, i, _ = oracle.compress(sub, ta, mode, mask=None if mask is None else mask[:rows])
        Csub = None if C is None else np.ascontiguousarray(C[:rows])
        if ta in ("s8", "u8"):
            oracle.mma_i64(v, i, Bb, Csub, ta, tb, K)
        else:
            oracle.mma_f64(v, i, Bb, Csub, ta, tb, K, tc="f32" if C is not None else "f32")
        return time.perf_counter() - t0

    rows = min(M, 16)
    dt = run(rows)
    while dt < budget_s / 4 and rows < M:
        rows = min(M, max(rows * 2, int(rows * budget_s / max(dt, 1e-3) * 0.9)))
        dt = run(rows)
    return 2.0 * rows * N * K / dt, rows, dt, oracle.num_threads()


def reference_arm(args, world, rank):
    """The oracle as the reference arm: each step a bounded row sample of the workload."""
    if rank != 0:
        return
    gen, ta, mode, out_dtype, desc = CONFIGS[args.config]
    c = gen()
    # per-step sample sized so that warm-up + timed steps take about 2.5 minutes in all
    total = float(os.environ.get("SP24_REF_TOTAL_SECONDS", "150"))
    budget = min(8.0, max(0.2, total / max(args.steps + args.warmup, 1)))
    # size the per-step sample once, then time warmup + steps on that sample
    _, rows, _, threads = oracle_sample(c, mode, budget)
    import oracle
    Ab = inputs.bits(c["A"])[:rows]
    mask = c["mask"].numpy()[:rows] if (mode == "mask" and c["mask"] is not None) else None
    Bb = inputs.bits(c["B"])
    C = None if c["C"] is None else np.ascontiguousarray(c["C"].numpy()[:rows])

    def step():
        v, i, _ = oracle.compress(np.ascontiguousarray(Ab), ta, mode, mask=mask)
        if ta in ("s8", "u8"):
            oracle.mma_i64(v, i, Bb, C, ta, c["tb"], c["K"])
        else:
            oracle.mma_f64(v, i, Bb, C, ta, c["tb"], c["K"])

    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step()
    dt = (time.perf_counter() - t0) / max(args.steps, 1)
    value = 2.0 * rows * c["N"] * c["K"] / dt / 1e12
    unit = "TOP/s" if ta in ("s8", "u8") else "TFLOP/s"
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": unit,
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": dt * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64" if ta not in ("s8", "u8") else "int64",
        "data": "synthetic", "config": {"workload": desc, "M": c["M"], "N": c["N"], "K": c["K"]},
        "cpu_baseline": {"value": value, "unit": unit, "cores": threads, "kind": "oracle",
                         "sample": f"first {rows} of {c['M']} rows per step (compress + product)"},
        "e2e": {"value": value, "unit": unit, "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------ GPU arm

def gpu_arm(args, world, rank, local):
    import structured_sparse_matrix_gb300 as sp
    gen, ta, mode, out_dtype, desc = CONFIGS[args.config]
    dev = torch.device("cuda", local if world > 1 else 0)
    base = gen()
    M, N, K = base["M"], base["N"], base["K"]
    flops = 2.0 * M * N * K
    tdt = base["A"].dtype

    # input sets resident in HBM, rotated so that the working set exceeds L2
    def make_set(c):
        s = {"A": c["A"].to(dev), "B": c["B"].to(dev),
             "C": None if c["C"] is None else c["C"].to(dev),
             "mask": None if c["mask"] is None else c["mask"].to(dev).to(torch.uint8)}
        s["values"] = torch.empty((M, K // 2), dtype=tdt, device=dev)
        s["index"] = torch.empty((M, K // 32), dtype=torch.int32, device=dev)
        s["meta"] = torch.empty(max(sp.meta_bytes(tdt, M, K), 16), dtype=torch.uint8, device=dev)
        s["D"] = torch.empty((M, N), dtype=out_dtype, device=dev)
        return s

    def set_bytes(s):
        return sum(t.numel() * t.element_size() for t in s.values() if t is not None)

    sets = [make_set(base)]
    # at least two sets, so that no step reads operands the step before it left in L2
    # (--sets 1: one set, for profiler captures that save and restore device memory)
    while (len(sets) < 2 or len(sets) * set_bytes(sets[0]) < 3 * L2_BYTES) and len(sets) < 16 \
            and (args.sets == 0 or len(sets) < args.sets):
        # distinct contents per set: roll the rows (cheap, same distribution)
        c2 = dict(base)
        shift = 37 * len(sets)
        c2["A"] = torch.roll(base["A"], shift, 0)
        if base["mask"] is not None:
            c2["mask"] = torch.roll(base["mask"], shift, 0)
        c2["B"] = torch.roll(base["B"], shift, 0)
        sets.append(make_set(c2))
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream(dev)
    L = sp.lib()
    codes = sp.DTYPE_CODES
    integer = ta in ("s8", "u8")
    cs = {"ta": codes[tdt], "tb": codes[base["B"].dtype], "td": codes[out_dtype],
          "tc": codes[torch.int32 if integer else torch.float32]}
    # scratch for the integer path (operands widened to bf16), reused by every step
    ws_bytes = sp.workspace_bytes(tdt, base["B"].dtype, M, N, K)
    ws = torch.empty(max(ws_bytes, 16), dtype=torch.uint8, device=dev) if ws_bytes else None

    fused = args.pass_mode == "fused"
    by_index = args.pass_mode == "index"  # the product reads the canonical index: no image
    # kernels one step launches: compression (+ re-layout), the product (+ two widening
    # passes for integer operands)
    launches_per_step = (1 if fused or by_index else 2) + (3 if integer else 1)

    def compress_call(s, st):
        m = s["mask"]
        if fused:
            return L.sp24_compress_meta(cs["ta"], M, K, sp._ptr(s["A"]), K, sp._ptr(m), K,
                                        sp.MODES[mode], sp._ptr(s["values"]), K // 2,
                                        sp._ptr(s["index"]), K // 32, sp._ptr(s["meta"]),
                                        sp._ptr(status), st)
        rc = L.sp24_compress(cs["ta"], M, K, sp._ptr(s["A"]), K, sp._ptr(m), K,
                             sp.MODES[mode], sp._ptr(s["values"]), K // 2,
                             sp._ptr(s["index"]), K // 32, sp._ptr(status), st)
        if by_index:
            return rc
        return rc | L.sp24_meta_prepare(cs["ta"], M, K, sp._ptr(s["index"]), K // 32,
                                        sp._ptr(s["meta"]), st)

    def product_call(s, st):
        if by_index:
            return L.sp24_mma_index(cs["ta"], cs["tb"], cs["tc"], cs["td"], M, N, K,
                                    sp._ptr(s["values"]), K // 2, sp._ptr(s["index"]), K // 32,
                                    sp._ptr(s["B"]), N, sp._ptr(s["C"]), N, sp._ptr(s["D"]), N,
                                    sp._ptr(ws), ws_bytes, sp._ptr(status), st)
        return L.sp24_mma(cs["ta"], cs["tb"], cs["tc"], cs["td"], M, N, K, sp._ptr(s["values"]),
                          K // 2, sp._ptr(s["meta"]), sp._ptr(s["B"]), N, sp._ptr(s["C"]), N,
                          sp._ptr(s["D"]), N, sp._ptr(ws), ws_bytes, sp._ptr(status), st)

    s_comp, s_prod = torch.cuda.Stream(dev), torch.cuda.Stream(dev)

    def launch_overlapped(nsteps):
        # the compression of step i on one stream, the products on another: step i+1's
        # compression runs while step i's product finishes (each step's product waits for
        # its own compression; a compression waits for the last product that read its
        # input set)
        cur = torch.cuda.current_stream(dev)
        s_comp.wait_stream(cur)
        s_prod.wait_stream(cur)
        comp_done = [torch.cuda.Event() for _ in range(nsteps)]
        prod_done = [torch.cuda.Event() for _ in range(nsteps)]
        for i in range(nsteps):
            s = sets[i % len(sets)]
            with torch.cuda.stream(s_comp):
                if i >= len(sets):
                    s_comp.wait_event(prod_done[i - len(sets)])
                rc = compress_call(s, sp._stream(s_comp))
                comp_done[i].record(s_comp)
            with torch.cuda.stream(s_prod):
                s_prod.wait_event(comp_done[i])
                rc |= product_call(s, sp._stream(s_prod))
                prod_done[i].record(s_prod)
            if rc != 0:
                raise RuntimeError(f"sp24 call failed (status bits {rc})")
        cur.wait_stream(s_comp)
        cur.wait_stream(s_prod)

    def launch(s, ev=None):
        # the C-ABI calls of one step, on the current stream (a graph's capture stream
        # while one is being recorded)
        st = sp._stream(torch.cuda.current_stream(dev))
        m = s["mask"]
        if ev is not None:
            ev[0].record(stream)
        if fused:
            # compression and the metadata image in one pass
            rc = L.sp24_compress_meta(cs["ta"], M, K, sp._ptr(s["A"]), K, sp._ptr(m), K,
                                      sp.MODES[mode], sp._ptr(s["values"]), K // 2,
                                      sp._ptr(s["index"]), K // 32, sp._ptr(s["meta"]),
                                      sp._ptr(status), st)
            if ev is not None:
                ev[1].record(stream)
        else:
            rc = L.sp24_compress(cs["ta"], M, K, sp._ptr(s["A"]), K, sp._ptr(m), K,
                                 sp.MODES[mode], sp._ptr(s["values"]), K // 2,
                                 sp._ptr(s["index"]), K // 32, sp._ptr(status), st)
            if ev is not None:
                ev[1].record(stream)
            if not by_index:
                rc |= L.sp24_meta_prepare(cs["ta"], M, K, sp._ptr(s["index"]), K // 32,
                                          sp._ptr(s["meta"]), st)
        if ev is not None:
            ev[2].record(stream)
        rc |= product_call(s, st)
        if ev is not None:
            ev[3].record(stream)
        if rc != 0:
            raise RuntimeError(f"sp24 call failed (status bits {rc})")

    for i in range(max(args.warmup, 3)):
        launch(sets[i % len(sets)])
    torch.cuda.synchronize(dev)
    if status.item() != 0:
        raise RuntimeError(f"device status {status.item()} during warm-up")

    # the K steps recorded once as a CUDA graph (launch overhead off the timed path; the
    # GEMM's programmatic dependency on the pass before it becomes a graph edge); eager
    # launches if capture is refused
    # Schedules: "overlapped" runs the steps' compressions on one stream and their products
    # on another, so step i+1's compression fills the SMs that step i's product leaves idle
    # in its last wave; "serial" runs each step's two calls back to back on one stream (the
    # product launched to overlap the compression's tail).  "auto" (the default) times one
    # untimed probe of each before the timed region and keeps the faster for the workload.
    schedule = "serial" if args.serial else args.schedule

    def capture(overlapped):
        g = torch.cuda.CUDAGraph()
        cap = torch.cuda.Stream(dev)
        cap.wait_stream(stream)
        with torch.cuda.graph(g, stream=cap):
            if overlapped:
                launch_overlapped(args.steps)
            else:
                for i in range(args.steps):
                    launch(sets[i % len(sets)])
        stream.wait_stream(cap)
        g.replay()  # untimed: uploads the graph
        torch.cuda.synchronize(dev)
        return g

    graphs = {"overlapped": None, "serial": None}
    if not args.eager:
        try:
            for name in graphs:
                graphs[name] = capture(name == "overlapped")
        except Exception as exc:  # noqa: BLE001 - any capture failure means eager timing
            log(f"graph capture failed, timing eager launches: {exc}")
            torch.cuda.synchronize(dev)
            graphs = {"overlapped": None, "serial": None}
    if status.item() != 0:
        raise RuntimeError(f"device status {status.item()} during warm-up")

    def run_schedule(name):
        # the K steps back to back, no events between the kernels (the GEMM may start
        # during the previous kernel's tail)
        if graphs[name] is not None:
            graphs[name].replay()
        elif name == "overlapped":
            launch_overlapped(args.steps)
        else:
            for i in range(args.steps):
                launch(sets[i % len(sets)])

    def probe(name, reps=3):
        # median ms of `reps` untimed runs of the K steps in one schedule
        out = []
        for _ in range(reps):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            run_schedule(name)
            b.record(stream)
            torch.cuda.synchronize(dev)
            out.append(a.elapsed_time(b))
        return max_over_ranks(statistics.median(out), world)

    probe_ms = {name: probe(name) for name in ("overlapped", "serial")}
    if schedule == "auto":
        schedule = min(probe_ms, key=probe_ms.get)

    def run_k_steps():
        run_schedule(schedule)

    # replays in the timed region: enough for at least --min-seconds
    replays = int(max(1, min(100000, -(-args.min_seconds * 1e3 // max(probe_ms[schedule], 1e-3)))))
    replays = int(max_over_ranks(float(replays), world))

    # timed region: `replays` replays of the K steps, each bracketed by events
    ev_rep = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(replays)]
    barrier(world)
    torch.cuda.synchronize(dev)
    with ClockSampler(dev.index) as clk:
        for a, b in ev_rep:
            a.record(stream)
            run_k_steps()
            b.record(stream)
        torch.cuda.synchronize(dev)
    barrier(world)
    rep_ms = [a.elapsed_time(b) for a, b in ev_rep]
    total_ms = max_over_ranks(statistics.median(rep_ms), world)
    timed_s = max_over_ranks(sum(rep_ms) * 1e-3, world)
    if status.item() != 0:
        raise RuntimeError(f"device status {status.item()} in the timed region")
    ms_step = total_ms / args.steps
    # per-kernel breakdown, two ways.  (1) Isolated: the same steps again with events
    # around each kernel; the GPU first spins for a while so that every launch is enqueued
    # before the first one runs (events then time the kernels, not the host's launch rate),
    # and each kernel's time includes its launch and ramp-up, which the timed steps overlap
    # with the kernel before (programmatic dependent launch).  (2) Back to back: one CUDA
    # graph of n launches of the kernel alone, each on its own operands (rotated through
    # enough copies that the launches' operands together exceed three L2 sizes, so no launch
    # reads what an earlier one left in L2), events around the graph, time / n: the
    # kernel's steady-state duration as a sequence of layers issues it.
    n_bd = max(3, min(args.steps, 200))
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(n_bd)]
    torch.cuda._sleep(int(n_bd * 400_000))  # ~0.2 ms of GPU clock per step to enqueue
    for i in range(n_bd):
        launch(sets[i % len(sets)], evs[i])
    torch.cuda.synchronize(dev)
    k_compress = statistics.mean(e[0].elapsed_time(e[1]) for e in evs)
    k_meta = statistics.mean(e[1].elapsed_time(e[2]) for e in evs)
    k_mma = statistics.mean(e[2].elapsed_time(e[3]) for e in evs)
    value = flops * world / (ms_step * 1e-3) / 1e12

    def nbytes(t):
        return 0 if t is None else t.numel() * t.element_size()

    def rotation(keys):
        # the sets, plus copies of the tensors `keys` of them, until the launches' operands
        # exceed three L2 sizes
        per = sum(nbytes(sets[0][k]) for k in keys)
        want = max(2, -(-3 * L2_BYTES // max(per, 1)))
        rot = [dict(x) for x in sets]
        while len(rot) < want:
            src = sets[len(rot) % len(sets)]
            rot.append(dict(src, **{k: (None if src[k] is None else src[k].clone())
                                    for k in keys}))
        return rot

    def back_to_back(call, rot, n):
        g = torch.cuda.CUDAGraph()
        cap = torch.cuda.Stream(dev)
        cap.wait_stream(stream)
        with torch.cuda.graph(g, stream=cap):
            for i in range(n):
                if call(rot[i % len(rot)], sp._stream(cap)) != 0:
                    raise RuntimeError("sp24 call failed")
        stream.wait_stream(cap)
        g.replay()  # untimed: uploads the graph
        torch.cuda.synchronize(dev)
        out = []
        for _ in range(5):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            g.replay()
            b.record(stream)
            torch.cuda.synchronize(dev)
            out.append(a.elapsed_time(b) / n)
        del g
        return statistics.median(out)

    n_b2b = max(8, min(args.steps, 60))
    prod_keys = ["values", "index" if by_index else "meta", "B", "C", "D"]
    comp_keys = ["A", "mask", "values", "index"] + ([] if by_index else ["meta"])
    b2b_mma = b2b_compress = None
    if not args.eager:
        try:
            rot = rotation(prod_keys)
            b2b_mma = back_to_back(product_call, rot, n_b2b)
            del rot
            if fused or by_index:
                rot = rotation(comp_keys)
                b2b_compress = back_to_back(compress_call, rot, n_b2b)
                del rot
            torch.cuda.empty_cache()
        except Exception as exc:  # noqa: BLE001 - capture refused: isolated times only
            log(f"back-to-back timing skipped: {exc}")
            torch.cuda.synchronize(dev)
    if status.item() != 0:
        raise RuntimeError(f"device status {status.item()} in the per-kernel timing")

    # --- rooflines.  The product: a tensor-bound sparse contraction, or HBM-bound when its
    # intensity is below the ridge (skinny N); the compression pass: HBM-bound.
    peaks, src = load_peaks()
    dense = peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"])
    hbm = peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"])
    # 8-bit integers run widened to bf16: their roof is the bf16 sparse rate
    dense_peak = dense * (FP8_OVER_BF16 if ta in ("e4m3", "e5m2") else 1.0)
    peak = dense_peak * SPARSE_OVER_DENSE
    esz = torch.empty((), dtype=tdt).element_size()
    osz = torch.empty((), dtype=out_dtype).element_size()
    # algorithmic bytes: compressed A, the sparsity metadata at its information size (the
    # canonical index, M*K/8 bytes, the size of the kernel's image), B, C (if any), D, once
    mma_bytes = (M * K // 2 * esz + M * K // 8 + K * N * esz +
                 (M * N * 4 if base["C"] is not None else 0) + M * N * osz)
    unit = "TOP/s" if integer else "TFLOP/s"
    intensity = flops / mma_bytes
    ridge = peak * 1e12 / (hbm * 1e9)
    how_b2b = (f"CUDA events around one graph of {n_b2b} back-to-back launches of the kernel "
               "alone on rotating operands (together > 3 L2 sizes), time / launches, median "
               "of 5 replays")
    how_iso = (f"CUDA events around each kernel over {n_bd} steps run right after the timed "
               "region (each time includes the kernel's launch and ramp-up)")

    def mma_roof(ms, how):
        tf = flops / (ms * 1e-3) / 1e12
        if intensity >= ridge:
            r = {"bound": "tensor", "achieved": tf, "peak": peak, "unit": unit, "frac": tf / peak,
                 "peak_source": (f"{src}: bf16 dense {dense} TFLOP/s"
                                 f"{' x2 (fp8/bf16 nominal)' if ta in ('e4m3', 'e5m2') else ''}"
                                 " x2 (2:4 sparse / dense nominal), burst figure"
                                 f"{'; int8 runs exactly on the bf16 path' if integer else ''}")}
        else:
            gbs = mma_bytes / (ms * 1e-3) / 1e9
            r = {"bound": "hbm", "achieved": gbs, "peak": hbm, "unit": "GB/s", "frac": gbs / hbm,
                 "peak_source": (f"{src}: HBM copy bandwidth; the product's intensity "
                                 f"{intensity:.0f} flop/B is below the sparse tensor ridge "
                                 f"{ridge:.0f} flop/B")}
        r.update({"traffic": profile_traffic(args.config), "kernel": "sp24_mma (spmma_kernel)",
                  "us": ms * 1e3, "timing": how, "algorithmic_bytes": mma_bytes})
        return r

    # compression kernel: HBM-bound, algorithmic bytes = A + mask read, values + index written
    cbytes = M * K * esz + (M * K if mode == "mask" else 0) + M * K // 2 * esz + M * K // 8
    # the fused pass also writes the metadata image (at its information size)
    fbytes = cbytes + (M * K // 8 if fused else 0)
    cname = ("sp24_compress_meta (compress_meta_kernel)" if fused else
             "sp24_compress (compress_kernel)")

    def comp_roof(ms, how):
        gbs = fbytes / (ms * 1e-3) / 1e9
        return {"bound": "hbm", "achieved": gbs, "peak": hbm, "unit": "GB/s", "frac": gbs / hbm,
                "traffic": profile_traffic(args.config, "compress_meta") if fused else None,
                "kernel": cname, "us": ms * 1e3, "timing": how,
                "algorithmic_bytes": fbytes, "peak_source": f"{src}: HBM copy bandwidth"}

    mma_ms, mma_how = (b2b_mma, how_b2b) if b2b_mma is not None else (k_mma, how_iso)
    roof_mma = mma_roof(mma_ms, mma_how)
    roof_comp = None
    if fused or by_index:
        c_ms, c_how = ((b2b_compress, how_b2b) if b2b_compress is not None
                       else (k_compress, how_iso))
        roof_comp = comp_roof(c_ms, c_how)
    # the line's roofline is the dominant kernel's: the one that takes longer
    roof = roof_mma
    if roof_comp is not None and roof_comp["us"] > roof_mma["us"]:
        roof = roof_comp
    kernels = {
        "note": "sp24_mma time includes the int8->bf16 widening pass" if integer else None,
        "sp24_mma_us": k_mma * 1e3,
        "sp24_mma_us_back_to_back": None if b2b_mma is None else b2b_mma * 1e3,
        "sp24_mma_tflops": flops / (mma_ms * 1e-3) / 1e12,
        "sp24_mma_roofline": roof_mma,
        "step_us_probe": {name: ms * 1e3 / args.steps for name, ms in probe_ms.items()},
    }
    if fused:
        kernels["sp24_compress_meta_us"] = k_compress * 1e3
        kernels["sp24_compress_meta_us_back_to_back"] = (None if b2b_compress is None
                                                         else b2b_compress * 1e3)
        kernels["sp24_compress_meta_gbs"] = roof_comp["achieved"]
        kernels["sp24_compress_meta_roofline"] = roof_comp
    else:
        kernels["sp24_compress_us"] = k_compress * 1e3
        kernels["sp24_compress_gbs"] = cbytes / (k_compress * 1e-3) / 1e9
        if by_index:
            kernels["sp24_compress_us_back_to_back"] = (None if b2b_compress is None
                                                        else b2b_compress * 1e3)
            kernels["sp24_compress_roofline"] = roof_comp
        else:
            kernels["sp24_meta_prepare_us"] = k_meta * 1e3

    # --- end to end through the C ABI with host buffers: every step copies its inputs from
    # pinned host memory, runs the calls and reads its result back.  Two device buffer
    # sets on three streams (H2D, compute, D2H), so step i's copies overlap step i-1's
    # compute and readback; each step waits for the buffers it reuses.
    e2e = None
    if not args.no_e2e:
        hs = {k: base[k].pin_memory() if base[k] is not None else None for k in ("A", "B", "C")}
        hmask = base["mask"].to(torch.uint8).pin_memory() if base["mask"] is not None else None
        hD = [torch.empty((M, N), dtype=out_dtype).pin_memory() for _ in range(2)]
        bufs = [sets[0], sets[1] if len(sets) > 1 else make_set(base)]
        h2d = sum(t.numel() * t.element_size() for t in (hs["A"], hs["B"], hs["C"], hmask)
                  if t is not None)
        d2h = hD[0].numel() * hD[0].element_size()
        s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
        ev_in = [torch.cuda.Event() for _ in range(2)]
        ev_run = [torch.cuda.Event() for _ in range(2)]
        ev_out = [torch.cuda.Event() for _ in range(2)]
        used = [False, False]

        def e2e_step(i):
            k = i % 2
            s = bufs[k]
            with torch.cuda.stream(s_in):
                if used[k]:
                    s_in.wait_event(ev_run[k])  # the previous step on these buffers has read them
                s["A"].copy_(hs["A"], non_blocking=True)
                if hmask is not None:
                    s["mask"].copy_(hmask, non_blocking=True)
                s["B"].copy_(hs["B"], non_blocking=True)
                if hs["C"] is not None:
                    s["C"].copy_(hs["C"], non_blocking=True)
                ev_in[k].record(s_in)
            stream.wait_event(ev_in[k])
            if used[k]:
                stream.wait_event(ev_out[k])  # its D has been read back
            launch(s)
            ev_run[k].record(stream)
            with torch.cuda.stream(s_out):
                s_out.wait_event(ev_run[k])
                hD[k].copy_(s["D"], non_blocking=True)
                ev_out[k].record(s_out)
            used[k] = True

        for i in range(4):
            e2e_step(i)
        torch.cuda.synchronize(dev)
        n_e2e = max(4, min(args.steps, 40))
        barrier(world)
        torch.cuda.synchronize(dev)
        t0 = time.perf_counter()
        for i in range(n_e2e):
            e2e_step(i)
        torch.cuda.synchronize(dev)
        e2e_ms = max_over_ranks((time.perf_counter() - t0) * 1e3 / n_e2e, world)
        e2e = {"value": flops * world / (e2e_ms * 1e-3) / 1e12, "unit": unit,
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms,
               "steps": n_e2e, "schedule": "copies of step i overlap step i-1 (two buffer "
                                           "sets; H2D, compute and D2H streams)"}

    # --- CPU baseline: the oracle on this host's cores, bounded sample, rank 0 at N=1
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu:
        fps, rows, dt, threads = oracle_sample(base, mode, float(os.environ.get(
            "SP24_CPU_SECONDS", "12")))
        cpu = {"value": fps / 1e12, "unit": unit, "cores": threads, "kind": "oracle",
               "sample": f"first {rows} of {M} rows (oracle compress + "
                         f"{'int64' if integer else 'float64'} product), {dt:.1f} s"}

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": unit, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_step,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": ta, "data": "synthetic",
            "config": {"workload": desc, "name": args.config, "M": M, "N": N, "K": K,
                       "step": (f"sp24_compress_meta({mode}) + sp24_mma" if fused else
                                f"sp24_compress({mode}) + sp24_mma_index" if by_index else
                                f"sp24_compress({mode}) + sp24_meta_prepare + sp24_mma"),
                       "l2": f"{len(sets)} rotating input sets, "
                             f"{len(sets) * set_bytes(sets[0]) / 2**20:.0f} MiB > L2",
                       "parallelism": f"replicas x{world}",
                       "launch": ("one CUDA graph of the K steps"
                                  if graphs[schedule] is not None else "eager launches"),
                       "timing": (f"median over {replays} replays of the K steps, each "
                                  f"bracketed by CUDA events; {timed_s:.2f} s timed in all"),
                       "replays": replays,
                       "schedule": ("overlapped: the K independent steps run their "
                                    "compressions on one stream and their products on "
                                    "another, so step i+1's compression overlaps step i's "
                                    "product" if schedule == "overlapped" else
                                    "serial: each step's calls back to back on one stream, "
                                    "the product overlapping the compression's tail")
                                   + ("; chosen as the faster of the two in an untimed probe"
                                      if args.schedule == "auto" and not args.serial else "")},
            "roofline": roof,
            "kernels": kernels,
            "cpu_baseline": cpu,
            "e2e": e2e,
            "gpu_launches": launches_per_step * args.steps * replays,
            "clocks": clk.summary(),
        }
        print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--config", default="e4m3-8192", choices=sorted(CONFIGS))
    ap.add_argument("--sets", type=int, default=0,
                    help="input sets rotated through the steps (0: as many as keep the "
                         "working set above three L2 sizes, at least two)")
    ap.add_argument("--min-seconds", type=float, default=2.0,
                    help="the timed region replays the K steps until it lasts this long")
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--schedule", default="auto", choices=["auto", "overlapped", "serial"],
                    help="overlapped: step i+1's compression on its own stream during step "
                         "i's product; serial: each step's calls back to back on one stream; "
                         "auto: the faster of the two in an untimed probe")
    ap.add_argument("--serial", action="store_true", help="same as --schedule serial")
    ap.add_argument("--eager", action="store_true",
                    help="launch the timed steps one by one instead of as a CUDA graph")
    ap.add_argument("--pass", dest="pass_mode", default="fused",
                    choices=["fused", "separate", "index"],
                    help="compression and metadata image in one kernel (fused), in two "
                         "(separate), or no image: the product reads the canonical index")
    args = ap.parse_args()
    world, rank, local = dist_setup()
    try:
        if args.impl == "reference":
            reference_arm(args, world, rank)
        else:
            gpu_arm(args, world, rank, local)
    finally:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
