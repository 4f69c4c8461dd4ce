"""Benchmark: one decode step of a synthetic Qwen3-8B-shaped BPDQ stack.

A step is every linear of 36 layers (qkv 4096->6144, o 4096->4096, gate_up
4096->24576, down 12288->4096) at ntok tokens: 144 GEMVs through the C ABI
(one q2_gemv_chain call), captured once in a CUDA graph and replayed.  The
weights (1.90 GB packed) are resident in HBM and larger than L2, so no flush
is needed between steps; the activations are one input and one output
buffer per projection, shared by the layers as an engine's activation
buffers are.  Prints one JSON line.

Besides the headline, the line carries per-format GEMV timings at the other
workloads (trellis 12288x4096 and 4096x12288, Leech 17408x5120 and
5120x17408, the fp16 control and the no-weights control at the 8B shapes),
each cycling enough distinct copies of its matrix to exceed L2 several times.

--impl reference times the CPU oracle (decode + f64 matvec) on a bounded
sample of the same workload and reports the same metric.

The JSON line ends with the other workloads, compact, so that they survive
a tail of the output ("frac" is the fraction of the measured HBM bandwidth):
  "stack8b":  the 8B stack at 1, 4 and 16 tokens  [ms/step, tok/s, frac]
  "sweep14b": the 14B stack (40 layers, 4 distinct layer copies cycled) per
              format, tok/s at each count of "ntok" (1, 2, 4, 8, 16, 32,
              64); "frac1": each format's frac at one token
  "fmt":      single GEMVs at batch 1 per format and shape, each cycling
              copies of its matrix over >= 4x L2   [us, frac]
  "rot":      activation rotation us at 1 and 64 tokens, and the 8B stack
              with every input rotated first
"""
from __future__ import annotations

import argparse
import json
import os
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "batch-1 GEMV µs and achieved HBM GB/s (% of byte bound) per format; decode tok/s"
HIDDEN, QKV, INTER, LAYERS = 4096, 6144, 12288, 36
SHAPES_8B = [("qkv", QKV, HIDDEN), ("o", HIDDEN, HIDDEN), ("gate_up", 2 * INTER, HIDDEN), ("down", HIDDEN, INTER)]
L2_BYTES = 126 * 1024 * 1024
SWEEP_NTOK = [1, 2, 4, 8, 16, 32, 64]     # token counts of the Qwen3-14B-shaped stack sweep

# DRAM traffic of the dominant kernel per launch, as a ratio to its
# algorithmic bytes, from an ncu capture (dram__bytes_read.sum +
# dram__bytes_write.sum) of a 24576x4096 launch of the kernel as it is now;
# the stack's traffic per launch is that ratio times the stack's algorithmic
# bytes per launch (traffic scales with the items processed).  A kernel with
# no entry has no capture of its current code, and reports null.
NCU_TRAFFIC_RATIO = {"k_bpdq1": 27780608 / 27525120}


def _peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


class Clocks:
    """nvidia-smi sampling of SM clock and throttle reasons during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.idx = gpu_index
        self.f = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
        self.p = None

    def start(self):
        try:
            self.p = subprocess.Popen(["nvidia-smi", "-i", str(self.idx), f"--query-gpu={self.FIELDS}",
                                       "--format=csv,noheader,nounits", "-lms", "100"],
                                      stdout=self.f, stderr=subprocess.DEVNULL)
        except OSError:
            self.p = None

    def stop(self) -> dict:
        if self.p is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.p.terminate()
        try:
            self.p.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.p.kill()
        self.f.flush()
        rows = [r.split(",") for r in open(self.f.name).read().strip().splitlines() if r.strip()]
        os.unlink(self.f.name)
        sm = [float(r[1]) for r in rows if len(r) >= 9 and r[1].strip().replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if len(r) >= 9 and r[2].strip().replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = set()
        for r in rows:
            if len(r) >= 9:
                for n, v in zip(names, r[5:9]):
                    if v.strip().lower() == "active":
                        reasons.add(n)
        return {"sm_mhz": float(np.median(sm)) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(sm)}


def _dist():
    import torch
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if ws > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    else:
        torch.cuda.set_device(local)
    return ws, rank, local


def _barrier(ws):
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()


def _max_over_ranks(v: float, ws: int) -> float:
    """The largest of every rank's v (a timing: the job ends with its slowest rank)."""
    if ws == 1:
        return v
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([v], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def _job_value(ws: int, ntok: int, steps: int, ms: float) -> float:
    """Whole-job tokens per second: every replica processes ntok tokens per
    step, so all ranks together do ws * ntok * steps tokens in the slowest
    rank's ms."""
    return ws * ntok * steps / (ms / 1e3)


def build_stack(q2, ntok: int, seed0: int = 1000):
    """36 layers x 4 BPDQ linears with distinct seeded weights.  The inputs
    are one seeded activation per projection (qkv, o, gate_up, down), shared
    by the 36 layers as an inference engine's activation buffers are: every
    layer's projection reads the same buffer, which therefore stays in L2
    (as the output of the kernel before it would be) while the weights
    stream from HBM.  Seeds: seed0 + 4*layer + projection for the weights,
    seed0 + 900 + projection for the activations."""
    import torch
    import synth
    xs = {name: torch.from_numpy(synth.activations(ntok, C, seed0 + 900 + j)).cuda()
          for j, (name, R, C) in enumerate(SHAPES_8B)}
    lin = []
    for layer in range(LAYERS):
        for j, (name, R, C) in enumerate(SHAPES_8B):
            seed = seed0 + 4 * layer + j
            d = synth.bpdq(R, C, seed)
            blob = q2.q2_pack_bpdq(d["plane0"], d["plane1"], d["coef"])
            del d
            lin.append({"name": name, "R": R, "C": C, "blob": blob, "x": xs[name]})
    return lin


def graph_of(calls, stream):
    """Capture the given closures (each launches through q2_gemv) in a CUDA graph."""
    import torch
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        for c in calls:           # warm once outside the graph
            c()
        stream.synchronize()
        with torch.cuda.graph(g, stream=stream):
            for c in calls:
                c()
    torch.cuda.synchronize()
    return g


def time_graph(g, stream, steps: int, warmup: int, ws: int = 1):
    import torch
    for _ in range(warmup):
        g.replay()
    torch.cuda.synchronize()
    _barrier(ws)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        e0.record(stream)
        for _ in range(steps):
            g.replay()
        e1.record(stream)
    torch.cuda.synchronize()
    _barrier(ws)
    return e0.elapsed_time(e1)          # ms


def per_format(q2, stream, hbm):
    """Batch-1 GEMV per format and shape: {label: [us, GB/s, frac of HBM]}
    (the no-weights control: [us]); each label cycles enough distinct copies
    of its matrix to read >= 4x L2 per pass, with one input vector."""
    import torch
    import synth
    out = {}

    def cycle(name, blob, R, C, fill=None):
        pk0 = q2.Packed(blob, ntok_max=1)
        if fill is not None:
            fill(pk0)
        nb = pk0.bytes_read(1)
        copies = 64 if nb == 0 else max(4, int(np.ceil(4 * L2_BYTES / nb)))
        pks = [pk0] + [q2.Packed(blob, ntok_max=1, workspace=pk0.ws) for _ in range(copies - 1)]
        if fill is not None:
            for p in pks[1:]:
                p.dev.copy_(pk0.dev)
        x = torch.from_numpy(synth.activations(1, C, 7)).cuda()
        y = torch.empty((1, R), dtype=torch.float16, device="cuda")
        g = graph_of([lambda p=p: p.gemv(x, y) for p in pks], stream)
        reps = max(3, int(2000 / copies))
        ms = time_graph(g, stream, reps, 3)
        us = ms * 1e3 / (reps * copies)
        gbs = nb / (us * 1e-6) / 1e9
        out[name] = [round(us, 2), round(gbs), round(gbs / hbm, 3)] if nb else [round(us, 2)]
        del pks, g

    for R, C in [(12288, 4096), (4096, 12288)]:
        d = synth.trellis(R, C, 2000 + (R > C))
        cycle(f"trl_{R}x{C}", q2.q2_pack_trellis(d["stream"], d["table"], d["scale"]), R, C)
    pool = synth._sample_shell(np.random.default_rng(3000), np.random.default_rng(3001).integers(2, 7, 200000))

    def fp16_fill(R, C, seed):
        blob = q2.q2_pack_fp16(np.zeros((R, C), dtype=np.float16))
        g = torch.Generator(device="cuda").manual_seed(seed)
        off = int(np.frombuffer(blob[56:64].tobytes(), dtype="<u8")[0])   # weight section offset

        def fill(p):
            w = torch.randn((R, C), generator=g, device="cuda", dtype=torch.float32).mul_(0.02).half()
            p.dev[off:off + R * C * 2].copy_(w.view(-1).view(torch.uint8))
        return blob, fill

    for R, C in [(17408, 5120), (5120, 17408)]:
        d = _leech_pool_matrix(R, C, 3000 + (R > C), pool)
        # the two in-memory layouts (bits per weight read is the design axis) and the fp16 control
        cycle(f"leech_{R}x{C}", q2.q2_pack_leech(d["v"], d["tail"], d["scale"], C, q2.LEECH_PLANES3), R, C)
        cycle(f"leech4_{R}x{C}", q2.q2_pack_leech(d["v"], d["tail"], d["scale"], C, q2.LEECH_OFFSET4), R, C)
        blob, fill = fp16_fill(R, C, R + C)
        cycle(f"fp16_{R}x{C}", blob, R, C, fill)
    d = synth.bpdq(1024, 1024, 0)
    cycle("bpdq_1024x1024", q2.q2_pack_bpdq(d["plane0"], d["plane1"], d["coef"]), 1024, 1024)
    for name, R, C in SHAPES_8B:
        blob, fill = fp16_fill(R, C, R + C)
        cycle(f"fp16_{name}", blob, R, C, fill)
        d = synth.bpdq(R, C, 1000 + R + C)
        cycle(f"bpdq_{name}", q2.q2_pack_bpdq(d["plane0"], d["plane1"], d["coef"]), R, C)
        cycle(f"nw_{name}", q2.q2_pack_noweights(R, C), R, C)
    return out


ROT_WIDTHS = [4096, 5120, 12288, 17408]


def _rotation(q2, C: int, seed: int):
    import synth
    nh, nq = q2.q2_rotate_split(C)
    inp = synth.rotation(C, nh, seed)
    return q2.Rotation(inp["signs"], inp["q"] if nq > 1 else None, nh, C), nh, nq


def rotations(q2, stream):
    """Latency of the activation rotation (H (x) Q)(S x) per input width, us
    at 1 and 64 tokens: 50 back-to-back rotations per graph replay."""
    import torch
    import synth
    out = {}
    for C in ROT_WIDTHS:
        rot, nh, nq = _rotation(q2, C, 900 + C % 1000)
        rec = []
        for ntok in (1, 64):
            x = torch.from_numpy(synth.activations(ntok, C, 901)).cuda()
            y = torch.empty_like(x)
            g = graph_of([lambda: rot.apply(x, y, stream=stream)] * 50, stream)
            ms = time_graph(g, stream, 20, 3)
            rec.append(round(ms * 1e3 / (20 * 50), 2))
        out[str(C)] = rec
    return out


SHAPES_14B = [("qkv", 7168, 5120), ("o", 5120, 5120), ("gate_up", 34816, 5120), ("down", 5120, 17408)]
LAYERS_14B = 40


def _leech_pool_matrix(R: int, C: int, seed: int, pool: np.ndarray) -> dict:
    """Leech weights whose blocks are drawn uniformly from a pool of points
    sampled exactly (uniform shell, uniform within shell); used only for the
    14B sweep, where exact sampling of every block would take hours."""
    import synth
    rng = np.random.default_rng((seed, 7))
    nb = C // 24
    idx = rng.integers(0, pool.shape[0], size=(R, nb))
    v = pool[idx]
    scale = rng.uniform(0.005, 0.03, size=R).astype(np.float16)
    tail = rng.normal(0.0, 0.01, size=(R, C % 24)).astype(np.float16)
    return {"v": v, "scale": scale, "tail": tail}


def sweep14b(q2, stream, formats, ntoks, distinct: int, steps: int, hbm: float) -> dict:
    """The Qwen3-14B-shaped stack (40 layers x qkv/o/gate_up/down)
    per format at each token count; `distinct` layer copies are cycled
    through the 40 layers (their footprint is several times L2).  Returns
    {fmt: {ntok: [ms/step, tok/s, frac of HBM]}}; "cublas" is torch.matmul
    on dense fp16 weights, "fp16" this library's dense control."""
    import torch
    import synth
    pool = None
    results = {}
    for fmt in formats:
        mats = []                                   # per distinct layer: 4 Packed (or cuBLAS weights)
        for layer in range(distinct):
            row = []
            for j, (name, R, C) in enumerate(SHAPES_14B):
                seed = 4000 + 4 * layer + j
                if fmt in ("fp16", "cublas"):
                    g = torch.Generator(device="cuda").manual_seed(seed)
                    w = torch.randn((R, C), generator=g, device="cuda").mul_(0.02).half()
                    if fmt == "cublas":
                        row.append(("cublas", w, R, C))
                        continue
                    blob = q2.q2_pack_fp16(np.zeros((R, C), dtype=np.float16))
                    pk = q2.Packed(blob, ntok_max=max(ntoks))
                    off = int(np.frombuffer(blob[56:64].tobytes(), dtype="<u8")[0])
                    pk.dev[off:off + R * C * 2].copy_(w.view(-1).view(torch.uint8))
                    del w
                elif fmt == "bpdq":
                    d = synth.bpdq(R, C, seed)
                    pk = q2.Packed(q2.q2_pack_bpdq(d["plane0"], d["plane1"], d["coef"]), ntok_max=max(ntoks),
                                   workspace=torch.zeros(16, dtype=torch.uint8, device="cuda"))
                elif fmt == "trellis":
                    d = synth.trellis(R, C, seed)
                    pk = q2.Packed(q2.q2_pack_trellis(d["stream"], d["table"], d["scale"]), ntok_max=max(ntoks),
                                   workspace=torch.zeros(16, dtype=torch.uint8, device="cuda"))
                else:
                    if pool is None:
                        pool = synth._sample_shell(np.random.default_rng(4242),
                                                   np.random.default_rng(4243).integers(2, 7, size=400_000))
                    d = _leech_pool_matrix(R, C, seed, pool)
                    pk = q2.Packed(q2.q2_pack_leech(d["v"], d["tail"], d["scale"], C), ntok_max=max(ntoks),
                                   workspace=torch.zeros(16, dtype=torch.uint8, device="cuda"))
                row.append(pk)
            mats.append(row)
        if fmt != "cublas":
            # the workspace a handle needs is not monotone in ntok: the largest over the counts timed
            need = max(1, max(p.workspace_bytes(nt) for row in mats for p in row for nt in ntoks))
            wsbuf = torch.zeros(need, dtype=torch.uint8, device="cuda")
            for row in mats:
                for p in row:
                    p.set_workspace(wsbuf)
        results[fmt] = {}
        for nt in ntoks:
            xs = {C: torch.from_numpy(synth.activations(nt, C, 9)).cuda() for _, _, C in SHAPES_14B}
            ys = {R: torch.empty((nt, R), dtype=torch.float16, device="cuda") for _, R, _ in SHAPES_14B}
            links, calls = [], []
            for layer in range(LAYERS_14B):
                for j, (name, R, C) in enumerate(SHAPES_14B):
                    item = mats[layer % distinct][j]
                    if fmt == "cublas":
                        w = item[1]
                        calls.append(lambda w=w, x=xs[C], y=ys[R]: torch.matmul(x, w.t(), out=y))
                    else:
                        links.append((item, xs[C], ys[R]))
            if links:
                chain = q2.Chain(links, nt, 0)
                calls = [chain.run]
            g = graph_of(calls, stream)
            ms = time_graph(g, stream, steps, 3)
            step_ms = ms / steps
            if fmt == "cublas":
                step_bytes = LAYERS_14B * sum(R * C * 2 for _, R, C in SHAPES_14B)
            else:
                step_bytes = sum(mats[l % distinct][j].bytes_read(nt) for l in range(LAYERS_14B) for j in range(4))
            gbs = step_bytes / (step_ms * 1e-3) / 1e9
            results[fmt][str(nt)] = [round(step_ms, 3), round(nt / (step_ms * 1e-3)), round(gbs / hbm, 3)]
            del g, calls, links
        del mats
        torch.cuda.empty_cache()
    return results


def sweep(args):
    """--sweep: the Qwen3-14B-shaped stack over the formats and token counts given on the command line."""
    import torch
    import dequant_gemv_q2_gb300 as q2
    q2.load()
    torch.cuda.set_device(0)
    stream = torch.cuda.Stream()
    hbm, _ = _peaks()
    res = sweep14b(q2, stream, args.sweep_formats.split(","), [int(t) for t in args.sweep_ntok.split(",")],
                   args.sweep_distinct, args.sweep_steps, hbm)
    print(json.dumps({"sweep": "Qwen3-14B-shaped stack, 40 layers x (qkv 5120->7168, o 5120->5120, "
                               "gate_up 5120->34816, down 17408->5120), linears only; [ms/step, tok/s, frac]",
                      "distinct_layer_copies": args.sweep_distinct, "results": res}), flush=True)


# Oracle cases timed on the host cores, per GEMV: BPDQ 1024x1024, the trellis
# and Leech shapes, and the four Qwen3-8B projections (one layer; the stack
# step is 36 times their sum).
CPU_CASES = [("bpdq_1024x1024", "bpdq", 1024, 1024),
             ("trellis_12288x4096", "trellis", 12288, 4096), ("trellis_4096x12288", "trellis", 4096, 12288),
             ("leech_17408x5120", "leech", 17408, 5120), ("leech_5120x17408", "leech", 5120, 17408)] + \
            [(f"bpdq_{n}", "bpdq", R, C) for n, R, C in SHAPES_8B]

_CPU_CASE_CACHE = {}
_CPU_BARRIER = None


def _cpu_case_inputs(fmt: str, R: int, C: int, seed: int):
    import synth
    if fmt == "bpdq":
        d = synth.bpdq(R, C, seed)
    elif fmt == "trellis":
        d = synth.trellis(R, C, seed)
    else:
        pool = synth._sample_shell(np.random.default_rng(seed), np.random.default_rng(seed + 1).integers(2, 7, 50000))
        d = _leech_pool_matrix(R, C, seed, pool)
    return d, synth.activations(1, C, seed)


def _cpu_rows(fmt: str, d: dict, r0: int, r1: int) -> dict:
    """The canonical arrays of rows [r0, r1) (rows are independent)."""
    if fmt == "bpdq":
        return {"plane0": d["plane0"][r0:r1], "plane1": d["plane1"][r0:r1], "coef": d["coef"][:, r0:r1]}
    if fmt == "trellis":
        return {"stream": d["stream"][r0:r1], "table": d["table"], "scale": d["scale"][r0:r1]}
    return {"v": d["v"][r0:r1], "scale": d["scale"][r0:r1], "tail": d["tail"][r0:r1]}


def _cpu_case_run(fmt: str, d, x):
    """One oracle GEMV: exact f64 decode of the canonical weights, then the
    f64 matvec."""
    from oracle import bpdq, leech, matvec, trellis
    if fmt == "bpdq":
        w = bpdq.decode_f64(d["plane0"], d["plane1"], d["coef"])
    elif fmt == "trellis":
        w = trellis.decode_f64(d["stream"], d["table"], d["scale"])
    else:
        w = leech.decode_f64(d["v"], d["scale"], d["tail"])
    return matvec.gemv(w, x)


def _cpu_init(barrier):
    global _CPU_BARRIER
    _CPU_BARRIER = barrier


def _cpu_worker(task):
    """Time the oracle on rows [k*R/n, (k+1)*R/n) of a case in this
    single-threaded process; the inputs are generated once per process and
    not timed.  With a barrier, every process starts its timed part together."""
    fmt, R, C, seed, k, n = task
    key = (fmt, R, C, seed)
    if key not in _CPU_CASE_CACHE:
        _CPU_CASE_CACHE.clear()
        _CPU_CASE_CACHE[key] = _cpu_case_inputs(fmt, R, C, seed)
    d, x = _CPU_CASE_CACHE[key]
    part = _cpu_rows(fmt, d, k * R // n, (k + 1) * R // n)
    if _CPU_BARRIER is not None:
        _CPU_BARRIER.wait(timeout=900)
    t0 = time.perf_counter()
    _cpu_case_run(fmt, part, x)
    return time.perf_counter() - t0


def _cpu_model() -> str:
    try:
        r = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10)
        for line in r.stdout.splitlines():
            if line.lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    try:
        for line in open("/proc/cpuinfo"):
            if line.lower().startswith(("model name", "cpu part", "hardware")):
                return line.split(":", 1)[1].strip()
    except OSError:
        pass
    import platform
    return platform.processor() or platform.machine()


def cpu_oracle_baseline() -> dict:
    """The oracle timed on the host cores, per case (us per GEMV): one
    process on one core (single-threaded BLAS), then the same GEMV split by
    rows over one process per core, all starting together (the GEMV's time
    is the slowest process's).  Spawned processes, before any GPU work."""
    import multiprocessing as mp
    ncores = os.cpu_count() or 1
    os.environ.update({"OMP_NUM_THREADS": "1", "OPENBLAS_NUM_THREADS": "1", "MKL_NUM_THREADS": "1"})
    ctx = mp.get_context("spawn")
    out = {"cores": ncores, "cpu": _cpu_model(), "per_gemv_us": {}}
    with ctx.Pool(1) as p1:
        for label, fmt, R, C in CPU_CASES:
            t = p1.map(_cpu_worker, [(fmt, R, C, 7000, 0, 1)])[0]
            out["per_gemv_us"][label] = [round(t * 1e6, 1)]
    bar = ctx.Barrier(ncores)
    with ctx.Pool(ncores, initializer=_cpu_init, initargs=(bar,)) as pn:
        for label, fmt, R, C in CPU_CASES:
            ts = pn.map(_cpu_worker, [(fmt, R, C, 7000, k, ncores) for k in range(ncores)], chunksize=1)
            out["per_gemv_us"][label].append(round(max(ts) * 1e6, 1))
    return out


def run_reference(args, ws, rank):
    """CPU oracle arm.  Each step is a bounded sample of the stack: one
    o-projection-shaped (4096x4096) oracle GEMV split by rows over every host
    core (one single-threaded process per core); tok/s is scaled from the
    weights the step covers to the stack's weights."""
    if rank != 0:
        return
    import multiprocessing as mp
    ncores = os.cpu_count() or 1
    os.environ.update({"OMP_NUM_THREADS": "1", "OPENBLAS_NUM_THREADS": "1", "MKL_NUM_THREADS": "1"})
    tasks = [("bpdq", HIDDEN, HIDDEN, 5000, k, ncores) for k in range(ncores)]
    ctx = mp.get_context("spawn")
    with ctx.Pool(ncores, initializer=_cpu_init, initargs=(ctx.Barrier(ncores),)) as pool:
        for _ in range(max(1, args.warmup)):
            pool.map(_cpu_worker, tasks, chunksize=1)
        t0 = time.perf_counter()
        for _ in range(args.steps):
            pool.map(_cpu_worker, tasks, chunksize=1)
        el = time.perf_counter() - t0
    step_s = el / args.steps
    frac = HIDDEN * HIDDEN / stack_weights()             # share of a stack step per timed step
    v = args.ntok * frac / step_s
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": v, "unit": "tok/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": step_s * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": "BPDQ Qwen3-8B-shaped decode stack: 36 layers x (qkv 4096->6144, o 4096->4096, "
                               "gate_up 4096->24576, down 12288->4096), linears only",
                   "ntok": args.ntok, "parallelism": "replicas"},
        "cpu_baseline": {"value": v, "unit": "tok/s", "cores": ncores, "kind": "oracle", "cpu": _cpu_model(),
                         "sample": f"each step: one oracle GEMV of a 4096x4096 BPDQ matrix (exact f64 decode + "
                                   f"f64 matvec) split by rows over {ncores} single-threaded processes; tok/s = "
                                   f"ntok x {frac:.5f} of a stack step per step time"},
        "e2e": {"value": v, "unit": "tok/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }), flush=True)


def stack_weights() -> int:
    return LAYERS * sum(R * C for _, R, C in SHAPES_8B)


def profile_case(fmt: str, launches: int = 4, ntok: int = 1):
    """A few launches of one layer-shaped matrix per format, for ncu captures
    (no timing): bpdq 24576x4096 and 4096x12288, trellis 12288x4096, leech
    17408x5120 in the three-plane then the offset-binary layout, fp16
    4096x4096, noweights 24576x4096; rotate: the activation
    rotation at widths 17408 and 4096."""
    import torch
    import dequant_gemv_q2_gb300 as q2
    import synth
    q2.load()
    mats = []
    if fmt == "bpdq":
        for R, C in [(24576, 4096), (4096, 12288)]:
            d = synth.bpdq(R, C, 1000 + R + C)
            mats.append((q2.q2_pack_bpdq(d["plane0"], d["plane1"], d["coef"]), C))
    elif fmt == "trellis":
        d = synth.trellis(12288, 4096, 2000)
        mats.append((q2.q2_pack_trellis(d["stream"], d["table"], d["scale"]), 4096))
    elif fmt == "leech":
        d = synth.leech(17408, 5120, 3001)
        for lay in (q2.LEECH_PLANES3, q2.LEECH_OFFSET4):
            mats.append((q2.q2_pack_leech(d["v"], d["tail"], d["scale"], 5120, layout=lay), 5120))
    elif fmt == "fp16":
        mats.append((q2.q2_pack_fp16(np.zeros((4096, 4096), dtype=np.float16)), 4096))
    elif fmt == "noweights":
        mats.append((q2.q2_pack_noweights(24576, 4096), 4096))
    elif fmt == "rotate":
        for C in (17408, 4096):
            rot = _rotation(q2, C, 970)[0]
            x = torch.from_numpy(synth.activations(ntok, C, 7)).cuda()
            for _ in range(launches):
                rot.apply(x)
        torch.cuda.synchronize()
        print(json.dumps({"profile_case": fmt, "widths": [17408, 4096], "launches_each": launches, "ntok": ntok}))
        return
    for blob, C in mats:
        pk = q2.Packed(blob, ntok_max=ntok)
        x = torch.from_numpy(synth.activations(ntok, C, 7)).cuda()
        for _ in range(launches):
            pk.gemv(x)
    torch.cuda.synchronize()
    print(json.dumps({"profile_case": fmt, "matrices": len(mats), "launches_each": launches, "ntok": ntok}))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=3000)
    ap.add_argument("--warmup", type=int, default=50)
    ap.add_argument("--ntok", type=int, default=1)
    ap.add_argument("--impl", default="q2", choices=["q2", "reference"])
    ap.add_argument("--lookahead", type=int, default=0,
                    help="q2_gemv_chain lookahead: GEMVs ahead whose weights each launch prefetches into L2")
    ap.add_argument("--no-extras", action="store_true", help="skip the per-format lines")
    ap.add_argument("--no-cpu", action="store_true", help="skip the CPU oracle baseline")
    ap.add_argument("--profile-case", default=None,
                    choices=["bpdq", "trellis", "leech", "fp16", "noweights", "rotate"],
                    help="run a few untimed launches of one format for an ncu capture")
    ap.add_argument("--sweep", action="store_true", help="sweep over the 14B layer stack: formats x tokens")
    ap.add_argument("--sweep-formats", default="fp16,cublas,bpdq,trellis,leech")
    ap.add_argument("--sweep-ntok", default="1,2,4,8,16,32,64")
    ap.add_argument("--sweep-distinct", type=int, default=4)
    ap.add_argument("--sweep-steps", type=int, default=20)
    args = ap.parse_args()
    args.warmup = max(3, args.warmup)
    if args.sweep:
        sweep(args)
        return
    if args.profile_case:
        profile_case(args.profile_case, ntok=args.ntok)
        return

    if args.impl == "reference":
        ws = int(os.environ.get("WORLD_SIZE", "1"))
        rank = int(os.environ.get("RANK", "0"))
        run_reference(args, ws, rank)
        return

    # the oracle baseline runs in spawned processes before any GPU work
    cpu = None
    ws_env = int(os.environ.get("WORLD_SIZE", "1"))
    if int(os.environ.get("RANK", "0")) == 0 and ws_env == 1 and not args.no_cpu:
        try:
            cpu = cpu_oracle_baseline()
        except Exception as e:                      # a failed baseline must not cost the GPU line
            cpu = {"error": repr(e)[:200]}

    import torch
    import dequant_gemv_q2_gb300 as q2
    ws, rank, local = _dist()
    q2.load()
    hbm, peak_kind = _peaks()
    stream = torch.cuda.Stream()

    lin = build_stack(q2, args.ntok)
    names = [n for n, _, _ in SHAPES_8B]
    shape = {n: (R, C) for n, R, C in SHAPES_8B}
    for L in lin:
        L["pk"] = q2.Packed(L["blob"], ntok_max=args.ntok, workspace=torch.zeros(16, dtype=torch.uint8, device="cuda"))
        del L["blob"]
    x0 = {n: next(L["x"] for L in lin if L["name"] == n) for n in names}

    def stack_graph(nt: int, xsrc=None):
        """The step at nt tokens as one q2_gemv_chain call in a CUDA graph: one
        input and one output buffer per projection, shared by the layers (the
        four inputs are views of one buffer and the four outputs of another,
        so the end-to-end leg moves a step's inputs and outputs with one copy
        each)."""
        xbuf = torch.empty(sum(nt * shape[n][1] for n in names), dtype=torch.float16, device="cuda")
        ybuf = torch.empty(sum(nt * shape[n][0] for n in names), dtype=torch.float16, device="cuda")
        xv, yv, xo, yo = {}, {}, 0, 0
        for j, n in enumerate(names):
            R, C = shape[n]
            xv[n] = xbuf[xo:xo + nt * C].view(nt, C)
            xv[n].copy_(xsrc[n] if xsrc is not None else
                        torch.from_numpy(__import__("synth").activations(nt, C, 1900 + j)).cuda())
            yv[n] = ybuf[yo:yo + nt * R].view(nt, R)
            xo += nt * C
            yo += nt * R
        need = max(L["pk"].workspace_bytes(nt) for L in lin)
        wsbuf = torch.zeros(need, dtype=torch.uint8, device="cuda")
        for L in lin:
            L["pk"].set_workspace(wsbuf)
        chain = q2.Chain([(L["pk"], xv[L["name"]], yv[L["name"]]) for L in lin], nt, args.lookahead)
        return graph_of([chain.run], stream), xbuf, ybuf, wsbuf, xv, yv

    def launches_per_gemv(nt: int) -> int:
        # one launch at 1 token; token pairs plus a single token at 2..6; one
        # tensor-core launch from 7 (the split-K reduction runs inside it for
        # every shape of this stack)
        return 1 if nt == 1 else (nt + 1) // 2 if nt <= 6 else 1

    g, xbuf, ybuf, wsbuf, xv, yv = stack_graph(args.ntok, x0)
    step_bytes = sum(L["pk"].bytes_read(args.ntok) for L in lin)

    clk = Clocks(torch.cuda.current_device())
    clk.start()
    time.sleep(0.3)
    ms = time_graph(g, stream, args.steps, args.warmup, ws)
    clocks = clk.stop()
    ms = _max_over_ranks(ms, ws)
    ms_step = ms / args.steps
    value = _job_value(ws, args.ntok, args.steps, ms)

    # end to end through the C ABI: every step copies the step's inputs from
    # pinned host memory (one copy) and reads its outputs back (one copy)
    xs_host = xbuf.cpu().pin_memory()
    ys_host = torch.empty_like(ybuf, device="cpu").pin_memory()
    h2d = xs_host.numel() * 2
    d2h = ys_host.numel() * 2
    e2e_steps = max(10, args.steps // 20)
    with torch.cuda.stream(stream):
        for _ in range(3):
            xbuf.copy_(xs_host, non_blocking=True)
            g.replay()
            ys_host.copy_(ybuf, non_blocking=True)
        torch.cuda.synchronize()
        _barrier(ws)
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(e2e_steps):
            xbuf.copy_(xs_host, non_blocking=True)
            g.replay()
            ys_host.copy_(ybuf, non_blocking=True)
        e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = _max_over_ranks(e0.elapsed_time(e1), ws)
    e2e_value = _job_value(ws, args.ntok, e2e_steps, e2e_ms)

    extras = {}
    if not args.no_extras and rank == 0:
        # the same 8B stack at the other token counts of its configuration
        st8 = {}
        for nt in (1, 4, 16):
            if nt == args.ntok:
                st8[str(nt)] = [round(ms_step, 4), round(value), round(step_bytes / (ms_step * 1e-3) / 1e9 / hbm, 3)]
                continue
            g2 = stack_graph(nt)[0]
            k = 40
            m2 = time_graph(g2, stream, k, 3) / k
            b2 = sum(L["pk"].bytes_read(nt) for L in lin)
            st8[str(nt)] = [round(m2, 4), round(nt / (m2 * 1e-3)), round(b2 / (m2 * 1e-3) / 1e9 / hbm, 3)]
            del g2
        extras["stack8b"] = st8
        # the same stack with every linear's input rotated first
        rots = {C: _rotation(q2, C, 950 + C % 1000)[0] for C in sorted({C for _, C in shape.values()})}
        g, xbuf, ybuf, wsbuf, xv, yv = stack_graph(args.ntok, x0)
        xr = {n: torch.empty_like(xv[n]) for n in names}
        rcalls = []
        for L in lin:
            n = L["name"]
            rcalls.append(lambda n=n: rots[shape[n][1]].apply(xv[n], xr[n], stream=stream))
            rcalls.append(lambda L=L, n=n: L["pk"].gemv(xr[n], yv[n]))
        gr = graph_of(rcalls, stream)
        rsteps = 40
        rms = time_graph(gr, stream, rsteps, 3) / rsteps
        del gr, rcalls
        rot = rotations(q2, stream)
        rot["stack_ms"] = round(rms, 4)
        del lin, g, xbuf, ybuf, wsbuf, xv, yv
        torch.cuda.empty_cache()
        sw = sweep14b(q2, stream, ["bpdq", "trellis", "leech", "cublas"], SWEEP_NTOK, 4, 10, hbm)
        sw["fp16"] = sweep14b(q2, stream, ["fp16"], SWEEP_NTOK, 4, 10, hbm)["fp16"]
        # compact: tok/s per format at each token count, and batch 1's fraction of HBM
        extras["sweep14b"] = {"ntok": SWEEP_NTOK,
                              **{f: [sw[f][str(nt)][1] for nt in SWEEP_NTOK] for f in sw},
                              "frac1": {f: sw[f]["1"][2] for f in sw}}
        extras["fmt"] = {k: [v[0], v[2]] if len(v) == 3 else v for k, v in per_format(q2, stream, hbm).items()}
        extras["rot"] = rot

    achieved = step_bytes / (ms_step * 1e-3) / 1e9
    kname = "k_bpdq1" if args.ntok == 1 else ("k_bpdqm" if args.ntok <= 6 else "k_tc")
    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "tok/s", "n_gpus": ws, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "fp16 weights-decoded, fp32 accumulate",
            "data": "synthetic (seeded BPDQ weights and N(0,1) fp16 activations of the Qwen3-8B shapes)",
            "config": {"workload": "BPDQ Qwen3-8B-shaped decode stack: 36 layers x (qkv 4096->6144, o 4096->4096, "
                                   "gate_up 4096->24576, down 12288->4096), linears only",
                       "ntok": args.ntok, "lookahead": args.lookahead,
                       "launches_per_step": len(SHAPES_8B) * LAYERS * launches_per_gemv(args.ntok),
                       "bytes_per_step": step_bytes,
                       "l2": "weights 1.9 GB > L2, no flush; activations: one buffer per projection, shared by "
                             "the layers (L2-resident)", "parallelism": "replicas" if ws > 1 else "single"},
            "roofline": {"bound": "hbm", "kernel": kname, "achieved": round(achieved, 1), "peak": hbm,
                         "peak_kind": peak_kind, "unit": "GB/s", "frac": round(achieved / hbm, 4),
                         "traffic": (round(NCU_TRAFFIC_RATIO[kname] * step_bytes / (len(SHAPES_8B) * LAYERS))
                                     if NCU_TRAFFIC_RATIO.get(kname) else None),
                         "traffic_unit": "bytes per launch"},
            "gpu_launches": len(SHAPES_8B) * LAYERS * launches_per_gemv(args.ntok) * args.steps,
            "clocks": clocks,
            "e2e": {"value": e2e_value, "unit": "tok/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
            "us_per_gemv_avg": round(ms_step * 1e3 / (len(SHAPES_8B) * LAYERS), 3),
        }
        if cpu is not None and "per_gemv_us" in cpu:
            us = cpu["per_gemv_us"]
            layer1 = sum(us[f"bpdq_{n}"][0] for n in names)
            layern = sum(us[f"bpdq_{n}"][-1] for n in names)
            line["cpu_baseline"] = {
                "value": args.ntok / (LAYERS * layer1 * 1e-6), "unit": "tok/s", "cores": 1, "kind": "oracle",
                "sample": "one oracle GEMV (exact f64 decode + f64 matvec) of each 8B projection shape, timed, "
                          "x 36 layers (extrapolated to the stack step)",
                "all_cores": {"cores": cpu["cores"], "value": args.ntok / (LAYERS * layern * 1e-6),
                              "how": "each GEMV split by rows over one single-threaded process per core, started "
                                     "together; its time is the slowest process's"},
                "cpu": cpu["cpu"],
                "us": us}
        elif cpu is not None:
            line["cpu_baseline"] = {"value": None, "unit": "tok/s", "cores": 1, "kind": "oracle",
                                    "sample": "failed: " + str(cpu.get("error", ""))[:200]}
        line.update(extras)                         # compact, and last: they survive a tail of the output
        print(json.dumps(line, separators=(",", ":")), flush=True)
    if ws > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
