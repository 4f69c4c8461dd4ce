"""Benchmark: one decode step of a synthetic Qwen3-8B-shaped BPDQ stack.

A step is every linear of 36 layers (qkv 4096->6144, o 4096->4096, gate_up
4096->24576, down 12288->4096) at ntok tokens: 144 q2_gemv launches through
the C ABI, captured once in a CUDA graph and replayed.  Weights (1.90 GB
packed) and activations are resident in HBM; the weights are larger than L2,
so no flush is needed between steps.  Prints one JSON line.

Besides the headline, the line carries per-format GEMV timings at the other
configurations (trellis 12288x4096 and 4096x12288, Leech 17408x5120 and
5120x17408, the fp16 control and the no-weights control at the 8B shapes),
each cycling enough distinct copies of its matrix to exceed L2 several times.

--impl reference times the CPU oracle (decode + f64 matvec) on a bounded
sample of the same workload and reports the same metric.
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

# DRAM traffic of the dominant kernel from the ncu capture summarised in
# profiles/bpdq_b1_qwen3_8b_stack.md: (dram__bytes_read.sum +
# dram__bytes_write.sum) / algorithmic bytes on a 24576x4096 launch.  The
# stack's traffic per launch is that ratio times the stack's algorithmic
# bytes per launch (traffic scales with the items processed).  Must be reset
# to None whenever the kernel changes.
NCU_TRAFFIC_RATIO = {"k_bpdq_b1": 27751936 / 27525120}


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


def build_stack(q2, ntok: int, config: int = 1):
    """36 layers x 4 BPDQ linears, distinct seeded weights and activations."""
    import torch
    import synth
    lin = []
    for layer in range(LAYERS):
        for j, (name, R, C) in enumerate(SHAPES_8B):
            seed = 1000 * config + 4 * layer + j
            d = synth.bpdq(R, C, seed)
            blob = q2.q2_pack_bpdq(d["plane0"], d["plane1"], d["coef"])
            del d
            x = torch.from_numpy(synth.activations(ntok, C, seed)).cuda()
            lin.append({"name": name, "R": R, "C": C, "blob": blob, "x": x})
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
    """GEMV us, GB/s and fraction of the byte bound per format (batch 1)."""
    import torch
    import synth
    out = {}

    def cycle(name, blob, R, C, fmt_label, fill=None):
        pk0 = q2.Packed(blob, ntok_max=1)
        if fill is not None:
            fill(pk0)
        nb = pk0.bytes_read(1)
        copies = max(4, int(np.ceil(4 * L2_BYTES / max(nb, 1))))
        copies = min(copies, 64)
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
        out[name] = {"format": fmt_label, "R": R, "C": C, "us_per_gemv": round(us, 3),
                     "bytes_per_gemv": nb, "bpw_read": round(8 * nb / (R * C), 4),
                     "gbs": round(gbs, 1), "frac_of_hbm": round(gbs / hbm, 4), "copies": copies}
        del pks, g

    for R, C in [(12288, 4096), (4096, 12288)]:
        d = synth.trellis(R, C, 2000 + (R > C))
        cycle(f"trellis_{R}x{C}", q2.q2_pack_trellis(d["stream"], d["table"], d["scale"]), R, C, "trellis")
    for R, C in [(17408, 5120), (5120, 17408)]:
        d = synth.leech(R, C, 3000 + (R > C))
        cycle(f"leech_{R}x{C}", q2.q2_pack_leech(d["v"], d["tail"], d["scale"], C), R, C, "leech")
    for name, R, C in SHAPES_8B:
        blob = q2.q2_pack_fp16(np.zeros((R, C), dtype=np.float16))
        g = torch.Generator(device="cuda").manual_seed(R + C)

        off = int(np.frombuffer(blob[56:64].tobytes(), dtype="<u8")[0])   # weight section offset

        def fill(p, R=R, C=C, g=g, off=off):
            w = torch.randn((R, C), generator=g, device="cuda", dtype=torch.float32).mul_(0.02).half()
            p.dev[off:off + R * C * 2].copy_(w.view(-1).view(torch.uint8))
        cycle(f"fp16_{name}_{R}x{C}", blob, R, C, "fp16", fill)
        d = synth.bpdq(R, C, 1000 + R + C)
        cycle(f"bpdq_{name}_{R}x{C}", q2.q2_pack_bpdq(d["plane0"], d["plane1"], d["coef"]), R, C, "bpdq")
        cycle(f"noweights_{name}_{R}x{C}", q2.q2_pack_noweights(R, C), R, C, "noweights")
    return out


ROT_WIDTHS = [4096, 5120, 12288, 17408]


def _rotation(q2, C: int, seed: int):
    import synth
    nh, nq = q2.q2_rotate_split(C)
    inp = synth.rotation(C, nh, seed)
    return q2.Rotation(inp["signs"], inp["q"] if nq > 1 else None, nh, C), nh, nq


def rotations(q2, stream):
    """Latency of the activation rotation (H (x) Q)(S x) per input width, at
    1, 16 and 64 tokens: 50 back-to-back rotations per graph replay."""
    import torch
    import synth
    out = {}
    for C in ROT_WIDTHS:
        rot, nh, nq = _rotation(q2, C, 900 + C % 1000)
        rec = {"C": C, "nh": nh, "nq": nq}
        for ntok in (1, 16, 64):
            x = torch.from_numpy(synth.activations(ntok, C, 901)).cuda()
            y = torch.empty_like(x)
            g = graph_of([lambda: rot.apply(x, y, stream=stream)] * 50, stream)
            ms = time_graph(g, stream, 20, 3)
            rec[f"us_ntok{ntok}"] = round(ms * 1e3 / (20 * 50), 3)
        out[f"rotation_{C}"] = rec
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


def sweep(args):
    """Config 4: Qwen3-14B-shaped stack (40 layers x qkv/o/gate_up/down) in each
    format, ntok in {1,2,4,8,16,32,64}; `distinct` layer copies are cycled
    through the 40 layers (their footprint is several times L2)."""
    import torch
    import dequant_gemv_q2_gb300 as q2
    import synth
    q2.load()
    torch.cuda.set_device(0)
    stream = torch.cuda.Stream()
    ntoks = [int(t) for t in args.sweep_ntok.split(",")]
    distinct = args.sweep_distinct
    pool = None
    results = {}
    for fmt in args.sweep_formats.split(","):
        mats = []                                   # per distinct layer: 4 Packed
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
                                                   np.random.default_rng(4243).integers(2, 7, size=2_000_000))
                    d = _leech_pool_matrix(R, C, seed, pool)
                    pk = q2.Packed(q2.q2_pack_leech(d["v"], d["tail"], d["scale"], C), ntok_max=max(ntoks),
                                   workspace=torch.zeros(16, dtype=torch.uint8, device="cuda"))
                row.append(pk)
            mats.append(row)
        if fmt != "cublas" and fmt != "fp16":
            need = max(p.workspace_bytes(max(ntoks)) for row in mats for p in row)
            wsbuf = torch.zeros(need, dtype=torch.uint8, device="cuda")
            for row in mats:
                for p in row:
                    p.set_workspace(wsbuf)
        layer_bytes = 0
        if fmt == "cublas":
            layer_bytes = sum(R * C * 2 for _, R, C in SHAPES_14B)
        results[fmt] = {}
        for nt in ntoks:
            xs = {C: torch.from_numpy(synth.activations(nt, C, 9)).cuda() for _, _, C in SHAPES_14B}
            ys = {R: torch.empty((nt, R), dtype=torch.float16, device="cuda") for _, R, _ in SHAPES_14B}
            calls = []
            for layer in range(LAYERS_14B):
                for j, (name, R, C) in enumerate(SHAPES_14B):
                    item = mats[layer % distinct][j]
                    if fmt == "cublas":
                        w = item[1]
                        calls.append(lambda w=w, x=xs[C], y=ys[R]: torch.matmul(x, w.t(), out=y))
                    else:
                        calls.append(lambda p=item, x=xs[C], y=ys[R]: p.gemv(x, y))
            g = graph_of(calls, stream)
            ms = time_graph(g, stream, args.sweep_steps, 3)
            step_ms = ms / args.sweep_steps
            if fmt == "cublas":
                step_bytes = layer_bytes * LAYERS_14B
            else:
                step_bytes = sum(mats[l % distinct][j].bytes_read(nt) for l in range(LAYERS_14B) for j in range(4))
            gbs = step_bytes / (step_ms * 1e-3) / 1e9
            results[fmt][nt] = {"ms_per_step": round(step_ms, 4), "tok_s": round(nt / (step_ms * 1e-3), 1),
                                "gbs": round(gbs, 1), "bytes_per_step": step_bytes}
            del g, calls
        del mats
        torch.cuda.empty_cache()
    print(json.dumps({"sweep": "Qwen3-14B-shaped stack, 40 layers x (qkv 5120->7168, o 5120->5120, "
                               "gate_up 5120->34816, down 17408->5120), linears only",
                      "distinct_layer_copies": distinct, "results": results}), flush=True)


def cpu_oracle_sample(seconds_target: float = 15.0) -> dict:
    """Oracle (decode + f64 matvec) on o-projection-shaped BPDQ matrices;
    returns seconds per weight and what was sampled.  Run in a subprocess
    with single-threaded numpy/BLAS."""
    code = r"""
import json, os, sys, time
sys.path.insert(0, %r)
import numpy as np
import synth
from oracle import bpdq, matvec
t0 = time.perf_counter(); n = 0; k = 0
while True:
    d = synth.bpdq(4096, 4096, 5000 + k)
    x = synth.activations(1, 4096, 5000 + k)
    t1 = time.perf_counter()
    w = bpdq.decode_f64(d["plane0"], d["plane1"], d["coef"])
    y = matvec.gemv(w, x)
    n += w.size; k += 1
    if time.perf_counter() - t0 > %f: break
el = time.perf_counter() - t0
print(json.dumps({"sec_per_weight": el / n, "matrices": k, "weights": n, "seconds": el}))
""" % (ROOT, seconds_target)
    env = dict(os.environ, OMP_NUM_THREADS="1", OPENBLAS_NUM_THREADS="1", MKL_NUM_THREADS="1")
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, env=env)
    if r.returncode != 0:
        return {"error": r.stderr[-500:]}
    return json.loads(r.stdout.strip().splitlines()[-1])


def stack_weights() -> int:
    return LAYERS * sum(R * C for _, R, C in SHAPES_8B)


def run_reference(args, ws, rank):
    """CPU oracle arm: each step is a bounded sample (one 4096x4096 BPDQ GEMV)."""
    if rank != 0:
        return
    import synth
    from oracle import bpdq, matvec
    d = synth.bpdq(4096, 4096, 5000)
    x = synth.activations(args.ntok, 4096, 5000)
    for _ in range(args.warmup):
        matvec.gemv(bpdq.decode_f64(d["plane0"], d["plane1"], d["coef"]), x)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        matvec.gemv(bpdq.decode_f64(d["plane0"], d["plane1"], d["coef"]), x)
    el = time.perf_counter() - t0
    sec_per_w = el / (args.steps * 4096 * 4096)
    step_s = sec_per_w * stack_weights()
    v = args.ntok / step_s
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": v, "unit": "tok/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": step_s * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": "BPDQ Qwen3-8B-shaped decode stack (36 layers x qkv/o/gate_up/down), linears only",
                   "ntok": args.ntok, "parallelism": "replicas"},
        "cpu_baseline": {"value": v, "unit": "tok/s", "cores": 1, "kind": "oracle",
                         "sample": f"{args.steps} oracle GEMVs of one 4096x4096 BPDQ matrix (decode + f64 matvec), "
                                   f"scaled to the stack's {stack_weights()} weights"},
        "e2e": {"value": v, "unit": "tok/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }), flush=True)


def profile_case(fmt: str, launches: int = 4, ntok: int = 1):
    """A few launches of one layer-shaped matrix per format, for ncu captures
    (no timing): bpdq 24576x4096 and 4096x12288, trellis 12288x4096, leech
    17408x5120, fp16 4096x4096, noweights 24576x4096; rotate: the activation
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
        mats.append((q2.q2_pack_leech(d["v"], d["tail"], d["scale"], 5120), 5120))
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

    # the oracle baseline runs in a subprocess started before any GPU work
    cpu = None
    ws_env = int(os.environ.get("WORLD_SIZE", "1"))
    if int(os.environ.get("RANK", "0")) == 0 and ws_env == 1 and not args.no_cpu:
        cpu = cpu_oracle_sample()

    import torch
    import dequant_gemv_q2_gb300 as q2
    ws, rank, local = _dist()
    q2.load()
    hbm, peak_kind = _peaks()
    stream = torch.cuda.Stream()

    lin = build_stack(q2, args.ntok)
    # every linear's x and y are views of one input and one output buffer, so
    # the end-to-end leg moves a step's inputs and outputs with one copy each
    xbuf = torch.empty(sum(L["x"].numel() for L in lin), dtype=torch.float16, device="cuda")
    ybuf = torch.empty(sum(args.ntok * L["R"] for L in lin), dtype=torch.float16, device="cuda")
    xo = yo = 0
    need = 0
    for L in lin:
        n = L["x"].numel()
        xbuf[xo:xo + n].copy_(L["x"].reshape(-1))
        L["x"] = xbuf[xo:xo + n].view(args.ntok, L["C"])
        xo += n
        L["pk"] = q2.Packed(L["blob"], ntok_max=args.ntok, workspace=torch.zeros(16, dtype=torch.uint8, device="cuda"))
        need = max(need, L["pk"].workspace_bytes(args.ntok))
        L["y"] = ybuf[yo:yo + args.ntok * L["R"]].view(args.ntok, L["R"])
        yo += args.ntok * L["R"]
    wsbuf = torch.zeros(need, dtype=torch.uint8, device="cuda")
    for L in lin:
        L["pk"].set_workspace(wsbuf)
        del L["blob"]
    step_bytes = sum(L["pk"].bytes_read(args.ntok) for L in lin)
    # the step is one q2_gemv_chain call: the 144 GEMVs in order, each launch
    # prefetching the weights of the next `lookahead` into L2
    chain = q2.Chain([(L["pk"], L["x"], L["y"]) for L in lin], args.ntok, args.lookahead)
    g = graph_of([chain.run], stream)

    clk = Clocks(torch.cuda.current_device())
    clk.start()
    time.sleep(0.3)
    ms = time_graph(g, stream, args.steps, args.warmup, ws)
    clocks = clk.stop()
    ms = _max_over_ranks(ms, ws)
    ms_step = ms / args.steps
    value = _job_value(ws, args.ntok, args.steps, ms)

    # end to end through the C ABI: every step copies all 144 inputs from
    # pinned host memory (one copy) and reads all outputs back (one copy)
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

    extras = rot_line = None
    if not args.no_extras and rank == 0:
        extras = per_format(q2, stream, hbm)
        extras.update(rotations(q2, stream))
        # the same stack with every linear's input rotated first (one rotation
        # per group of projections sharing an input: qkv and gate_up are fused)
        rots = {C: _rotation(q2, C, 950 + C % 1000)[0] for C in sorted({L["C"] for L in lin})}
        for L in lin:
            L["xr"] = torch.empty_like(L["x"])
        rcalls = []
        for L in lin:
            rcalls.append(lambda L=L: rots[L["C"]].apply(L["x"], L["xr"], stream=stream))
            rcalls.append(lambda L=L: L["pk"].gemv(L["xr"], L["y"]))
        gr = graph_of(rcalls, stream)
        rsteps = max(10, args.steps // 4)
        rms = time_graph(gr, stream, rsteps, 3) / rsteps
        rot_line = {"workload": "the same stack, each linear's input rotated by q2_rotate first",
                    "rotations_per_step": len(lin), "ms_per_step": round(rms, 4),
                    "tok_s": round(args.ntok / (rms * 1e-3), 1),
                    "rotation_share": round(1.0 - ms_step / rms, 3)}
        del gr

    achieved = step_bytes / (ms_step * 1e-3) / 1e9
    kname = "k_bpdq_b1" if args.ntok == 1 else ("k_bpdq_mt" if args.ntok <= 6 else "k_tc")
    # launches of one BPDQ GEMV: one at 1 token; token pairs plus a single
    # token at 2..6; one tensor-core launch from 7 (the split-K reduction runs
    # inside it for every shape of this stack)
    launches_per_gemv = 1 if args.ntok == 1 else (args.ntok + 1) // 2 if args.ntok <= 6 else 1
    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "tok/s", "n_gpus": ws, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "fp16 weights-decoded, fp32 accumulate",
            "data": "synthetic (seeded BPDQ weights and N(0,1) fp16 activations of the Qwen3-8B shapes)",
            "config": {"workload": "BPDQ Qwen3-8B-shaped decode stack: 36 layers x (qkv 4096->6144, o 4096->4096, "
                                   "gate_up 4096->24576, down 12288->4096), linears only",
                       "ntok": args.ntok, "lookahead": args.lookahead,
                       "launches_per_step": len(lin) * launches_per_gemv,
                       "bytes_per_step": step_bytes,
                       "l2": "weights 1.9 GB > L2, no flush", "parallelism": "replicas" if ws > 1 else "single"},
            "roofline": {"bound": "hbm", "kernel": kname, "achieved": round(achieved, 1), "peak": hbm,
                         "peak_kind": peak_kind, "unit": "GB/s", "frac": round(achieved / hbm, 4),
                         "traffic": (round(NCU_TRAFFIC_RATIO[kname] * step_bytes / len(lin))
                                     if NCU_TRAFFIC_RATIO.get(kname) else None),
                         "traffic_unit": "bytes per launch"},
            "gpu_launches": len(lin) * launches_per_gemv * args.steps,
            "clocks": clocks,
            "e2e": {"value": e2e_value, "unit": "tok/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
            "us_per_gemv_avg": round(ms_step * 1e3 / len(lin), 3),
        }
        if cpu is not None and "sec_per_weight" in cpu:
            step_s = cpu["sec_per_weight"] * stack_weights()
            line["cpu_baseline"] = {"value": args.ntok / step_s, "unit": "tok/s", "cores": 1, "kind": "oracle",
                                    "sample": f"{cpu['matrices']} oracle GEMVs of 4096x4096 BPDQ matrices "
                                              f"(decode + f64 matvec, {cpu['seconds']:.1f} s), scaled to the "
                                              f"stack's {stack_weights()} weights"}
        elif cpu is not None:
            line["cpu_baseline"] = {"value": None, "unit": "tok/s", "cores": 1, "kind": "oracle",
                                    "sample": "failed: " + cpu.get("error", "")[:200]}
        if extras is not None:
            line["per_format"] = extras
        if rot_line is not None:
            line["stack_with_rotation"] = rot_line
        print(json.dumps(line), flush=True)
    if ws > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
