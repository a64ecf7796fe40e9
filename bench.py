"""Benchmark of the groupwise int4/int5 dequant-GEMM on GB300.

Default workload (N=1): decode/verify widths of the o_proj-shaped int4 matrix,
N=5120 rows, K=6144, T in {1, 2, 4, 8}.  One step = one call at each of the
four widths, each on a different copy of the packed weights (24 copies,
401 MB, rotate so every call streams cold weights from HBM -- the regime the
"ninfer-3080 docs/performance.md" route boundaries section calls production).

Metric: achieved HBM GB/s = algorithmic bytes (packed weights + bf16
activations) per step / step time, with the roofline fraction against the
measured HBM copy bandwidth, and microseconds per call per T.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                  [--workload decode|batched|multi|prefill_a|prefill_b|tiny]

Under torchrun (N > 1) every rank runs its own replica (weak scaling; the path
needs no collective) and rank 0 prints the line with the max time over ranks.
``--impl reference`` times the fp64 CPU oracle on the host instead.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from bit_weight_only_groupwise_gb300 import synth  # noqa: E402

METRIC = "W4/W5 dequant-GEMM µs/call and achieved HBM GB/s vs roofline, by token width T"
L2_BYTES = 129 * 1024 * 1024
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0
PROFILES = os.path.join(ROOT, "profiles")

WORKLOADS = {
    # name: (config name in the generator, widths timed per step)
    "decode": ("decode", [1, 2, 4, 8]),
    "batched": ("batched", [16, 32, 64, 256]),
    "multi": ("multi", [4, 16, 64]),
    "prefill_a": ("prefill_a", [256, 1024, 4096]),
    "prefill_b": ("prefill_b", [256, 1024, 4096]),
    "tiny": ("tiny", [1]),
    "linear_add": ("linear_add", [1, 2, 4, 8]),
    "swiglu": ("swiglu", [1, 2, 4, 8]),
    "decode_fp8": ("decode_fp8", [1, 2, 4, 8]),
    "prefill_fp8": ("prefill_fp8", [256, 1024, 4096]),
}


def describe(name: str) -> dict:
    cfg = synth.CONFIGS[WORKLOADS[name][0]]
    parents = [{"N": N, "K": cfg["K"], "codec": "fp8" if b == 8 else f"int{b}"} for N, b in cfg["parents"]]
    return {"name": name, "K": cfg["K"], "parents": parents, "T": WORKLOADS[name][1],
            "outliers": cfg["outliers"], "epilogue": cfg.get("epilogue", "store")}


def codec_bits(codec: str) -> int:
    return 8 if codec == "fp8" else int(codec[3:])


def weight_bytes(N: int, K: int, bits: int) -> int:
    # algorithmic: packed codes + fp16 group scales, read once per call
    return N * K * bits // 8 + 2 * N * (K // 64)


def step_bytes(desc) -> int:
    K = desc["K"]
    total = 0
    for T in desc["T"]:
        total += sum(weight_bytes(p["N"], K, codec_bits(p["codec"])) for p in desc["parents"]) + 2 * T * K
    return total


def hbm_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def tensor_peak():
    """Dense bf16 tensor throughput (burst: each call is a short kernel)."""
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["bf16_tflops"]), "measured"
    except Exception:
        return FALLBACK_BF16_TFLOPS, "fallback"


def route_kernel(route: str, K: int) -> tuple:
    """(kernel name, source file, bound) of the kernel a route launches."""
    if route.startswith("tcgen05"):
        return "qg::wide_kernel", "wide.cu", "tensor"
    full = (K // 64) % 8 == 0 and 1 <= (K // 64) // 8 <= 16
    return ("qg::skinny_line_kernel" if full else "qg::skinny_kernel"), "skinny.cu", "hbm"


def recorded_traffic(kernel_src: str, profile_name: str):
    """Per-launch DRAM bytes from a committed ncu summary, if it was taken on this kernel source."""
    path = os.path.join(PROFILES, profile_name)
    if not os.path.exists(path):
        return None
    want = hashlib.sha256(open(kernel_src, "rb").read()).hexdigest()
    rec = {}
    for line in open(path):
        if ":" in line:
            k, v = line.split(":", 1)
            rec[k.strip().lstrip("-* ")] = v.strip()
    if rec.get("kernel_source_sha256") != want:
        return None
    try:
        return json.loads(rec["dram_bytes_per_launch"])
    except Exception:
        return None


class ClockSampler:
    """nvidia-smi clock and throttle-reason samples during the timed region."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.path = os.path.join("/tmp", f"qgemm_clocks_{os.getpid()}.csv")

    def __enter__(self):
        try:
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.QUERY}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=self.fh, stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            self.fh.close()

    def summary(self):
        if self.proc is None or not os.path.exists(self.path):
            return None
        rows = []
        for line in open(self.path):
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                rows.append((float(f[1]), float(f[2]), f[5:9]))
            except ValueError:
                continue
        if not rows:
            return None
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for _, _, fl in rows for i, v in enumerate(fl) if v.lower() == "active"})
        return {"sm_mhz": statistics.median(r[0] for r in rows), "sm_max_mhz": max(r[1] for r in rows),
                "reasons": reasons, "samples": len(rows)}


# ---------------------------------------------------------------- distributed plumbing

def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def max_over_ranks(value: float, world: int) -> float:
    if world == 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device="cuda" if torch.cuda.is_available() else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


# ---------------------------------------------------------------- CPU oracle baseline

def oracle_sample(desc, seconds: float = 12.0):
    """Time the fp64 oracle on whole calls of the workload for about `seconds`."""
    import oracle
    wl = synth.workload(desc["name"] if desc["name"] in synth.CONFIGS else WORKLOADS[desc["name"]][0],
                        max(desc["T"]))
    lib = oracle.load()
    done_bytes, elapsed, calls = 0, 0.0, []
    K = desc["K"]
    # narrow widths first; wide ones on a column subset (cost is linear in T)
    while elapsed < seconds:
        for T in desc["T"]:
            cols = min(T, 8)
            x = wl["x"][:cols]
            t0 = time.perf_counter()
            for p in wl["parents"]:
                oracle.gemm_parent(p, x, lib=lib)
            dt = time.perf_counter() - t0
            # the row dequantisation costs about one column's dot products
            scale = (T + 1) / (cols + 1)
            elapsed += dt * scale
            calls.append((T, cols))
            done_bytes += sum(weight_bytes(p["N"], K, p["bits"]) for p in wl["parents"]) + 2 * T * K
            if elapsed >= seconds:
                break
    extrap = any(T != c for T, c in calls)
    sample = (f"{len(calls)} oracle calls of workload '{desc['name']}' at T in {desc['T']}"
              + ("; wide T timed on 8 columns and scaled by (T+1)/9 (cost is linear in T)" if extrap else ""))
    return done_bytes / elapsed / 1e9, elapsed, sample


def oracle_rows(desc, wl, lib, r0: int, nrows: int):
    """Time the oracle on rows [r0, r0 + nrows) (cyclic) of every parent at
    every width of the step; returns (seconds, algorithmic bytes of that share
    of the step).  Wide widths run on 8 columns and scale by (T+1)/9."""
    import oracle
    K = desc["K"]
    elapsed, done = 0.0, 0.0
    for T in desc["T"]:
        cols = min(T, 8)
        x = wl["x"][:cols]
        for p in wl["parents"]:
            N = p["N"]
            n = min(nrows, N)
            idx = (r0 + np.arange(n)) % N
            t0 = time.perf_counter()
            oracle.gemm(p["bits"], p["packed"][idx], p["scales"][idx], x, n, K, lib=lib)
            elapsed += (time.perf_counter() - t0) * (T + 1) / (cols + 1)
            done += weight_bytes(n, K, p["bits"]) + 2 * T * K * n / N
    return elapsed, done


def run_reference(args, desc):
    """The fp64 oracle on the host cores, as it stands: each step times it on
    a slice of the weight rows (every parent, every width), sized so that the
    whole --warmup + --steps run takes about --ref-seconds; the value is the
    median over the timed steps of the slice's algorithmic bytes per second."""
    world, rank, _ = dist_env()
    if rank != 0:
        return 0
    import oracle
    lib = oracle.load()
    wl = synth.workload(WORKLOADS[desc["name"]][0], max(desc["T"]))
    n_steps = args.warmup + args.steps
    # calibrate: seconds per weight row of a step
    t_cal, _ = oracle_rows(desc, wl, lib, 0, 32)
    per_row = max(t_cal / 32, 1e-7)
    rows = int(max(1, min(max(p["N"] for p in wl["parents"]), args.ref_seconds / n_steps / per_row)))
    gbs_vals = []
    r0 = 0
    for i in range(n_steps):
        el, done = oracle_rows(desc, wl, lib, r0, rows)
        r0 += rows
        if i >= args.warmup:
            gbs_vals.append(done / max(el, 1e-9) / 1e9)
    value = statistics.median(gbs_vals)
    sample = (f"{n_steps} steps of {rows} weight rows per parent of workload '{desc['name']}' at T in "
              f"{desc['T']} (wide T on 8 columns, scaled by (T+1)/9), about {args.ref_seconds:.0f} s in all")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * step_bytes(desc) / (value * 1e9),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": desc["name"], "parents": desc["parents"], "K": desc["K"], "T": desc["T"]},
        "cpu_baseline": {"value": value, "unit": "GB/s", "cores": 1, "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# ---------------------------------------------------------------- GPU arm

def run_ours(args, desc):
    import torch
    import bit_weight_only_groupwise_gb300 as qg

    world, rank, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    dev = torch.device("cuda", torch.cuda.current_device())
    stream = torch.cuda.current_stream()
    K = desc["K"]
    Ts = desc["T"]
    T_max = max(Ts)

    # weights: each parent packed once, then copied so that the rotation exceeds 3x L2
    wl = synth.workload(WORKLOADS[desc["name"]][0], T_max, seed=0)
    parents = wl["parents"]
    epi = desc["epilogue"]
    epi_code = {"store": qg.QGEMM_EPILOGUE_STORE, "add": qg.QGEMM_EPILOGUE_ADD,
                "swiglu": qg.QGEMM_EPILOGUE_SWIGLU}[epi]
    if epi == "swiglu":
        # the gate/up pair (parents 0 and 1) packed as one matrix with one output
        g, u = parents
        base = [qg.SwiGLUPair(g["bits"], g["N"], K, g["packed"], g["scales"], u["packed"], u["scales"], T_max)]
        set_bytes = qg.qgemm_pair_packed_bytes(g["N"], K, g["bits"])
        out_cols = [g["N"]]
    else:
        base = [qg.GroupwiseWeights(p["bits"], p["N"], K, p["packed"], p["scales"], T_max, epilogue=epi_code)
                for p in parents]
        set_bytes = sum(qg.qgemm_packed_bytes(p["N"], K, p["bits"]) for p in parents)
        out_cols = [p["N"] for p in parents]
    copies = max(2, int(np.ceil(3 * L2_BYTES / set_bytes)))
    weight_sets = []
    for i in range(copies):
        ws = []
        for b in base:
            w = type(b).__new__(type(b))
            w.codec, w.N, w.K, w.T_max, w.epilogue, w.out = b.codec, b.N, b.K, b.T_max, b.epilogue, b.out
            w.packed = b.packed.clone() if i else b.packed
            st, w.plan = qg.qgemm_plan(b.N, K, b.codec, T_max)
            qg.check(st, "qgemm_plan")
            if epi != "store":
                qg.check(qg.qgemm_plan_set_epilogue(w.plan, epi_code, qg.QGEMM_OUT_F32), "set_epilogue")
            wsb = qg.qgemm_plan_workspace_bytes(w.plan)
            w.workspace = torch.zeros(max(wsb, 16), dtype=torch.uint8, device=dev)
            qg.check(qg.qgemm_plan_bind(w.plan, w.packed, w.workspace, w.workspace.numel()), "bind")
            qg.check(qg.qgemm_plan_set_pdl(w.plan, not args.no_pdl), "set_pdl")
            ws.append(w)
        weight_sets.append(ws)
    xs = {T: torch.from_numpy(wl["x"][:T].view(np.int16).copy()).to(dev) for T in Ts}
    ys = {T: [torch.empty((T, n), dtype=torch.float32, device=dev) for n in out_cols] for T in Ts}
    # the residual of a LinearAdd: fp32 [T, N], seeded
    rs = {T: torch.from_numpy(np.random.default_rng(T).normal(0, 8, (T, out_cols[0])).astype(np.float32)).to(dev)
          for T in Ts} if epi == "add" else {}
    torch.cuda.synchronize()

    def call(ws, T, X=None, Ys=None, Rt=None):
        X = xs[T] if X is None else X
        Ys = ys[T] if Ys is None else Ys
        if epi != "store":
            Rt = (rs[T] if Rt is None else Rt) if epi == "add" else None
            st = qg.qgemm_run_ex(ws[0].plan, X, T, Rt, Ys[0], torch.cuda.current_stream())
        elif len(ws) == 1:
            st = qg.qgemm_run(ws[0].plan, X, T, Ys[0], torch.cuda.current_stream())
        else:
            st = qg.qgemm_run_multi([w.plan for w in ws], X, T, Ys, torch.cuda.current_stream())
        if st != qg.QGEMM_OK:
            raise qg.QgemmError(st, "run")

    # eager warm-up (loads the kernels), then one CUDA graph per (T, chunk of the
    # copy rotation) holding R calls, so that host launch cost stays off the clock
    for T in Ts:
        for ws in weight_sets[:2]:
            call(ws, T)
    torch.cuda.synchronize()
    assert qg.qgemm_device_status(stream) == qg.QGEMM_OK
    R = max(d for d in range(1, min(copies, args.steps) + 1) if args.steps % d == 0)
    n_chunks = (copies + R - 1) // R
    graphs = {}
    cap_stream = torch.cuda.Stream()
    for T in Ts:
        graphs[T] = []
        for ci in range(n_chunks):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=cap_stream):
                for r in range(R):
                    call(weight_sets[(ci * R + r) % copies], T)
            graphs[T].append(g)
    torch.cuda.synchronize()
    blocks = args.steps // R

    def replay_block(b, evs=None):
        for j, T in enumerate(Ts):
            if evs is not None:
                evs[j][0].record(stream)
            graphs[T][b % n_chunks].replay()
            if evs is not None:
                evs[j][1].record(stream)

    with torch.cuda.stream(stream):
        for b in range(max(1, (args.warmup + R - 1) // R)):
            replay_block(b)
    torch.cuda.synchronize()

    # timed region: exactly K steps = K/R replays of every width's R-call graph;
    # events around each replay on the launching stream give per-T call times
    ev = [[(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in Ts]
          for _ in range(blocks)]
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    n_launch0 = qg.qgemm_launch_count()
    barrier(world)
    torch.cuda.synchronize()
    with ClockSampler(torch.cuda.current_device()) as clocks:
        with torch.cuda.stream(stream):
            start.record(stream)
            for b in range(blocks):
                replay_block(b, ev[b])
            stop.record(stream)
        torch.cuda.synchronize()
    barrier(world)
    # graph replays do not pass through the host entry points: count the
    # kernels the replayed graphs hold: one per call, except that the tcgen05
    # route launches once per codec among the parents
    n_codecs = len({p["codec"] for p in desc["parents"]})
    launches = blocks * R * sum(n_codecs if weight_sets[0][0].route(T).startswith("tcgen05") else 1 for T in Ts)
    elapsed_ms = max_over_ranks(start.elapsed_time(stop), world)
    per_T_ms = {T: [ev[b][j][0].elapsed_time(ev[b][j][1]) / R for b in range(blocks)] for j, T in enumerate(Ts)}
    assert qg.qgemm_device_status(stream) == qg.QGEMM_OK
    del n_launch0

    sb = step_bytes(desc)
    value = world * args.steps * sb / (elapsed_ms * 1e-3) / 1e9
    peak, peak_kind = hbm_peak()
    per_T = {}
    by_kernel = {}          # kernel -> [time ms, bytes, flops, launches] over the timed region
    for T in Ts:
        b = sum(weight_bytes(p["N"], K, codec_bits(p["codec"])) for p in desc["parents"]) + 2 * T * K
        flops = sum(2 * T * p["N"] * K for p in desc["parents"])
        med = statistics.median(per_T_ms[T])
        mean = statistics.fmean(per_T_ms[T])
        route = ",".join(w.route(T) for w in weight_sets[0])
        per_T[str(T)] = {"us_per_call": 1e3 * med, "gbs": b / (med * 1e-3) / 1e9,
                         "frac": b / (med * 1e-3) / 1e9 / peak,
                         "tflops": flops / (med * 1e-3) / 1e12, "route": route}
        kern = route_kernel(weight_sets[0][0].route(T), K)
        acc = by_kernel.setdefault(kern, [0.0, 0, 0, 0])
        acc[0] += mean * blocks * R
        acc[1] += b * blocks * R
        acc[2] += flops * blocks * R
        acc[3] += blocks * R
    # the roofline of the kernel that takes most of the timed region: HBM bytes
    # for the weight-streaming kernels, tensor FLOPs for the tcgen05 route
    (kname, ksrc, bound), (k_ms, k_bytes, k_flops, k_launches) = max(by_kernel.items(), key=lambda kv: kv[1][0])
    profile_stem = kname.split("::")[-1]
    traffic = recorded_traffic(os.path.join(ROOT, "bit_weight_only_groupwise_gb300", "csrc", ksrc),
                               f"{profile_stem}_{desc['name']}_traffic.md")
    if bound == "hbm":
        achieved = k_bytes / (k_ms * 1e-3) / 1e9
        roof = {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                "traffic": traffic, "peak_source": peak_kind, "kernel": kname,
                "algorithmic_bytes_per_launch": k_bytes / k_launches}
    else:
        tpeak, tkind = tensor_peak()
        achieved = k_flops / (k_ms * 1e-3) / 1e12
        roof = {"bound": "tensor", "achieved": achieved, "peak": tpeak, "unit": "TFLOP/s",
                "frac": achieved / tpeak, "traffic": traffic, "peak_source": tkind, "kernel": kname,
                "algorithmic_flops_per_launch": k_flops / k_launches}

    # end to end: pinned host X -> device, the call, device Y -> pinned host, every step
    e2e = None
    if not args.no_e2e:
        hx = {T: torch.from_numpy(wl["x"][:T].view(np.int16).copy()).pin_memory() for T in Ts}
        hy = {T: [torch.empty((T, n), dtype=torch.float32).pin_memory() for n in out_cols] for T in Ts}
        dx = {T: torch.empty_like(xs[T]) for T in Ts}
        hr = {T: rs[T].cpu().pin_memory() for T in rs}
        dr = {T: torch.empty_like(rs[T]) for T in rs}
        h2d = sum(hx[T].numel() * 2 for T in Ts) + sum(hr[T].numel() * 4 for T in hr)
        d2h = sum(y.numel() * 4 for T in Ts for y in hy[T])
        e_steps = max(1, min(args.steps, 2000))
        barrier(world)
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for i in range(e_steps):
            for T in Ts:
                dx[T].copy_(hx[T], non_blocking=True)
                if epi == "add":
                    dr[T].copy_(hr[T], non_blocking=True)
                call(weight_sets[i % copies], T, X=dx[T], Rt=dr.get(T))
                for y, h in zip(ys[T], hy[T]):
                    h.copy_(y, non_blocking=True)
            stream.synchronize()          # the step's results are on the host
        e1.record(stream)
        torch.cuda.synchronize()
        e_ms = max_over_ranks(max(e0.elapsed_time(e1), 1e3 * (time.perf_counter() - t0)), world)
        e2e = {"value": world * e_steps * sb / (e_ms * 1e-3) / 1e9, "unit": "GB/s",
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
               "ms_per_step": e_ms / e_steps}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu:
        gbs, el, sample = oracle_sample(desc, seconds=args.cpu_seconds)
        cpu = {"value": gbs, "unit": "GB/s", "cores": 1, "kind": "oracle", "sample": sample,
               "seconds": el, "host_cores": os.cpu_count()}

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": elapsed_ms / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": desc["name"], "parents": desc["parents"], "K": desc["K"], "T": Ts,
                       "epilogue": epi,
                       "l2": f"rotating {copies} packed-weight copies ({copies * set_bytes / 1e6:.0f} MB > 3x L2)",
                       "parallelism": "replicas" if world > 1 else "single",
                       "pdl": not args.no_pdl},
            "per_T": per_T,
            "roofline": roof,
            "cpu_baseline": cpu,
            "e2e": e2e,
            "gpu_launches": launches,
            "clocks": clocks.summary(),
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=48000)
    ap.add_argument("--warmup", type=int, default=50)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=sorted(WORKLOADS), default="decode")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-pdl", action="store_true", help="launch without programmatic dependent launch")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--ref-seconds", type=float, default=90.0,
                    help="total host time of the reference arm, split over its steps")
    args = ap.parse_args()
    desc = describe(args.workload)
    if args.impl == "reference":
        return run_reference(args, desc)
    return run_ours(args, desc)


if __name__ == "__main__":
    sys.exit(main())
