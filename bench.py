"""Benchmark of the groupwise int4/int5 dequant-GEMM on GB300.

Default workload (N=1): every configuration of the metric, one call at each
of its token widths per step:

  tiny       int4   256 x 512,   T = 1
  decode     int4  5120 x 6144,  T = 1, 2, 4, 8   (decode and verify widths)
  batched    int4 12288 x 5120,  T = 16, 32, 64, 256
  multi      int4  4096 x 5120 + int5 12288 x 5120 over one shared X, T = 4, 16, 64
  prefill_a  int4  7168 x 5120,  T = 256, 1024, 4096
  prefill_b  int4  5120 x 6144,  T = 256, 1024, 4096

Each (configuration, width) runs as a CUDA graph of R back-to-back calls, each
call on its own copy of the packed weights, so no call finds its weights in L2
(between two replays of one graph the rest of the step streams far more than
the 129 MB L2) -- the cold regime the "ninfer-3080 docs/performance.md" route
boundaries section calls production.

Metric: achieved HBM GB/s = algorithmic bytes (packed weights + bf16
activations, every call of the step) / step time, with per-call microseconds,
GB/s, TFLOP/s and the fraction of each call's roofline, max((W + X) / HBM,
2NKT / bf16 tensor peak), and the roofline of every kernel.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                  [--workload all|decode|batched|multi|prefill_a|prefill_b|tiny|...]

Under torchrun (N > 1) every rank runs its own replica (weak scaling; the path
needs no collective) and rank 0 prints the line with the max time over ranks.
``--impl reference`` times the fp64 CPU oracle on the host instead.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
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
CSRC = os.path.join(ROOT, "bit_weight_only_groupwise_gb300", "csrc")

# the widths timed per configuration of the input generator
WIDTHS = {
    "tiny": [1],
    "decode": [1, 2, 4, 8],
    "batched": [16, 32, 64, 256],
    "multi": [4, 16, 64],
    "prefill_a": [256, 1024, 4096],
    "prefill_b": [256, 1024, 4096],
    "linear_add": [1, 2, 4, 8],
    "swiglu": [1, 2, 4, 8],
    "decode_fp8": [1, 2, 4, 8],
    "prefill_fp8": [256, 1024, 4096],
    "decode_nvfp4": [1, 2, 4, 8],
    "prefill_nvfp4": [256, 1024, 4096],
    "decode_ring": [1, 8, 16],
}
# a workload is a list of configurations; one step is one call at every width of each
WORKLOADS = {"all": ["tiny", "decode", "batched", "multi", "prefill_a", "prefill_b"]}
WORKLOADS.update({name: [name] for name in WIDTHS})


def codec_name(bits: int) -> str:
    return {8: "fp8", synth.NVFP4: "nvfp4"}.get(bits, f"int{bits}")


def codec_bits(codec: str) -> int:
    return {"fp8": 8, "nvfp4": synth.NVFP4}.get(codec) or int(codec[3:])


def describe(name: str) -> dict:
    configs = []
    for c in WORKLOADS[name]:
        cfg = synth.CONFIGS[c]
        configs.append({"config": c, "K": cfg["K"], "T": WIDTHS[c], "outliers": cfg["outliers"],
                        "epilogue": cfg.get("epilogue", "store"),
                        "parents": [{"N": N, "K": cfg["K"], "codec": codec_name(b)} for N, b in cfg["parents"]]})
    return {"name": name, "configs": configs}


def weight_bytes(N: int, K: int, bits: int) -> int:
    # algorithmic: packed codes + their scales, read once per call (fp16 per
    # 64 columns; NVFP4: 4-bit codes and one byte per 16 columns)
    if bits == synth.NVFP4:
        return N * K // 2 + N * (K // 16)
    return N * K * bits // 8 + 2 * N * (K // 64)


def call_bytes(cfg, T) -> int:
    K = cfg["K"]
    return sum(weight_bytes(p["N"], K, codec_bits(p["codec"])) for p in cfg["parents"]) + 2 * T * K


def call_flops(cfg, T) -> int:
    return sum(2 * T * p["N"] * cfg["K"] for p in cfg["parents"])


def calls(desc):
    """(config index, config, T) of every call of one step."""
    return [(i, c, T) for i, c in enumerate(desc["configs"]) for T in c["T"]]


def step_bytes(desc) -> int:
    return sum(call_bytes(c, T) for _, c, T in calls(desc))


def config_summary(desc) -> dict:
    return {"workload": desc["name"],
            "calls": {c["config"]: {"parents": c["parents"], "K": c["K"], "T": c["T"], "epilogue": c["epilogue"]}
                      for c in desc["configs"]}}


def _peak(key, fallback):
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)[key]), "measured"
    except Exception:
        return fallback, "fallback"


def hbm_peak():
    return _peak("hbm_gbs", FALLBACK_HBM_GBS)


def tensor_peak():
    """Dense bf16 tensor throughput (burst: each call is a short kernel)."""
    return _peak("bf16_tflops", FALLBACK_BF16_TFLOPS)


def call_bound(cfg, T, hbm, tens) -> tuple:
    """(bound, roofline seconds) of one call by the metric's formula."""
    t_mem = call_bytes(cfg, T) / (hbm * 1e9)
    t_tc = call_flops(cfg, T) / (tens * 1e12)
    return ("hbm", t_mem) if t_mem >= t_tc else ("tensor", t_tc)


def route_kernel(route: str, K: int) -> tuple:
    """(kernel name, source file) of the kernel a route launches."""
    if route.startswith("tcgen05"):
        return "qg::wide_kernel", "wide.cu"
    full = (K // 64) % 8 == 0 and 1 <= (K // 64) // 8 <= 16
    return ("qg::skinny_line_kernel" if full else "qg::skinny_kernel"), "skinny.cu"


def kernel_code_sha256(path: str) -> str:
    """sha256 of a kernel source's code: comments removed and runs of
    whitespace collapsed, so that an edit of comments alone keeps the hash
    (the kernel's instructions, and so its DRAM traffic, are unchanged) and
    any change of code does not."""
    src = open(path, encoding="utf-8").read()
    src = re.sub(r"/\*.*?\*/", " ", src, flags=re.S)
    src = re.sub(r"//[^\n]*", " ", src)
    return hashlib.sha256(" ".join(src.split()).encode()).hexdigest()


def recorded_traffic(kernel_src: str, profile_name: str, keys):
    """Mean per-launch DRAM bytes over the calls `keys` ("config:T") from a
    committed ncu summary, if it was taken on this kernel's code and covers
    every one of them; else None."""
    path = os.path.join(PROFILES, profile_name)
    if not os.path.exists(path):
        return None
    want = kernel_code_sha256(kernel_src)
    rec = {}
    for line in open(path):
        if ":" in line:
            k, v = line.split(":", 1)
            rec[k.strip().lstrip("-* ")] = v.strip()
    if rec.get("kernel_code_sha256") != want:
        return None
    try:
        by_call = json.loads(rec["dram_bytes_by_call"])
        return statistics.fmean(by_call[k] for k in keys)
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

def _oracle_call(lib, wl, cfg, T, rows=None, r0=0):
    """Seconds of the oracle on one call (every parent) at width T, on
    min(T, 8) columns scaled by (T + 1) / (cols + 1) (the row dequantisation
    costs about one column; the rest is linear in T by column independence),
    optionally on `rows` weight rows (cyclic from r0) of each parent; returns
    (seconds, algorithmic bytes of that share of the call)."""
    import oracle
    K = cfg["K"]
    cols = min(T, 8)
    x = wl["x"][:cols]
    elapsed, done = 0.0, 0.0
    for p in wl["parents"]:
        N = p["N"]
        if rows is None:
            t0 = time.perf_counter()
            oracle.gemm_parent(p, x, lib=lib)
            dt = time.perf_counter() - t0
            n = N
        else:
            n = min(rows, N)
            idx = (r0 + np.arange(n)) % N
            t0 = time.perf_counter()
            if p["bits"] == synth.NVFP4:
                oracle.gemm_nvfp4(p["packed"][idx], p["scales"][idx], p["tscale"], x, n, K, lib=lib)
            else:
                oracle.gemm(p["bits"], p["packed"][idx], p["scales"][idx], x, n, K, lib=lib)
            dt = time.perf_counter() - t0
        elapsed += dt * (T + 1) / (cols + 1)
        done += weight_bytes(n, K, p["bits"]) + 2 * T * K * n / N
    return elapsed, done


def _oracle_inputs(desc):
    # the oracle runs on at most 8 columns (activations are prefix-consistent)
    return [synth.workload(c["config"], min(8, max(c["T"]))) for c in desc["configs"]]


def oracle_sample(desc, seconds: float = 12.0):
    """Time the fp64 oracle on whole calls of the workload for about `seconds`."""
    import oracle
    lib = oracle.load()
    wls = _oracle_inputs(desc)
    done_bytes, elapsed, n = 0.0, 0.0, 0
    while elapsed < seconds:
        for ci, c, T in calls(desc):
            dt, b = _oracle_call(lib, wls[ci], c, T)
            elapsed += dt
            done_bytes += b
            n += 1
            if elapsed >= seconds:
                break
    sample = (f"{n} oracle calls of workload '{desc['name']}' in step order (every parent, whole weight "
              f"matrices); widths above 8 timed on 8 columns and scaled by (T+1)/9 (cost is linear in T)")
    return done_bytes / elapsed / 1e9, elapsed, sample


def run_reference(args, desc):
    """The fp64 oracle on the host cores, as it stands: each step times it on
    a slice of the weight rows of every call of the step, sized so that the
    whole --warmup + --steps run takes about --ref-seconds; the value is the
    median over the timed steps of the slice's algorithmic bytes per second."""
    world, rank, _ = dist_env()
    if rank != 0:
        return 0
    import oracle
    lib = oracle.load()
    wls = _oracle_inputs(desc)
    n_steps = args.warmup + args.steps

    def step(rows, r0):
        el, done = 0.0, 0.0
        for ci, c, T in calls(desc):
            dt, b = _oracle_call(lib, wls[ci], c, T, rows=rows, r0=r0)
            el += dt
            done += b
        return el, done

    # calibrate: seconds per weight row of a step
    t_cal, _ = step(16, 0)
    per_row = max(t_cal / 16, 1e-7)
    max_rows = max(p["N"] for c in desc["configs"] for p in c["parents"])
    rows = int(max(1, min(max_rows, args.ref_seconds / n_steps / per_row)))
    gbs_vals = []
    r0 = 0
    for i in range(n_steps):
        el, done = step(rows, r0)
        r0 += rows
        if i >= args.warmup:
            gbs_vals.append(done / max(el, 1e-9) / 1e9)
    value = statistics.median(gbs_vals)
    sample = (f"{n_steps} steps of {rows} weight rows per parent of every call of workload '{desc['name']}' "
              f"(widths above 8 on 8 columns, scaled by (T+1)/9), about {args.ref_seconds:.0f} s in all")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * step_bytes(desc) / (value * 1e9),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": config_summary(desc),
        "cpu_baseline": {"value": value, "unit": "GB/s", "cores": 1, "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# ---------------------------------------------------------------- GPU arm

class Config:
    """One configuration's weights (R packed copies, one plan each), inputs and outputs."""

    def __init__(self, qg, torch, dev, cfg, copies, pdl, force_route=-1):
        self.cfg = cfg
        K = cfg["K"]
        Ts = cfg["T"]
        T_max = max(Ts)
        wl = synth.workload(cfg["config"], T_max, seed=0)
        self.wl = wl
        parents = wl["parents"]
        self.epi = cfg["epilogue"]
        epi_code = {"store": qg.QGEMM_EPILOGUE_STORE, "add": qg.QGEMM_EPILOGUE_ADD,
                    "swiglu": qg.QGEMM_EPILOGUE_SWIGLU}[self.epi]
        if self.epi == "swiglu":
            # the gate/up pair (parents 0 and 1) packed as one matrix with one output
            g, u = parents
            base = [qg.SwiGLUPair(g["bits"], g["N"], K, g["packed"], g["scales"], u["packed"], u["scales"], T_max)]
            self.set_bytes = qg.qgemm_pair_packed_bytes(g["N"], K, g["bits"])
            self.out_cols = [g["N"]]
        else:
            base = [qg.GroupwiseWeights(p["bits"], p["N"], K, p["packed"], p["scales"], T_max, epilogue=epi_code,
                                        tensor_scale=p.get("tscale"))
                    for p in parents]
            self.set_bytes = sum(qg.qgemm_packed_bytes(p["N"], K, p["bits"]) for p in parents)
            self.out_cols = [p["N"] for p in parents]
        self.sets = []
        for i in range(copies):
            ws = []
            for b in base:
                w = type(b).__new__(type(b))
                w.codec, w.N, w.K, w.T_max, w.epilogue, w.out = b.codec, b.N, b.K, b.T_max, b.epilogue, b.out
                w.device = dev
                w.packed = b.packed.clone() if i else b.packed
                st, w.plan = qg.qgemm_plan(b.N, K, b.codec, T_max)
                qg.check(st, "qgemm_plan")
                if self.epi != "store":
                    qg.check(qg.qgemm_plan_set_epilogue(w.plan, epi_code, qg.QGEMM_OUT_F32), "set_epilogue")
                wsb = qg.qgemm_plan_workspace_bytes(w.plan)
                w.workspace = torch.zeros(max(wsb, 16), dtype=torch.uint8, device=dev)
                qg.check(qg.qgemm_plan_bind(w.plan, w.packed, w.workspace, w.workspace.numel()), "bind")
                qg.check(qg.qgemm_plan_set_pdl(w.plan, pdl), "set_pdl")
                if getattr(b, "tensor_scale", None) is not None:
                    qg.check(qg.qgemm_plan_set_tensor_scale(w.plan, b.tensor_scale), "set_tensor_scale")
                if force_route >= 0:
                    qg.check(qg.qgemm_plan_force_route(w.plan, force_route), "force_route")
                ws.append(w)
            self.sets.append(ws)
        self.xs = {T: torch.from_numpy(wl["x"][:T].view(np.int16).copy()).to(dev) for T in Ts}
        self.ys = {T: [torch.empty((T, n), dtype=torch.float32, device=dev) for n in self.out_cols] for T in Ts}
        # the residual of a LinearAdd: fp32 [T, N], seeded
        self.rs = {T: torch.from_numpy(np.random.default_rng(T).normal(0, 8, (T, self.out_cols[0]))
                                       .astype(np.float32)).to(dev) for T in Ts} if self.epi == "add" else {}

    def call(self, qg, torch, i, T, X=None, Ys=None, Rt=None):
        ws = self.sets[i % len(self.sets)]
        X = self.xs[T] if X is None else X
        Ys = self.ys[T] if Ys is None else Ys
        s = torch.cuda.current_stream()
        if self.epi != "store":
            Rt = (self.rs[T] if Rt is None else Rt) if self.epi == "add" else None
            st = qg.qgemm_run_ex(ws[0].plan, X, T, Rt, Ys[0], s)
        elif len(ws) == 1:
            st = qg.qgemm_run(ws[0].plan, X, T, Ys[0], s)
        else:
            st = qg.qgemm_run_multi([w.plan for w in ws], X, T, Ys, s)
        if st != qg.QGEMM_OK:
            raise qg.QgemmError(st, "run")

    def launches(self, T) -> int:
        """Kernels one call at width T launches: one on every route (the
        parents of a multi-parent call share one launch, whatever their
        codecs)."""
        return 1


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

    # R calls per graph, each on its own packed copy; a single small
    # configuration rotates enough copies to exceed 3x L2 on its own
    R = max(d for d in range(1, min(args.calls_per_graph, args.steps) + 1) if args.steps % d == 0)
    blocks = args.steps // R
    cfgs = []
    for c in desc["configs"]:
        set_bytes = sum(qg.qgemm_packed_bytes(p["N"], c["K"], codec_bits(p["codec"])) for p in c["parents"])
        copies = R if len(desc["configs"]) > 1 else max(R, min(256, int(np.ceil(3 * L2_BYTES / set_bytes))))
        cfgs.append(Config(qg, torch, dev, c, copies, not args.no_pdl, args.force_route))
    torch.cuda.synchronize()

    # eager warm-up (loads the kernels), then one CUDA graph per (call, chunk
    # of the copy rotation) holding R calls, so that host launch cost stays
    # off the clock
    for ci, c, T in calls(desc):
        for i in range(2):
            cfgs[ci].call(qg, torch, i, T)
    torch.cuda.synchronize()
    assert qg.qgemm_device_status(stream) == qg.QGEMM_OK
    graphs = {}
    cap_stream = torch.cuda.Stream()
    for ci, c, T in calls(desc):
        n_chunks = (len(cfgs[ci].sets) + R - 1) // R
        gl = []
        for ch in range(n_chunks):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=cap_stream):
                for r in range(R):
                    cfgs[ci].call(qg, torch, ch * R + r, T)
            gl.append(g)
        graphs[(ci, T)] = gl
    torch.cuda.synchronize()
    keys = [(ci, T) for ci, _, T in calls(desc)]

    def replay_block(b, evs=None):
        for j, k in enumerate(keys):
            if evs is not None:
                evs[j][0].record(stream)
            gl = graphs[k]
            gl[b % len(gl)].replay()
            if evs is not None:
                evs[j][1].record(stream)

    with torch.cuda.stream(stream):
        for b in range(max(1, (args.warmup + R - 1) // R)):
            replay_block(b)
    torch.cuda.synchronize()

    # timed region: exactly K steps = K/R replays of every call's R-call graph;
    # events around each replay on the launching stream give per-call times
    ev = [[(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in keys]
          for _ in range(blocks)]
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
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
    elapsed_ms = max_over_ranks(start.elapsed_time(stop), world)
    per_call_ms = {k: [ev[b][j][0].elapsed_time(ev[b][j][1]) / R for b in range(blocks)] for j, k in enumerate(keys)}
    assert qg.qgemm_device_status(stream) == qg.QGEMM_OK
    # graph replays do not pass through the host entry points: the kernels the
    # replayed graphs hold
    launches = blocks * R * sum(cfgs[ci].launches(T) for ci, T in keys)

    sb = step_bytes(desc)
    value = world * args.steps * sb / (elapsed_ms * 1e-3) / 1e9
    hbm, hbm_kind = hbm_peak()
    tens, tens_kind = tensor_peak()
    per_call = {}
    groups = {}         # (kernel, bound) -> [time ms, bytes, flops, launches, call keys]
    for ci, c, T in calls(desc):
        k = (ci, T)
        b = call_bytes(c, T)
        fl = call_flops(c, T)
        med = statistics.median(per_call_ms[k])
        mean = statistics.fmean(per_call_ms[k])
        route = ",".join(w.route(T) for w in cfgs[ci].sets[0])
        bound, t_roof = call_bound(c, T, hbm, tens)
        name = f"{c['config']}:{T}"
        per_call[name] = {"us_per_call": 1e3 * med, "gbs": b / (med * 1e-3) / 1e9, "hbm_frac": b / (med * 1e-3) / 1e9 / hbm,
                          "tflops": fl / (med * 1e-3) / 1e12, "tensor_frac": fl / (med * 1e-3) / 1e12 / tens,
                          "bound": bound, "roofline_us": 1e6 * t_roof, "frac": 1e6 * t_roof / (1e3 * med),
                          "columns_per_s": T / (med * 1e-3), "route": route}
        kname, ksrc = route_kernel(cfgs[ci].sets[0][0].route(T), c["K"])
        acc = groups.setdefault((kname, ksrc, bound), [0.0, 0, 0, 0, []])
        n = blocks * R * cfgs[ci].launches(T)
        acc[0] += mean * blocks * R
        acc[1] += b * blocks * R
        acc[2] += fl * blocks * R
        acc[3] += n
        acc[4].append(name)

    def roofline(kname, ksrc, bound, g):
        k_ms, k_bytes, k_flops, k_launches, names = g
        traffic = recorded_traffic(os.path.join(CSRC, ksrc), f"{kname.split('::')[-1]}_{desc['name']}_traffic.md",
                                   names)
        if bound == "hbm":
            achieved = k_bytes / (k_ms * 1e-3) / 1e9
            return {"bound": "hbm", "achieved": achieved, "peak": hbm, "unit": "GB/s", "frac": achieved / hbm,
                    "traffic": traffic, "peak_source": hbm_kind, "kernel": kname, "calls": names,
                    "algorithmic_bytes_per_launch": k_bytes / k_launches, "share_of_step": 0.0}
        achieved = k_flops / (k_ms * 1e-3) / 1e12
        return {"bound": "tensor", "achieved": achieved, "peak": tens, "unit": "TFLOP/s", "frac": achieved / tens,
                "traffic": traffic, "peak_source": tens_kind, "kernel": kname, "calls": names,
                "algorithmic_flops_per_launch": k_flops / k_launches, "share_of_step": 0.0}

    total_ms = sum(g[0] for g in groups.values())
    rooflines = []
    for (kname, ksrc, bound), g in sorted(groups.items(), key=lambda kv: -kv[1][0]):
        r = roofline(kname, ksrc, bound, g)
        r["share_of_step"] = g[0] / total_ms
        rooflines.append(r)
    # the roofline of the kernel (and bound) taking most of the timed region
    roof = rooflines[0]

    # end to end: pinned host X -> device, the call, device Y -> pinned host,
    # for every call of the step
    e2e = None
    if not args.no_e2e:
        hx, hy, dx, hr, dr = {}, {}, {}, {}, {}
        for ci, c, T in calls(desc):
            cf = cfgs[ci]
            hx[(ci, T)] = torch.from_numpy(cf.wl["x"][:T].view(np.int16).copy()).pin_memory()
            hy[(ci, T)] = [torch.empty((T, n), dtype=torch.float32).pin_memory() for n in cf.out_cols]
            dx[(ci, T)] = torch.empty_like(cf.xs[T])
            if cf.epi == "add":
                hr[(ci, T)] = cf.rs[T].cpu().pin_memory()
                dr[(ci, T)] = torch.empty_like(cf.rs[T])
        h2d = sum(h.numel() * 2 for h in hx.values()) + sum(h.numel() * 4 for h in hr.values())
        d2h = sum(y.numel() * 4 for ys in hy.values() for y in ys)
        e_steps = max(1, min(args.steps, args.e2e_steps))
        # three streams: the upload of a call's X (and residual), the call
        # itself, the download of its Y; each waits for the stage before it
        # (events), so one call's copies overlap the next calls' work.  Every
        # call has its own device and pinned host buffers, and its own three
        # events (landed, done, downloaded), recorded again every step: a wait
        # takes the event as last recorded when the wait is issued.  The host
        # consumes results one step behind: before it issues step i + 1, the
        # results of step i - 1 are on the host, so at most two steps are in
        # flight and every step's Y is read back inside the timed region.
        up, down = torch.cuda.Stream(), torch.cuda.Stream()
        evs = {k: (torch.cuda.Event(), torch.cuda.Event(), torch.cuda.Event()) for k in hx}
        barrier(world)
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        prev_step = None                  # event: the previous step's results are on the host
        for i in range(e_steps):
            for ci, c, T in calls(desc):
                k = (ci, T)
                landed, done, downloaded = evs[k]
                with torch.cuda.stream(up):
                    if i > 0:
                        up.wait_event(downloaded)     # this call's buffers of the step before are free
                    dx[k].copy_(hx[k], non_blocking=True)
                    if k in hr:
                        dr[k].copy_(hr[k], non_blocking=True)
                    landed.record(up)
                stream.wait_event(landed)
                with torch.cuda.stream(stream):
                    cfgs[ci].call(qg, torch, i, T, X=dx[k], Rt=dr.get(k))
                    done.record(stream)
                down.wait_event(done)
                with torch.cuda.stream(down):
                    for y, h in zip(cfgs[ci].ys[T], hy[k]):
                        h.copy_(y, non_blocking=True)
                    downloaded.record(down)
            if prev_step is not None:
                prev_step.synchronize()       # step i - 1's results are on the host
            prev_step = torch.cuda.Event()
            prev_step.record(down)
        down.synchronize()                    # every step's results are on the host
        stream.wait_stream(down)
        e1.record(stream)
        torch.cuda.synchronize()
        e_ms = max_over_ranks(max(e0.elapsed_time(e1), 1e3 * (time.perf_counter() - t0)), world)
        e2e = {"value": world * e_steps * sb / (e_ms * 1e-3) / 1e9, "unit": "GB/s",
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": e_ms / e_steps,
               "steps": e_steps}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu:
        gbs, el, sample = oracle_sample(desc, seconds=args.cpu_seconds)
        cpu = {"value": gbs, "unit": "GB/s", "cores": 1, "kind": "oracle", "sample": sample,
               "seconds": el, "host_cores": os.cpu_count()}

    if rank == 0:
        l2 = (f"each call of a graph streams its own packed copy ({R} copies per configuration); between two "
              f"replays of a graph the rest of the step streams more than 3x the L2")
        if len(desc["configs"]) == 1:
            cf = cfgs[0]
            rot = len(cf.sets) * cf.set_bytes
            l2 = (f"rotating {len(cf.sets)} packed-weight copies ({rot / 1e6:.0f} MB"
                  + (" > 3x L2)" if rot > 3 * L2_BYTES else ", warm: less than 3x L2)"))
        config = config_summary(desc)
        config.update({"l2": l2, "parallelism": "replicas" if world > 1 else "single", "pdl": not args.no_pdl,
                       "calls_per_graph": R})
        if args.force_route >= 0:
            config["forced_route"] = args.force_route
        line = {
            "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": elapsed_ms / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": config,
            "per_call": per_call,
            "roofline": roof,
            "rooflines": rooflines,
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
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=sorted(WORKLOADS), default="all")
    ap.add_argument("--calls-per-graph", type=int, default=10,
                    help="R: calls of one (configuration, width) per CUDA graph (a divisor of --steps)")
    ap.add_argument("--force-route", type=int, default=-1,
                    help="route sweeps and profiles: force this route (qgemm_plan_force_route) where it covers T")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--e2e-steps", type=int, default=20)
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
