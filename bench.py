"""Throughput of the k-quant routed-MoE layer on GB300 (one JSON line).

A step is one forward of the whole layer (router, top-k, permutation, grouped
gate/up + SwiGLU, grouped down, slot-order combine with the shared expert and
the residual) over one batch of T rows. The default workload is the decode row
of the Qwen3.5-35B-A3B-shaped layer: T=1, H=2048, E=256, top-8, F=512, shared
expert, Q4_K gate/up, Q5_K down, fp32 hidden rows, seeded synthetic weights.

L2 (129 MB) is defeated with 16 distinct layer instances, rotated step by step,
7.8 GB in total: the weights one step touches are evicted before that instance
comes round again. Steps are CUDA-graph replays on one stream, timed with CUDA
events. The dominant unit is timed inside the graph replay too: on the decode
path it is the whole layer step (its kernels overlap by design); on the
tensor-core path the gate/up kernel, between event-record nodes that the
library places around its launches while the stream is capturing. The default
run also measures the 64-row batched decode and the 4096-row prefill on the
same layer instances and adds them to its line (``decode_t64``,
``prefill_t4096``). ``--impl reference`` times the fp64 CPU oracle on a
bounded sample of the same workload instead.
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

H, E, K_TOP, F = 2048, 256, 8, 512
EXPERT_BYTES = 2 * F * (H // 256) * 144 + H * (F // 256) * 176   # 1 900 544
QTYPE_BYTES = {"q4k": 144, "q5k": 176, "q6k": 210, "mxfp4": 136}
DOWN_TYPE = "q5k"  # the down projection's format (set from --down-type)


def expert_bytes():
    return 2 * F * (H // 256) * 144 + H * (F // 256) * QTYPE_BYTES[DOWN_TYPE]
GATEUP_EXPERT_BYTES = 2 * F * (H // 256) * 144                    # 1 179 648
KERNEL_SOURCES = {
    "decode": ["quantized_moe_transformer_gb300/csrc/moe_decode.cu",
               "quantized_moe_transformer_gb300/csrc/common.cuh",
               "quantized_moe_transformer_gb300/csrc/tc.cuh"],
    "gemv": ["quantized_moe_transformer_gb300/csrc/moe_gemv.cu",
             "quantized_moe_transformer_gb300/csrc/common.cuh"],
    "gemm_tc": ["quantized_moe_transformer_gb300/csrc/moe_gemm_tc.cu",
                "quantized_moe_transformer_gb300/csrc/common.cuh",
                "quantized_moe_transformer_gb300/csrc/tc.cuh"],
}
WORKLOADS = {
    "decode": dict(T=1, routing="uniform"),
    "decode64": dict(T=64, routing="uniform"),
    "decode64-zipf": dict(T=64, routing="zipf"),
    "prefill512": dict(T=512, routing="uniform"),
    "prefill4096": dict(T=4096, routing="uniform"),
    # the whole attention + MoE block (16 query heads, 2 KV heads, head_dim 128)
    "block1": dict(T=1, routing="uniform", block=True, pos0=4095),
    "block4096": dict(T=4096, routing="uniform", block=True, pos0=0),
}


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=1000)
    p.add_argument("--warmup", type=int, default=20)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--workload", choices=sorted(WORKLOADS), default="decode")
    p.add_argument("--layers", type=int, default=16)
    p.add_argument("--down-type", choices=["q5k", "q6k", "mxfp4"], default="q5k",
                   help="format of the down projections (q6k and mxfp4 run on the grouped GEMV kernels)")
    p.add_argument("--T", type=int, default=None, help="override the workload's row count")
    p.add_argument("--routing", choices=["uniform", "zipf"], default=None)
    p.add_argument("--gemm-threshold", type=int, default=None,
                   help="rows above which the tensor-core path is taken (library default if unset)")
    p.add_argument("--cpu-seconds", type=float, default=24.0)
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--stage-split", action="store_true",
                   help="add each stage's time per layer step inside graph replays (router, route, gateup, "
                        "down, combine, decode: event-record nodes around each stage's launches, which add a "
                        "few us each) to the line as stages_in_graph_us")
    p.add_argument("--no-extras", action="store_true",
                   help="skip the T=64 and T=4096 points the default decode run adds to its line")
    p.add_argument("--cpu-sample", type=str, default=None, help=argparse.SUPPRESS)
    p.add_argument("--record-traffic", type=str, default=None, metavar="CSV",
                   help="read an ncu --csv log with dram__bytes_read.sum / dram__bytes_write.sum of this "
                        "workload's kernels and store the dominant kernel's DRAM bytes per launch in "
                        "profiles/ncu_traffic.json (no GPU work)")
    return p.parse_args()


def workload_config(name, T, routing, layers):
    what = ("attention (16 q heads, 2 kv heads, hd 128, bf16 cache of 4096) + routed-MoE block"
            if WORKLOADS[name].get("block") else "routed-MoE layer")
    return {"workload": f"{name}: {what}, T={T} rows, H={H}, E={E}, top-{K_TOP}, F={F}, "
                        f"shared expert, Q4_K gate/up, {DOWN_TYPE.upper().replace('K', '_K')} down, "
                        f"fp32 hidden, {routing} routing",
            "T": T, "H": H, "E": E, "top_k": K_TOP, "F": F, "routing": routing,
            "down_type": DOWN_TYPE,
            "l2": f"{layers} distinct layer instances rotated ({layers * expert_bytes() * 257 / 1e9:.1f} GB "
                  f"> 129 MB L2)",
            "parallelism": "replicas"}


# ---------------------------------------------------------------- CPU oracle

def cpu_sample_main(spec: str):
    """Runs in a child process: times the oracle on forwards of ``T`` rows of
    layer instance 0 for about ``seconds`` (at least one forward) and prints
    timings, row counts and the single-row outputs as JSON."""
    from oracle import qmoe_oracle as oracle
    from quantized_moe_transformer_gb300 import inputs
    cfg = json.loads(spec)
    T = cfg["T"]
    arr = inputs.moe_layer(0, H, E, F, shared=True, routing=cfg["routing"])
    X = inputs.hidden(1000, max(64, T), H, cfg["routing"])
    times, rows, outs = [], [], []
    t_end = time.perf_counter() + cfg["seconds"]
    i = 0
    while True:
        x = X[i:i + 1] if T == 1 else X[:T]
        t0 = time.perf_counter()
        out = oracle.moe_forward(x, arr, K_TOP)
        times.append(time.perf_counter() - t0)
        rows.append(x.shape[0])
        if T == 1:
            outs.append(out[0].tolist())
        i += 1
        if T > 1 or time.perf_counter() > t_end or i >= 64:
            break
    print(json.dumps({"times": times, "rows": rows, "outs": outs}))


def run_cpu_sample(routing, T, seconds, threads=1):
    env = dict(os.environ)
    for v in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
        env[v] = str(threads)
    spec = json.dumps({"routing": routing, "T": T, "seconds": seconds})
    r = subprocess.run([sys.executable, os.path.abspath(__file__), "--cpu-sample", spec],
                       capture_output=True, text=True, env=env, cwd=ROOT)
    if r.returncode != 0:
        raise RuntimeError(r.stderr)
    return json.loads(r.stdout.strip().splitlines()[-1])


def reference_main(args, rank, world):
    """The oracle as the reference arm: each step is one row through the layer."""
    if rank != 0:
        return
    from oracle import qmoe_oracle as oracle
    from quantized_moe_transformer_gb300 import inputs
    wl = WORKLOADS[args.workload]
    arr = inputs.moe_layer(0, H, E, F, shared=True, routing=wl["routing"])
    n = args.warmup + args.steps
    X = inputs.hidden(1000, n, H, wl["routing"])
    for i in range(args.warmup):
        oracle.moe_forward(X[i:i + 1], arr, K_TOP)
    t0 = time.perf_counter()
    for i in range(args.warmup, n):
        oracle.moe_forward(X[i:i + 1], arr, K_TOP)
    dt = time.perf_counter() - t0
    value = args.steps / dt
    cores = len(os.sched_getaffinity(0))
    line = {"metric": "MoE-layer tokens/s", "value": value, "unit": "tokens/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * dt / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "impl": "reference",
            "config": workload_config(args.workload, wl["T"], wl["routing"], 1),
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                             "sample": f"one row per step of the {args.workload} workload "
                                       f"(numpy fp64 oracle, {cores} cores visible)",
                             "cpu_model": cpu_model()},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line))


# ---------------------------------------------------------------- GPU arm

class ClockSampler:
    def __init__(self, index):
        self.p = None
        self.index = index

    def __enter__(self):
        q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
        try:
            self.p = subprocess.Popen(["nvidia-smi", "-i", str(self.index), f"--query-gpu={q}",
                                       "--format=csv,noheader,nounits", "-lms", "100"],
                                      stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.p = None
        time.sleep(0.3)
        return self

    def __exit__(self, *a):
        self.summary = None
        if self.p is None:
            return
        time.sleep(0.2)
        self.p.terminate()
        out, _ = self.p.communicate(timeout=10)
        sm, mx, reasons = [], 0.0, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = max(mx, float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if sm:
            self.summary = {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx,
                            "reasons": sorted(reasons), "samples": len(sm)}


def make_layer_on_device(torch, seed, routing, device, from_arrays=None):
    """Layer instance from device RNG (instances 1..N-1) or host arrays (0)."""
    from quantized_moe_transformer_gb300 import binding as qb
    if from_arrays is not None:
        return qb.MoeLayer.from_arrays(from_arrays, K_TOP, device)
    g = torch.Generator(device=device)
    g.manual_seed(seed)

    def blocks(n, nb):
        # the distributions of inputs.packed_blocks: Q4_K/Q5_K d, dmin in
        # [2^-12, 2^-10]; Q6_K d in [2^-14, 2^-12]; MXFP4 exponents 119..124
        b = torch.randint(0, 256, (n, nb), dtype=torch.uint8, device=device, generator=g)
        if nb in (144, 176):
            dd = torch.empty((n, 2), device=device).uniform_(2.0**-12, 2.0**-10, generator=g)
            b[:, 0:4] = dd.half().view(torch.uint8).reshape(n, 4)
        elif nb == 210:
            dd = torch.empty((n, 1), device=device).uniform_(2.0**-14, 2.0**-12, generator=g)
            b[:, 0:2] = dd.half().view(torch.uint8).reshape(n, 2)
        else:
            b[:, 0:8] = torch.randint(119, 125, (n, 8), dtype=torch.uint8, device=device, generator=g)
        return b

    Wr = torch.randn((H, E), device=device, generator=g) * 0.02
    if routing == "zipf":
        rank = torch.randperm(E, device=device, generator=g).double()
        Wr[0] = (-1.1 * torch.log1p(rank)).float()
    nb = H // 256
    Wg = blocks(E * F * nb, 144).reshape(E, F, nb, 144)
    Wu = blocks(E * F * nb, 144).reshape(E, F, nb, 144)
    db = QTYPE_BYTES[DOWN_TYPE]
    Wd = blocks(E * H * (F // 256), db).reshape(E, H, F // 256, db)
    Sg = blocks(F * nb, 144).reshape(F, nb, 144)
    Su = blocks(F * nb, 144).reshape(F, nb, 144)
    Sd = blocks(H * (F // 256), db).reshape(H, F // 256, db)
    return qb.MoeLayer(H, E, K_TOP, F, Wr.contiguous(), Wg, Wu, Wd, Sg, Su, Sd, "q4k", DOWN_TYPE)


CTX = 4096


def make_block_on_device(torch, qb, seed, moe_layer, device):
    """Attention weights (Q4_K) and RMSNorm gains of one block instance."""
    g = torch.Generator(device=device)
    g.manual_seed(seed)

    def blocks(rows, nb):
        b = torch.randint(0, 256, (rows * nb, 144), dtype=torch.uint8, device=device, generator=g)
        dd = torch.empty((rows * nb, 2), device=device).uniform_(2.0**-12, 2.0**-10, generator=g)
        b[:, 0:4] = dd.half().view(torch.uint8).reshape(rows * nb, 4)
        return b.reshape(rows, nb, 144)

    g1 = 1.0 + 0.1 * torch.randn(H, device=device, generator=g)
    g2 = 1.0 + 0.1 * torch.randn(H, device=device, generator=g)
    return qb.Block(H, 16, 2, 128, g1, g2, blocks(2048, 8), blocks(256, 8), blocks(256, 8), blocks(H, 8),
                    moe_layer)


def block_moe_ws_offset(qb, blk, T, pos0):
    """Byte offset of the MoE layer's workspace inside a block workspace."""
    a = int(qb._block_lib().qmoe_attn_workspace_bytes(__import__("ctypes").byref(blk.desc), T, pos0))
    row = (4 * T * H + 255) // 256 * 256
    return a + 2 * row


def max_over_ranks(ms, world, device):
    """The slowest rank's timed-region milliseconds (every rank gets it)."""
    if world == 1:
        return ms
    import torch
    import torch.distributed as dist
    t = torch.tensor([ms], device=device, dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(rows_per_step, steps, world, ms):
    """Whole-job rows per second: every rank runs its own replica of the
    workload (rows_per_step rows per step), timed by the slowest rank."""
    return rows_per_step * steps * world / (ms / 1e3)


def source_sha(paths):
    h = hashlib.sha256()
    for p in paths:
        with open(os.path.join(ROOT, p), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def cpu_model() -> str:
    """The host CPU's model name (lscpu, else /proc/cpuinfo, else platform)."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    try:
        for line in open("/proc/cpuinfo"):
            if line.lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except OSError:
        pass
    import platform
    return platform.processor() or platform.machine()


def cpu_baseline(routing, seconds):
    """The oracle (numpy fp64) on the host cores: single-row forwards (T=1) and
    one 64-row forward (T=64), each on one thread and on every core this
    process may run on. Returns the cpu_baseline record and the T=1 outputs
    (for the parity spot check)."""
    cores = len(os.sched_getaffinity(0))
    points, outs1 = [], None
    for T in (1, 64):
        for threads in sorted({1, cores}):
            res = run_cpu_sample(routing, T, seconds / 4, threads=threads)
            n_rows = sum(res["rows"])
            tps = n_rows / sum(res["times"])
            points.append({"T": T, "threads": threads, "tokens_per_s": tps, "rows": n_rows,
                           "seconds": sum(res["times"])})
            if T == 1 and threads == 1:
                outs1 = res
    best1 = max(p["tokens_per_s"] for p in points if p["T"] == 1)
    cores_best = max((p for p in points if p["T"] == 1), key=lambda p: p["tokens_per_s"])["threads"]
    rec = {"value": best1, "unit": "tokens/s", "cores": cores_best, "kind": "oracle",
           "sample": "numpy fp64 oracle on layer instance 0: single-row forwards (T=1) for about "
                     f"{seconds / 4:.0f} s and one 64-row forward (T=64), each on 1 thread and on all "
                     f"{cores} cores; value = the faster T=1 rate",
           "cpu_model": cpu_model(), "cores_visible": cores, "points": points}
    return rec, outs1


def make_inputs(torch, NL, T, H_, routing, device, seed):
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    Xs = torch.randn((NL, T, H_), device=device, generator=g)
    if routing == "zipf":
        Xs[:, :, 0] = 1.0
    return Xs


def time_graphs(torch, step, NL, steps, warmup, stream, world, device, clock_index=None):
    """Captures one graph of NL steps (and one per step for the remainder),
    replays warmup steps, then times ``steps`` steps with CUDA events on
    ``stream``. Returns (ms over the timed region, max over ranks; clocks)."""
    import torch.distributed as dist
    macro = torch.cuda.CUDAGraph()
    with torch.cuda.graph(macro, stream=stream):
        for i in range(NL):
            step(i, stream)
    singles = []
    for i in range(steps % NL):
        gph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gph, stream=stream):
            step(i, stream)
        singles.append(gph)
    for _ in range(max(1, -(-warmup // NL))):
        macro.replay()
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    clk = ClockSampler(clock_index) if clock_index is not None else None
    if clk:
        clk.__enter__()
    with torch.cuda.stream(stream):
        ev0.record(stream)
        for _ in range(steps // NL):
            macro.replay()
        for gph in singles:
            gph.replay()
        ev1.record(stream)
    torch.cuda.synchronize()
    if clk:
        clk.__exit__()
    ms = max_over_ranks(ev0.elapsed_time(ev1), world, device)
    if world > 1:
        dist.barrier()
    return ms, (clk.summary if clk else None)


def gateup_in_graph_us(torch, qb, step, NL, stream, replays=3):
    """Average duration of the gate/up kernel inside a graph replay: the
    library brackets each gate/up launch with events, which stream capture turns
    into event-record nodes of the graph; after each replay the times of that
    replay's launches are read back."""
    return stage_in_graph_us(torch, qb, step, NL, stream, "gateup", replays)


def stage_in_graph_us(torch, qb, step, NL, stream, stage, replays=3):
    """(Average time per bracketed launch group of ``stage`` inside graph
    replays of NL layer steps, number of groups read.)"""
    with torch.cuda.stream(stream):
        qb.profile_start(stage)             # events created outside the capture
        for i in range(NL):
            step(i, stream)
        qb.profile_stop()
        torch.cuda.synchronize()
        qb.profile_start(stage)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for i in range(NL):
                step(i, stream)
    tot, n = 0.0, 0
    for _ in range(replays):
        g.replay()
        torch.cuda.synchronize()
        ms, k = qb.profile_read()
        tot += ms
        n += k
    qb.profile_stop()
    return (1e3 * tot / n if n else 0.0), n


def stages_per_step_us(torch, qb, step, NL, stream, replays=3):
    """Each stage's time per layer step inside graph replays (a stage with no
    launches on the path reads 0)."""
    out = {}
    for stage in ("router", "route", "gateup", "down", "combine", "decode"):
        us, n = stage_in_graph_us(torch, qb, step, NL, stream, stage, replays)
        out[stage] = round(us * n / (replays * NL), 2)
    return out


def distinct_experts(torch, qb, layers, step, ws, ws_off, T, NL, stream):
    L = layers[0].workspace_layout(T)
    U = []
    with torch.cuda.stream(stream):
        for i in range(NL):
            step(i, stream)
            o = ws_off + L.ids
            ids = ws[o:o + 4 * T * K_TOP].view(torch.int32)
            U.append(int(torch.unique(ids).numel()))
    torch.cuda.synchronize()
    return float(np.mean(U))


def layer_bytes(u_mean, T):
    return (u_mean + 1) * expert_bytes() + H * E * 4 + 2 * T * H * 4


def layer_flops(T):
    return 2.0 * T * (H * E + 3 * H * F * (K_TOP + 1))


def measure_layer(torch, qb, layers, T, routing, steps, warmup, stream, world, device, peaks, rank, clocks=False):
    """One workload of the MoE layer: step time from graph replays, the
    dominant unit's time, roofline fractions."""
    NL = len(layers)
    Xs = make_inputs(torch, NL, T, H, routing, device, 7 + rank + 131 * T)
    outs = torch.empty_like(Xs)
    ws = layers[0].workspace(T)

    def step(i, s=None):
        qb.moe_forward(layers[i % NL], Xs[i % NL], Xs[i % NL], out=outs[i % NL], ws=ws, stream=s)

    with torch.cuda.stream(stream):
        n0 = qb.launch_count()
        step(0, stream)
        launches_per_step = qb.launch_count() - n0
        for i in range(max(warmup, 3)):
            step(i, stream)
    torch.cuda.synchronize()
    if qb.query_status(stream) != 0:
        raise RuntimeError("device status word set during warm-up")
    path = qb.last_path()
    ms, clk = time_graphs(torch, step, NL, steps, warmup, stream, world, device,
                          clock_index=device.index if clocks else None)
    step_s = ms / steps / 1e3
    u_mean = distinct_experts(torch, qb, layers, step, ws, 0, T, NL, stream)
    lb = layer_bytes(u_mean, T)
    hbm_peak = peaks.get("hbm_gbs") or 6800.0
    hbm_src = "measured hbm_gbs (burst copy)" if peaks.get("hbm_gbs") else "fallback 6.8 TB/s"
    rows_h = T * K_TOP + T
    rec = {"T": T, "routing": routing, "path": path, "steps": steps, "ms_per_step": ms / steps,
           "tokens_per_s": T / step_s, "launches_per_step": launches_per_step,
           "distinct_experts_mean": u_mean,
           "layer_hbm": {"achieved": lb / step_s / 1e9, "unit": "GB/s", "frac": lb / step_s / 1e9 / hbm_peak,
                         "alg_bytes_per_step": lb},
           "layer_tflops": {"achieved": layer_flops(T) / step_s / 1e12, "unit": "TFLOP/s"}}
    if path == "gemm_tc":
        us, n = gateup_in_graph_us(torch, qb, step, NL, stream)
        alg = 2.0 * rows_h * H * 2 * F
        peak = peaks.get("bf16_tflops") or 1900.0
        rec["roofline"] = {"bound": "tensor", "kernel": "moe_tc_kernel<gate/up> (tcgen05)",
                           "achieved": alg / (us / 1e6) / 1e12, "peak": peak,
                           "peak_source": "measured bf16_tflops (burst cuBLAS)" if peaks.get("bf16_tflops")
                           else "fallback 1.9 PFLOP/s",
                           "unit": "TFLOP/s", "frac": alg / (us / 1e6) / 1e12 / peak,
                           "algorithmic_per_launch": alg, "avg_launch_us": us, "launches_timed": n,
                           "timing": "event-record nodes around each gate/up launch inside the graph replay"}
        rec["layer_tflops"]["frac"] = rec["layer_tflops"]["achieved"] / peak
    else:
        # the decode path's kernels overlap by design (programmatic dependent
        # launch), so its dominant unit is the whole layer step
        kname = ("decode chain: router + expert kernels (whole layer step inside the graph replay)"
                 if path == "decode" else "whole layer step (grouped GEMV path) inside the graph replay")
        rec["roofline"] = {"bound": "hbm", "kernel": kname, "achieved": lb / step_s / 1e9, "peak": hbm_peak,
                           "peak_source": hbm_src, "unit": "GB/s", "frac": lb / step_s / 1e9 / hbm_peak,
                           "algorithmic_per_launch": lb, "avg_launch_us": step_s * 1e6,
                           "launches_timed": steps, "timing": "graph replay of the whole layer"}
    return rec, clk, step, ws, outs


def ours_main(args, rank, world, local_rank):
    import torch

    from quantized_moe_transformer_gb300 import binding as qb
    from quantized_moe_transformer_gb300 import build, inputs

    build.build()
    if args.gemm_threshold is not None:
        qb.set_gemm_threshold(args.gemm_threshold)
    device = torch.device("cuda", local_rank)
    torch.cuda.set_device(device)
    wl = WORKLOADS[args.workload]
    T, routing = wl["T"], wl["routing"]
    if args.T is not None:
        T = args.T
    if args.routing is not None:
        routing = args.routing
    NL = args.layers
    peaks = {}
    pk = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(pk):
        peaks = json.load(open(pk))
    hbm_peak = peaks.get("hbm_gbs") or 6800.0

    is_block = wl.get("block", False)
    pos0 = wl.get("pos0", 0)
    arr0 = inputs.moe_layer(0, H, E, F, shared=True, routing=routing, down_type=DOWN_TYPE)
    layers = [make_layer_on_device(torch, 1000 * rank + i, routing, device,
                                   arr0 if i == 0 else None) for i in range(NL)]
    stream = torch.cuda.Stream(device=device)

    if is_block:
        rec, clk, e2e = measure_block(torch, qb, layers, T, pos0, args, stream, world, device, rank, peaks)
        path = rec["path"]
    else:
        rec, clk, step, ws, outs = measure_layer(torch, qb, layers, T, routing, args.steps, args.warmup, stream,
                                                 world, device, peaks, rank, clocks=True)
        path = rec["path"]
        attach_traffic(rec, args.workload)
        if args.stage_split:
            rec["stages_in_graph_us"] = stages_per_step_us(torch, qb, step, len(layers), stream)

        # end to end through the C ABI on host buffers (pinned), copies inside
        Xh = torch.randn((NL, T, H), generator=torch.Generator().manual_seed(11)).pin_memory()
        if routing == "zipf":
            Xh[:, :, 0] = 1.0
        Oh = torch.empty_like(Xh).pin_memory()
        hws = torch.empty(qb.host_workspace_bytes(layers[0], T), dtype=torch.uint8, device=device)
        n_e2e = min(args.steps, 400)
        calls = [(layers[i], Xh[i], Oh[i]) for i in range(NL)]  # each layer instance's own buffers
        # warm-up: every layer's host call twice (the second captures the graph
        # that later calls with the same arguments replay)
        for i in range(2 * NL + 1):
            lay, xi, oi = calls[i % NL]
            qb.moe_forward_host(lay, xi, out=oi, ws=hws, stream=stream)
        t0 = time.perf_counter()
        for i in range(n_e2e):
            lay, xi, oi = calls[i % NL]
            qb.moe_forward_host(lay, xi, out=oi, ws=hws, stream=stream)
        dt = time.perf_counter() - t0
        e2e = {"value": T * n_e2e * world / dt, "unit": "tokens/s", "h2d_bytes_per_step": T * H * 4,
               "d2h_bytes_per_step": T * H * 4, "steps": n_e2e,
               "api": "qmoe_moe_forward_host (pinned host buffers, one call per step)"}

    ms = rec["ms_per_step"] * args.steps
    value = job_throughput(T, args.steps, world, ms)

    # the other two points of the metric (batched decode at 64 rows, prefill
    # at 4096 rows) on the same layer instances, when the default runs
    extras = {}
    if not is_block and not args.no_extras and args.workload == "decode" and args.T is None:
        for key, Tx, st in (("decode_t64", 64, 400), ("prefill_t4096", 4096, 48)):
            r, _, _, _, _ = measure_layer(torch, qb, layers, Tx, routing, st, 3 * NL // 2, stream, world, device,
                                          peaks, rank)
            r["tokens_per_s"] *= world
            attach_traffic(r, {"decode_t64": "decode64", "prefill_t4096": "prefill4096"}[key])
            extras[key] = r
        torch.cuda.empty_cache()

    # CPU baseline and a parity spot check of instance 0 on the same rows
    cpu = None
    parity = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline and not is_block:
        cpu, res = cpu_baseline(routing, args.cpu_seconds)
        n = len(res["outs"])
        Xp = torch.from_numpy(inputs.hidden(1000, 64, H, routing)[:n]).to(device)
        got = np.stack([qb.moe_forward(layers[0], Xp[i:i + 1]).cpu().numpy()[0] for i in range(n)])
        ref = np.array(res["outs"])
        parity = {"rows": n, "max_abs_err_over_max_ref": float(np.max(np.abs(got - ref)) / np.max(np.abs(ref)))}

    if rank == 0:
        line = {"metric": "MoE-layer tokens/s", "value": value, "unit": "tokens/s", "n_gpus": world,
                "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms / args.steps,
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
                "dtype": "bf16" if path == "gemm_tc" else "f32", "data": "synthetic",
                "config": workload_config(args.workload, T, routing, NL),
                "path": path, "roofline": rec["roofline"],
                "layer_hbm": rec.get("layer_hbm"), "layer_tflops": rec.get("layer_tflops"),
                "cpu_baseline": cpu, "e2e": e2e, "gpu_launches": rec["launches_per_step"] * args.steps,
                "launches_per_step": rec["launches_per_step"], "clocks": clk, "parity": parity}
        if "stages_in_graph_us" in rec:
            line["stages_in_graph_us"] = rec["stages_in_graph_us"]
        line.update(extras)
        print(json.dumps(line))


def measure_block(torch, qb, layers, T, pos0, args, stream, world, device, rank, peaks):
    """The attention + MoE block (config of the block workloads)."""
    NL = len(layers)
    blocks_ = [make_block_on_device(torch, qb, 5000 * rank + i, layers[i], device) for i in range(NL)]
    g = torch.Generator(device=device)
    g.manual_seed(7 + rank)
    Xs = torch.randn((NL, T, H), device=device, generator=g)
    outs = torch.empty_like(Xs)
    kcs = [torch.randn((CTX, 2, 128), device=device, generator=g).to(torch.bfloat16) for _ in range(NL)]
    vcs = [torch.randn((CTX, 2, 128), device=device, generator=g).to(torch.bfloat16) for _ in range(NL)]
    ws = blocks_[0].workspace(T, pos0)

    def step(i, s=None):
        j = i % NL
        qb.block_forward(blocks_[j], Xs[j], kcs[j], vcs[j], pos0, out=outs[j], ws=ws, stream=s)

    with torch.cuda.stream(stream):
        n0 = qb.launch_count()
        step(0, stream)
        launches_per_step = qb.launch_count() - n0
        for i in range(max(args.warmup, 3)):
            step(i, stream)
    torch.cuda.synchronize()
    path = qb.last_path()
    ms, clk = time_graphs(torch, step, NL, args.steps, args.warmup, stream, world, device,
                          clock_index=device.index)
    step_s = ms / args.steps / 1e3
    rec = {"path": path, "ms_per_step": ms / args.steps, "launches_per_step": launches_per_step,
           "roofline": {"bound": "tensor" if path == "gemm_tc" else "hbm", "kernel": "whole block step",
                        "achieved": None, "peak": None, "unit": None, "frac": None, "traffic": None,
                        "avg_launch_us": step_s * 1e6,
                        "note": "block steps are reported, not gated; the MoE layer carries the roofline"}}
    Xh = torch.randn((NL, T, H), generator=torch.Generator().manual_seed(11)).pin_memory()
    Oh = torch.empty_like(Xh).pin_memory()
    Xd = torch.empty((T, H), device=device)
    n_e2e = min(args.steps, 200)
    with torch.cuda.stream(stream):
        for i in range(3 + n_e2e):
            if i == 3:
                torch.cuda.synchronize()
                t0 = time.perf_counter()
            j = i % NL
            Xd.copy_(Xh[j], non_blocking=True)
            qb.block_forward(blocks_[j], Xd, kcs[j], vcs[j], pos0, out=outs[j], ws=ws, stream=stream)
            Oh[j].copy_(outs[j], non_blocking=True)
            stream.synchronize()
    dt = time.perf_counter() - t0
    e2e = {"value": T * n_e2e * world / dt, "unit": "tokens/s", "h2d_bytes_per_step": T * H * 4,
           "d2h_bytes_per_step": T * H * 4, "steps": n_e2e,
           "api": "binding.block_forward with pinned host copies on the same stream"}
    return rec, clk, e2e


# kernels whose DRAM bytes make up the dominant unit of each path: the decode
# path's chained kernels per step, the grouped gate/up kernel otherwise
TRAFFIC_KERNELS = {
    "decode": ("decode_router_kernel", ("decode_router_kernel", "decode_experts_kernel")),
    "gemm_tc": ("moe_tc_kernel<1,", ("moe_tc_kernel<1,",)),
    "gemv": ("gateup_gemv_kernel", ("gateup_gemv_kernel",)),
}


def attach_traffic(rec, workload):
    """rec["roofline"]["traffic"]: the dominant kernel's DRAM bytes per launch
    recorded in profiles/ncu_traffic.json for this path and workload, when the
    record was taken on the current kernel sources (else None)."""
    path = rec["path"]
    kernel_sha = source_sha(KERNEL_SOURCES[path])
    traffic = None
    tf = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    if os.path.exists(tf):
        r = json.load(open(tf)).get(f"{path}:{workload}")
        if r and r.get("source_sha") == kernel_sha:
            traffic = r["dram_bytes_per_launch"]
    rec["roofline"]["traffic"] = traffic
    rec["roofline"]["kernel_source_sha"] = kernel_sha


def record_traffic(args):
    """profiles/ncu_traffic.json["path:workload"] = DRAM bytes per dominant
    launch (per step for the decode chain), from an ncu CSV log."""
    import csv
    path = "decode" if WORKLOADS[args.workload].get("T", 1) <= 4 else "gemm_tc"
    first, names = TRAFFIC_KERNELS[path]
    per_launch = {}
    with open(args.record_traffic) as f:
        rows = [r for r in csv.reader(f) if len(r) > 5]
    hdr = rows[0]
    ki, mi, vi, ii = hdr.index("Kernel Name"), hdr.index("Metric Name"), hdr.index("Metric Value"), hdr.index("ID")
    ui = hdr.index("Metric Unit") if "Metric Unit" in hdr else None
    scale = {"byte": 1.0, "Kbyte": 1e3, "Mbyte": 1e6, "Gbyte": 1e9}
    for r in rows[1:]:
        name = r[ki].replace(" ", "")
        if not any(n.replace(" ", "") in name for n in names):
            continue
        if r[mi] not in ("dram__bytes_read.sum", "dram__bytes_write.sum"):
            continue
        d = per_launch.setdefault(r[ii], {"name": name, "bytes": 0.0})
        d["bytes"] += float(r[vi].replace(",", "")) * (scale[r[ui]] if ui is not None else 1.0)
    units = sum(1 for d in per_launch.values() if first.replace(" ", "") in d["name"])
    total = sum(d["bytes"] for d in per_launch.values())
    if units == 0:
        raise SystemExit(f"no {first} launch in {args.record_traffic}")
    tf = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    data = json.load(open(tf)) if os.path.exists(tf) else {}
    data[f"{path}:{args.workload}"] = {"dram_bytes_per_launch": total / units, "launches": units,
                                       "source_sha": source_sha(KERNEL_SOURCES[path]),
                                       "kernels": sorted({d["name"][:60] for d in per_launch.values()})}
    with open(tf, "w") as f:
        json.dump(data, f, indent=1, sort_keys=True)
    print(json.dumps(data[f"{path}:{args.workload}"]))


def main():
    global DOWN_TYPE
    args = parse()
    DOWN_TYPE = args.down_type
    if args.record_traffic:
        record_traffic(args)
        return
    if args.cpu_sample:
        cpu_sample_main(args.cpu_sample)
        return
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.gpus != world:
        # one process per GPU: N replicas need N ranks from a launcher
        sys.exit(f"bench.py: --gpus {args.gpus} but WORLD_SIZE={world}; launch N ranks with "
                 f"python -m torch.distributed.run --nproc-per-node {args.gpus} bench.py --gpus {args.gpus}")
    if args.impl == "reference":
        reference_main(args, rank, world)
        return
    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl")
    ours_main(args, rank, world, local_rank)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
