"""Benchmark of the weight-only MXFP4 decode matvec path on one GB300.

One step = the 24 MXFP4 gate/up SwiGLU layers (layers 0:24) of the
SmolLM3-3B-shaped decode stack at batch 1: each layer K=2048, N=11008, fp32
row postscale, its own weights and its own bf16 activation vector, the 24
calls chained with programmatic dependent launch in one CUDA graph.  The
layers' weights (577 MB) exceed L2 several times, so every step streams from
HBM.

Prints one JSON line.  `value` is the MXFP4 layer's algorithmic weight
traffic per second (GB/s; µs per layer beside it) and `roofline` is that
kernel's.  The full 36-layer stack (with the 12 bf16 layers), the other
workloads (single layer over rotating copies, batch sweep, MoE, INT4) and
the CPU oracle baseline (one thread, and all host cores) ride along in the
same line.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl thinmx|reference]

Under torchrun (N > 1) each rank runs an independent replica (the path has no
exchange step); the step time is the max over ranks.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0


# ---------------------------------------------------------------------------
def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        try:
            d = json.load(open(p))
            hbm = d.get("hbm_gbs") or d.get("hbm_GBs")
            if hbm:
                return float(hbm), "measured", d
        except Exception:
            pass
    return FALLBACK_HBM_GBS, "fallback", {}


def tensor_peak_tflops():
    """Dense f16/bf16 tensor peak (TFLOP/s): the measured bf16 burst figure
    when the pool's measurements exist, else the fallback."""
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        try:
            d = json.load(open(p))
            v = d.get("bf16_tflops")
            if v:
                return float(v)
        except Exception:
            pass
    return FALLBACK_BF16_TFLOPS


class Clocks:
    """nvidia-smi sampling during the timed region."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *a):
        self.lines = []
        if self.proc is not None:
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except Exception:
                self.proc.kill()
                out = ""
            self.lines = [l for l in out.splitlines() if l.strip()]

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for l in getattr(self, "lines", []):
            f = [x.strip() for x in l.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx.append(float(f[2]))
            except ValueError:
                continue
            for nm, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(nm)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx),
                "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------------------
def build_stack(torch, synth, loader, cfg, device):
    """Device-resident weights of the 36-layer stack (seeded synthetic draws)."""
    layers = []
    for l in range(cfg.layers):
        x = synth.torch_normal((1, cfg.k), 1.0, cfg.wid, l, 2, device).to(torch.bfloat16)
        h = torch.empty((1, cfg.n), dtype=torch.bfloat16, device=device)
        if l < cfg.mxfp4_layers:
            wg = synth.torch_normal((cfg.n, cfg.k), synth.WEIGHT_STD, cfg.wid, l, 0, device)
            wu = synth.torch_normal((cfg.n, cfg.k), synth.WEIGHT_STD, cfg.wid, l, 1, device)
            pg = synth.torch_uniform((cfg.n,), 0.9, 1.1, cfg.wid, l, 3, device)
            pu = synth.torch_uniform((cfg.n,), 0.9, 1.1, cfg.wid, l, 4, device)
            packed = loader.mxfp4_gate_up_from_f32(wg, wu, pg, pu)
            del wg, wu
            layers.append(("mxfp4", packed, x, h))
        else:
            wg = synth.torch_normal((cfg.n, cfg.k), synth.WEIGHT_STD, cfg.wid, l, 0,
                                    device).to(torch.bfloat16)
            wu = synth.torch_normal((cfg.n, cfg.k), synth.WEIGHT_STD, cfg.wid, l, 1,
                                    device).to(torch.bfloat16)
            layers.append(("bf16", (wg, wu), x, h))
    torch.cuda.synchronize()
    return layers


def run_layer(thinmx, cfg, layer, x=None, h=None):
    kind, w, x0, h0 = layer
    x = x0 if x is None else x
    h = h0 if h is None else h
    if kind == "mxfp4":
        thinmx.tt_mxfp4_swiglu_matvec(w, cfg.n, cfg.k, x, 1, h)
    else:
        thinmx.tt_bf16_swiglu_matvec(w[0], w[1], cfg.n, cfg.k, x, 1, h)


def capture(torch, fn):
    fn()  # eager warm-up (sets kernel attributes outside capture)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fn()
    torch.cuda.synchronize()
    return g


def replay_times(torch, g, reps):
    """Per-replay CUDA-event times (ms) of `reps` back-to-back replays on the
    current stream; the events sit between replays and add no sync."""
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(reps + 1)]
    ev[0].record()
    for i in range(reps):
        g.replay()
        ev[i + 1].record()
    torch.cuda.synchronize()
    return [ev[i].elapsed_time(ev[i + 1]) for i in range(reps)]


def time_graph(torch, g, reps=20, warm=3):
    """Median of at least 20 timed replays (ms per replay), after `warm`."""
    for _ in range(warm):
        g.replay()
    torch.cuda.synchronize()
    return statistics.median(replay_times(torch, g, max(20, reps)))


def stack_bytes(cfg):
    mx = 2 * (cfg.n * cfg.k // 2 + cfg.n * cfg.k // 32 + 4 * cfg.n) + 2 * cfg.k + 2 * cfg.n
    bf = 2 * (cfg.n * cfg.k * 2) + 2 * cfg.k + 2 * cfg.n
    return mx, bf


def gate_up_bytes(n, k, m, postscale=True):
    return 2 * (n * k // 2 + n * k // 32 + (4 * n if postscale else 0)) + 2 * m * k + 2 * m * n


# ---------------------------------------------------------------------------
def host_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:  # pragma: no cover
        return os.cpu_count() or 1


def oracle_layer(rows=None):
    """One MXFP4 gate/up layer of the headline workload (K=2048, N=11008,
    with postscales), drawn and quantised by the oracle (setup, not timed).
    `rows` keeps only the first rows (a bounded sample)."""
    import oracle
    from bit_weight_only_mxfp4_gb300 import synth
    cfg = synth.STACK
    rows = rows or cfg.n
    d = synth.gate_up_inputs(cfg.wid, 0, rows, cfg.k)
    gc, gs, _ = oracle.mxfp4_quantize(d["wg"])
    uc, us, _ = oracle.mxfp4_quantize(d["wu"])
    return {"gate": (gc, gs, d["pg"]), "up": (uc, us, d["pu"]), "x": d["x"], "rows": rows,
            "n": cfg.n, "k": cfg.k, "bytes": gate_up_bytes(rows, cfg.k, 1)}


def oracle_layer_call(L, threads, pool=None):
    """The oracle's SwiGLU matvec over the layer's rows: one call, or (threads
    > 1) contiguous row ranges on `threads` host threads, the oracle's own
    parallelisation over output rows (the C calls release the GIL)."""
    import oracle
    if threads <= 1:
        return oracle.mxfp4_swiglu_matvec(L["gate"], L["up"], L["x"])
    rows = L["rows"]
    cuts = [rows * i // threads for i in range(threads + 1)]

    def part(i):
        a, b = cuts[i], cuts[i + 1]
        return oracle.mxfp4_swiglu_matvec(tuple(v[a:b] for v in L["gate"]),
                                          tuple(v[a:b] for v in L["up"]), L["x"])
    return list(pool.map(part, range(threads)))


def oracle_leg(L, threads, target_s):
    """Times the oracle on layer L until about target_s seconds have passed."""
    import concurrent.futures as cf
    pool = cf.ThreadPoolExecutor(max_workers=threads) if threads > 1 else None
    try:
        oracle_layer_call(L, threads, pool)  # first touch of the pages
        t_total, calls = 0.0, 0
        while t_total < target_s or calls < 2:
            t0 = time.perf_counter()
            oracle_layer_call(L, threads, pool)
            t_total += time.perf_counter() - t0
            calls += 1
    finally:
        if pool is not None:
            pool.shutdown()
    return {"value": L["bytes"] * calls / t_total / 1e9, "unit": "GB/s", "cores": threads,
            "kind": "oracle", "us_per_layer": round(t_total / calls * 1e6, 1),
            "sample": f"MXFP4 gate/up layer 0 of the stack ({L['rows']} of {L['n']} rows, "
                      f"K={L['k']}), {calls} calls, {t_total:.1f} s, fp64, "
                      + ("1 thread" if threads == 1 else
                         f"{threads} threads over output rows"),
            "seconds": round(t_total, 2)}


def cpu_baseline(target_s: float = 8.0):
    """The fp64 CPU oracle, as it stands, on the headline workload's unit (one
    MXFP4 gate/up layer), timed (i) on one thread and (ii) over output rows on
    every host core.  The all-cores leg is the reported value."""
    L = oracle_layer()
    single = oracle_leg(L, 1, target_s)
    cores = host_cores()
    allc = oracle_leg(L, cores, target_s) if cores > 1 else dict(single)
    out = dict(allc)
    out["legs"] = [single, allc]
    return out


# ---------------------------------------------------------------------------
# dram__bytes_read.sum + dram__bytes_write.sum of one launch, from an ncu
# capture of the current kernel on the same shape (K = 2048, N = 11008, m = 1);
# set an entry back to None whenever its kernel changes.
DRAM_TRAFFIC = {
    "swiglu_mxfp4_m1r_kernel": 24148480,
    "swiglu_bf16_kernel": 92470784,
}
# The kernel that serves the batch-1 MXFP4 gate/up layer at K = 2048.
MXFP4_M1_KERNEL = "swiglu_mxfp4_m1r_kernel"

# The other workloads' kernels: (kernel(s), bound, DRAM read + write of one
# launch (summed over a call's kernels) from an ncu capture of the current
# code on the same shape, or None where no such capture exists).
WORKLOAD_KERNELS = {
    "fp8_gate_up_k2048_n11008_m1": ("fp8_swiglu_k_kernel", "hbm", 45198848),
    "bf16_down_k11008_n2048_m1": ("bf16_rows_k_kernel", "hbm", 45119744),
    "fp8_down_k11008_n2048_m1": ("fp8_pair_kernel", "hbm", 22598656),
    "mxfp4_down_k11008_n2048_m1": ("mxfp4_rows_k_kernel", "hbm", 12020736),
    "gptoss20b_int4_qkv_k2880_n5120_g128": ("int4_mma_kernel", "hbm", 7704832),
    "gptoss20b_moe_h2880_e32_top4": ("moe_fused_kernel", "hbm", 53517824),
    "gptoss20b_moe_q1_h2880_e32_top4": ("lowbit_router_kernel + lowbit_swiglu_kernel + "
                                        "lowbit_down_kernel", "hbm", 14180864),
    "gptoss20b_moe_q2_h2880_e32_top4": ("lowbit_router_kernel + lowbit_swiglu_kernel + "
                                        "lowbit_down_kernel", "hbm", None),
    # time per call (split + merge kernels); traffic of the split kernel (the
    # merge kernel's reads of the split partials hit L2)
    "gqa_decode_smollm3_3b_h16_kv4_d128_len32768": ("gqa_decode_kernel + gqa_merge_kernel",
                                                    "hbm", 67459072),
    "gqa_decode_gptoss20b_h64_kv8_d64_len32768": ("gqa_decode_kernel + gqa_merge_kernel",
                                                  "hbm", 67426560),
}
NOMINAL_HBM_GBS = 8000.0


def max_over_ranks(dist, vals, device=None):
    """Element-wise max of per-rank timings over all ranks (identity for one
    process): with independent replicas the slowest one sets the step time."""
    if dist is None:
        return [float(v) for v in vals]
    import torch
    t = torch.tensor([float(v) for v in vals], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(v) for v in t.tolist()]


def job_throughput(bytes_per_step, world, ms):
    """Whole-job GB/s: every replica moves bytes_per_step per step of ms."""
    return bytes_per_step * world / (ms * 1e-3) / 1e9


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="thinmx", choices=["thinmx", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--quick", action="store_true", help="skip the secondary workloads")
    ap.add_argument("--only", default=None,
                    choices=["gate_up", "bf16", "moe", "int4", "sweep", "fp8", "mlp", "gqa",
                             "lowbit"],
                    help="run one small workload only (for profiler captures)")
    ap.add_argument("--layers", type=int, default=None,
                    help="with --only moe / lowbit: MoE layers to build (default: the full stack)")
    ap.add_argument("--gqa", default=None,
                    help="with --only gqa: one case, model:len (e.g. gptoss20b:32768)")
    ap.add_argument("--ms", default=None,
                    help="with --only sweep: comma-separated batch sizes (default: all)")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))

    if args.impl == "reference":
        return reference_arm(args, world, rank)

    import torch
    from bit_weight_only_mxfp4_gb300 import build as tt_build
    from bit_weight_only_mxfp4_gb300 import loader, synth, thinmx

    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    pg = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=device)
        pg = dist
    if rank == 0:
        tt_build.build()
    if pg:
        pg.barrier()
    thinmx.load()

    if args.only:
        hbm, peak_kind, _ = peaks()
        if args.only == "gate_up":
            r = single_gate_up(torch, synth, loader, thinmx, device, hbm, copies=4,
                               reps=args.steps)
        elif args.only == "bf16":
            r = single_bf16(torch, synth, thinmx, device, hbm, copies=2, reps=args.steps)
        elif args.only == "sweep":
            ms = tuple(int(v) for v in args.ms.split(",")) if args.ms else None
            r = secondary_sweep(torch, synth, loader, thinmx, device, hbm, ms=ms)
        elif args.only == "int4":
            l2 = torch.cuda.get_device_properties(device).L2_cache_size
            r = int4_workload(torch, synth, thinmx, device, hbm, l2, reps=args.steps)
        elif args.only == "lowbit":
            r = moe_lowbit_workload(torch, synth, loader, thinmx, device, hbm, reps=args.steps,
                                    layers=args.layers)
        elif args.only == "gqa":
            l2 = torch.cuda.get_device_properties(device).L2_cache_size
            r = gqa_workload(torch, synth, thinmx, device, hbm, l2, reps=args.steps,
                             case=args.gqa)
        elif args.only == "mlp":
            r = mlp_stack_workload(torch, synth, loader, thinmx, device, hbm, reps=args.steps)
        elif args.only == "fp8":
            l2 = torch.cuda.get_device_properties(device).L2_cache_size
            r = fp8_workload(torch, synth, thinmx, device, hbm, l2, reps=args.steps)
        else:
            r = moe_workload(torch, synth, loader, thinmx, device, hbm, reps=args.steps,
                             layers=args.layers)
        print(json.dumps({"only": args.only, **r}))
        return 0

    cfg = synth.STACK
    layers = build_stack(torch, synth, loader, cfg, device)
    mx_b, bf_b = stack_bytes(cfg)
    mx_layers = [L for L in layers if L[0] == "mxfp4"]
    bf_layers = [L for L in layers if L[0] == "bf16"]
    n_mx = len(mx_layers)
    step_bytes = n_mx * mx_b  # the step: the stack's 24 MXFP4 layers

    g_mx = capture(torch, lambda: [run_layer(thinmx, cfg, L) for L in mx_layers])
    g_bf = capture(torch, lambda: [run_layer(thinmx, cfg, L) for L in bf_layers])
    g_stack = capture(torch, lambda: [run_layer(thinmx, cfg, L) for L in layers])

    # ---- timed region: K steps (24 PDL-chained MXFP4 layers each) ----------
    for _ in range(args.warmup):
        g_mx.replay()
    torch.cuda.synchronize()
    if pg:
        pg.barrier()
    torch.cuda.synchronize()
    with Clocks(local) as clk:
        step_ms = replay_times(torch, g_mx, args.steps)
    if pg:
        pg.barrier()
    torch.cuda.synchronize()
    ms_med = statistics.median(step_ms)
    ms_mean = sum(step_ms) / len(step_ms)

    # the bf16 layers and the whole 36-layer stack, medians of >= 20 replays
    ms_bf = time_graph(torch, g_bf) / len(bf_layers)
    ms_stack = time_graph(torch, g_stack)

    # ---- end to end through the public API with host buffers --------------
    x_host = torch.empty((n_mx, cfg.k), dtype=torch.bfloat16).pin_memory()
    h_host = torch.empty((n_mx, cfg.n), dtype=torch.bfloat16).pin_memory()
    for i, lay in enumerate(mx_layers):
        x_host[i].copy_(lay[2][0].cpu())
    x_dev = torch.empty((n_mx, cfg.k), dtype=torch.bfloat16, device=device)
    h_dev = torch.empty((n_mx, cfg.n), dtype=torch.bfloat16, device=device)

    # each layer's call with its device addresses, resolved once (the binding
    # takes raw addresses as well as tensors)
    stream = torch.cuda.current_stream().cuda_stream
    calls = [(thinmx.tt_mxfp4_swiglu_matvec,
              (w.data_ptr(), cfg.n, cfg.k, x_dev[i:i + 1].data_ptr(), 1,
               h_dev[i:i + 1].data_ptr(), stream))
             for i, (_, w, _, _) in enumerate(mx_layers)]

    def e2e_calls():
        for fn, a in calls:
            fn(*a)

    # The step captured once into a CUDA graph (how a decode loop runs its
    # layer stack, and how the pages' runtime does): the host -> device copy
    # of x, the same 24 calls and the device -> host copy of h, replayed
    # every step; each call's stream argument is the capturing stream while
    # the graph is recorded.  The copies read and write the pinned host
    # buffers when the graph runs.
    def e2e_capture_step():
        cs = torch.cuda.current_stream().cuda_stream
        x_dev.copy_(x_host, non_blocking=True)
        for fn, a in calls:
            fn(*a[:-1], cs)
        h_host.copy_(h_dev, non_blocking=True)

    g_e2e = capture(torch, e2e_capture_step)

    def e2e_step(graph):
        if graph:
            g_e2e.replay()
        else:
            x_dev.copy_(x_host, non_blocking=True)
            e2e_calls()
            h_host.copy_(h_dev, non_blocking=True)
        torch.cuda.current_stream().synchronize()

    def e2e_time(graph):
        for _ in range(args.warmup):
            e2e_step(graph)
        torch.cuda.synchronize()
        t = []
        for _ in range(args.steps):
            t0 = time.perf_counter()
            e2e_step(graph)
            t.append((time.perf_counter() - t0) * 1e3)
        return statistics.median(t)

    e2e_med = e2e_time(True)
    e2e_ng_med = e2e_time(False)
    # the slowest replica sets every step time
    ms_med, ms_mean, e2e_med, e2e_ng_med = max_over_ranks(
        pg, [ms_med, ms_mean, e2e_med, e2e_ng_med], device)

    # ---- secondary workloads (rank 0 only) -----------------------------------
    others = {}
    hbm, peak_kind, _ = peaks()
    if rank == 0 and not args.quick:
        others = secondary(torch, synth, loader, thinmx, device, hbm, peak_kind)
    others["smollm3_3b_gate_up_stack_36l_mxfp4_0_24"] = {
        "us": round(ms_stack * 1e3, 2),
        "GBps": round(job_throughput(n_mx * mx_b + len(bf_layers) * bf_b, 1, ms_stack), 1),
        "bytes": n_mx * mx_b + len(bf_layers) * bf_b,
        "us_per_layer": {"mxfp4": round(ms_med * 1e3 / n_mx, 3), "bf16": round(ms_bf * 1e3, 3)},
        "timing": "one CUDA graph of the 36 PDL-chained calls; median of 20 replays"}

    # ---- cpu baseline ---------------------------------------------------------
    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        cpu = cpu_baseline()

    err = thinmx.tt_device_error_read()
    if rank != 0:
        if pg:
            pg.destroy_process_group()
        return 0

    gbs = job_throughput(step_bytes, world, ms_med)
    us_mx = ms_med * 1e3 / n_mx
    mx_ach = mx_b / (us_mx * 1e-6) / 1e9
    bf_ach = bf_b / (ms_bf * 1e-3) / 1e9
    mx_kernel = MXFP4_M1_KERNEL
    kernels = [
        {"kernel": mx_kernel, "bound": "hbm", "achieved": round(mx_ach, 1),
         "peak": hbm, "unit": "GB/s", "frac": round(mx_ach / hbm, 4),
         "frac_of_nominal_8tbs": round(mx_ach / NOMINAL_HBM_GBS, 4),
         "bytes_per_launch": mx_b, "us_per_launch": round(us_mx, 3),
         "traffic": DRAM_TRAFFIC.get(mx_kernel)},
        {"kernel": "swiglu_bf16_kernel", "bound": "hbm", "achieved": round(bf_ach, 1),
         "peak": hbm, "unit": "GB/s", "frac": round(bf_ach / hbm, 4),
         "frac_of_nominal_8tbs": round(bf_ach / NOMINAL_HBM_GBS, 4),
         "bytes_per_launch": bf_b, "us_per_launch": round(ms_bf * 1e3, 3),
         "traffic": DRAM_TRAFFIC.get("swiglu_bf16_kernel")},
    ]
    for name, (kern, bound, traffic) in WORKLOAD_KERNELS.items():
        o = others.get(name)
        if not isinstance(o, dict) or "GBps" not in o:
            continue
        kernels.append({"kernel": kern, "workload": name, "bound": bound, "achieved": o["GBps"],
                        "peak": hbm, "unit": "GB/s", "frac": round(o["GBps"] / hbm, 4),
                        "bytes_per_launch": o.get("bytes", o.get("bytes_per_layer")),
                        "us_per_launch": o.get("us", o.get("us_per_layer")),
                        "traffic": traffic})
    roofline = {k: kernels[0][k] for k in ("bound", "achieved", "peak", "unit", "frac",
                                           "traffic")}
    roofline["kernel"] = mx_kernel
    roofline["frac_of_nominal_8tbs"] = kernels[0]["frac_of_nominal_8tbs"]
    roofline["peak_source"] = f"{peak_kind} HBM copy bandwidth (of {peak_kind})"
    roofline["target_frac"] = 0.75
    roofline["target_met"] = bool(mx_ach / hbm >= 0.75)
    line = {
        "metric": "batch-1 MXFP4 SwiGLU matvec µs/layer, weight GB/s and % of GB300 HBM roofline",
        "value": round(gbs, 1),
        "unit": "GB/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms_med, 5),
        "ms_per_step_mean": round(ms_mean, 5),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "mxfp4(e2m1+e8m0) x bf16 -> fp32 acc -> bf16",
        "data": "synthetic: W ~ N(0,0.02^2) quantised to MXFP4 on the GPU, x ~ N(0,1) bf16, "
                "postscale ~ U[0.9,1.1]; seeded",
        "config": {"workload": "smollm3_3b_mxfp4_gate_up_layers_0_24_k2048_n11008_m1",
                   "layers_per_step": n_mx, "k": cfg.k, "n": cfg.n, "m": 1,
                   "bytes_per_step": step_bytes, "bytes_per_layer": mx_b,
                   "l2_policy": "inputs larger than L2 (577 MB of MXFP4 weights per step)",
                   "timing": "CUDA graph of the 24 PDL-chained calls; CUDA events on the replay "
                             "stream around every step; median of the K steps"},
        "us_per_layer": {"mxfp4": round(us_mx, 3), "bf16": round(ms_bf * 1e3, 3)},
        "roofline": roofline,
        "roofline_by_kernel": kernels,
        "e2e": {"value": round(job_throughput(step_bytes, world, e2e_med), 1), "unit": "GB/s",
                "ms_per_step": round(e2e_med, 4),
                "h2d_bytes_per_step": n_mx * cfg.k * 2, "d2h_bytes_per_step": n_mx * cfg.n * 2,
                "path": "pinned host x -> device, the 24 C-ABI calls, h -> pinned host, "
                        "captured once in a CUDA graph and replayed; host wall clock around "
                        "each step (replay and synchronize inside); median of the K steps",
                "no_graph": {"value": round(job_throughput(step_bytes, world, e2e_ng_med), 1),
                             "unit": "GB/s", "ms_per_step": round(e2e_ng_med, 4),
                             "path": "the same copies, with the 24 C-ABI calls issued one by "
                                     "one from Python every step"}},
        "gpu_launches": n_mx * args.steps,
        "clocks": clk.summary(),
        "others": others,
        "cpu_baseline": cpu,
        "device_error": err,
    }
    print(json.dumps(line))
    if pg:
        pg.destroy_process_group()
    return 0


def single_gate_up(torch, synth, loader, thinmx, device, hbm, copies=None, reps=50):
    """One SmolLM3 gate/up layer at M=1, cycling through enough weight copies
    that their total exceeds twice the L2 size."""
    c = synth.GATE_UP
    per = gate_up_bytes(c.n, c.k, 1)
    if copies is None:
        l2 = torch.cuda.get_device_properties(device).L2_cache_size
        copies = max(4, int(2 * l2 // per) + 2)
    bufs = []
    for i in range(copies):
        wg = synth.torch_normal((c.n, c.k), synth.WEIGHT_STD, c.wid, i, 0, device)
        wu = synth.torch_normal((c.n, c.k), synth.WEIGHT_STD, c.wid, i, 1, device)
        pgv = synth.torch_uniform((c.n,), 0.9, 1.1, c.wid, i, 3, device)
        puv = synth.torch_uniform((c.n,), 0.9, 1.1, c.wid, i, 4, device)
        packed = loader.mxfp4_gate_up_from_f32(wg, wu, pgv, puv)
        del wg, wu
        x = synth.torch_normal((1, c.k), 1.0, c.wid, i, 2, device).to(torch.bfloat16)
        h = torch.empty((1, c.n), dtype=torch.bfloat16, device=device)
        bufs.append((packed, x, h))
    g = capture(torch, lambda: [thinmx.tt_mxfp4_swiglu_matvec(p, c.n, c.k, x, 1, h)
                                for p, x, h in bufs])
    ms = time_graph(torch, g, reps) / copies
    del bufs, g
    torch.cuda.empty_cache()
    return {c.name: {"us": round(ms * 1e3, 3), "GBps": round(per / (ms * 1e-3) / 1e9, 1),
                     "frac": round(per / (ms * 1e-3) / 1e9 / hbm, 4), "bytes": per,
                     "rotating_copies": copies}}


def single_bf16(torch, synth, thinmx, device, hbm, copies=2, reps=50):
    """One SmolLM3 bf16 gate/up layer at M=1 (90 MB of weights per copy)."""
    c = synth.STACK
    per = 4 * c.n * c.k + 2 * c.k + 2 * c.n
    bufs = []
    for i in range(copies):
        wg = synth.torch_normal((c.n, c.k), synth.WEIGHT_STD, c.wid, 24 + i, 0,
                                device).to(torch.bfloat16)
        wu = synth.torch_normal((c.n, c.k), synth.WEIGHT_STD, c.wid, 24 + i, 1,
                                device).to(torch.bfloat16)
        x = synth.torch_normal((1, c.k), 1.0, c.wid, 24 + i, 2, device).to(torch.bfloat16)
        h = torch.empty((1, c.n), dtype=torch.bfloat16, device=device)
        bufs.append((wg, wu, x, h))
    g = capture(torch, lambda: [thinmx.tt_bf16_swiglu_matvec(wg, wu, c.n, c.k, x, 1, h)
                                for wg, wu, x, h in bufs])
    ms = time_graph(torch, g, reps) / copies
    del bufs, g
    return {"bf16_gate_up_k2048_n11008_m1": {
        "us": round(ms * 1e3, 3), "GBps": round(per / (ms * 1e-3) / 1e9, 1),
        "frac": round(per / (ms * 1e-3) / 1e9 / hbm, 4), "bytes": per, "rotating_copies": copies}}


def secondary(torch, synth, loader, thinmx, device, hbm, peak_kind):
    """Single gate/up layer (rotating copies > 2x L2), the Phi-4 batch sweep,
    the INT4 QKV projection and the MoE stack."""
    out = dict(single_gate_up(torch, synth, loader, thinmx, device, hbm))
    l2 = torch.cuda.get_device_properties(device).L2_cache_size
    out.update(secondary_sweep(torch, synth, loader, thinmx, device, hbm))
    torch.cuda.empty_cache()
    out.update(int4_workload(torch, synth, thinmx, device, hbm, l2))
    torch.cuda.empty_cache()
    out.update(fp8_workload(torch, synth, thinmx, device, hbm, l2))
    torch.cuda.empty_cache()
    out.update(mlp_stack_workload(torch, synth, loader, thinmx, device, hbm))
    torch.cuda.empty_cache()
    out.update(gqa_workload(torch, synth, thinmx, device, hbm, l2))
    torch.cuda.empty_cache()
    out.update(moe_workload(torch, synth, loader, thinmx, device, hbm))
    torch.cuda.empty_cache()
    out.update(moe_lowbit_workload(torch, synth, loader, thinmx, device, hbm))
    torch.cuda.empty_cache()
    out["peak"] = {"hbm_gbs": hbm, "source": peak_kind,
                   "tensor_tflops": tensor_peak_tflops()}
    return out


def secondary_sweep(torch, synth, loader, thinmx, device, hbm, reps=20, ms=None):
    """Phi-4 gate/up (K=5120, N=17920) over the batch sizes: the CUDA-core
    streaming kernel at m = 1, the tile kernel with mma.sync multiply-adds
    for m = 2..8, the tcgen05 tensor-core kernel above; weight copies > 2x
    L2."""
    tensor_peak = tensor_peak_tflops()
    l2 = torch.cuda.get_device_properties(device).L2_cache_size
    s = synth.SWEEP
    wg = synth.torch_normal((s.n, s.k), synth.WEIGHT_STD, s.wid, 0, 0, device)
    wu = synth.torch_normal((s.n, s.k), synth.WEIGHT_STD, s.wid, 0, 1, device)
    pgv = synth.torch_uniform((s.n,), 0.9, 1.1, s.wid, 0, 3, device)
    puv = synth.torch_uniform((s.n,), 0.9, 1.1, s.wid, 0, 4, device)
    base = loader.mxfp4_gate_up_from_f32(wg, wu, pgv, puv)
    del wg, wu
    per_w = base.numel()
    copies = max(3, int(2 * l2 // per_w) + 1)
    packs = [base] + [base.clone() for _ in range(copies - 1)]
    sweep = {}
    for m in (ms or s.ms):
        xs = [synth.torch_normal((m, s.k), 1.0, s.wid, 0, 2, device).to(torch.bfloat16)
              for _ in range(copies)]
        hs = [torch.empty((m, s.n), dtype=torch.bfloat16, device=device) for _ in range(copies)]
        g = capture(torch, lambda: [thinmx.tt_mxfp4_swiglu_matvec(p, s.n, s.k, x, m, h)
                                    for p, x, h in zip(packs, xs, hs)])
        ms = time_graph(torch, g, reps) / copies
        b = gate_up_bytes(s.n, s.k, m)
        tflops = 4 * m * s.n * s.k / (ms * 1e-3) / 1e12
        # the library's dispatch at this size (k = 5120)
        path = ("tcgen05 kind::f16" if m > 8 else
                "mma.sync tile kernel" if m >= 2 else "cuda-core streaming (FMA)")
        sweep[str(m)] = {"us": round(ms * 1e3, 3), "GBps": round(b / (ms * 1e-3) / 1e9, 1),
                         "frac": round(b / (ms * 1e-3) / 1e9 / hbm, 4),
                         "TFLOPs": round(tflops, 2),
                         "path": path}
        if m > 8:  # against the dense f16/bf16 tensor peak as well
            sweep[str(m)]["tensor_frac"] = round(tflops / tensor_peak, 4)
        del g
    del packs, base
    return {s.name: sweep}


def fp8_workload(torch, synth, thinmx, device, hbm, l2, reps=50):
    """The MLP matvecs at SmolLM3 sizes, M=1, each over rotating weight
    copies whose total exceeds twice the L2 size: the quality-FP8 profile's
    gate/up SwiGLU (K=2048, N=11008) and down projection (K=11008, N=2048),
    and the down projection in bf16 and in MXFP4."""
    c = synth.GATE_UP
    out = {}
    cases = {"fp8_gate_up_k2048_n11008_m1": ("fp8", c.n, c.k, True),
             "fp8_down_k11008_n2048_m1": ("fp8", c.k, c.n, False),
             "bf16_down_k11008_n2048_m1": ("bf16", c.k, c.n, False),
             "mxfp4_down_k11008_n2048_m1": ("mxfp4", c.k, c.n, False)}
    for name, (kind, n, k, swiglu) in cases.items():
        mats = 2 if swiglu else 1
        if kind == "fp8":
            per = mats * (n * k + 4 * n) + 2 * k + 2 * n
        elif kind == "bf16":
            per = 2 * n * k + 2 * k + 2 * n
        else:
            per = n * k // 2 + n * k // 32 + 2 * k + 2 * n
        copies = max(4, int(2 * l2 // per) + 2)
        bufs = []
        for i in range(copies):
            ws = []
            for j in range(mats):
                w = synth.torch_normal((n, k), synth.WEIGHT_STD, 20, i, j, device)
                if kind == "fp8":
                    codes = torch.empty((n, k), dtype=torch.uint8, device=device)
                    scales = torch.empty(n, dtype=torch.float32, device=device)
                    thinmx.tt_quantize_fp8(w, n, k, codes, scales)
                    ws.append((codes, scales))
                elif kind == "bf16":
                    ws.append(w.to(torch.bfloat16))
                else:
                    codes = torch.empty((n, k // 2), dtype=torch.uint8, device=device)
                    scales = torch.empty((n, k // 32), dtype=torch.uint8, device=device)
                    thinmx.tt_quantize_mxfp4(w, n, k, codes, scales)
                    ws.append((codes, scales))
                del w
            x = synth.torch_normal((1, k), 1.0, 20, i, 9, device).to(torch.bfloat16)
            y = torch.empty((1, n), dtype=torch.bfloat16, device=device)
            bufs.append((ws, x, y))
        if kind == "fp8" and swiglu:
            fn = lambda: [thinmx.tt_fp8_swiglu_matvec(w[0][0], w[0][1], w[1][0], w[1][1], n, k, x,
                                                      1, y) for w, x, y in bufs]
        elif kind == "fp8":
            fn = lambda: [thinmx.tt_fp8_matvec(w[0][0], w[0][1], n, k, x, 1, y)
                          for w, x, y in bufs]
        elif kind == "bf16":
            fn = lambda: [thinmx.tt_bf16_matvec(w[0], n, k, x, 1, y) for w, x, y in bufs]
        else:
            fn = lambda: [thinmx.tt_mxfp4_matvec(w[0][0], w[0][1], None, n, k, x, 1, y)
                          for w, x, y in bufs]
        g = capture(torch, fn)
        ms = time_graph(torch, g, reps) / copies
        del bufs, g
        torch.cuda.empty_cache()
        out[name] = {"us": round(ms * 1e3, 3), "GBps": round(per / (ms * 1e-3) / 1e9, 1),
                     "frac": round(per / (ms * 1e-3) / 1e9 / hbm, 4), "bytes": per,
                     "rotating_copies": copies}
    return out


def mlp_stack_workload(torch, synth, loader, thinmx, device, hbm, reps=20):
    """The SmolLM3-3B-shaped decode MLP stack at M=1 (36 layers, hidden 2048,
    intermediate 11008), every layer gate/up SwiGLU then the down projection,
    layer l + 1 reading layer l's output: 72 PDL-chained calls in one CUDA
    graph, in two profiles -- the selective one (MXFP4 gate/up in layers
    0:24, bf16 elsewhere, bf16 down projections) and the FP8 one (FP8
    everywhere).  All weights resident (3.3 GB and 2.4 GB, far beyond L2)."""
    c = synth.STACK
    H, I = c.k, c.n
    out = {}
    b_mx = 2 * (I * H // 2 + I * H // 32 + 4 * I) + 2 * H + 2 * I
    b_bf = 4 * I * H + 2 * H + 2 * I
    b_bfd = 2 * H * I + 2 * I + 2 * H
    b_f8 = 2 * (I * H + 4 * I) + 2 * H + 2 * I
    b_f8d = H * I + 4 * H + 2 * I + 2 * H

    def fp8(w, n, k):
        codes = torch.empty((n, k), dtype=torch.uint8, device=device)
        scales = torch.empty(n, dtype=torch.float32, device=device)
        thinmx.tt_quantize_fp8(w, n, k, codes, scales)
        return codes, scales

    for profile in ("selective_mxfp4", "fp8"):
        layers, nbytes = [], 0
        for l in range(c.layers):
            wg = synth.torch_normal((I, H), synth.WEIGHT_STD, 30, l, 0, device)
            wu = synth.torch_normal((I, H), synth.WEIGHT_STD, 30, l, 1, device)
            wd = synth.torch_normal((H, I), synth.WEIGHT_STD, 30, l, 2, device)
            h = torch.empty((1, I), dtype=torch.bfloat16, device=device)
            y = torch.empty((1, H), dtype=torch.bfloat16, device=device)
            if profile == "fp8":
                layers.append(("fp8", fp8(wg, I, H), fp8(wu, I, H), fp8(wd, H, I), h, y))
                nbytes += b_f8 + b_f8d
            elif l < c.mxfp4_layers:
                pg = synth.torch_uniform((I,), 0.9, 1.1, 30, l, 3, device)
                pu = synth.torch_uniform((I,), 0.9, 1.1, 30, l, 4, device)
                layers.append(("mxfp4", loader.mxfp4_gate_up_from_f32(wg, wu, pg, pu), None,
                               wd.to(torch.bfloat16), h, y))
                nbytes += b_mx + b_bfd
            else:
                layers.append(("bf16", wg.to(torch.bfloat16), wu.to(torch.bfloat16),
                               wd.to(torch.bfloat16), h, y))
                nbytes += b_bf + b_bfd
            del wg, wu, wd
        x0 = synth.torch_normal((1, H), 1.0, 30, 99, 0, device).to(torch.bfloat16)

        def step():
            x = x0
            for kind, a, b, d, h, y in layers:
                if kind == "fp8":
                    thinmx.tt_fp8_swiglu_matvec(a[0], a[1], b[0], b[1], I, H, x, 1, h)
                    thinmx.tt_fp8_matvec(d[0], d[1], H, I, h, 1, y)
                else:
                    if kind == "mxfp4":
                        thinmx.tt_mxfp4_swiglu_matvec(a, I, H, x, 1, h)
                    else:
                        thinmx.tt_bf16_swiglu_matvec(a, b, I, H, x, 1, h)
                    thinmx.tt_bf16_matvec(d, H, I, h, 1, y)
                x = y

        g = capture(torch, step)
        ms = time_graph(torch, g, reps)
        out[f"smollm3_3b_mlp_stack_36l_{profile}"] = {
            "us": round(ms * 1e3, 2), "us_per_layer": round(ms * 1e3 / c.layers, 3),
            "GBps": round(nbytes / (ms * 1e-3) / 1e9, 1),
            "frac": round(nbytes / (ms * 1e-3) / 1e9 / hbm, 4), "bytes": nbytes,
            "kernels": 2 * c.layers}
        del layers, g
        torch.cuda.empty_cache()
    return out


def int4_workload(torch, synth, thinmx, device, hbm, l2, reps=50):
    """Grouped INT4 QKV projection (K=2880, N=5120, G=128) at M=1, cycling
    through weight copies whose total exceeds twice the L2 size."""
    c = synth.QKV
    ng = (c.k + c.group - 1) // c.group
    w = synth.torch_normal((c.n, c.k), synth.WEIGHT_STD, c.wid, 0, 0, device)
    codes = torch.empty((c.n, c.k // 2), dtype=torch.uint8, device=device)
    scales = torch.empty((c.n, ng), dtype=torch.int16, device=device)
    zp = torch.empty((c.n, (ng + 1) // 2), dtype=torch.uint8, device=device)
    thinmx.tt_quantize_int4_grouped(w, c.n, c.k, c.group, codes, scales, zp)
    del w
    per = c.n * c.k // 2 + c.n * ng * 2 + c.n * ((ng + 1) // 2) + 2 * c.k + 2 * c.n
    copies = max(4, int(2 * l2 // per) + 2)
    bufs = []
    for i in range(copies):
        x = synth.torch_normal((1, c.k), 1.0, c.wid, i, 1, device).to(torch.bfloat16)
        y = torch.empty((1, c.n), dtype=torch.bfloat16, device=device)
        bufs.append((codes.clone(), scales.clone(), zp.clone(), x, y))
    g = capture(torch, lambda: [thinmx.tt_int4_grouped_matvec(a, b, z, c.n, c.k, c.group, x, 1, y)
                                for a, b, z, x, y in bufs])
    ms = time_graph(torch, g, reps) / copies
    del bufs, g
    return {c.name: {"us": round(ms * 1e3, 3), "GBps": round(per / (ms * 1e-3) / 1e9, 1),
                     "frac": round(per / (ms * 1e-3) / 1e9 / hbm, 4), "bytes": per,
                     "rotating_copies": copies}}


def gqa_bytes(heads, kvh, d, length):
    """Algorithmic bytes of one decode attention call: the K and V rows read
    once, q read, out written (bf16)."""
    return 2 * kvh * length * d * 2 + 2 * heads * d * 2


def gqa_workload(torch, synth, thinmx, device, hbm, l2, reps=50, case=None):
    """Single-token GQA attention over a bf16 KV cache (SmolLM3-3B heads
    16/4/128 and gpt-oss-20b heads 64/8/64; 4096 and 32768 cached tokens),
    each over rotating caches whose total exceeds twice the L2 size; one
    workspace shared by the stream-ordered calls.  `case` ("model:len")
    keeps one of them."""
    c = synth.GQA
    out = {}
    for model, heads, kvh, d in c.shapes:
        if case and not case.startswith(model + ":"):
            continue
        ws_bytes = thinmx.tt_gqa_decode_workspace_bytes(heads, kvh, d)
        ws = torch.zeros(ws_bytes, dtype=torch.uint8, device=device)
        for length in c.lens:
            if case and case != f"{model}:{length}":
                continue
            per = gqa_bytes(heads, kvh, d, length)
            copies = max(3, int(2 * l2 // per) + 2)
            bufs = []
            for i in range(copies):
                k = synth.torch_normal((kvh, length, d), 1.0, c.wid, i, 1, device).to(torch.bfloat16)
                v = synth.torch_normal((kvh, length, d), 1.0, c.wid, i, 2, device).to(torch.bfloat16)
                q = synth.torch_normal((heads, d), 1.0, c.wid, i, 0, device).to(torch.bfloat16)
                o = torch.empty((heads, d), dtype=torch.bfloat16, device=device)
                bufs.append((q, k, v, o))
            scale = 1.0 / d ** 0.5
            g = capture(torch, lambda: [thinmx.tt_gqa_decode_attention(
                q, k, v, heads, kvh, d, length, length, scale, o, ws, ws_bytes)
                for q, k, v, o in bufs])
            ms = time_graph(torch, g, reps) / copies
            del bufs, g
            torch.cuda.empty_cache()
            gbs = per / (ms * 1e-3) / 1e9
            out[f"gqa_decode_{model}_h{heads}_kv{kvh}_d{d}_len{length}"] = {
                "us": round(ms * 1e3, 3), "GBps": round(gbs, 1), "frac": round(gbs / hbm, 4),
                "bytes": per, "rotating_copies": copies}
    return out


def moe_workload(torch, synth, loader, thinmx, device, hbm, reps=20, layers=None):
    """gpt-oss-20b-shaped MoE stack: 24 layers, 32 MXFP4 experts each
    (hidden = inter = 2880), top-4; one call per layer, all weights resident
    (~10 GB, far beyond L2)."""
    c = synth.MOE
    H, I, E, K = c.hidden, c.inter, c.experts, c.top_k
    n_layers = layers or c.layers
    layers = []
    for l in range(n_layers):
        gbufs, dbufs = [], []
        for e in range(E):  # every expert in buffers of its own
            wgu = synth.torch_normal((2 * I, H), synth.WEIGHT_STD, c.wid, l, 100 + 2 * e, device)
            wdn = synth.torch_normal((H, I), synth.WEIGHT_STD, c.wid, l, 101 + 2 * e, device)
            g, d = loader.moe_expert_from_f32(wgu, wdn)
            gbufs.append(g)
            dbufs.append(d)
            del wgu, wdn
        wr = synth.torch_normal((E, H), synth.WEIGHT_STD, c.wid, l, 1, device).to(torch.bfloat16)
        x = synth.torch_normal((H,), 1.0, c.wid, l, 0, device).to(torch.bfloat16)
        layers.append((loader.expert_table(gbufs), loader.expert_table(dbufs), wr, x,
                       (gbufs, dbufs)))
    out = torch.empty(H, dtype=torch.bfloat16, device=device)
    idx = torch.empty(K, dtype=torch.int32, device=device)
    prob = torch.empty(K, dtype=torch.float32, device=device)
    wsb = thinmx.tt_moe_workspace_bytes(H, I, E, K)
    ws = torch.zeros(wsb, dtype=torch.uint8, device=device)  # counters start at zero
    torch.cuda.synchronize()

    def step():
        for gt, dt, wr, x, _ in layers:
            thinmx.tt_moe_mxfp4_topk_mlp(x, H, I, wr, E, K, gt, dt, out, idx, prob, ws, wsb)

    g = capture(torch, step)
    ms = time_graph(torch, g, reps) / n_layers
    per = E * H * 2 + K * (2 * I * (H // 2 + H // 32) + H * (I // 2 + I // 32)) + 2 * H + 2 * H
    del layers, g
    return {c.name: {"us_per_layer": round(ms * 1e3, 3),
                     "GBps": round(per / (ms * 1e-3) / 1e9, 1),
                     "frac": round(per / (ms * 1e-3) / 1e9 / hbm, 4), "bytes_per_layer": per,
                     "layers": n_layers, "kernels_per_layer": 1}}


def moe_lowbit_workload(torch, synth, loader, thinmx, device, hbm, reps=20, layers=None):
    """The gpt-oss-20b-shaped MoE stack with Q1 and with Q2 experts (the
    pages' packed_expert_q1_layers="0:24"): 24 layers, 32 experts each
    (hidden = inter = 2880), top-4; each layer three PDL-chained kernels.
    One layer's experts are quantised on the GPU and copied into every
    layer's own buffers (all resident, far beyond L2)."""
    c = synth.MOE
    H, I, E, K = c.hidden, c.inter, c.experts, c.top_k
    n_layers = layers or c.layers
    out = {}
    for bits in (1, 2):
        gnb = thinmx.tt_lowbit_matrix_bytes(bits, 2 * I, H)
        dnb = thinmx.tt_lowbit_matrix_bytes(bits, H, I)
        base_g, base_d = [], []
        for e in range(E):
            wgu = synth.torch_normal((2 * I, H), synth.WEIGHT_STD, c.wid, 0, 100 + 2 * e, device)
            wdn = synth.torch_normal((H, I), synth.WEIGHT_STD, c.wid, 0, 101 + 2 * e, device)
            g = torch.empty(gnb, dtype=torch.uint8, device=device)
            d = torch.empty(dnb, dtype=torch.uint8, device=device)
            thinmx.tt_quantize_lowbit(bits, wgu, 2 * I, H, g, gnb)
            thinmx.tt_quantize_lowbit(bits, wdn, H, I, d, dnb)
            base_g.append(g)
            base_d.append(d)
            del wgu, wdn
        stack = []
        for l in range(n_layers):
            gb = [b.clone() for b in base_g]
            db = [b.clone() for b in base_d]
            wr = synth.torch_normal((E, H), synth.WEIGHT_STD, c.wid, l, 1, device).to(torch.bfloat16)
            x = synth.torch_normal((H,), 1.0, c.wid, l, 0, device).to(torch.bfloat16)
            stack.append((loader.expert_table(gb), loader.expert_table(db), wr, x, (gb, db)))
        del base_g, base_d
        o = torch.empty(H, dtype=torch.bfloat16, device=device)
        idx = torch.empty(K, dtype=torch.int32, device=device)
        prob = torch.empty(K, dtype=torch.float32, device=device)
        wsb = thinmx.tt_moe_lowbit_workspace_bytes(I, E, K)
        ws = torch.empty(wsb, dtype=torch.uint8, device=device)
        torch.cuda.synchronize()

        def step():
            for gt, dt, wr, x, _ in stack:
                thinmx.tt_moe_lowbit_topk_mlp(bits, x, H, I, wr, E, K, gt, dt, o, idx, prob, ws,
                                              wsb)

        g = capture(torch, step)
        ms = time_graph(torch, g, reps) / n_layers
        per = E * H * 2 + 2 * H + K * (gnb + dnb) + 2 * H
        del stack, g
        torch.cuda.empty_cache()
        out[f"gptoss20b_moe_q{bits}_h2880_e32_top4"] = {
            "us_per_layer": round(ms * 1e3, 3), "GBps": round(per / (ms * 1e-3) / 1e9, 1),
            "frac": round(per / (ms * 1e-3) / 1e9 / hbm, 4), "bytes_per_layer": per,
            "layers": n_layers, "kernels_per_layer": 3}
    return out


def reference_arm(args, world, rank):
    """The CPU oracle timed as the reference arm (the pages ship no runnable
    implementation).  Each step is a bounded sample of the headline workload:
    one full MXFP4 gate/up layer (K=2048, N=11008), the oracle's matvec over
    output rows on every host core."""
    if rank != 0:
        return 0
    import concurrent.futures as cf
    L = oracle_layer()
    cores = host_cores()
    pool = cf.ThreadPoolExecutor(max_workers=cores) if cores > 1 else None
    try:
        for _ in range(args.warmup):
            oracle_layer_call(L, cores, pool)
        times = []
        for _ in range(args.steps):
            t0 = time.perf_counter()
            oracle_layer_call(L, cores, pool)
            times.append(time.perf_counter() - t0)
    finally:
        if pool is not None:
            pool.shutdown()
    med = statistics.median(times)
    v = L["bytes"] / med / 1e9
    sample = (f"MXFP4 gate/up layer 0 of the stack (all {L['rows']} rows, K={L['k']}) per step, "
              f"fp64 oracle over output rows on {cores} host threads; median of {args.steps}")
    line = {
        "impl": "reference",
        "metric": "batch-1 MXFP4 SwiGLU matvec µs/layer, weight GB/s and % of GB300 HBM roofline",
        "value": round(v, 4), "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(med * 1e3, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic, seeded (the same distributions as the GPU arm)",
        "config": {"workload": "smollm3_3b_mxfp4_gate_up_layers_0_24_k2048_n11008_m1",
                   "sample": "one layer per step"},
        "us_per_layer": {"mxfp4": round(med * 1e6, 1)},
        "cpu_baseline": {"value": round(v, 4), "unit": "GB/s", "cores": cores, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": round(v, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))
    return 0


if __name__ == "__main__":
    sys.exit(main())
