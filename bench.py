"""Benchmark of the fused GPTQ W4A16 linear layer on one GB300 (or N replicas).

Headline workload (sweep_70b, M = 1): the Llama-70B projection shapes
(K, N) in {(8192, 28672), (28672, 8192), (8192, 10240)} x groupsize in
{32, 64, 128, -1} x {trivial, act-order g_idx} = 24 layer configurations,
scales log-uniform [1e-3, 5e-2], x ~ N(0, 1) fp16, no bias.  Every layer
configuration is made R times (R weight replicas, at least 3x the 129 MB L2
per configuration), and one step is one M = 1 call on every replica of every
configuration, captured once into a CUDA graph and replayed: each layer is
touched once per step and ~10 GB of weights stream from HBM per step.

Metric: effective HBM bandwidth of decode, algorithmic bytes (qweight +
qzeros + scales as stored) per second, whole job.  Also on the line, kept
short enough to be read whole: the roofline fraction of the decode kernels,
the end-to-end figure through the C ABI with host buffers, the CPU oracle
timed on this host (a seeded column sample of the same workload), SM clocks
during the timed region, the binding-roofline fraction of the whole
sweep_70b workload at every M (M = 2048 is the prefill), the prefill
tensor-core numbers (sweep_70b M = 2048 and prefill_7b M = 512), and the
decode_7b / actorder_7b workloads.  Per-case detail goes to stderr as one
JSON line, with the rows past the hot path (fused Q/K/V projections, GPTQ_V2,
8-bit codes, bf16 and fp32 activations, the GPU packer).

--impl reference times the CPU oracle (the plain dequantize-then-matmul
route) on the same workload: each step one layer configuration in turn, on a
seeded sample of 256 of its columns.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import synthetic  # noqa: E402

METRIC = "W4A16 GEMM: decode eff. HBM TB/s (% roofline), prefill TFLOPS (% FP16 peak)"
L2_BYTES = 129 * 2**20
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0
SAMPLE_COLS = 256                     # columns per layer in the oracle's bounded sample


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=20)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--impl", default="native", choices=["native", "reference"])
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-extra", action="store_true", help="headline only (no sweep/prefill/7B legs)")
    p.add_argument("--soak-s", type=float, default=1.0)
    p.add_argument("--sweep70b", action="store_true",
                   help="also time every one of the 240 sweep_70b cases on its own (per-case detail on stderr)")
    p.add_argument("--single", default=None, metavar="K,N,M[,PATH[,G[,ACT]]]",
                   help="profiling target instead of the bench: one synthetic layer (groupsize G, default 128; "
                        "ACT 1 for act-order), a 256 MB L2 flush before each of four calls on PATH (a "
                        "GPTQ_Q4_PATH_* suffix, default AUTO)")
    return p.parse_args()


def run_single(spec: str) -> None:
    """Four calls of one layer, each after an L2 flush: a short, fixed launch
    sequence for ncu captures (-s <launches before> -c 1 takes the fourth call)."""
    import torch
    import gptq_bit_weight_gb300 as q4
    parts = spec.split(",")
    K, N, M = int(parts[0]), int(parts[1]), int(parts[2])
    path = getattr(q4, "GPTQ_Q4_PATH_" + (parts[3].upper() if len(parts) > 3 and parts[3] else "AUTO"))
    gs = int(parts[4]) if len(parts) > 4 else 128
    act = len(parts) > 5 and parts[5] == "1"
    layer = synthetic.make_layer(K, N, gs, act_order=act, bias=True, key=(77, K, N, gs & 0xFFFF, int(act)))
    dev = torch.device("cuda", 0)
    t = lambda a: None if a is None else torch.from_numpy(np.ascontiguousarray(a)).to(dev)
    mat = q4.Q4Matrix(t(layer.qweight), t(layer.qzeros), t(layer.scales), t(layer.g_idx), t(layer.bias), gs)
    mat.set_path(path)
    mat.reserve(M)
    x = t(synthetic.activations(M, K, key=(77, K, N, M)))
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    for _ in range(4):
        flush.zero_()
        y = mat(x)
    torch.cuda.synchronize()
    mat.device_error()
    print(json.dumps({"single": spec, "max_abs_y": float(y.float().abs().max())}))


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return (float(d["hbm_gbs"]), float(d["bf16_tflops"]),
                float(d.get("bf16_tflops_sustained", d["bf16_tflops"])), "measured")
    except Exception:
        return FALLBACK_HBM_GBS, FALLBACK_BF16_TFLOPS, 1700.0, "fallback"


def dist_env():
    return int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")), int(os.environ.get("LOCAL_RANK", "0"))


def r3(v, n=3):
    return None if v is None else round(float(v), n)


# --------------------------------------------------------- replicas (N > 1)
# Every rank runs the same workload on its own GPU (weak scaling); there is no
# data-path collective.  The only cross-rank traffic is the barrier around the
# timed region and the max of the per-rank times.

def rank_barrier(world: int) -> None:
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks_value(v: float, world: int, device) -> float:
    if world == 1:
        return float(v)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(v)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(bytes_per_rank_per_step: float, steps: int, world: int, seconds: float) -> float:
    """Whole-job rate in TB/s: the units all ranks processed over the slowest rank's time."""
    return bytes_per_rank_per_step * steps * world / seconds / 1e12


# ------------------------------------------------------------------ clocks

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        self.out = ""
        if self.proc is not None:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                self.out, _ = self.proc.communicate(timeout=5)
            except Exception:
                self.proc.kill()
                self.out = ""

    def summary(self):
        sm, smax, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in (self.out or "").splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax = float(parts[2])
            except ValueError:
                continue
            for name, val in zip(names, parts[5:9]):
                if val.lower() == "active":
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": smax, "reasons": sorted(reasons), "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": smax, "reasons": sorted(reasons),
                "samples": len(sm)}


# --------------------------------------------------------------- the oracle

SWEEP_CONFIGS = [(K, N, g, a) for (K, N) in synthetic.SWEEP_70B_SHAPES for g in synthetic.SWEEP_70B_G
                 for a in (False, True)]


def sample_columns(N: int, key) -> np.ndarray:
    """A seeded sample of SAMPLE_COLS columns in whole 8-column blocks (one
    qzeros word each), so the oracle runs on exactly those columns."""
    blocks = np.sort(synthetic.rng(*key).choice(N // 8, size=SAMPLE_COLS // 8, replace=False))
    return (blocks[:, None] * 8 + np.arange(8)[None, :]).reshape(-1), blocks


def oracle_step(cfg, cores, L=None):
    """The oracle as it stands on one sweep_70b M = 1 configuration, on a
    column sample: unpack + dequantize the sampled columns, then y in fp64.
    Returns the sampled columns' weight bytes (qweight + qzeros + scales) and
    the seconds that took (input generation is not timed)."""
    import oracle
    K, N, g, act = cfg
    if L is None:
        L = synthetic.workload_layer("sweep_70b", K, N, g, act)
    cols, blocks = sample_columns(N, (90, K, N, g & 0xFFFF, int(act)))
    qw = np.ascontiguousarray(L.qweight[:, cols])
    qz = np.ascontiguousarray(L.qzeros[:, blocks])
    sc = np.ascontiguousarray(L.scales[:, cols])
    x = synthetic.workload_x("sweep_70b", K, N, g, act, 1)
    t0 = time.perf_counter()
    dq = oracle.dequantize_layer(qw, qz, sc, L.g_idx, K, cols.size, g)
    oracle.reference_output(x, dq, None, nthreads=cores)
    return qw.nbytes + qz.nbytes + sc.nbytes, time.perf_counter() - t0


def run_reference(args):
    """The CPU oracle on the headline workload (sweep_70b, M = 1): each step
    one layer configuration in turn, on a seeded sample of its columns."""
    rank, world, _ = dist_env()
    if rank != 0:
        return
    import oracle
    oracle.build()
    cores = os.cpu_count() or 1
    for i in range(args.warmup):
        oracle_step(SWEEP_CONFIGS[i % len(SWEEP_CONFIGS)], cores)
    nbytes, secs = 0, 0.0
    for i in range(args.steps):
        b, s = oracle_step(SWEEP_CONFIGS[(args.warmup + i) % len(SWEEP_CONFIGS)], cores)
        nbytes += b
        secs += s
    value = nbytes / secs / 1e12
    sample = (f"each step: one sweep_70b M=1 layer configuration in turn, {SAMPLE_COLS} seeded columns "
              f"(unpack, dequantize, fp64 products on {cores} threads; input generation untimed)")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": secs / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": headline_config(),
        "cpu_baseline": {"value": value, "unit": "TB/s", "cores": cores, "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": "TB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line, separators=(",", ":")), flush=True)


def cpu_baseline_sample(layers, budget_s: float = 12.0):
    """The oracle as it stands, timed on this host's cores, on column samples
    of the headline configurations in turn (round robin) until the budget is
    spent.  layers: the configurations' host tensors, already drawn."""
    import oracle
    oracle.build()
    cores = os.cpu_count() or 1
    nbytes, secs, n = 0, 0.0, 0
    while secs < budget_s and n < 50 * len(SWEEP_CONFIGS):
        i = n % len(SWEEP_CONFIGS)
        b, s = oracle_step(SWEEP_CONFIGS[i], cores, layers[i])
        nbytes += b
        secs += s
        n += 1
    return {"value": nbytes / secs / 1e12, "unit": "TB/s", "cores": cores, "kind": "oracle",
            "sample": f"{n} sweep_70b M=1 configs x {SAMPLE_COLS} cols, {secs:.1f} s"}


def headline_config():
    return {"workload": "sweep_70b", "M": 1, "layer_configs": "3 shapes x g{32,64,128,-1} x {trivial,act-order}"}


# The roofline's traffic: DRAM bytes (read + write) of one launch of the
# dominant decode kernel, from an ncu capture of
#   bench.py --single 8192,28672,1,DECODE,128   (the fourth call, after an L2 flush)
# whose algorithmic bytes are 122,028,032; ncu read 122.15 MB and wrote 2.95 MB.
DECODE_TRAFFIC = {"bytes": 125_114_368, "launch": "decode_kernel<1,0,1,0>, 8192x28672 g128 M=1",
                  "algorithmic_bytes": 122_028_032}


# ------------------------------------------------------------------ native

class Sweep:
    """The 24 sweep_70b layer configurations on the device, R replicas each
    (R * weight bytes >= 3x L2)."""

    def __init__(self, q4, torch, dev, reserve_m):
        t = lambda a: None if a is None else torch.from_numpy(np.ascontiguousarray(a)).to(dev)
        self.cfgs = []
        for (K, N, g, act) in SWEEP_CONFIGS:
            L = synthetic.workload_layer("sweep_70b", K, N, g, act)
            qw, qz, sc, gi = t(L.qweight), t(L.qzeros), t(L.scales), t(L.g_idx)
            R = max(2, int(np.ceil(3 * L2_BYTES / L.weight_bytes)))
            mats = [q4.Q4Matrix(qw, qz, sc, gi, None, g) for _ in range(R)]
            for m in mats:
                m.reserve(reserve_m)
            del qw, qz, sc, gi
            self.cfgs.append({"K": K, "N": N, "g": g, "act": act, "mats": mats, "wb": L.weight_bytes,
                              "x": {}, "o": {}, "L": L})
        self.torch, self.dev = torch, dev

    def xo(self, c, M):
        if M not in c["x"]:
            t = self.torch
            c["x"][M] = t.from_numpy(synthetic.workload_x("sweep_70b", c["K"], c["N"], c["g"], c["act"], M)).to(self.dev)
            c["o"][M] = t.empty((M, c["N"]), dtype=t.float16, device=self.dev)
        return c["x"][M], c["o"][M]

    def drop_m(self, M):
        for c in self.cfgs:
            c["x"].pop(M, None)
            c["o"].pop(M, None)


def capture(torch, q4, issue):
    """One CUDA graph of issue(stream_ptr); returns (graph, our launches in it)."""
    issue(torch.cuda.current_stream().cuda_stream)     # nothing allocates during capture
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    n0 = q4.gptq_q4_launch_count()
    with torch.cuda.graph(g):
        issue(torch.cuda.current_stream().cuda_stream)
    return g, q4.gptq_q4_launch_count() - n0


def graph_seconds(torch, stream, g, reps):
    for _ in range(3):
        g.replay()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for _ in range(reps):
        g.replay()
    b.record(stream)
    torch.cuda.synchronize()
    return a.elapsed_time(b) * 1e-3 / reps


def run_native(args):
    import torch

    import gptq_bit_weight_gb300 as q4

    rank, world, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    stream = torch.cuda.current_stream()
    hbm_gbs, bf16_tf, bf16_tf_sus, peak_src = peaks()
    detail = {}

    sw = Sweep(q4, torch, dev, reserve_m=256)
    step_bytes = sum(c["wb"] * len(c["mats"]) for c in sw.cfgs)

    def issue_m(M, cfgs):
        def issue(sp):
            for c in cfgs:
                x, o = sw.xo(c, M)
                for m in c["mats"]:
                    q4.gptq_q4_matmul(m.handle, x.data_ptr(), M, o.data_ptr(), sp)
        return issue

    def barrier():
        rank_barrier(world)
        torch.cuda.synchronize()

    def max_over_ranks(v):
        return max_over_ranks_value(v, world, dev)

    step_graph, launches_per_step = capture(torch, q4, issue_m(1, sw.cfgs))
    with ClockSampler(local) as clk:
        t_end = time.perf_counter() + args.soak_s
        for _ in range(max(3, args.warmup)):
            step_graph.replay()
        torch.cuda.synchronize()
        while time.perf_counter() < t_end:      # clock soak: more untimed warm-up
            step_graph.replay()
            torch.cuda.synchronize()
        # ---- timed region: exactly K steps (graph replays)
        barrier()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(args.steps):
            step_graph.replay()
        e1.record(stream)
        barrier()
        ms = max_over_ranks(e0.elapsed_time(e1))
    clocks = clk.summary()
    launches = launches_per_step * args.steps
    value = job_throughput(step_bytes, args.steps, world, ms * 1e-3)

    # ---- roofline of the decode kernels: a graph of the trivial-g_idx configs
    # (only decode kernels launch there; act-order calls add the x gather)
    triv = [c for c in sw.cfgs if not c["act"]]
    g_triv, n_triv = capture(torch, q4, issue_m(1, triv))
    triv_bytes = sum(c["wb"] * len(c["mats"]) for c in triv)
    triv_s = graph_seconds(torch, stream, g_triv, max(5, args.steps // 2))
    del g_triv
    achieved_gbs = triv_bytes / triv_s / 1e9

    # ---- per layer configuration at M = 1: a graph of its R replicas
    m1 = {}
    for c in sw.cfgs:
        g1, _ = capture(torch, q4, issue_m(1, [c]))
        s = graph_seconds(torch, stream, g1, 10) / len(c["mats"])
        m1[(c["K"], c["N"], c["g"], c["act"])] = s
        del g1
    fr1 = {k: sw_cfg_bytes(k) / s / 1e9 / hbm_gbs for k, s in m1.items()}
    detail["m1_us"] = {cfg_name(k): round(s * 1e6, 2) for k, s in m1.items()}
    detail["m1_frac"] = {cfg_name(k): r3(f) for k, f in fr1.items()}

    # ---- end to end through the C ABI with host buffers (pinned), copies
    # inside the timed region: every step copies each configuration's x host ->
    # device, runs every C-ABI call, and copies every output device -> host;
    # one CUDA graph per step, timed on the host clock to the completed copies
    hx = {id(c): sw.xo(c, 1)[0].cpu().pin_memory() for c in sw.cfgs}
    ho = {id(c): torch.empty((1, c["N"]), dtype=torch.float16).pin_memory() for c in sw.cfgs}
    dx = {id(c): torch.empty_like(sw.xo(c, 1)[0]) for c in sw.cfgs}
    h2d = sum(t.numel() * 2 for t in hx.values())
    d2h = sum(t.numel() * 2 for t in ho.values())

    def e2e_issue(sp):
        for c in sw.cfgs:
            dx[id(c)].copy_(hx[id(c)], non_blocking=True)
        for c in sw.cfgs:
            o = sw.xo(c, 1)[1]
            for m in c["mats"]:
                q4.gptq_q4_matmul(m.handle, dx[id(c)].data_ptr(), 1, o.data_ptr(), sp)
        for c in sw.cfgs:
            ho[id(c)].copy_(sw.xo(c, 1)[1], non_blocking=True)

    e2e_graph, _ = capture(torch, q4, e2e_issue)
    for _ in range(max(3, args.warmup)):
        e2e_graph.replay()
    torch.cuda.synchronize()
    barrier()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        e2e_graph.replay()
    torch.cuda.synchronize()
    barrier()
    e2e_s = max_over_ranks(time.perf_counter() - t0)
    e2e_value = job_throughput(step_bytes, args.steps, world, e2e_s)
    assert all(torch.equal(ho[id(c)], sw.xo(c, 1)[1].cpu()) for c in sw.cfgs), "e2e results did not reach the host"
    del e2e_graph

    line_extra = {}
    if not args.no_extra:
        line_extra, d2 = run_extra_legs(q4, torch, dev, stream, sw, hbm_gbs, bf16_tf, issue_m, args)
        detail.update(d2)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline_sample([c["L"] for c in sw.cfgs])

    if rank == 0:
        fr = list(fr1.values())
        cfg = headline_config()
        cfg.update({"bytes_per_step": step_bytes,
                    "l2": f"inputs > L2: {step_bytes / 1e9:.1f} GB weights/step (>=3x L2 per config), each once",
                    "launch": "CUDA graph of C-ABI calls", "parallelism": f"replicas x{world}"})
        line = {
            "metric": METRIC, "value": r3(value, 4), "unit": "TB/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": r3(ms / args.steps, 4), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f16 x int4 -> f32 accumulate", "data": "synthetic",
            "config": cfg,
            "roofline": {"bound": "hbm", "achieved": r3(achieved_gbs, 1), "peak": hbm_gbs, "unit": "GB/s",
                         "frac": r3(achieved_gbs / hbm_gbs), "traffic": DECODE_TRAFFIC["bytes"],
                         "traffic_launch": DECODE_TRAFFIC["launch"], "peak_source": peak_src,
                         "kernel": "decode, 12 trivial-g_idx configs"},
            "m1_frac": {"min": r3(min(fr)), "mean": r3(float(np.mean(fr))), "max": r3(max(fr)),
                        "by_g": {str(g): r3(float(np.mean([f for k, f in fr1.items() if k[2] == g])))
                                 for g in synthetic.SWEEP_70B_G},
                        "act": r3(float(np.mean([f for k, f in fr1.items() if k[3]])))},
            "e2e": {"value": r3(e2e_value, 4), "unit": "TB/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
            "gpu_launches": launches,
            "clocks": clocks,
        }
        line.update(line_extra)
        if cpu:
            line["cpu_baseline"] = cpu
        print(json.dumps({"detail": detail}, separators=(",", ":")), file=sys.stderr, flush=True)
        print(json.dumps(line, separators=(",", ":")), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def sw_cfg_bytes(k):
    K, N, g, _ = k
    G = 1 if g == -1 else K // g
    return K * N // 2 + G * N * 2 + G * N // 2


def cfg_name(k):
    K, N, g, act = k
    return f"{K}x{N} g{g}{' act' if act else ''}"


def run_extra_legs(q4, torch, dev, stream, sw, hbm_gbs, bf16_tf, issue_m, args):
    """The rest of the workloads, summarised for the JSON line (detail for stderr)."""
    line, detail = {}, {}
    # sweep_70b at every M: binding-roofline fraction summed over the 24 configs,
    # sum(max(bytes / HBM, flops / tensor)) / sum(time), one graph of every
    # replica of every config per M (M = 2048: the prefill leg below)
    by_m = {}
    for M in synthetic.SWEEP_70B_M:
        if M == 2048:
            continue
        g, _ = capture(torch, q4, issue_m(M, sw.cfgs))
        s = graph_seconds(torch, stream, g, 5)
        del g
        bound = sum(max(c["wb"] / (hbm_gbs * 1e9), 2.0 * M * c["K"] * c["N"] / (bf16_tf * 1e12)) * len(c["mats"])
                    for c in sw.cfgs)
        by_m[M] = bound / s
        if M > 1:
            sw.drop_m(M)
    # prefill: sweep_70b M = 2048 on one replica of each config
    pf = {}
    tot_f, tot_s = 0.0, 0.0
    for c in sw.cfgs:
        M = 2048
        m = c["mats"][0]
        x = torch.from_numpy(synthetic.workload_x("sweep_70b", c["K"], c["N"], c["g"], c["act"], M)).to(dev)
        o = torch.empty((M, c["N"]), dtype=torch.float16, device=dev)
        m.reserve(M)
        g, _ = capture(torch, q4, lambda sp: q4.gptq_q4_matmul(m.handle, x.data_ptr(), M, o.data_ptr(), sp))
        s = graph_seconds(torch, stream, g, 10)
        del g, x, o
        fl = 2.0 * M * c["K"] * c["N"]
        pf[(c["K"], c["N"], c["g"], c["act"])] = fl / s / 1e12
        tot_f += fl
        tot_s += s
    by_m[2048] = tot_f / tot_s / 1e12 / bf16_tf
    pfr = [v / bf16_tf for v in pf.values()]
    detail["prefill_70b_m2048_tflops"] = {cfg_name(k): round(v, 1) for k, v in pf.items()}
    line["sweep_frac_by_M"] = {str(M): r3(f) for M, f in sorted(by_m.items())}
    p7, d7 = run_prefill_7b(q4, torch, dev, stream, bf16_tf)
    detail["prefill_7b"] = d7
    line["prefill"] = {"fields": "TFLOP/s,frac,min,max", "m2048_70b": [r3(tot_f / tot_s / 1e12, 1),
                                                                        r3(tot_f / tot_s / 1e12 / bf16_tf),
                                                                        r3(min(pfr)), r3(max(pfr))],
                       "m512_7b": p7["m512"], "m2048_7b": p7["m2048"], "unfused_7b": p7["unfused"],
                       "peak": bf16_tf}
    # 7B decode workloads (secondary)
    line["decode_7b"], detail["decode_7b"] = run_7b_decode(q4, torch, dev, stream, hbm_gbs, "decode_7b",
                                                           synthetic.DECODE_7B_SHAPES, synthetic.DECODE_7B_M, False)
    line["actorder_7b"], detail["actorder_7b"] = run_7b_decode(q4, torch, dev, stream, hbm_gbs, "actorder_7b",
                                                               synthetic.ACTORDER_7B_SHAPES, synthetic.ACTORDER_7B_M,
                                                               True)
    detail["next_rows"] = run_next_rows(q4, torch, dev, stream, hbm_gbs)
    if args.sweep70b:
        detail["sweep_70b_cases"] = run_sweep_70b_cases(q4, torch, dev, stream, sw, hbm_gbs, bf16_tf)
    return line, detail


def _graph_time(torch, stream, issue, reps=20):
    """Per-replay seconds of a CUDA graph of issue(stream_ptr)."""
    issue(stream.cuda_stream)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        issue(torch.cuda.current_stream().cuda_stream)
    for _ in range(3):
        g.replay()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for _ in range(reps):
        g.replay()
    b.record(stream)
    torch.cuda.synchronize()
    return a.elapsed_time(b) * 1e-3 / reps


def run_next_rows(q4, torch, dev, stream, hbm_gbs):
    """Measurements of the rows added past the hot path, on Llama-7B shapes:
    projection fusion (Q, K, V of one input as one handle vs three), the
    GPTQ_V2 zero convention (same kernels; must cost the same), and the GPU
    packer (float weights -> checkpoint words)."""
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(dev)
    res = {}
    K, Nq = 4096, 4096
    R = 6                                                   # 6 x 3 x 8.7 MB = 157 MB of weights > 129 MB L2
    layers = [synthetic.workload_layer("decode_7b", K, Nq, 128, False) for _ in range(3)]
    sep = [[q4.Q4Matrix(t(L.qweight), t(L.qzeros), t(L.scales), None, None, 128) for L in layers] for _ in range(R)]
    fused = [q4.Q4Matrix.fused([(t(L.qweight), t(L.qzeros), t(L.scales)) for L in layers], None, None, 128)
             for _ in range(R)]
    wbytes = 3 * layers[0].weight_bytes
    for M in (1, 8):
        x = t(synthetic.workload_x("decode_7b", K, Nq, 128, False, M))
        o1 = torch.empty((M, Nq), dtype=torch.float16, device=dev)
        o3 = torch.empty((M, 3 * Nq), dtype=torch.float16, device=dev)

        def issue_sep(sp):
            for r in range(R):
                for m in sep[r]:
                    q4.gptq_q4_matmul(m.handle, x.data_ptr(), M, o1.data_ptr(), sp)

        def issue_fused(sp):
            for r in range(R):
                q4.gptq_q4_matmul(fused[r].handle, x.data_ptr(), M, o3.data_ptr(), sp)

        ts = _graph_time(torch, stream, issue_sep) / R
        tf = _graph_time(torch, stream, issue_fused) / R
        res[f"qkv_7b M={M}"] = {"separate_us": round(ts * 1e6, 2), "fused_us": round(tf * 1e6, 2),
                                "separate_TB/s": round(wbytes / ts / 1e12, 3), "fused_TB/s": round(wbytes / tf / 1e12, 3)}
    del sep, fused
    # GPTQ_V2: the same layer read as a V2 checkpoint
    L = synthetic.workload_layer("decode_7b", 4096, 11008, 128, False)
    mats = [q4.Q4Matrix(t(L.qweight), t(L.qzeros), t(L.scales), None, None, 128) for _ in range(6)]
    x = t(synthetic.workload_x("decode_7b", 4096, 11008, 128, False, 1))
    o = torch.empty((1, 11008), dtype=torch.float16, device=dev)

    def issue(sp):
        for m in mats:
            q4.gptq_q4_matmul(m.handle, x.data_ptr(), 1, o.data_ptr(), sp)

    t1 = _graph_time(torch, stream, issue) / len(mats)
    for m in mats:
        m.set_format(q4.GPTQ_Q4_FORMAT_GPTQ_V2)
    t2 = _graph_time(torch, stream, issue) / len(mats)
    res["gptq_v2 4096x11008 M=1"] = {"gptq_us": round(t1 * 1e6, 2), "gptq_v2_us": round(t2 * 1e6, 2),
                                     "gptq_v2_TB/s": round(L.weight_bytes / t2 / 1e12, 3)}
    del mats
    # 8-bit checkpoint of the same shape (two 4-bit halves along K): decode
    # at M = 1 (weight bytes / time) and the fused prefill at M = 512
    L8 = synthetic.make_layer8(4096, 11008, 128, key=(33, 4096, 11008))
    mats = [q4.Q4Matrix(t(L8.qweight), t(L8.qzeros), t(L8.scales), None, None, 128, bits=8) for _ in range(6)]
    t8 = _graph_time(torch, stream, issue) / len(mats)
    bytes8 = 4096 * 11008 + (4096 // 128) * 11008 * 3   # codes + fp16 scales + 8-bit zeros
    x512 = t(synthetic.activations(512, 4096, key=(33, 512)))
    o512 = torch.empty((512, 11008), dtype=torch.float16, device=dev)
    mats[0].reserve(512)

    def issue512(sp):
        q4.gptq_q4_matmul(mats[0].handle, x512.data_ptr(), 512, o512.data_ptr(), sp)

    t512 = _graph_time(torch, stream, issue512)
    res["8bit 4096x11008"] = {"M=1_us": round(t8 * 1e6, 2), "M=1_TB/s": round(bytes8 / t8 / 1e12, 3),
                              "M=512_us": round(t512 * 1e6, 2),
                              "M=512_TFLOP/s": round(2 * 512 * 4096 * 11008 / t512 / 1e12, 1)}
    del mats
    # bf16 activations and outputs on the 4-bit layer (one preparation launch
    # per call scales and rounds x to fp16): decode at M = 1, prefill at M = 512
    mats = [q4.Q4Matrix(t(L.qweight), t(L.qzeros), t(L.scales), None, None, 128) for _ in range(6)]
    for m in mats:
        m.set_act_dtype(torch.bfloat16)
        m.reserve(512)
    xb1 = t(synthetic.activations_bf16(1, 4096, key=(35, 1)).view(np.int16)).view(torch.bfloat16)
    xb512 = t(synthetic.activations_bf16(512, 4096, key=(35, 512)).view(np.int16)).view(torch.bfloat16)
    ob1 = torch.empty((1, 11008), dtype=torch.bfloat16, device=dev)
    ob512 = torch.empty((512, 11008), dtype=torch.bfloat16, device=dev)

    def issue_b1(sp):
        for m in mats:
            q4.gptq_q4_matmul(m.handle, xb1.data_ptr(), 1, ob1.data_ptr(), sp)

    def issue_b512(sp):
        q4.gptq_q4_matmul(mats[0].handle, xb512.data_ptr(), 512, ob512.data_ptr(), sp)

    tb1 = _graph_time(torch, stream, issue_b1) / len(mats)
    tb512 = _graph_time(torch, stream, issue_b512)
    res["bf16 4096x11008"] = {"M=1_us": round(tb1 * 1e6, 2), "M=1_TB/s": round(L.weight_bytes / tb1 / 1e12, 3),
                              "M=512_us": round(tb512 * 1e6, 2),
                              "M=512_TFLOP/s": round(2 * 512 * 4096 * 11008 / tb512 / 1e12, 1)}
    del mats
    # fp32 activations and outputs on the 4-bit layer (hi/lo fp16 rows, raw
    # fp32 sums, one combine launch): decode at M = 1, prefill at M = 512
    mats = [q4.Q4Matrix(t(L.qweight), t(L.qzeros), t(L.scales), None, None, 128) for _ in range(6)]
    for m in mats:
        m.set_act_dtype(torch.float32)
        m.reserve(512)
    xf1 = t(synthetic.activations_f32(1, 4096, key=(39, 1)).view(np.float32))
    xf512 = t(synthetic.activations_f32(512, 4096, key=(39, 512)).view(np.float32))
    of1 = torch.empty((1, 11008), dtype=torch.float32, device=dev)
    of512 = torch.empty((512, 11008), dtype=torch.float32, device=dev)

    def issue_f1(sp):
        for m in mats:
            q4.gptq_q4_matmul(m.handle, xf1.data_ptr(), 1, of1.data_ptr(), sp)

    def issue_f512(sp):
        q4.gptq_q4_matmul(mats[0].handle, xf512.data_ptr(), 512, of512.data_ptr(), sp)

    tf1 = _graph_time(torch, stream, issue_f1) / len(mats)
    tf512 = _graph_time(torch, stream, issue_f512)
    res["fp32 4096x11008"] = {"M=1_us": round(tf1 * 1e6, 2), "M=1_TB/s": round(L.weight_bytes / tf1 / 1e12, 3),
                              "M=512_us": round(tf512 * 1e6, 2),
                              "M=512_TFLOP/s": round(2 * 512 * 4096 * 11008 / tf512 / 1e12, 1)}
    del mats
    # GPU packer: float weights (fp16) + scales + zeros -> qweight/qzeros
    K, N, gs = 4096, 11008, 128
    g = np.random.default_rng(5)
    w = torch.from_numpy(g.normal(0, 0.05, (K, N)).astype(np.float16)).to(dev)
    sc = torch.from_numpy(g.uniform(0.002, 0.02, (K // gs, N)).astype(np.float16)).to(dev)
    zs = torch.from_numpy(g.integers(0, 16, (K // gs, N)).astype(np.int32)).to(dev)
    qw = torch.empty((K // 8, N), dtype=torch.int32, device=dev)
    qz = torch.empty((K // gs, N // 8), dtype=torch.int32, device=dev)

    def issue_pack(sp):
        q4.gptq_q4_pack(w.data_ptr(), sc.data_ptr(), zs.data_ptr(), None, K, N, gs, 0, qw.data_ptr(), qz.data_ptr(), sp)

    tp = _graph_time(torch, stream, issue_pack, reps=10)
    moved = K * N * 2 + K * N // 2 + (K // gs) * N * 6 + (K // gs) * N // 2
    res["pack 4096x11008"] = {"us": round(tp * 1e6, 2), "TB/s": round(moved / tp / 1e12, 3),
                              "frac_of_hbm_peak": round(moved / tp / 1e9 / hbm_gbs, 3),
                              "bytes": "w fp16 read + qweight written + scales/zeros read + qzeros written"}
    return res


def run_7b_decode(q4, torch, dev, stream, hbm_gbs, workload, shapes, Ms, act):
    """A 7B decode workload through the default path: per shape, replicas
    >= 3x L2, one graph per M over the replicas; TB/s on the weight bytes
    (any x gather inside the calls)."""
    t = lambda a: None if a is None else torch.from_numpy(a).to(dev)
    tot_b, tot_s, cases = 0.0, 0.0, {}
    for (K, N) in shapes:
        L = synthetic.workload_layer(workload, K, N, 128, act)
        R = max(2, int(np.ceil(3 * L2_BYTES / L.weight_bytes)))
        qw, qz, sc, gi, b = t(L.qweight), t(L.qzeros), t(L.scales), t(L.g_idx), t(L.bias)
        mats = [q4.Q4Matrix(qw, qz, sc, gi, b, 128) for _ in range(R)]
        for m in mats:
            m.reserve(max(Ms))
        for M in Ms:
            x = t(synthetic.workload_x(workload, K, N, 128, act, M))
            o = torch.empty((M, N), dtype=torch.float16, device=dev)

            def issue(sp):
                for m in mats:
                    q4.gptq_q4_matmul(m.handle, x.data_ptr(), M, o.data_ptr(), sp)

            g, _ = capture(torch, q4, issue)
            s = graph_seconds(torch, stream, g, 10) / R
            del g
            cases[f"{K}x{N} M={M}"] = round(s * 1e6, 2)
            tot_b += L.weight_bytes
            tot_s += s
        del mats
    v = tot_b / tot_s / 1e12
    return {"TB/s": r3(v), "frac": r3(v * 1e3 / hbm_gbs)}, cases


def run_prefill_7b(q4, torch, dev, stream, bf16_tf):
    """prefill_7b: fused (shared-memory dequantization inside the tcgen05
    GEMM) at M in {512, 2048} x the three 7B shapes x {trivial, act-order};
    the unfused route (dequantize to temp_dq, then the tcgen05 GEMM) beside it
    on the trivial cases.  One call per graph, replayed back to back."""
    out, detail = {}, {}
    f_tot = {512: [0.0, 0.0], 2048: [0.0, 0.0]}
    u_tot = [0.0, 0.0]
    fr = {512: [], 2048: []}
    for act in (False, True):
        for (K, N) in synthetic.PREFILL_7B_SHAPES:
            L = synthetic.workload_layer("prefill_7b", K, N, 128, act)
            t = lambda a: None if a is None else torch.from_numpy(a).to(dev)
            mat = q4.Q4Matrix(t(L.qweight), t(L.qzeros), t(L.scales), t(L.g_idx), None, 128)
            mat.reserve(max(synthetic.PREFILL_7B_M))
            temp_dq = torch.empty((K, N), dtype=torch.float16, device=dev)
            for M in synthetic.PREFILL_7B_M:
                x = t(synthetic.workload_x("prefill_7b", K, N, 128, act, M))
                o = torch.empty((M, N), dtype=torch.float16, device=dev)
                g, _ = capture(torch, q4, lambda sp: q4.gptq_q4_matmul(mat.handle, x.data_ptr(), M, o.data_ptr(), sp))
                s = graph_seconds(torch, stream, g, 10)
                del g
                fl = 2.0 * M * K * N
                f_tot[M][0] += fl
                f_tot[M][1] += s
                fr[M].append(fl / s / 1e12 / bf16_tf)
                name = f"{K}x{N} M={M}{' act' if act else ''}"
                detail[name] = {"us": round(s * 1e6, 1), "TFLOP/s": round(fl / s / 1e12, 1)}
                if not act:
                    g, _ = capture(torch, q4, lambda sp: q4.gptq_q4_matmul_unfused(
                        mat.handle, x.data_ptr(), M, temp_dq.data_ptr(), o.data_ptr(), sp))
                    su = graph_seconds(torch, stream, g, 10)
                    del g
                    u_tot[0] += fl
                    u_tot[1] += su
                    detail[name]["unfused_us"] = round(su * 1e6, 1)
            mat.close()
            del temp_dq
    for M in (512, 2048):
        v = f_tot[M][0] / f_tot[M][1] / 1e12
        out[f"m{M}"] = [r3(v, 1), r3(v / bf16_tf), r3(min(fr[M])), r3(max(fr[M]))]
    out["unfused"] = r3(u_tot[0] / u_tot[1] / 1e12, 1)
    return out, detail


def run_sweep_70b_cases(q4, torch, dev, stream, sw, hbm_gbs, tf_peak):
    """Every sweep_70b case on its own: per (config, M) a graph over the
    config's replicas; binding-roofline fraction per case."""
    cases = {}
    for c in sw.cfgs:
        for M in synthetic.SWEEP_70B_M:
            mats = c["mats"] if M < 2048 else c["mats"][:1]
            x = torch.from_numpy(synthetic.workload_x("sweep_70b", c["K"], c["N"], c["g"], c["act"], M)).to(dev)
            o = torch.empty((M, c["N"]), dtype=torch.float16, device=dev)
            for m in mats:
                m.reserve(M)

            def issue(sp):
                for m in mats:
                    q4.gptq_q4_matmul(m.handle, x.data_ptr(), M, o.data_ptr(), sp)

            g, _ = capture(torch, q4, issue)
            s = graph_seconds(torch, stream, g, 5) / len(mats)
            del g
            t_bw = c["wb"] / (hbm_gbs * 1e9)
            t_tc = 2.0 * M * c["K"] * c["N"] / (tf_peak * 1e12)
            cases[f"{cfg_name((c['K'], c['N'], c['g'], c['act']))} M={M}"] = {
                "us": round(s * 1e6, 2), "frac": round(max(t_bw, t_tc) / s, 3)}
    return cases


def main():
    args = parse()
    if args.single:
        run_single(args.single)
    elif args.impl == "reference":
        run_reference(args)
    else:
        run_native(args)


if __name__ == "__main__":
    main()
