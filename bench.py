"""Benchmark of the fused GPTQ W4A16 linear layer on one GB300 (or N replicas).

Workload (decode_7b): Llama-7B-shaped projection layers (K,N) in
{(4096,4096), (4096,11008), (11008,4096), (4096,12288)}, groupsize 128,
trivial g_idx, fp16 bias, x ~ N(0,1) fp16, with M in {1,2,4,8} rows.  One
step runs every (shape, M) case once on each of R weight replicas, so that a
weight set is touched once per step and the per-step working set (R * 81.7 MB)
is several times the 129 MB L2: every call streams its weights from HBM.

Metric: effective HBM bandwidth of decode, algorithmic bytes (qweight +
qzeros + scales as stored) per second, whole job.  Also reported: the
decode kernel's roofline fraction (per-launch CUDA events), the end-to-end
figure through the C ABI with host buffers, the CPU oracle timed on this
host, SM clocks during the run, the prefill_7b tensor-core numbers, the
Llama-70B M = 1 layers and the act-order decode workload, and (next_rows)
the rows past the hot path: fused Q/K/V projections, GPTQ_V2, 8-bit codes,
bf16 activations and the GPU packer.

--impl reference times the CPU oracle (the plain dequantize-then-matmul
route) on the same workload, one shape per step.
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


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=20)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--impl", default="native", choices=["native", "reference"])
    p.add_argument("--replicas", type=int, default=8)
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-prefill", action="store_true")
    p.add_argument("--soak-s", type=float, default=1.0)
    p.add_argument("--only", choices=["decode", "prefill"], default=None,
                   help="run one leg only (for profiling); the JSON line is then partial")
    p.add_argument("--sweep70b", action="store_true",
                   help="also time all 240 sweep_70b cases (several minutes); adds a sweep_70b key")
    p.add_argument("--single", default=None, metavar="K,N,M[,PATH]",
                   help="profiling target instead of the bench: one synthetic g=128 layer, a 256 MB L2 "
                        "flush before each of four calls on PATH (a GPTQ_Q4_PATH_* suffix, default DECODE)")
    return p.parse_args()


def run_single(spec: str) -> None:
    """Four calls of one layer, each after an L2 flush: a short, fixed launch
    sequence for ncu captures (-s 3 -c 1 takes the fourth call)."""
    import torch
    import gptq_bit_weight_gb300 as q4
    parts = spec.split(",")
    K, N, M = int(parts[0]), int(parts[1]), int(parts[2])
    path = getattr(q4, "GPTQ_Q4_PATH_" + (parts[3].upper() if len(parts) > 3 else "DECODE"))
    layer = synthetic.make_layer(K, N, 128, bias=True, key=(77, K, N))
    dev = torch.device("cuda", 0)
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(dev)
    mat = q4.Q4Matrix(t(layer.qweight), t(layer.qzeros), t(layer.scales), None, t(layer.bias), 128)
    mat.set_path(path)
    x = t(synthetic.activations(M, K, key=(77, K, N, M)))
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    for _ in range(4):
        flush.zero_()
        y = mat(x)
    torch.cuda.synchronize()
    mat.device_error()
    print(json.dumps({"single": spec, "max_abs_y": float(y.float().abs().max())}))


# DRAM bytes the decode kernels move per algorithmic byte, from an ncu launch
# list of the decode_7b leg (dram__bytes_read.sum + dram__bytes_write.sum over
# 1216 launches / their K*N/2 + G*N*2.5 bytes); the kernels read every packed
# word, scale and zero once.
DECODE_DRAM_PER_ALGORITHMIC_BYTE = 24957.7e6 / 24841.4e6


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), float(d.get("bf16_tflops_sustained", d["bf16_tflops"])), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, FALLBACK_BF16_TFLOPS, 1700.0, "fallback"


def dist_env():
    return int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")), int(os.environ.get("LOCAL_RANK", "0"))


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


# --------------------------------------------------------------- reference

def run_reference(args):
    """The CPU oracle on the decode_7b workload: one shape (all four M) per step."""
    rank, world, _ = dist_env()
    if rank != 0:
        return
    import oracle
    oracle.build()
    cores = os.cpu_count() or 1
    shapes = synthetic.DECODE_7B_SHAPES
    layers = {s: synthetic.workload_layer("decode_7b", s[0], s[1], 128, False) for s in shapes}
    xs = {(s, M): synthetic.workload_x("decode_7b", s[0], s[1], 128, False, M) for s in shapes
          for M in synthetic.DECODE_7B_M}

    def step(i):
        s = shapes[i % len(shapes)]
        L = layers[s]
        dq = oracle.dequantize_layer(L.qweight, L.qzeros, L.scales, None, s[0], s[1], 128)
        for M in synthetic.DECODE_7B_M:
            oracle.reference_output(xs[(s, M)], dq, L.bias, nthreads=cores)
        return L.weight_bytes * len(synthetic.DECODE_7B_M)

    for i in range(args.warmup):
        step(i)
    t0 = time.perf_counter()
    nbytes = 0
    for i in range(args.steps):
        nbytes += step(args.warmup + i)
    dt = time.perf_counter() - t0
    value = nbytes / dt / 1e12
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": {"workload": "decode_7b", "shapes": [list(s) for s in shapes], "M": synthetic.DECODE_7B_M,
                   "groupsize": 128, "step": "one shape, all four M, dequantize once then fp64 products"},
        "cpu_baseline": {"value": value, "unit": "TB/s", "cores": cores, "kind": "oracle",
                         "sample": "each step: one decode_7b shape, all four M (shapes in turn)"},
        "e2e": {"value": value, "unit": "TB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def cpu_baseline_sample(budget_s: float = 25.0):
    """The oracle as it stands on the decode_7b cases, shape by shape, within a time budget."""
    import oracle
    oracle.build()
    cores = os.cpu_count() or 1
    t0 = time.perf_counter()
    nbytes, ncases, shapes_done = 0, 0, []
    for (K, N) in synthetic.DECODE_7B_SHAPES:
        L = synthetic.workload_layer("decode_7b", K, N, 128, False)
        dq = oracle.dequantize_layer(L.qweight, L.qzeros, L.scales, None, K, N, 128)
        for M in synthetic.DECODE_7B_M:
            x = synthetic.workload_x("decode_7b", K, N, 128, False, M)
            oracle.reference_output(x, dq, L.bias, nthreads=cores)
            nbytes += L.weight_bytes
            ncases += 1
        shapes_done.append([K, N])
        if time.perf_counter() - t0 > budget_s:
            break
    dt = time.perf_counter() - t0
    return {"value": nbytes / dt / 1e12, "unit": "TB/s", "cores": cores, "kind": "oracle",
            "sample": f"{ncases} decode_7b cases (shapes {shapes_done}, M 1/2/4/8; dequantize once per shape, "
                      f"fp64 products on {cores} threads), {dt:.1f} s"}


# ------------------------------------------------------------------ native

def run_native(args):
    import torch

    import gptq_bit_weight_gb300 as q4

    if args.only == "prefill":
        dev = torch.device("cuda", 0)
        torch.cuda.set_device(dev)
        _, bf16_tf, _, peak_src = peaks()
        print(json.dumps({"prefill": run_prefill(q4, torch, dev, torch.cuda.current_stream(), bf16_tf, peak_src)}),
              flush=True)
        return

    rank, world, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    stream = torch.cuda.current_stream()
    sptr = stream.cuda_stream
    hbm_gbs, bf16_tf, bf16_tf_sus, peak_src = peaks()

    shapes = synthetic.DECODE_7B_SHAPES
    Ms = synthetic.DECODE_7B_M
    R = args.replicas
    mats, wbytes = {}, {}
    for (K, N) in shapes:
        L = synthetic.workload_layer("decode_7b", K, N, 128, False)
        qw = torch.from_numpy(L.qweight).to(dev)
        qz = torch.from_numpy(L.qzeros).to(dev)
        sc = torch.from_numpy(L.scales).to(dev)
        b = torch.from_numpy(L.bias).to(dev)
        mats[(K, N)] = [q4.Q4Matrix(qw, qz, sc, None, b, 128) for _ in range(R)]
        for m in mats[(K, N)]:
            m.reserve(max(Ms))
        wbytes[(K, N)] = L.weight_bytes
        del qw, qz, sc
    xs = {(s, M): torch.from_numpy(synthetic.workload_x("decode_7b", s[0], s[1], 128, False, M)).to(dev)
          for s in shapes for M in Ms}
    outs = {(s, M): torch.empty((M, s[1]), dtype=torch.float16, device=dev) for s in shapes for M in Ms}
    calls = [(s, M, r) for r in range(R) for M in Ms for s in shapes]
    step_bytes = sum(wbytes[s] for (s, M, r) in calls)
    l2_defeated = R * sum(wbytes.values()) > 2 * L2_BYTES

    def issue(call_list, stream_ptr):
        for (s, M, r) in call_list:
            q4.gptq_q4_matmul(mats[s][r].handle, xs[(s, M)].data_ptr(), M, outs[(s, M)].data_ptr(), stream_ptr)

    def barrier():
        rank_barrier(world)
        torch.cuda.synchronize()

    def max_over_ranks(v):
        return max_over_ranks_value(v, world, dev)

    # One step is captured once into a CUDA graph and replayed: the kernels
    # then run back to back as in a model's decode loop, instead of waiting
    # on Python + ctypes + the launch API for every call (~11 us a call).
    def capture(call_list):
        g = torch.cuda.CUDAGraph()
        issue(call_list, sptr)                  # make sure nothing allocates during capture
        torch.cuda.synchronize()
        n0 = q4.gptq_q4_launch_count()
        with torch.cuda.graph(g):
            issue(call_list, torch.cuda.current_stream().cuda_stream)
        return g, q4.gptq_q4_launch_count() - n0

    step_graph, launches_per_step = capture(calls)

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
        launches = launches_per_step * args.steps
        ms = max_over_ranks(e0.elapsed_time(e1))
        # ---- the same steps launched eagerly, call by call, for comparison
        barrier()
        e2, e3 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e2.record(stream)
        for _ in range(args.steps):
            issue(calls, sptr)
        e3.record(stream)
        barrier()
        eager_ms = max_over_ranks(e2.elapsed_time(e3))
    clocks = clk.summary()

    value = job_throughput(step_bytes, args.steps, world, ms * 1e-3)
    eager_value = job_throughput(step_bytes, args.steps, world, eager_ms * 1e-3)
    # The timed region holds nothing but decode kernels, back to back: the
    # average launch duration is the region's time over its launches.
    achieved_gbs = step_bytes * args.steps / (ms * 1e-3) / 1e9

    # per-case figures: a graph of the R replicas of one case, replayed
    per_case = {}
    for s in shapes:
        for M in Ms:
            g, n = capture([(s, M, r) for r in range(R)])
            for _ in range(3):
                g.replay()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            reps = 20
            a.record(stream)
            for _ in range(reps):
                g.replay()
            b.record(stream)
            torch.cuda.synchronize()
            us = a.elapsed_time(b) * 1e3 / (reps * R)
            per_case[f"{s[0]}x{s[1]} M={M}"] = {"us": round(us, 2), "TB/s": round(wbytes[s] / (us * 1e-6) / 1e12, 3)}
            del g

    # ---- end to end through the C ABI with host buffers (pinned), copies inside the timed region.
    # One step, as a decode loop would run it: the step's inputs copied host -> device (one copy
    # per distinct input; the replicas of a case share it), every C-ABI matmul, the results copied
    # device -> host, all captured once into a CUDA graph and replayed; timed on the host clock
    # up to the completed device -> host copies.
    hx = {k: v.cpu().pin_memory() for k, v in xs.items()}
    ho = {k: torch.empty(v.shape, dtype=torch.float16).pin_memory() for k, v in outs.items()}
    dx = {k: torch.empty_like(v) for k, v in xs.items()}
    h2d = sum(t.numel() * 2 for t in hx.values())
    d2h = sum(t.numel() * 2 for t in ho.values())

    def e2e_issue(stream_ptr):
        for k in hx:
            dx[k].copy_(hx[k], non_blocking=True)
        for (s, M, r) in calls:
            q4.gptq_q4_matmul(mats[s][r].handle, dx[(s, M)].data_ptr(), M, outs[(s, M)].data_ptr(), stream_ptr)
        for k in ho:
            ho[k].copy_(outs[k], non_blocking=True)

    e2e_issue(sptr)
    torch.cuda.synchronize()
    e2e_graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(e2e_graph):
        e2e_issue(torch.cuda.current_stream().cuda_stream)
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
    assert all(torch.equal(ho[k], outs[k].cpu()) for k in ho), "e2e results did not reach the host"

    decode_70b = None
    if args.only is None:
        decode_70b = run_decode_70b(q4, torch, dev, stream, hbm_gbs)
        actorder = run_actorder_decode(q4, torch, dev, stream, hbm_gbs, bf16_tf)
        next_rows = run_next_rows(q4, torch, dev, stream, hbm_gbs)
        sweep70 = run_sweep_70b(q4, torch, dev, stream, hbm_gbs, bf16_tf) if args.sweep70b else None

    prefill = None
    if not args.no_prefill and args.only != "decode":
        prefill = run_prefill(q4, torch, dev, stream, bf16_tf, peak_src)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline and args.only is None:
        cpu = cpu_baseline_sample()

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "TB/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms / args.steps, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f16 x int4 -> f32 accumulate", "data": "synthetic",
            "config": {"workload": "decode_7b", "shapes": [list(s) for s in shapes], "M": Ms, "groupsize": 128,
                       "g_idx": "trivial", "bias": True, "replicas": R,
                       "calls_per_step": len(calls), "launch": "one CUDA graph per step (captured C-ABI calls)",
                       "l2": (f"inputs larger than L2: {R} weight replicas, {R * sum(wbytes.values()) / 1e6:.0f} MB "
                              f"per step vs 129 MB L2, each replica touched once per step") if l2_defeated else
                             f"NOT defeated: {R} replicas = {R * sum(wbytes.values()) / 1e6:.0f} MB (profiling run)",
                       "bytes_per_step": step_bytes, "soak_s": args.soak_s,
                       "parallelism": f"replicas x{world}"},
            "roofline": {"bound": "hbm", "achieved": achieved_gbs, "peak": hbm_gbs, "unit": "GB/s",
                         "frac": achieved_gbs / hbm_gbs,
                         # DRAM bytes (read + write) per step: the algorithmic bytes times the ratio
                         # ncu measured over every decode_7b launch of the bench
                         "traffic": round(step_bytes * DECODE_DRAM_PER_ALGORITHMIC_BYTE),
                         "traffic_unit": "bytes per step",
                         "kernel": ("decode_kernel<1,*> (register-streaming with a shared-memory weight ring; "
                                    "every decode_7b case)"),
                         "peak_source": peak_src,
                         "how": "algorithmic bytes of the timed region / its CUDA-event time (only decode kernels run in it)"},
            "eager": {"value": eager_value, "unit": "TB/s",
                      "how": "the same steps launched call by call from Python through the C ABI"},
            "per_case": per_case,
            "e2e": {"value": e2e_value, "unit": "TB/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
            "gpu_launches": launches,
            "clocks": clocks,
        }
        if decode_70b:
            line["decode_70b"] = decode_70b
            line["actorder_7b"] = actorder
            line["next_rows"] = next_rows
            if sweep70:
                line["sweep_70b"] = sweep70
        if prefill:
            line["prefill"] = prefill
        if cpu:
            line["cpu_baseline"] = cpu
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def run_decode_70b(q4, torch, dev, stream, hbm_gbs, reps=10):
    """M=1 decode on the Llama-70B projection shapes (sweep_70b, g=128,
    trivial g_idx): per shape, enough weight replicas to exceed L2, captured
    in one CUDA graph and replayed; eff. TB/s on the stored weight bytes."""
    out = {}
    tot_bytes, tot_s = 0.0, 0.0
    for (K, N) in synthetic.SWEEP_70B_SHAPES:
        L = synthetic.workload_layer("sweep_70b", K, N, 128, False)
        qw, qz, sc = (torch.from_numpy(a).to(dev) for a in (L.qweight, L.qzeros, L.scales))
        R = max(2, int(np.ceil(3 * L2_BYTES / L.weight_bytes)))
        mats = [q4.Q4Matrix(qw, qz, sc, None, None, 128) for _ in range(R)]
        del qw, qz, sc
        x = torch.from_numpy(synthetic.workload_x("sweep_70b", K, N, 128, False, 1)).to(dev)
        o = torch.empty((1, N), dtype=torch.float16, device=dev)
        for m in mats:
            q4.gptq_q4_matmul(m.handle, x.data_ptr(), 1, o.data_ptr(), stream.cuda_stream)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            for m in mats:
                q4.gptq_q4_matmul(m.handle, x.data_ptr(), 1, o.data_ptr(), torch.cuda.current_stream().cuda_stream)
        for _ in range(3):
            g.replay()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(reps):
            g.replay()
        b.record(stream)
        torch.cuda.synchronize()
        us = a.elapsed_time(b) * 1e3 / (reps * R)
        tbs = L.weight_bytes / (us * 1e-6) / 1e12
        out[f"{K}x{N} M=1"] = {"us": round(us, 2), "TB/s": round(tbs, 3), "frac": round(tbs * 1e3 / hbm_gbs, 3)}
        tot_bytes += L.weight_bytes
        tot_s += us * 1e-6
        del g, mats
    return {"workload": "sweep_70b M=1, g=128, trivial g_idx", "value": tot_bytes / tot_s / 1e12, "unit": "TB/s",
            "frac_of_hbm_peak": tot_bytes / tot_s / 1e9 / hbm_gbs, "cases": out,
            "how": "weight bytes / per-call time from CUDA-graph replays of >= 3x L2 of weight replicas"}


def time_layer_cases(q4, torch, dev, stream, workload, K, N, g, act, Ms, hbm_gbs, tf_peak, reps=10):
    """One layer configuration of a workload at several M through the default
    path (GPTQ_Q4_PATH_AUTO): enough weight replicas to exceed L2 three times,
    each M captured in one CUDA graph over the replicas and replayed.  Per
    case: time per call, eff. TB/s on the stored weight bytes, TFLOP/s, and the
    fraction of the roofline that binds, max(bytes/HBM, flops/tensor)/time."""
    L = synthetic.workload_layer(workload, K, N, g, act)
    t = lambda a: None if a is None else torch.from_numpy(a).to(dev)
    qw, qz, sc, gi = t(L.qweight), t(L.qzeros), t(L.scales), t(L.g_idx)
    R = max(2, int(np.ceil(3 * L2_BYTES / L.weight_bytes)))
    mats = [q4.Q4Matrix(qw, qz, sc, gi, None, g) for _ in range(R)]
    del qw, qz, sc, gi
    for m in mats:
        m.reserve(max(Ms))
    res = {}
    for M in Ms:
        x = t(synthetic.workload_x(workload, K, N, g, act, M))
        o = torch.empty((M, N), dtype=torch.float16, device=dev)
        for m in mats:
            q4.gptq_q4_matmul(m.handle, x.data_ptr(), M, o.data_ptr(), stream.cuda_stream)
        torch.cuda.synchronize()
        gr = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gr):
            for m in mats:
                q4.gptq_q4_matmul(m.handle, x.data_ptr(), M, o.data_ptr(), torch.cuda.current_stream().cuda_stream)
        for _ in range(3):
            gr.replay()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(reps):
            gr.replay()
        b.record(stream)
        torch.cuda.synchronize()
        sec = a.elapsed_time(b) * 1e-3 / (reps * R)
        flops = 2.0 * M * K * N
        t_bw, t_tc = L.weight_bytes / (hbm_gbs * 1e9), flops / (tf_peak * 1e12)
        res[M] = {"us": round(sec * 1e6, 2), "TB/s": round(L.weight_bytes / sec / 1e12, 3),
                  "TFLOP/s": round(flops / sec / 1e12, 1), "bound": "hbm" if t_bw >= t_tc else "tensor",
                  "frac": round(max(t_bw, t_tc) / sec, 3)}
        del gr
    del mats
    torch.cuda.empty_cache()
    return L.weight_bytes, res


def run_actorder_decode(q4, torch, dev, stream, hbm_gbs, tf_peak):
    """actorder_7b: decode with a scattered act-order g_idx, M in {1, 4, 16},
    on (4096, 11008) and (11008, 4096); the x reorder runs inside each call."""
    cases, tot_b, tot_s = {}, 0.0, 0.0
    for (K, N) in synthetic.ACTORDER_7B_SHAPES:
        wb, res = time_layer_cases(q4, torch, dev, stream, "actorder_7b", K, N, 128, True, synthetic.ACTORDER_7B_M,
                                   hbm_gbs, tf_peak)
        for M, r in res.items():
            cases[f"{K}x{N} M={M}"] = r
            tot_b += wb
            tot_s += r["us"] * 1e-6
    return {"workload": "actorder_7b", "value": tot_b / tot_s / 1e12, "unit": "TB/s",
            "frac_of_hbm_peak": tot_b / tot_s / 1e9 / hbm_gbs, "cases": cases,
            "how": "weight bytes / per-call time (x reorder included) from CUDA-graph replays of >= 3x L2 of replicas"}


def run_sweep_70b(q4, torch, dev, stream, hbm_gbs, tf_peak):
    """sweep_70b in full: 3 shapes x 4 group sizes x {trivial, act-order} x
    10 values of M (240 cases), through the default path."""
    cases = {}
    for (K, N) in synthetic.SWEEP_70B_SHAPES:
        for g in synthetic.SWEEP_70B_G:
            for act in (False, True):
                _, res = time_layer_cases(q4, torch, dev, stream, "sweep_70b", K, N, g, act, synthetic.SWEEP_70B_M,
                                          hbm_gbs, tf_peak, reps=5)
                for M, r in res.items():
                    cases[f"{K}x{N} g={g} act={int(act)} M={M}"] = r
    fr = [r["frac"] for r in cases.values()]
    return {"workload": "sweep_70b (all 240 cases)", "cases": cases, "median_frac": float(np.median(fr)),
            "min_frac": float(np.min(fr)), "max_frac": float(np.max(fr))}


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


def run_prefill(q4, torch, dev, stream, bf16_tf, peak_src, reps=10):
    """prefill_7b: M in {512, 2048} x the three 7B shapes x {trivial, act-order}.

    Fused (shared-memory dequantization inside the tcgen05 GEMM) against the
    unfused route (dequantize to temp_dq, then the tcgen05 GEMM on it).  Each
    case is one call captured in a CUDA graph, replayed `reps` times back to
    back after a warm-up and timed with CUDA events around the replays; the
    work is compute-bound, so the 129 MB L2 does not flatter it."""
    sptr = stream.cuda_stream
    cases, tot_flops, tot_fused, tot_unf = {}, 0.0, 0.0, 0.0
    per_launch = []
    for act in (False, True):
        for (K, N) in synthetic.PREFILL_7B_SHAPES:
            L = synthetic.workload_layer("prefill_7b", K, N, 128, act)
            mat = q4.Q4Matrix(torch.from_numpy(L.qweight).to(dev), torch.from_numpy(L.qzeros).to(dev),
                              torch.from_numpy(L.scales).to(dev),
                              None if L.g_idx is None else torch.from_numpy(L.g_idx).to(dev), None, 128)
            mat.reserve(max(synthetic.PREFILL_7B_M))
            temp_dq = torch.empty((K, N), dtype=torch.float16, device=dev)
            for M in synthetic.PREFILL_7B_M:
                x = torch.from_numpy(synthetic.workload_x("prefill_7b", K, N, 128, act, M)).to(dev)
                out = torch.empty((M, N), dtype=torch.float16, device=dev)

                def fused(sp):
                    q4.gptq_q4_matmul(mat.handle, x.data_ptr(), M, out.data_ptr(), sp)

                def unfused(sp):
                    q4.gptq_q4_matmul_unfused(mat.handle, x.data_ptr(), M, temp_dq.data_ptr(), out.data_ptr(), sp)

                mat.set_path(q4.GPTQ_Q4_PATH_PREFILL)
                times = {}
                for name, fn in (("fused", fused), ("unfused", unfused)):
                    # one call captured in a CUDA graph and replayed back to back, so that the
                    # host's launch cost does not show as device time on the short cases
                    for _ in range(3):
                        fn(sptr)
                    torch.cuda.synchronize()
                    g = torch.cuda.CUDAGraph()
                    with torch.cuda.graph(g):
                        fn(torch.cuda.current_stream().cuda_stream)
                    g.replay()
                    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                    a.record(stream)
                    for _ in range(reps):
                        g.replay()
                    b.record(stream)
                    torch.cuda.synchronize()
                    times[name] = a.elapsed_time(b) / reps
                    del g
                flops = 2.0 * M * K * N
                tot_flops += flops
                tot_fused += times["fused"]
                tot_unf += times["unfused"]
                if not act:
                    per_launch.append((flops, times["fused"]))
                cases[f"{K}x{N} M={M}{' act' if act else ''}"] = {
                    "fused_us": round(times["fused"] * 1e3, 1),
                    "fused_TFLOPS": round(flops / (times["fused"] * 1e-3) / 1e12, 1),
                    "unfused_us": round(times["unfused"] * 1e3, 1),
                    "unfused_TFLOPS": round(flops / (times["unfused"] * 1e-3) / 1e12, 1)}
            mat.close()
            del temp_dq
    fused_tf = tot_flops / (tot_fused * 1e-3) / 1e12
    kern_flops = sum(f for f, _ in per_launch)
    kern_ms = sum(t for _, t in per_launch)
    achieved = kern_flops / (kern_ms * 1e-3) / 1e12
    return {
        "workload": "prefill_7b", "metric": "prefill TFLOPS (2*M*K*N / time)", "value": fused_tf,
        "unit": "TFLOP/s", "unfused_value": tot_flops / (tot_unf * 1e-3) / 1e12,
        "roofline": {"bound": "tensor", "achieved": achieved, "peak": bf16_tf, "unit": "TFLOP/s",
                     "frac": achieved / bf16_tf, "traffic": None, "kernel": "prefill_kernel (fused prefill)",
                     "peak_source": f"{peak_src} bf16 burst x 1 (fp16 and bf16 dense rates are equal)",
                     "how": "trivial-g_idx cases: 2*M*K*N summed / per-call time (CUDA-graph replays) summed"},
        "cases": cases,
    }


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
