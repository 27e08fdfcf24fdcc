#!/usr/bin/env python
"""Benchmark of the flow-matching action-expert denoise loop on GB300.

One bench step = one whole denoise (T Euler steps over one batch of action
chunks) through the C ABI, inputs resident in HBM.  Prints ONE JSON line:
chunks/s (value), microseconds per denoise step, the dominant kernel's
roofline fraction (CUDA-event timed inside the captured graph), the same
metric end to end through host buffers (e2e), and the CPU oracle as a
baseline.

    python bench.py [--gpus N --steps K --warmup W] [--workload pi05] [--impl ours|reference]

Multi-GPU (torchrun, N > 1): replicas only -- every rank runs its own
independent denoise loops (the loop has no exchange step); value = chunks of
all ranks / the slowest rank's time.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import synth  # noqa: E402

METRIC = "action chunks/s & µs per denoise step (1 GB300); % of HBM/tensor roofline"
UNIT = "chunks/s"
L2_BYTES = 129 * 1024 * 1024

WORKLOAD_TEXT = {
    "pi05": "pi0.5-shaped expert, bf16: 18 layers, hidden 1024, 8x256 q heads, 1 KV head, GeGLU 4096, "
            "37 AdaRMS sites (hoisted [3072,1024] Denses), prefix 968, horizon 50, action_dim 32, batch 1, 10 steps",
    "gr00t": "GR00T-N1.7-shaped DiT head, bf16: 32 blocks alternating cross-attention (300 VL tokens, "
             "32x48 heads) and self-attention (1 state + 16 action tokens), hidden 1536, FF 6144, batch 1, 4 steps",
    "pi05_b32": "pi0.5-shaped expert as above at batch 32 (per-sample prefix 968), 10 steps",
    "pi05_long": "pi0.5-shaped expert, batch 8, prefix 4096 per sample, horizon 50, 10 steps",
    "pi05_fp8": "pi0.5-shaped expert as pi05 with the per-layer projections streamed as E4M3 codes + fp32 "
                "row scales (bf16 activations), batch 1, 10 steps",
    "gr00t_fp8": "GR00T-N1.7-shaped DiT head as gr00t with E4M3 per-layer projections, batch 1, 4 steps",
    "tiny": "tiny expert, fp32: 2 layers, hidden 256, 4x64 heads, GeLU 1024, prefix 64, horizon 16, batch 1, 4 steps",
}


# ----------------------------------------------------------------------------
# algorithmic work (bytes and FLOPs a kernel must move / do, no re-reads)
# ----------------------------------------------------------------------------

def kernel_work(g: dict, batch: int, prefix: int):
    """Per kernel class: (launches per denoise step, bytes per launch, FLOPs per launch)."""
    es = 2 if g["dtype"] == synth.DTYPE_BF16 else 4
    fp8 = g.get("weight_format", synth.WFMT_NATIVE) == synth.WFMT_FP8
    ws = 1 if fp8 else es            # bytes per element of the per-layer projections
    sc = 4 if fp8 else 0             # FP8: one fp32 scale per output row
    D, L, F, H, A = g["hidden"], g["layers"], g["mlp_dim"], g["horizon"], g["action_dim"]
    Hq, Dh = g["q_heads"], g["head_dim"]
    tok = H + g["state_tokens"]
    M = batch * tok
    qd = Hq * Dh
    dit = g["family"] == synth.FAMILY_DIT
    up_rows = synth.up_rows(g)
    out = {}

    def add(name, n, by, fl):
        c, b0, f0 = out.get(name, (0, 0.0, 0.0))
        out[name] = (c + n, b0 + by * n, f0 + fl * n)

    for l in range(L):
        nq = synth.qkv_rows(g, l)
        add("qkv_gemm", 1, nq * (D * ws + sc) + M * D * es + M * nq * es, 2.0 * M * nq * D)
        add("o_gemm", 1, D * (qd * ws + sc) + M * qd * es + M * D * 8 + batch * D * es, 2.0 * M * D * qd)
        add("up_gemm", 1, up_rows * (D * ws + sc) + M * D * es + M * F * es, 2.0 * M * up_rows * D)
        add("down_gemm", 1, D * (F * ws + sc) + M * F * es + M * D * 8 + batch * D * es, 2.0 * M * D * F)
        if dit and l % 2 == 0:
            keys, kv = prefix, batch * prefix * g["kv_heads"] * Dh * 2 * es
        elif dit:
            keys, kv = tok, 0
        else:
            keys, kv = prefix + H, batch * prefix * Dh * 2 * es
        add("attention", 1, kv + 2 * M * qd * es + (0 if dit else batch * H * Dh * 2 * es),
            4.0 * batch * Hq * tok * keys * Dh)
    # convert totals to per-launch averages
    return {k: (n, b / n, f / n) for k, (n, b, f) in out.items()}


def step_work(g: dict, batch: int, prefix: int):
    """Algorithmic bytes and FLOPs of one denoise step (every weight + K/V read once)."""
    w = kernel_work(g, batch, prefix)
    return sum(n * b for n, b, f in w.values()), sum(n * f for n, b, f in w.values())


KCLASS = {"qkv_gemm": 1, "attention": 2, "o_gemm": 3, "up_gemm": 4, "down_gemm": 5}

# DRAM bytes (read + write) per launch of a kernel class, from one `ncu --set full`
# capture (profiles/pi05_b1_kernels_full.md, profiles/pi05_b32_kernels_full.md),
# with the SHA-1 prefixes of the sources those kernels were built from: a value
# is reported only while every listed source is unchanged.
_GEMM_SRC = {"gemm_tc.cu": "394de066eb6a04ef", "epilogue.cuh": "8f28ff6cb7f33192"}
_ATTN_SRC = {"attention_tc5.cu": "3179e2d1ae18a24c"}
TRAFFIC = {
    ("pi05", "attention"): (1.28e6 + 3.56e6, _ATTN_SRC),   # attention + split merge
    ("pi05", "o_gemm"): (4.47e6, _GEMM_SRC),
    ("pi05", "up_gemm"): (16.96e6, _GEMM_SRC),
    ("pi05", "down_gemm"): (8.87e6, _GEMM_SRC),
    ("pi05_b32", "qkv_gemm"): (8.67e6, _GEMM_SRC),
    ("pi05_b32", "attention"): (39.95e6, _ATTN_SRC),
    ("pi05_b32", "o_gemm"): (10.82e6, _GEMM_SRC),
    ("pi05_b32", "up_gemm"): (20.15e6, _GEMM_SRC),
    ("pi05_b32", "down_gemm"): (21.57e6, _GEMM_SRC),
}


def measured_traffic(workload: str, kernel: str):
    """Per-launch DRAM bytes of ``kernel`` from the committed capture, or None when
    there is none for this workload or a listed source changed since."""
    import hashlib
    ent = TRAFFIC.get((workload, kernel))
    if ent is None:
        return None
    nbytes, srcs = ent
    csrc = os.path.join(ROOT, "flow_matching_vla_gb300", "csrc")
    for name, digest in srcs.items():
        try:
            with open(os.path.join(csrc, name), "rb") as f:
                if hashlib.sha1(f.read()).hexdigest()[:16] != digest:
                    return None
        except OSError:
            return None
    return nbytes


# ----------------------------------------------------------------------------
# clocks during the timed region
# ----------------------------------------------------------------------------

class Clocks:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.dev = device_index
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.dev), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"], stdout=self.f, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if not self.proc:
            return None
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.f.close()
        rows = []
        for line in open(self.path):
            p = [x.strip() for x in line.split(",")]
            if len(p) < 9:
                continue
            try:
                rows.append((float(p[1]), float(p[2]), p[5:9]))
            except ValueError:
                continue
        os.unlink(self.path)
        if not rows:
            return None
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for _, _, r in rows for i in range(4) if r[i].lower().startswith("active")})
        mx = max(r[1] for r in rows)
        loaded = [r[0] for r in rows]
        return {"sm_mhz": statistics.median(loaded), "sm_max_mhz": mx, "reasons": reasons,
                "samples": len(rows)}


# ----------------------------------------------------------------------------
# CPU oracle baseline (bounded sample)
# ----------------------------------------------------------------------------

def oracle_rate(case, budget_s: float = 15.0, max_evals: int | None = None):
    """Chunks/s of the fp64 CPU oracle, from whole velocity evaluations of one sample."""
    import oracle
    g = case["geom"]
    T = g["steps"]
    sub = dict(case)
    sub["x_noise"] = case["x_noise"][:1]
    sub["K"] = [None if k is None else k[:1] for k in case["K"]]
    sub["V"] = [None if v is None else v[:1] for v in case["V"]]
    for key in ("text_mask", "image_mask", "state"):
        if case.get(key) is not None:
            sub[key] = case[key][:1]
    sub["geom"] = dict(g, batch=1)
    x = sub["x_noise"].astype(np.float64)
    from oracle.schedule import modulation_table
    from oracle.dit import action_time_bias
    mod = modulation_table(sub["geom"], sub["weights"], T, 1)
    atb = action_time_bias(sub["geom"], sub["weights"], T) if g["family"] == synth.FAMILY_DIT else None
    times = []
    t_end = time.perf_counter() + budget_s
    k = 0
    while True:
        t0 = time.perf_counter()
        v = oracle.velocity(sub, x, k % T, steps=T, mod=mod, atb=atb)
        times.append(time.perf_counter() - t0)
        k += 1
        if time.perf_counter() > t_end or (max_evals and k >= max_evals):
            break
    t_step = float(np.mean(times))
    cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
    return {"value": 1.0 / (T * t_step), "unit": UNIT, "cores": cores, "kind": "oracle",
            "sample": f"{len(times)} velocity evaluation(s) of 1 sample (numpy fp64, "
                      f"{t_step:.3f} s each) scaled to a {T}-step chunk"}, t_step


# ----------------------------------------------------------------------------

def dist_setup(impl: str):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if impl == "ours" else "gloo"
        if impl == "ours":
            import torch
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    return world, rank, local


def max_over_ranks(v: float, world: int) -> float:
    if world == 1:
        return v
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([v], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def run_reference(args, world, rank):
    if rank != 0:
        return 0
    case = synth.make_case(args.workload)
    g = case["geom"]
    budget = max(1.0, args.ref_seconds / max(1, args.steps + args.warmup))
    for _ in range(args.warmup):
        oracle_rate(case, budget_s=0.0, max_evals=1)
    t0 = time.perf_counter()
    rates = []
    for _ in range(args.steps):
        cb, t_step = oracle_rate(case, budget_s=0.0, max_evals=1)
        rates.append(t_step)
    el = time.perf_counter() - t0
    t_step = float(np.mean(rates))
    value = 1.0 / (g["steps"] * t_step)
    cores = cb["cores"]
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": el * 1000 / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded)", "config": config_obj(args, g),
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                             "sample": f"each step: 1 velocity evaluation of 1 sample of the workload "
                                       f"(numpy fp64 oracle on the host cores), scaled to a "
                                       f"{g['steps']}-step chunk"},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def config_obj(args, g):
    return {"workload": WORKLOAD_TEXT.get(args.workload, args.workload), "name": args.workload,
            "batch": g["batch"], "prefix": g["prefix"], "horizon": g["horizon"],
            "denoise_steps": g["steps"], "parallelism": f"replicas x{args.gpus}",
            "l2": "inputs larger than L2 (weights read every denoise step exceed 129 MB); no flush"}


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="pi05", choices=sorted(synth.CONFIGS))
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--ref-seconds", type=float, default=120.0)
    ap.add_argument("--no-kernel-timing", action="store_true")
    ap.add_argument("--profile", action="store_true",
                    help="warm up, then run one denoise inside the NVTX range 'denoise' (for ncu) and exit")
    args = ap.parse_args(argv)
    if args.warmup < 3 and args.impl == "ours":
        ap.error("--warmup must be >= 3")
    world, rank, local = dist_setup(args.impl)
    if args.impl == "reference":
        return run_reference(args, world, rank)

    import torch
    import flow_matching_vla_gb300 as fmv

    peaks = {}
    pk = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(pk):
        peaks = json.load(open(pk))
    hbm_peak = peaks.get("hbm_gbs", 6800.0)
    tc_peak = peaks.get("bf16_tflops_sustained", 1700.0)
    peak_src = "of measured" if peaks else "of fallback"

    case = synth.make_case(args.workload)
    g = case["geom"]
    B, T, P = g["batch"], g["steps"], g["prefix"]
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    stream = torch.cuda.Stream(device=dev)
    loop, held = fmv.from_case(case, stream=stream)
    x = torch.from_numpy(case["x_noise"]).to(dev)
    out = torch.empty_like(x)
    torch.cuda.synchronize()

    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            loop.denoise(x, out)
        stream.synchronize()
        kernels_per_step = loop.info(fmv.INFO_KERNELS_PER_STEP)
        if args.profile:
            torch.cuda.nvtx.range_push("denoise")
            loop.denoise(x, out)
            stream.synchronize()
            torch.cuda.nvtx.range_pop()
            print(json.dumps({"profile": args.workload, "kernels_per_denoise_step": kernels_per_step,
                              "denoise_steps": T}), flush=True)
            return 0
        barrier(world)
        clocks = fmv_clocks = Clocks(local)
        clocks.start()
        t0 = torch.cuda.Event(enable_timing=True)
        t1 = torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        t0.record(stream)
        for _ in range(args.steps):
            loop.denoise(x, out)
        t1.record(stream)
        t1.synchronize()
        torch.cuda.synchronize()
        clk = clocks.stop()
        ms = t0.elapsed_time(t1)
    ms = max_over_ranks(ms, world)
    chunks = B * args.steps * world
    value = chunks / (ms / 1000.0)
    ms_per_step = ms / args.steps
    us_per_denoise_step = ms_per_step * 1000.0 / T

    # e2e: the same loop through host buffers (H2D of the noise, D2H of the chunk, every step)
    xh = torch.from_numpy(case["x_noise"]).pin_memory()
    oh = torch.empty_like(xh).pin_memory()
    for _ in range(max(1, args.warmup // 2)):
        loop.denoise_host(xh, oh)
    barrier(world)
    e0 = time.perf_counter()
    for _ in range(args.steps):
        loop.denoise_host(xh, oh)
    e_el = max_over_ranks(time.perf_counter() - e0, world)
    e2e = {"value": chunks / e_el, "unit": UNIT, "h2d_bytes_per_step": int(xh.numel() * 4),
           "d2h_bytes_per_step": int(oh.numel() * 4)}

    # per-kernel durations inside the captured graph (event-record nodes)
    work = kernel_work(g, B, P)
    roofline, kernel_table = None, {}
    if not args.no_kernel_timing:
        with torch.cuda.stream(stream):
            for name, cls in KCLASS.items():
                if name not in work:
                    continue
                loop.set_option(fmv.OPT_TIME_KERNEL, cls)
                for _ in range(3):
                    loop.denoise(x, out)
                ts = loop.kernel_times()
                loop.set_option(fmv.OPT_TIME_KERNEL, 0)
                if not ts:
                    continue
                n, by, fl = work[name]
                avg = float(np.mean(ts)) / 1000.0
                kernel_table[name] = {"launches_per_step": n, "avg_us": avg * 1e6,
                                      "share_est": None, "bytes": by, "flops": fl}
            loop.denoise(x, out)
            stream.synchronize()
        total = sum(v["avg_us"] * v["launches_per_step"] for v in kernel_table.values())
        for v in kernel_table.values():
            v["share_est"] = v["avg_us"] * v["launches_per_step"] / total if total else None
        if kernel_table:
            dom = max(kernel_table, key=lambda k: kernel_table[k]["avg_us"] * kernel_table[k]["launches_per_step"])
            d = kernel_table[dom]
            ridge = tc_peak * 1e12 / (hbm_peak * 1e9)
            tensor = d["flops"] / d["bytes"] > ridge
            t = d["avg_us"] / 1e6
            if tensor:
                achieved, peak, unit = d["flops"] / t / 1e12, tc_peak, "TFLOP/s"
            else:
                achieved, peak, unit = d["bytes"] / t / 1e9, hbm_peak, "GB/s"
            roofline = {"kernel": dom, "bound": "tensor" if tensor else "hbm", "achieved": achieved,
                        "peak": peak, "unit": unit, "frac": achieved / peak,
                        "traffic": measured_traffic(args.workload, dom),
                        "peak_source": peak_src, "avg_launch_us": d["avg_us"],
                        "algorithmic_bytes_per_launch": d["bytes"],
                        "algorithmic_flops_per_launch": d["flops"]}

    step_bytes, step_flops = step_work(g, B, P)
    t_hbm = step_bytes / (hbm_peak * 1e9)
    t_tc = step_flops / (tc_peak * 1e12)
    t_min = max(t_hbm, t_tc)
    if rank != 0:
        return 0
    cpu = None
    if not args.no_cpu_baseline and world == 1:
        cpu, _ = oracle_rate(case, budget_s=args.cpu_seconds)
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "us_per_denoise_step": us_per_denoise_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16" if g["dtype"] == synth.DTYPE_BF16 else "f32",
        "data": "synthetic (seeded; weights ~N(0,0.02), K/V and noise ~N(0,1))",
        "config": config_obj(argparse.Namespace(**{**vars(args), "gpus": world}), g),
        "roofline": roofline,
        "step_roofline": {"bytes_per_denoise_step": step_bytes, "flops_per_denoise_step": step_flops,
                          "t_min_us": t_min * 1e6, "frac": t_min * 1e6 / us_per_denoise_step,
                          "bound": "tensor" if t_tc > t_hbm else "hbm", "peak_source": peak_src},
        "kernels": kernel_table,
        "cpu_baseline": cpu,
        "e2e": e2e,
        "gpu_launches": int(kernels_per_step * T * args.steps),
        "clocks": clk,
    }
    print(json.dumps(line), flush=True)
    return 0


if __name__ == "__main__":
    sys.exit(main())
