#!/usr/bin/env python
"""Benchmark of the flow-matching action-expert denoise loop on GB300.

One bench step = one whole denoise (T Euler steps over one batch of action
chunks) through the C ABI, inputs resident in HBM.  The headline workload is
the pi0.5-shaped expert at batch 32 (per-sample 968-token prefix, 10 steps),
the largest single-GPU configuration.  Prints ONE JSON line: chunks/s
(value), microseconds per denoise step, the dominant kernel class against its
roofline (per-launch times from dependency-release stamps taken inside the
captured graph, so the programmatic-launch chain is the one timed), the whole
step against its roofline, the same metric end to end through host buffers
(e2e), the per-step slope of a step-count sweep, the hoisted cond
re-evaluation, the other workloads as extra keys, and the CPU oracle as a
baseline.

    python bench.py [--gpus N --steps K --warmup W] [--workload pi05_b32] [--impl ours|reference]

Multi-GPU (torchrun, N > 1): replicas only -- every rank runs its own
independent denoise loops (the loop has no exchange step); value = chunks of
all ranks / the slowest rank's time.
"""
from __future__ import annotations

import argparse
import json
import os
import platform
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
HEADLINE = "pi05_b32"
EXTRAS = ("pi05", "gr00t", "pi05_long")

WORKLOAD_TEXT = {
    "pi05": "pi0.5-shaped expert, bf16: 18 layers, hidden 1024, 8x256 q heads, 1 KV head, GeGLU 4096, "
            "37 AdaRMS sites (hoisted [3072,1024] Denses), prefix 968, horizon 50, action_dim 32, batch 1, 10 steps",
    "gr00t": "GR00T-N1.7-shaped DiT head, bf16: 32 blocks alternating cross-attention (300 VL tokens, "
             "32x48 heads) and self-attention (1 state + 16 action tokens), hidden 1536, FF 6144, batch 1, 4 steps",
    "pi05_b32": "pi0.5-shaped expert, bf16, batch 32 (per-sample prefix K/V of 968 tokens): 18 layers, hidden "
                "1024, 8x256 q heads, 1 KV head, GeGLU 4096, horizon 50, action_dim 32, 10 steps",
    "pi05_long": "pi0.5-shaped expert, bf16, batch 8, prefix 4096 per sample, horizon 50, 10 steps",
    "pi05_fp8": "pi0.5-shaped expert as pi05 with the per-layer projections streamed as E4M3 codes + fp32 "
                "row scales (bf16 activations), batch 1, 10 steps",
    "gr00t_fp8": "GR00T-N1.7-shaped DiT head as gr00t with E4M3 per-layer projections, batch 1, 4 steps",
    "tiny": "tiny expert, fp32: 2 layers, hidden 256, 4x64 heads, GeLU 1024, prefix 64, horizon 16, batch 1, 4 steps",
}

KCLASS_NAMES = {1: "qkv_gemm", 2: "attention", 3: "o_gemm", 4: "up_gemm", 5: "down_gemm", 6: "norm",
                7: "other"}


# ----------------------------------------------------------------------------
# algorithmic work
#
# Bytes are the step's unavoidable reads: every weight, the prefix / VL K/V and
# the modulation rows, each once per denoise step (activations excluded).
# FLOPs are 2 * rows * parameters of every projection plus 4 * rows * keys * Dh
# of the attention.
# ----------------------------------------------------------------------------

def kernel_work(g: dict, batch: int, prefix: int):
    """Per kernel class: (launches per denoise step, algorithmic bytes per launch,
    FLOPs per launch) -- bytes = the weights (+ FP8 row scales) a GEMM streams,
    the K/V an attention reads, the modulation rows a norm reads."""
    es = 2 if g["dtype"] == synth.DTYPE_BF16 else 4
    fp8 = g.get("weight_format", synth.WFMT_NATIVE) == synth.WFMT_FP8
    ws = 1 if fp8 else es            # bytes per element of the per-layer projections
    sc = 4 if fp8 else 0             # FP8: one fp32 scale per output row
    D, L, F, H = g["hidden"], g["layers"], g["mlp_dim"], g["horizon"]
    Hq, Dh = g["q_heads"], g["head_dim"]
    tok = H + g["state_tokens"]
    M = batch * tok
    qd = Hq * Dh
    dit = g["family"] == synth.FAMILY_DIT
    up_rows = synth.up_rows(g)
    R = synth.row_width(g)
    out = {}

    def add(name, n, by, fl):
        c, b0, f0 = out.get(name, (0, 0.0, 0.0))
        out[name] = (c + n, b0 + by * n, f0 + fl * n)

    for l in range(L):
        nq = synth.qkv_rows(g, l)
        add("qkv_gemm", 1, nq * (D * ws + sc), 2.0 * M * nq * D)
        add("o_gemm", 1, D * (qd * ws + sc), 2.0 * M * D * qd)
        add("up_gemm", 1, up_rows * (D * ws + sc), 2.0 * M * up_rows * D)
        add("down_gemm", 1, D * (F * ws + sc), 2.0 * M * D * F)
        if dit and l % 2 == 0:
            keys, kv = prefix, batch * prefix * g["kv_heads"] * Dh * 2 * es
        elif dit:
            keys, kv = tok, 0
        else:
            keys, kv = prefix + H, batch * prefix * Dh * 2 * es
        add("attention", 1, kv, 4.0 * batch * Hq * tok * keys * Dh)
    # norms: the modulation rows of the step (per sample)
    sites = synth.norm_sites(g)
    add("norm", sites, batch * R * es, 0.0)
    return {k: (n, b / n, f / n) for k, (n, b, f) in out.items()}


def step_work(g: dict, batch: int, prefix: int):
    """Algorithmic bytes and FLOPs of one denoise step: every weight the step reads
    (per-layer projections, action in/out projections, DiT encoder), the prefix /
    VL K/V and the step's modulation rows, once each."""
    es = 2 if g["dtype"] == synth.DTYPE_BF16 else 4
    w = kernel_work(g, batch, prefix)
    by = sum(n * b for n, b, f in w.values())
    fl = sum(n * f for n, b, f in w.values())
    D, A, H = g["hidden"], g["action_dim"], g["horizon"]
    if g["family"] == synth.FAMILY_DIT:
        extra_w = D * A + D * D + D * D + A * D        # W1, W2's action half, W3, W_out
        fl += 2.0 * batch * H * (D * A + 2 * D * D + A * D)
    else:
        extra_w = D * A + A * D                        # action_in_proj, action_out_proj
        fl += 2.0 * batch * H * 2 * D * A
    return by + extra_w * es, fl


def load_peaks():
    pk = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(pk):
        p = json.load(open(pk))
        return (p.get("hbm_gbs", 6800.0), p.get("bf16_tflops", 1900.0), p.get("bf16_tflops_sustained", 1700.0),
                "of measured")
    return 6800.0, 1900.0, 1700.0, "of fallback"


# DRAM traffic per launch of a kernel class from ncu captures (profiles/traffic.json,
# written with `python bench.py --record-traffic ...`): reported only while the
# sources of that class's kernels, hashed there, are unchanged.
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "traffic.json")
KERNEL_SOURCES = {
    "attention": ("attention_tc5.cu", "attention_dit.cu", "tc_ptx.cuh", "common.cuh", "launch.cuh"),
    "gemm": ("gemm_tc.cu", "gemm_tc_impl.cuh", "gemm_tc_pers.cu", "gemm_tc_spec.cu", "epilogue.cuh", "tc_ptx.cuh",
             "common.cuh", "launch.cuh"),
    "norm": ("norm.cu", "common.cuh", "launch.cuh"),
}


def source_group(kernel: str) -> str:
    return kernel if kernel in ("attention", "norm") else "gemm"


def source_digest(kernel: str = "attention"):
    import hashlib
    h = hashlib.sha1()
    csrc = os.path.join(ROOT, "flow_matching_vla_gb300", "csrc")
    for name in KERNEL_SOURCES[source_group(kernel)]:
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def measured_traffic(workload: str, kernel: str):
    """Per-launch DRAM bytes of ``kernel`` from the recorded capture, or None when none
    is recorded for this workload or the class's kernel sources changed since."""
    try:
        t = json.load(open(TRAFFIC_FILE))
    except (OSError, ValueError):
        return None
    src = t.get("sources")
    if not isinstance(src, dict) or src.get(kernel) != source_digest(kernel):
        return None
    return t.get("bytes_per_launch", {}).get(workload, {}).get(kernel)


def record_traffic(csv_path: str, workload: str, kernel: str, command: str):
    """Store the mean dram read+write bytes per captured launch of an ncu CSV
    (`--metrics dram__bytes_read.sum,dram__bytes_write.sum --csv`) for one kernel class."""
    import csv
    vals = {}
    with open(csv_path) as f:
        rows = [r for r in csv.reader(f) if len(r) >= 5]
    hdr = rows[0]
    i_id, i_name, i_val = hdr.index("ID"), hdr.index("Metric Name"), hdr.index("Metric Value")
    i_unit = hdr.index("Metric Unit")
    scale = {"byte": 1, "Kbyte": 1e3, "Mbyte": 1e6, "Gbyte": 1e9}
    for r in rows[1:]:
        if r[i_name] in ("dram__bytes_read.sum", "dram__bytes_write.sum"):
            v = float(r[i_val].replace(",", "")) * scale.get(r[i_unit], 1)
            vals[r[i_id]] = vals.get(r[i_id], 0.0) + v
    if not vals:
        raise SystemExit("no dram__bytes metrics in " + csv_path)
    try:
        t = json.load(open(TRAFFIC_FILE))
    except (OSError, ValueError):
        t = {}
    if not isinstance(t.get("sources"), dict):
        t = {"sources": {}, "bytes_per_launch": {}, "commands": {}}
    if t["sources"].get(kernel) != source_digest(kernel):
        # the class's kernels changed: its earlier numbers (every workload) are stale
        for w in t["bytes_per_launch"].values():
            w.pop(kernel, None)
        for w in t["commands"].values():
            w.pop(kernel, None)
        t["sources"][kernel] = source_digest(kernel)
    t["bytes_per_launch"].setdefault(workload, {})[kernel] = float(np.mean(list(vals.values())))
    t["commands"].setdefault(workload, {})[kernel] = command
    with open(TRAFFIC_FILE, "w") as f:
        json.dump(t, f, indent=1, sort_keys=True)
    print(json.dumps({"recorded": workload, "kernel": kernel, "launches": len(vals),
                      "bytes_per_launch": t["bytes_per_launch"][workload][kernel]}))


# ----------------------------------------------------------------------------
# clocks during the timed region
# ----------------------------------------------------------------------------

class Clocks:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int, period_ms: int = 50):
        self.dev = device_index
        self.period = period_ms
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.dev), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", str(self.period)], stdout=self.f,
                stderr=subprocess.DEVNULL)
            time.sleep(0.3)   # let the sampler come up before the timed region
        except Exception:
            self.proc = None

    def stop(self):
        if not self.proc:
            return None
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
                rows.append((float(p[1]), float(p[2]), float(p[3]), p[5:9]))
            except ValueError:
                continue
        os.unlink(self.path)
        if not rows:
            return None
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for *_, r in rows for i in range(4) if r[i].lower().startswith("active")})
        mx = max(r[1] for r in rows)
        # samples under load: power above the idle floor
        pw = [r[2] for r in rows]
        floor = min(pw)
        loaded = [r[0] for r in rows if r[2] > floor + 0.25 * (max(pw) - floor)] or [r[0] for r in rows]
        return {"sm_mhz": statistics.median(loaded), "sm_max_mhz": mx, "reasons": reasons,
                "samples": len(rows), "samples_under_load": len(loaded), "period_ms": self.period,
                "power_w_max": max(pw)}


# ----------------------------------------------------------------------------
# CPU oracle baseline (bounded sample)
# ----------------------------------------------------------------------------

def _host_cores():
    return len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()


def oracle_rate(case, budget_s: float = 15.0, max_evals: int | None = None):
    """Chunks/s of the fp64 CPU oracle, from whole velocity evaluations of one sample."""
    import oracle
    g = case["geom"]
    T = g["steps"]
    sub = dict(case)
    sub["x_noise"] = case["x_noise"][:1]
    sub["K"] = [None if k is None else k[:1] for k in case["K"]]
    sub["V"] = [None if v is None else v[:1] for v in case["V"]]
    for key in ("text_mask", "image_mask", "state", "state_raw", "features"):
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
        oracle.velocity(sub, x, k % T, steps=T, mod=mod, atb=atb)
        times.append(time.perf_counter() - t0)
        k += 1
        if time.perf_counter() > t_end or (max_evals and k >= max_evals):
            break
    t_step = float(np.mean(times))
    threads = int(os.environ.get("OPENBLAS_NUM_THREADS", "0") or 0) or _host_cores()
    return {"value": 1.0 / (T * t_step), "unit": UNIT, "cores": threads, "kind": "oracle",
            "machine": platform.machine(),
            "sample": f"{len(times)} velocity evaluation(s) of 1 sample (numpy fp64, "
                      f"{t_step:.3f} s each) scaled to a {T}-step chunk"}, t_step


def oracle_one_thread(workload: str, budget_s: float):
    """The oracle on one host thread (BLAS pinned to one thread in a child process)."""
    env = dict(os.environ, OMP_NUM_THREADS="1", OPENBLAS_NUM_THREADS="1", MKL_NUM_THREADS="1",
               BLIS_NUM_THREADS="1")
    code = ("import json, bench, synth; r, _ = bench.oracle_rate(synth.make_case(%r), budget_s=%r); "
            "r['cores'] = 1; print(json.dumps(r))" % (workload, budget_s))
    try:
        out = subprocess.run([sys.executable, "-c", code], env=env, cwd=ROOT, capture_output=True, text=True,
                             timeout=budget_s * 6 + 120)
        return json.loads(out.stdout.strip().splitlines()[-1])
    except Exception as e:  # reported, not fatal
        return {"error": str(e)[:200]}


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


def config_obj(args, g, world):
    return {"workload": WORKLOAD_TEXT.get(args.workload, args.workload), "name": args.workload,
            "batch": g["batch"], "prefix": g["prefix"], "horizon": g["horizon"],
            "denoise_steps": g["steps"], "parallelism": f"replicas x{world}",
            "l2": "inputs larger than L2 (weights + K/V read every denoise step exceed 129 MB); no flush"}


def run_reference(args, world, rank):
    if rank != 0:
        return 0
    case = synth.make_case(args.workload)
    g = case["geom"]
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
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": el * 1000 / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded)", "config": config_obj(args, g, args.gpus),
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": cb["cores"], "kind": "oracle",
                             "machine": platform.machine(),
                             "sample": f"each step: 1 velocity evaluation of 1 sample of the workload "
                                       f"(numpy fp64 oracle on the host cores), scaled to a "
                                       f"{g['steps']}-step chunk"},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


# ----------------------------------------------------------------------------
# GPU measurement of one workload
# ----------------------------------------------------------------------------

def time_denoise(loop, x, out, stream, n):
    import torch
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    t0.record(stream)
    for _ in range(n):
        loop.denoise(x, out)
    t1.record(stream)
    t1.synchronize()
    return t0.elapsed_time(t1) / n   # ms per denoise


def kernel_table(loop, fmv, x, out, stream, g, B, P, replays=3):
    """Per kernel class from launch stamps of ``replays`` graph replays: launches per
    denoise step, average in-chain microseconds per launch, share of the step."""
    import torch
    T = g["steps"]
    loop.set_option(fmv.OPT_TIME_KERNELS, 1)
    with torch.cuda.stream(stream):
        loop.denoise(x, out)              # capture with stamps
        sums, totals = {}, []
        for _ in range(replays):
            loop.denoise(x, out)
            us, cls = loop.kernel_times()
            totals.append(sum(us))
            for u, c in zip(us, cls):
                n, t = sums.get(c, (0, 0.0))
                sums[c] = (n + 1, t + u)
    loop.set_option(fmv.OPT_TIME_KERNELS, 0)
    work = kernel_work(g, B, P)
    table = {}
    total_us = float(np.mean(totals)) / T
    for c, (n, t) in sums.items():
        name = KCLASS_NAMES.get(c, str(c))
        launches = n / replays / T
        per_step = t / replays / T
        row = {"launches_per_step": launches, "us_per_step": per_step, "avg_us": per_step / launches,
               "share": per_step / total_us if total_us else None}
        if name in work:
            nw, by, fl = work[name]
            row.update(algorithmic_bytes=by, algorithmic_flops=fl, work_launches_per_step=nw)
        table[name] = row
    return table, total_us


def roofline_of(name, row, peaks, workload):
    hbm, tc_burst, tc_sust, src = peaks
    by, fl = row.get("algorithmic_bytes", 0.0), row.get("algorithmic_flops", 0.0)
    # per launch of the work unit (the attention's split merge is part of its launch)
    t = row["us_per_step"] / row.get("work_launches_per_step", row["launches_per_step"]) * 1e-6
    ridge = tc_burst * 1e12 / (hbm * 1e9)
    tensor = by == 0 or (fl / by) > ridge
    if tensor:
        achieved = fl / t / 1e12
        r = {"bound": "tensor", "achieved": achieved, "peak": tc_burst, "unit": "TFLOP/s",
             "frac": achieved / tc_burst, "frac_of_sustained_peak": achieved / tc_sust}
    else:
        achieved = by / t / 1e9
        r = {"bound": "hbm", "achieved": achieved, "peak": hbm, "unit": "GB/s", "frac": achieved / hbm}
    r.update({"kernel": name, "traffic": measured_traffic(workload, name), "peak_source": src,
              "peak_kind": "burst", "avg_launch_us": t * 1e6,
              "algorithmic_bytes_per_launch": by, "algorithmic_flops_per_launch": fl})
    return r


def measure_workload(fmv, name, args, stream, dev, world, peaks, e2e=True, sweep=False, timed=None):
    """Time one workload: denoise rate, per-kernel attribution, rooflines, e2e."""
    import torch
    case = synth.make_case(name)
    g = case["geom"]
    B, T, P = g["batch"], g["steps"], g["prefix"]
    kw = {"max_steps": 16} if sweep else {}
    loop, held = fmv.from_case(case, stream=stream, **kw)
    x = torch.from_numpy(case["x_noise"]).to(dev)
    out = torch.empty_like(x)
    res = {"name": name, "workload": WORKLOAD_TEXT.get(name, name)}
    n = timed or args.steps
    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            loop.denoise(x, out)
        stream.synchronize()
        kernels_per_step = loop.info(fmv.INFO_KERNELS_PER_STEP)
        ms = time_denoise(loop, x, out, stream, n)
    res.update(ms_per_denoise=ms, us_per_denoise_step=ms * 1000.0 / T, chunks_per_s=B / (ms / 1000.0),
               kernels_per_denoise_step=kernels_per_step, batch=B, denoise_steps=T)
    sb, sf = step_work(g, B, P)
    t_hbm, t_tc = sb / (peaks[0] * 1e9), sf / (peaks[1] * 1e12)
    t_min = max(t_hbm, t_tc)
    res["step_roofline"] = {"bytes_per_denoise_step": sb, "flops_per_denoise_step": sf,
                            "t_min_us": t_min * 1e6, "frac": t_min * 1e6 / res["us_per_denoise_step"],
                            "bound": "tensor" if t_tc > t_hbm else "hbm", "peak_source": peaks[3],
                            "peak_kind": "burst",
                            "bytes_are": "weights + prefix/VL K/V + modulation rows, once per step"}
    if not args.no_kernel_timing:
        table, stamped_us = kernel_table(loop, fmv, x, out, stream, g, B, P)
        res["kernels"] = table
        res["stamped_us_per_denoise_step"] = stamped_us
        cand = {k: v for k, v in table.items() if k not in ("norm", "other")}
        if cand:
            dom = max(cand, key=lambda k: cand[k]["us_per_step"])
            res["roofline"] = roofline_of(dom, cand[dom], peaks, name)
    if e2e:
        xh = torch.from_numpy(case["x_noise"]).pin_memory()
        oh = torch.empty_like(xh).pin_memory()
        for _ in range(max(1, args.warmup // 2)):
            loop.denoise_host(xh, oh)
        barrier(world)
        e0 = time.perf_counter()
        for _ in range(n):
            loop.denoise_host(xh, oh)
        e_el = max_over_ranks(time.perf_counter() - e0, world)
        res["e2e"] = {"value": B * n * world / e_el, "unit": UNIT, "h2d_bytes_per_step": int(xh.numel() * 4),
                      "d2h_bytes_per_step": int(oh.numel() * 4),
                      "api": "gr00t_denoise_host (pinned host noise in, chunk out, stream synchronised)"}
    if sweep:
        # per-step slope t(T) = P + T * E over T in {1, 2, 4, 8, 16} (vla.cpp Eq. (3))
        Ts, ts = [1, 2, 4, 8, 16], []
        with torch.cuda.stream(stream):
            for Tk in Ts:
                loop.set_schedule(Tk, B)
                for _ in range(3):
                    loop.denoise(x, out)
                ts.append(time_denoise(loop, x, out, stream, 5) * 1000.0)
            loop.set_schedule(T, B)
        slope, icpt = np.polyfit(np.array(Ts, float), np.array(ts), 1)
        res["step_sweep"] = {"steps": Ts, "us_per_denoise": ts, "fit_us_per_step": float(slope),
                             "fit_intercept_us": float(icpt)}
    loop.close()
    del held, x, out, loop
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    return res, case


def cond_reevaluation(fmv, stream, dev, peaks):
    """The hoisted cond on a step-count change for the long-prefix workload: the
    [80, 1024] x [1024, 37 * 3072] Dense (plus the time MLP), timed on its own."""
    import torch
    case = synth.make_case("pi05_long")
    g = case["geom"]
    loop, held = fmv.from_case(case, stream=stream)
    T, B = g["steps"], g["batch"]
    ev = []
    with torch.cuda.stream(stream):
        for i in range(12):
            loop.set_schedule(T - 1, B)           # a different count, so the next call re-evaluates
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            a.record(stream)
            loop.set_schedule(T, B)
            b.record(stream)
            b.synchronize()
            if i >= 2:
                ev.append(a.elapsed_time(b) * 1000.0)
    E, S, R, D = g["time_dim"], synth.norm_sites(g), synth.row_width(g), g["hidden"]
    rows = T * B
    by = (S * R * E + 2 * E * E) * 2 + rows * S * R * 2
    fl = 2.0 * rows * (S * R * E + 2 * E * E)
    us = float(np.median(ev))
    loop.close()
    del held, loop
    torch.cuda.empty_cache()
    return {"what": f"gr00t_set_schedule on a step-count change, pi05_long (T={T}, B={B}): time embedding, "
                    f"time MLP and the [{rows}, {E}] x [{E}, {S * R}] cond Dense",
            "us": us, "bytes": by, "flops": fl, "achieved_gbs": by / us * 1e-3,
            "frac_hbm": by / us * 1e-3 / peaks[0], "peak_source": peaks[3]}


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=40)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=HEADLINE, choices=sorted(synth.CONFIGS))
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--ref-seconds", type=float, default=120.0,
                    help="reference arm: upper bound on its total run time (each step is one oracle evaluation)")
    ap.add_argument("--no-kernel-timing", action="store_true")
    ap.add_argument("--no-extras", action="store_true", help="skip the other workloads, the sweep and the cond timing")
    ap.add_argument("--profile", action="store_true",
                    help="warm up, then run one denoise inside the NVTX range 'denoise' (for ncu) and exit")
    ap.add_argument("--record-traffic", nargs=3, metavar=("CSV", "WORKLOAD", "KERNEL"),
                    help="store the dram bytes per launch of an ncu CSV capture in profiles/traffic.json")
    ap.add_argument("--traffic-command", default="", help="the ncu command line recorded with --record-traffic")
    args = ap.parse_args(argv)
    if args.record_traffic:
        record_traffic(*args.record_traffic, command=args.traffic_command)
        return 0
    if args.warmup < 3 and args.impl == "ours":
        ap.error("--warmup must be >= 3")
    world, rank, local = dist_setup(args.impl)
    if args.impl == "reference":
        return run_reference(args, world, rank)

    import torch
    import flow_matching_vla_gb300 as fmv

    peaks = load_peaks()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    stream = torch.cuda.Stream(device=dev)

    if args.profile:
        case = synth.make_case(args.workload)
        loop, held = fmv.from_case(case, stream=stream)
        x = torch.from_numpy(case["x_noise"]).to(dev)
        out = torch.empty_like(x)
        with torch.cuda.stream(stream):
            for _ in range(args.warmup):
                loop.denoise(x, out)
            stream.synchronize()
            torch.cuda.nvtx.range_push("denoise")
            loop.denoise(x, out)
            stream.synchronize()
            torch.cuda.nvtx.range_pop()
        print(json.dumps({"profile": args.workload, "kernels_per_denoise_step": loop.info(fmv.INFO_KERNELS_PER_STEP),
                          "denoise_steps": case["geom"]["steps"]}), flush=True)
        return 0

    # ---- headline: K timed denoise calls, clocks sampled meanwhile ----
    case = synth.make_case(args.workload)
    g = case["geom"]
    B, T, P = g["batch"], g["steps"], g["prefix"]
    loop, held = fmv.from_case(case, stream=stream)
    x = torch.from_numpy(case["x_noise"]).to(dev)
    out = torch.empty_like(x)
    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            loop.denoise(x, out)
        stream.synchronize()
        kernels_per_step = loop.info(fmv.INFO_KERNELS_PER_STEP)
        barrier(world)
        clocks = Clocks(local)
        clocks.start()
        ms = time_denoise(loop, x, out, stream, args.steps) * args.steps
        torch.cuda.synchronize()
        clk = clocks.stop()
    loop.close()
    del held, loop, x, out
    torch.cuda.empty_cache()
    ms = max_over_ranks(ms, world)
    chunks = B * args.steps * world
    value = chunks / (ms / 1000.0)
    ms_per_step = ms / args.steps
    us_per_denoise_step = ms_per_step * 1000.0 / T

    # ---- the same workload again for attribution, e2e and the step sweep ----
    detail, _ = measure_workload(fmv, args.workload, args, stream, dev, world, peaks, e2e=True,
                                 sweep=not args.no_extras and world == 1)
    extras = {}
    cond = None
    if not args.no_extras and world == 1:
        for name in EXTRAS:
            if name == args.workload:
                continue
            r, _ = measure_workload(fmv, name, args, stream, dev, world, peaks, e2e=False, timed=10)
            extras[name] = {k: r[k] for k in ("workload", "us_per_denoise_step", "chunks_per_s", "step_roofline",
                                              "roofline", "kernels", "stamped_us_per_denoise_step",
                                              "kernels_per_denoise_step") if k in r}
        cond = cond_reevaluation(fmv, stream, dev, peaks)
    if rank != 0:
        return 0
    cpu = None
    cpu_1t = {}
    if not args.no_cpu_baseline and world == 1:
        cpu, _ = oracle_rate(case, budget_s=args.cpu_seconds)
        for name in ("tiny", "pi05"):
            cpu_1t[name] = oracle_one_thread(name, budget_s=min(8.0, args.cpu_seconds))
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "us_per_denoise_step": us_per_denoise_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16" if g["dtype"] == synth.DTYPE_BF16 else "f32",
        "data": "synthetic (seeded; weights ~N(0,0.02), K/V and noise ~N(0,1))",
        "config": config_obj(args, g, world),
        "roofline": detail.get("roofline"),
        "step_roofline": dict(detail["step_roofline"],
                              frac=detail["step_roofline"]["t_min_us"] / us_per_denoise_step),
        "kernels": detail.get("kernels"),
        "stamped_us_per_denoise_step": detail.get("stamped_us_per_denoise_step"),
        "step_sweep": detail.get("step_sweep"),
        "cond_reevaluation": cond,
        "extra_workloads": extras,
        "cpu_baseline": cpu,
        "cpu_baseline_one_thread": cpu_1t or None,
        "e2e": detail.get("e2e"),
        "gpu_launches": int(kernels_per_step * T * args.steps),
        "clocks": clk,
    }
    print(json.dumps(line), flush=True)
    return 0


if __name__ == "__main__":
    sys.exit(main())
