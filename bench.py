#!/usr/bin/env python3
"""Benchmark of the block-scaled FP8 hot path on one GB300 (or N replicas).

Default workload: the decode-shaped FP8 linear layer, X bf16 [8, 2048] ~ N(0, 1)
with 1% outlier channels x20, W e4m3 [10944, 2048] from N(0, 0.02) with
per-128x128 fp32 scales. One step = act_quant(X) then fp8_gemm (the
"Administrator & Developer Guide" 6.3 fp8 path of linear()), on inputs
resident in HBM. The metric is HBM throughput in GB/s of algorithmic bytes
(decode is HBM-bound); the GEMM-shaped workloads report TFLOP/s.

Timing: steps are captured in CUDA graphs (chunks of up to 100 steps) and the
timed region is the replay of exactly --steps steps between CUDA events on the
launching stream, with a device synchronise and a barrier on both sides. The
weights rotate over enough copies to exceed 3x the L2 size, so no step finds
its weight in L2. nvidia-smi samples clocks during the timed region.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

With --impl reference the CPU oracle is timed on the host cores on a bounded
sample of the same workload (there is no GPU reference implementation to run:
the pages hold no code).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import re
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import synthetic  # noqa: E402

# name -> (kind, shape dict). Shapes from the workload list: decode-shaped
# linear (M in 1, 8, 64), the 16x320x256 case, the prefill FFN GEMMs, the
# attention projections, weight_dequant of an [18432, 7168] weight.
WORKLOADS = {
    "decode_linear_m8": ("linear", dict(M=8, N=10944, K=2048, frac=0.01, seed=synthetic.SEED_DECODE)),
    "decode_linear_m1": ("linear", dict(M=1, N=10944, K=2048, frac=0.01, seed=synthetic.SEED_DECODE)),
    "decode_linear_m64": ("linear", dict(M=64, N=10944, K=2048, frac=0.01, seed=synthetic.SEED_DECODE)),
    "pr1_linear_16x320x256": ("linear", dict(M=16, N=320, K=256, frac=0.0, seed=synthetic.SEED_PR1)),
    "prefill_gemm_w1": ("linear", dict(M=4096, N=18432, K=7168, frac=0.0, seed=synthetic.SEED_PREFILL)),
    "prefill_gemm_w2": ("linear", dict(M=4096, N=7168, K=18432, frac=0.0, seed=synthetic.SEED_PREFILL)),
    # power-of-two (UE8M0) scales on activations and weights: the tensor core applies them
    "prefill_gemm_w1_ue8m0": ("linear", dict(M=4096, N=18432, K=7168, frac=0.0, seed=synthetic.SEED_PREFILL, fmt=1)),
    "prefill_gemm_w2_ue8m0": ("linear", dict(M=4096, N=7168, K=18432, frac=0.0, seed=synthetic.SEED_PREFILL, fmt=1)),
    "attn_wq_b_m2048": ("linear", dict(M=2048, N=24576, K=1536, frac=0.0, seed=synthetic.SEED_ATTN)),
    "attn_wkv_b_m2048": ("linear", dict(M=2048, N=32768, K=512, frac=0.0, seed=synthetic.SEED_ATTN)),
    "attn_wq_a_m2048": ("linear", dict(M=2048, N=1536, K=7168, frac=0.0, seed=synthetic.SEED_ATTN)),
    "attn_wkv_a_m2048": ("linear", dict(M=2048, N=576, K=7168, frac=0.0, seed=synthetic.SEED_ATTN)),
    "attn_wq_b_m64": ("linear", dict(M=64, N=24576, K=1536, frac=0.0, seed=synthetic.SEED_ATTN)),
    "attn_wkv_b_m64": ("linear", dict(M=64, N=32768, K=512, frac=0.0, seed=synthetic.SEED_ATTN)),
    "attn_wq_a_m64": ("linear", dict(M=64, N=1536, K=7168, frac=0.0, seed=synthetic.SEED_ATTN)),
    "attn_wkv_a_m64": ("linear", dict(M=64, N=576, K=7168, frac=0.0, seed=synthetic.SEED_ATTN)),
    "weight_dequant_18432x7168": ("dequant", dict(N=18432, K=7168, seed=synthetic.SEED_ATTN)),
    "prefill_ffn_4096": ("ffn", dict(M=4096, dim=7168, inter=18432, seed=synthetic.SEED_PREFILL)),
    "prefill_ffn_4096_ue8m0": ("ffn", dict(M=4096, dim=7168, inter=18432, seed=synthetic.SEED_PREFILL, fmt=1)),
    "moe_t4096_uniform": ("moe", dict(T=4096, E=256, dim=7168, inter=2048, k=8, zipf=0.0, seed=synthetic.SEED_MOE)),
    "moe_t4096_uniform_ue8m0": ("moe", dict(T=4096, E=256, dim=7168, inter=2048, k=8, zipf=0.0, fmt=1,
                                            seed=synthetic.SEED_MOE)),
    "moe_t4096_zipf": ("moe", dict(T=4096, E=256, dim=7168, inter=2048, k=8, zipf=1.2, seed=synthetic.SEED_MOE)),
    "moe_t4096_uniform_shared": ("moe", dict(T=4096, E=256, dim=7168, inter=2048, k=8, zipf=0.0, shared=1,
                                             seed=synthetic.SEED_MOE)),
    # The same expert shapes and rows per expert (128) with 32 experts: a
    # 1.4 GB step small enough for a full ncu capture of the grouped GEMMs.
    "moe_t512_e32_uniform": ("moe", dict(T=512, E=32, dim=7168, inter=2048, k=8, zipf=0.0, seed=synthetic.SEED_MOE)),
    "mla_absorb_m64": ("mla", dict(T=64, H=128, C=512, seed=synthetic.SEED_ATTN)),
    "mla_absorb_m2048": ("mla", dict(T=2048, H=128, C=512, seed=synthetic.SEED_ATTN)),
    "moe_gate_t4096_e256": ("gate", dict(T=4096, E=256, groups=8, kept=4, k=8, route_scale=2.5,
                                         seed=synthetic.SEED_GATE)),
}
DEFAULT = "decode_linear_m8"
FP8_OVER_BF16 = 2.0   # nominal dense fp8 / bf16 tensor rate (4.5 / 2.25 PFLOP/s)


def parse():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=None)
    ap.add_argument("--warmup", type=int, default=None)
    ap.add_argument("--workload", default=DEFAULT, choices=sorted(WORKLOADS))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true", help="skip the oracle timing leg")
    ap.add_argument("--no-e2e", action="store_true", help="skip the host-buffer end-to-end leg")
    ap.add_argument("--no-soak", action="store_true",
                    help="no untimed replays before the timed region (for profilers; clocks then cover it alone)")
    ap.add_argument("--no-other", action="store_true",
                    help="skip the other_workloads key (prefill GEMM and MoE step, fp32 and UE8M0 scales)")
    ap.add_argument("--eager", action="store_true",
                    help="launch every step from the host instead of replaying CUDA graphs (for profilers)")
    return ap.parse_args()


# ---------------------------------------------------------------------------
# algorithmic work
# ---------------------------------------------------------------------------

def linear_bytes(M, N, K):
    """Bytes the FP8 linear layer must move, whatever the kernels: read x
    (bf16), the e4m3 weight and its 128x128 scales, write y (bf16)."""
    kb = K // 128
    nb = -(-N // 128)
    return M * K * 2 + N * K + nb * kb * 4 + M * N * 2


def gemm_kernel_bytes(M, N, K):
    """Bytes of the stand-alone fp8_gemm kernel: the quantised activation and
    its scales, the weight and its scales, the bf16 output."""
    kb = K // 128
    nb = -(-N // 128)
    return M * K + M * kb * 4 + N * K + nb * kb * 4 + M * N * 2


def linear_flops(M, N, K):
    return 2.0 * M * N * K


def dequant_bytes(N, K):
    return N * K + (-(-N // 128)) * (-(-K // 128)) * 4 + N * K * 2


# ---------------------------------------------------------------------------
# environment: peaks, clocks, ranks
# ---------------------------------------------------------------------------

def tensor_peak(peaks):
    """The FP8 dense peak a tensor-bound kernel is held to: the sustained bf16
    rate x the nominal fp8/bf16 ratio when the kernel is timed after the soak
    (seconds of load, the regime of a long run, under the power cap), the burst
    rate otherwise. Returns (peak, its description, the burst peak)."""
    burst = peaks["bf16"] * FP8_OVER_BF16
    if _SOAK[0] > 0:
        return (peaks["bf16_sus"] * FP8_OVER_BF16,
                f"bf16_tflops_sustained ({peaks['src']}) x {FP8_OVER_BF16} nominal fp8/bf16 ratio: timed after "
                f"{_SOAK[0]:.0f} s of load", burst)
    return burst, f"bf16_tflops ({peaks['src']}) x {FP8_OVER_BF16} nominal fp8/bf16 ratio", burst


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return dict(hbm=float(d["hbm_gbs"]), bf16=float(d["bf16_tflops"]),
                    bf16_sus=float(d.get("bf16_tflops_sustained", d["bf16_tflops"])), src="measured")
    return dict(hbm=6800.0, bf16=1900.0, bf16_sus=1700.0, src="fallback")


class ClockSampler:
    """nvidia-smi clocks and throttle reasons, sampled while running."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int, period_ms: int = 50):
        self.cmd = ["nvidia-smi", f"--id={gpu_index}", f"--query-gpu={self.FIELDS}",
                    "--format=csv,noheader,nounits", f"-lms={period_ms}"]
        self.lines = []
        self.proc = None
        self.t = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(self.cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except OSError:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def __exit__(self, *exc):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.t.join(timeout=2)

    def summary(self, t0=None, t1=None):
        rows = [ln for (t, ln) in self.lines if (t0 is None or t >= t0) and (t1 is None or t <= t1)]
        if not rows:
            rows = [ln for (_, ln) in self.lines]
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in rows:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
            except ValueError:
                continue
            for name, v in zip(names, parts[4:8]):
                if v.lower() == "active":
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    return ws, int(os.environ.get("RANK", "0")), int(os.environ.get("LOCAL_RANK", "0"))


def reduce_over_ranks(elapsed_s: float, units: float, device=None):
    """(max elapsed over ranks, sum of units over ranks). With one process it
    returns its arguments; under torch.distributed it all-reduces."""
    import torch
    import torch.distributed as dist

    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return elapsed_s, units
    t = torch.tensor([elapsed_s], dtype=torch.float64, device=device)
    u = torch.tensor([units], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    dist.all_reduce(u, op=dist.ReduceOp.SUM)
    return float(t.item()), float(u.item())


def barrier():
    import torch.distributed as dist

    if dist.is_available() and dist.is_initialized():
        dist.barrier()


# ---------------------------------------------------------------------------
# traffic figures recorded from ncu captures, valid only for unchanged sources
# ---------------------------------------------------------------------------

_COMMENT = re.compile(r"//[^\n]*|/\*.*?\*/", re.S)


# The library sources whose code makes up each recorded kernel: the kernel,
# the device helpers it includes and the host code that plans its launch.
# None: every source (a workload of several kernels).
KERNEL_SOURCES = {
    "fp8_gemm": ("gemm.cu", "gemm_decode.cu", "ptx.cuh", "quotient.cuh", "host.cuh"),
    "swiglu_gemm": ("gemm.cu", "ptx.cuh", "quotient.cuh", "host.cuh"),
    "linear_fused": ("api.cu", "gemm.cu", "gemm_decode.cu", "ptx.cuh", "quotient.cuh", "host.cuh"),
    "weight_dequant": ("quant.cu", "ptx.cuh", "quotient.cuh", "host.cuh"),
    "mla": ("mla.cu", "ptx.cuh", "host.cuh"),
    "moe_step": None,
}


def kernel_source_digest(kernel: str | None = None) -> str:
    """Digest of the code of the sources that make up `kernel` (all sources if
    None): comments and whitespace removed, so an edit to a comment keeps a
    profile's traffic record valid and any change to that code invalidates it.
    (A string literal holding "//" would lose its tail here; the sources have
    none that matters to the digest.)"""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "fp8_block_scaled_quant_gb300", "csrc")
    files = KERNEL_SOURCES.get(kernel) if kernel else None
    for name in sorted(os.listdir(csrc)):
        if not name.endswith((".cu", ".cuh", ".h")) or (files is not None and name not in files):
            continue
        with open(os.path.join(csrc, name), encoding="utf-8") as f:
            code = "".join(_COMMENT.sub(" ", f.read()).split())
        h.update(name.encode() + code.encode())
    return h.hexdigest()[:16]


def recorded_traffic(workload: str, kernel: str):
    """DRAM bytes per launch that an ncu capture of this workload recorded in
    profiles/traffic.json, if the kernel's sources are unchanged since (else None)."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        records = json.load(f).get("records", [])
    digest = kernel_source_digest(kernel)
    for r in records:
        if r.get("workload") == workload and r.get("kernel") == kernel and r.get("sources") == digest:
            return int(r["bytes_per_launch"])
    return None


# ---------------------------------------------------------------------------
# our arm
# ---------------------------------------------------------------------------

def graph_chunks(fn_step, n_steps, chunk, torch):
    """CUDA graphs that run fn_step(i) for i in [0, n_steps), up to `chunk` per graph."""
    graphs = []
    i = 0
    while i < n_steps:
        n = min(chunk, n_steps - i)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            for j in range(i, i + n):
                fn_step(j)
        graphs.append(g)
        i += n
    return graphs


class Eager:
    """Stands in for a captured graph: replay() runs the steps from the host."""

    def __init__(self, fn_step, begin, n):
        self.fn, self.begin, self.n = fn_step, begin, n

    def replay(self):
        for j in range(self.begin, self.begin + self.n):
            self.fn(j)


def make_runs(fn_step, n_steps, chunk, torch, eager):
    if eager:
        return [Eager(fn_step, i, min(chunk, n_steps - i)) for i in range(0, n_steps, chunk)]
    return graph_chunks(fn_step, n_steps, chunk, torch)


def upload_graphs(graphs, stream, torch) -> bool:
    """Upload captured graphs to the device before they are timed, so that a
    graph's first replay does not pay for its upload inside the timed region
    (cuGraphUpload through the driver; False where it is not available)."""
    import ctypes

    try:
        upload = ctypes.CDLL("libcuda.so.1").cuGraphUpload
    except (OSError, AttributeError):
        return False
    upload.argtypes = [ctypes.c_void_p, ctypes.c_void_p]
    upload.restype = ctypes.c_int
    ok = True
    for g in graphs:
        if not hasattr(g, "raw_cuda_graph_exec"):
            return False
        ok = upload(ctypes.c_void_p(g.raw_cuda_graph_exec()), ctypes.c_void_p(stream.cuda_stream)) == 0 and ok
    torch.cuda.synchronize()
    return ok


SOAK_S = 2.0   # untimed replays right before each timed region, so clock samplers see the GPU under load
_SOAK = [SOAK_S]   # set to 0 by --no-soak


def timed_runs(dev, stream, torch, main, extras=(), soak=None, soak_s=None):
    """Times `main` (graphs of exactly the --steps steps) and then each list of
    graphs in `extras` (kernel-only passes), with nvidia-smi sampling clocks.
    Before the timed region the `soak` graphs are replayed for soak_s seconds
    (untimed), so that the clocks sampled -- by this process and by anyone
    watching the GPU -- are those of the GPU under this load. Returns
    (elapsed of main, [elapsed of each extra], clock summary over soak + main,
    whether the graphs were uploaded before timing)."""
    if soak_s is None:
        soak_s = _SOAK[0]
    if soak_s <= 0:
        soak = None
    graphs = list(main) + [g for e in extras for g in e] + list(soak or [])
    uploaded = upload_graphs(graphs, stream, torch)
    with ClockSampler(dev.index) as clk:
        time.sleep(0.3)
        ts = time.time()
        if soak:
            while time.time() - ts < soak_s:
                for g in soak:
                    g.replay()
                torch.cuda.synchronize()
        el, t0, t1 = timed_replay(main, stream, torch)
        els = [timed_replay(e, stream, torch)[0] for e in extras]
    clocks = clk.summary(ts, t1)
    clocks["window"] = f"{soak_s if soak else 0:.1f} s of untimed replays of the step, then the timed region"
    return el, els, clocks, uploaded


def timed_replay(graphs, stream, torch):
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    barrier()
    t0 = time.time()
    start.record(stream)
    for g in graphs:
        g.replay()
    end.record(stream)
    torch.cuda.synchronize()
    t1 = time.time()
    barrier()
    return start.elapsed_time(end) / 1e3, t0, t1


def run_linear(args, shape, dev, torch, fb, peaks, steps, warmup, rank, world):
    M, N, K, frac, seed = shape["M"], shape["N"], shape["K"], shape["frac"], shape["seed"]
    fmt = shape.get("fmt", 0)
    props = torch.cuda.get_device_properties(dev)
    l2 = int(getattr(props, "L2_cache_size", 0) or 132 * 2 ** 20)
    w_bytes = N * K
    R = max(2, math.ceil(3 * l2 / w_bytes))
    R = min(R, 64)
    w = synthetic.device_normal((N, K), seed + 1, 0.02, dev)
    q0, s0 = fb.weight_quant(w, fmt)
    del w
    qs = [q0] + [q0.clone() for _ in range(R - 1)]
    ss = [s0] + [s0.clone() for _ in range(R - 1)]
    xs = [synthetic.device_activations(M, K, seed + i, dev, outlier_frac=frac) for i in range(R)]
    ys = [torch.empty((M, N), dtype=torch.bfloat16, device=dev) for _ in range(R)]
    aqs = [fb.act_quant(x, fmt) for x in xs]   # for the GEMM-only pass
    ws = fb.workspace(fb.linear_workspace_bytes(M, N, K), dev, "bench")
    gws = fb.workspace(fb.gemm_workspace_bytes(M, N, K), dev, "bench_gemm")
    aq_buf = [(torch.empty((M, K), dtype=torch.float8_e4m3fn, device=dev),
               torch.empty((M, K // 128), dtype=torch.float32, device=dev)) for _ in range(R)]

    def step(i):
        r = i % R
        fb.linear(xs[r], qs[r], ss[r], scale_fmt=fmt, out=ys[r], ws=ws)

    def gemm_only(i):
        r = i % R
        fb.fp8_gemm(aqs[r][0], aqs[r][1], qs[r], ss[r], scale_fmt=fmt, out=ys[r], ws=gws)

    def aq_only(i):
        r = i % R
        fb.act_quant(xs[r], fmt, q=aq_buf[r][0], s=aq_buf[r][1])

    for i in range(3):   # eager warm-up: sets kernel attributes, loads modules
        step(i)
        gemm_only(i)
        aq_only(i)
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream(dev)
    chunk = 100
    g_warm = make_runs(step, warmup, chunk, torch, args.eager)
    g_main = make_runs(step, steps, chunk, torch, args.eager)
    g_gemm = make_runs(gemm_only, steps, chunk, torch, args.eager)
    g_aq = make_runs(aq_only, steps, chunk, torch, args.eager)
    g_soak = make_runs(step, chunk, chunk, torch, args.eager)
    for g in g_warm:
        g.replay()
    torch.cuda.synchronize()

    el, (el_gemm, el_aq), clocks, uploaded = timed_runs(dev, stream, torch, g_main, (g_gemm, g_aq), g_soak)
    assert fb.last_device_error(dev) == 0, "a kernel reported a wait timeout"

    # One kernel where the library fuses act_quant into the GEMM (M <= 2 on
    # shapes the decode GEMM does not take); otherwise act_quant then fp8_gemm.
    fused = fb.linear_kernels(M, N, K) == 1
    step_bytes = linear_bytes(M, N, K)
    gemm_b = gemm_kernel_bytes(M, N, K)
    flops = linear_flops(M, N, K)
    el_max, units = reduce_over_ranks(el, steps * step_bytes, dev)
    hbm_bound = flops / step_bytes < 400
    gemm_s = el_gemm / steps
    kern_s, kern_b = (el / steps, step_bytes) if fused else (gemm_s, gemm_b)
    kern_name = "fp8blk_linear (act_quant fused into the GEMM)" if fused else "fp8_gemm"
    if fmt and not fused and M > 128:
        kern_name += " (UE8M0 scales applied by the tensor core)"
    if hbm_bound:
        metric_val = units / el_max / 1e9
        unit = "GB/s"
        achieved = kern_b / kern_s / 1e9
        roof = {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm"], "unit": "GB/s",
                "frac": achieved / peaks["hbm"], "peak_source": f"hbm_gbs ({peaks['src']})"}
    else:
        metric_val = steps * flops * world / el_max / 1e12
        unit = "TFLOP/s"
        peak, peak_src, burst = tensor_peak(peaks)
        achieved = flops / kern_s / 1e12
        roof = {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                "frac": achieved / peak, "peak_source": peak_src, "frac_of_burst_peak": achieved / burst}
    roof["kernel"] = kern_name
    roof["traffic"] = recorded_traffic(args.workload, "linear_fused" if fused else "fp8_gemm")
    roof["algorithmic_bytes_per_launch"] = kern_b
    roof["kernel_us"] = kern_s * 1e6

    e2e = None
    if not args.no_e2e:
        e2e = run_e2e(shape, dev, torch, fb, qs, ss, min(steps, 20000), hbm_bound, step_bytes, flops)

    out = {
        "value": metric_val, "unit": unit, "ms_per_step": el_max / steps * 1e3,
        "clocks": clocks, "roofline": roof, "e2e": e2e,
        "gpu_launches": (1 if fused else 2) * steps,
        "kernels_us": {"linear_step": el / steps * 1e6, "act_quant_alone": el_aq / steps * 1e6,
                       "fp8_gemm_alone": gemm_s * 1e6},
        "config": {"workload": args.workload, "M": M, "N": N, "K": K, "outlier_channels": frac,
                   "x": "bf16 N(0,1)",
                   "w": "e4m3 from N(0,0.02), " + ("power-of-two (UE8M0)" if fmt else "fp32") + " 128x128 block scales",
                   "scale_fmt": "ue8m0" if fmt else "fp32",
                   "l2": f"weights rotate over {R} copies ({R * w_bytes / 1e6:.0f} MB > 3x L2 {l2 / 1e6:.0f} MB)",
                   "launch": "host loop" if args.eager else
                   f"CUDA graphs of up to {chunk} steps" + (", uploaded before timing" if uploaded else "")},
        "dtype": "e4m3 x e4m3 -> f32 accumulate, bf16 out",
    }
    return out


def run_e2e(shape, dev, torch, fb, qs, ss, n, hbm_bound, step_bytes, flops):
    """End to end through fp8blk_linear_host on pinned host buffers: each step's
    X comes from host memory and its Y lands in host memory (the layer's
    kernels read and write the pinned buffers over the chip-to-chip link);
    timed on the stream and by the wall clock (the larger counts). The weight
    rotates over the same copies as the device-timed leg, so no step finds its
    weight in L2."""
    M, N, K = shape["M"], shape["N"], shape["K"]
    fmt = shape.get("fmt", 0)
    xh = [synthetic.device_activations(M, K, shape["seed"] + 7 + i, dev, shape["frac"]).cpu().pin_memory()
          for i in range(4)]
    yh = [torch.empty((M, N), dtype=torch.bfloat16).pin_memory() for _ in range(4)]
    ws = fb.workspace(fb.linear_host_workspace_bytes(M, N, K), dev, "bench_e2e")
    R = len(qs)
    for i in range(3):
        fb.linear_host(xh[i % 4], qs[i % R], ss[i % R], yh[i % 4], scale_fmt=fmt, ws=ws)
    stream = torch.cuda.current_stream(dev)
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    barrier()
    t0 = time.time()
    start.record(stream)
    for i in range(n):
        fb.linear_host(xh[i % 4], qs[i % R], ss[i % R], yh[i % 4], scale_fmt=fmt, ws=ws)
    end.record(stream)
    torch.cuda.synchronize()
    wall = time.time() - t0
    el = max(start.elapsed_time(end) / 1e3, wall)
    el, units = reduce_over_ranks(el, n * (step_bytes if hbm_bound else flops), dev)
    val = units / el / (1e9 if hbm_bound else 1e12)
    return {"value": val, "unit": "GB/s" if hbm_bound else "TFLOP/s", "h2d_bytes_per_step": M * K * 2,
            "d2h_bytes_per_step": M * N * 2, "steps": n, "ms_per_step": el / n * 1e3,
            "api": "fp8blk_linear_host (pinned host buffers)", "weights": f"rotating over {R} copies"}


def run_ffn(args, shape, dev, torch, fb, peaks, steps, warmup, rank, world):
    """Dense SwiGLU FFN: act_quant(x), the fused w1/w3 GEMM (SwiGLU + act_quant
    epilogue), the w2 GEMM. Tensor-bound: 3 * 2 * M * dim * inter flops."""
    M, dim, inter, seed = shape["M"], shape["dim"], shape["inter"], shape["seed"]
    fmt = shape.get("fmt", 0)
    x = synthetic.device_activations(M, dim, seed, dev)
    sets = []
    for c in range(2):   # two weight copies: 792 MB > 3x L2 between consecutive steps
        ws_ = [synthetic.device_normal(sh, seed + 10 + i, 0.02, dev) for i, sh in
               enumerate([(inter, dim), (inter, dim), (dim, inter)])]
        sets.append([fb.weight_quant(w, fmt) for w in ws_])
        del ws_
    y = torch.empty((M, dim), dtype=torch.bfloat16, device=dev)
    xq, xs = fb.act_quant(x, fmt)
    wsp = fb.workspace(0, dev, "ffn")

    def step(i):
        (q1, s1), (q3, s3), (q2, s2) = sets[i % 2]
        fb.ffn(x, q1, s1, q3, s3, q2, s2, scale_fmt=fmt, out=y)

    def swiglu_only(i):
        (q1, s1), (q3, s3), _ = sets[i % 2]
        fb.swiglu_gemm(xq, xs, q1, s1, q3, s3, scale_fmt=fmt)

    for i in range(3):
        step(i)
        swiglu_only(i)
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream(dev)
    g_warm = make_runs(step, warmup, 10, torch, args.eager)
    g_main = make_runs(step, steps, 10, torch, args.eager)
    g_swi = make_runs(swiglu_only, steps, 10, torch, args.eager)
    g_soak = make_runs(step, 10, 10, torch, args.eager)
    for g in g_warm:
        g.replay()
    el, (el_swi,), clocks, _ = timed_runs(dev, stream, torch, g_main, (g_swi,), g_soak)
    assert fb.last_device_error(dev) == 0
    flops = 3 * 2.0 * M * dim * inter
    el_max, units = reduce_over_ranks(el, steps * flops, dev)
    peak, peak_src, burst = tensor_peak(peaks)
    swi_flops = 2 * 2.0 * M * dim * inter
    achieved = swi_flops / (el_swi / steps) / 1e12
    del wsp
    return {
        "value": units / el_max / 1e12, "unit": "TFLOP/s", "ms_per_step": el_max / steps * 1e3,
        "clocks": clocks, "gpu_launches": 3 * steps,
        "roofline": {"bound": "tensor", "kernel": "fused w1/w3 GEMM + SwiGLU + act_quant", "achieved": achieved,
                     "peak": peak, "unit": "TFLOP/s", "frac": achieved / peak, "frac_of_burst_peak": achieved / burst,
                     "traffic": recorded_traffic(args.workload, "swiglu_gemm"),
                     "peak_source": peak_src,
                     "kernel_us": el_swi / steps * 1e6},
        "e2e": None, "kernels_us": {"swiglu_gemm": el_swi / steps * 1e6},
        "config": {"workload": args.workload, "M": M, "dim": dim, "inter": inter,
                   "scale_fmt": "ue8m0" if fmt else "fp32",
                   "l2": "two weight sets (792 MB) alternate between steps"},
        "dtype": "e4m3 x e4m3 -> f32 accumulate; SwiGLU in fp32/bf16; e4m3 re-quantisation",
    }


def moe_weight_bytes(E_touched, dim, inter):
    kbd, kbi = dim // 128, inter // 128
    return E_touched * (2 * inter * dim + dim * inter + 4 * (2 * (inter // 128) * kbd + (dim // 128) * kbi))


def run_moe(args, shape, dev, torch, fb, peaks, steps, warmup, rank, world):
    """Routed experts: permutation, gather, grouped w1/w3 GEMM with the SwiGLU
    + act_quant epilogue, grouped w2 GEMM scattered to slots, weighted combine.
    HBM-bound on the touched experts' weights at this token count."""
    T, E, dim, inter, k, seed = (shape[n] for n in ("T", "E", "dim", "inter", "k", "seed"))
    ns = shape.get("shared", 0)
    fmt = shape.get("fmt", 0)
    x = synthetic.device_activations(T, dim, seed, dev)
    xq, xs = fb.act_quant(x, fmt)
    idx_np, w_np = synthetic.moe_routing(T, E, k, seed, zipf_s=shape["zipf"])
    idx = torch.from_numpy(idx_np).to(dev)
    wts = torch.from_numpy(w_np).to(dev)
    stacks = []
    for which in range(3):
        sh = (inter, dim) if which < 2 else (dim, inter)
        qs, ss = zip(*[fb.weight_quant(synthetic.device_normal(sh, seed * 100000 + 3 * e + which, 0.02, dev), fmt)
                       for e in range(E + ns)])
        stacks.append((torch.cat(qs), torch.cat(ss)))
        del qs, ss
    y = torch.empty((T, dim), dtype=torch.bfloat16, device=dev)
    (q1, s1), (q3, s3), (q2, s2) = stacks

    def step(i):
        fb.moe_grouped_gemm(xq, xs, idx, wts, q1, s1, q3, s3, q2, s2, E, scale_fmt=fmt, out=y, n_shared=ns)

    for i in range(3):
        step(i)
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream(dev)
    g_warm = make_runs(step, warmup, 10, torch, args.eager)
    g_main = make_runs(step, steps, 10, torch, args.eager)
    g_soak = make_runs(step, 10, 10, torch, args.eager)
    for g in g_warm:
        g.replay()
    el, _, clocks, _ = timed_runs(dev, stream, torch, g_main, (), g_soak)
    assert fb.last_device_error(dev) == 0
    touched = int(np.unique(idx_np).size) + ns
    b = moe_weight_bytes(touched, dim, inter) + T * dim + T * (dim // 128) * 4 + T * dim * 2 + T * k * 8
    flops = 3 * 2.0 * T * (k + ns) * dim * inter
    el_max, units = reduce_over_ranks(el, steps * b, dev)
    achieved = b / (el / steps) / 1e9
    return {
        "value": units / el_max / 1e9, "unit": "GB/s", "ms_per_step": el_max / steps * 1e3,
        "tflops": steps * flops / el / 1e12,
        "clocks": clocks, "gpu_launches": (7 + (1 if ns else 0)) * steps,
        "roofline": {"bound": "hbm", "kernel": f"whole routed-expert step ({7 + (1 if ns else 0)} kernels)",
                     "achieved": achieved,
                     "peak": peaks["hbm"], "unit": "GB/s", "frac": achieved / peaks["hbm"],
                     "traffic": recorded_traffic(args.workload, "moe_step"),
                     "peak_source": f"hbm_gbs ({peaks['src']})", "algorithmic_bytes_per_launch": b},
        "e2e": None,
        "config": {"workload": args.workload, "T": T, "E": E, "dim": dim, "inter": inter, "topk": k,
                   "routing": "Zipf(1.2)" if shape["zipf"] else "uniform", "shared_experts": ns,
                   "scale_fmt": "ue8m0" if fmt else "fp32",
                   "experts_touched": touched,
                   "l2": f"{touched} experts' weights ({moe_weight_bytes(touched, dim, inter) / 1e9:.2f} GB) per step"},
        "dtype": "e4m3 x e4m3 -> f32 accumulate; SwiGLU in fp32/bf16; e4m3 re-quantisation",
    }


def run_dequant(args, shape, dev, torch, fb, peaks, steps, warmup, rank, world):
    N, K, seed = shape["N"], shape["K"], shape["seed"]
    w = synthetic.device_normal((N, K), seed, 0.02, dev)
    q, s = fb.weight_quant(w)
    del w
    outs = [torch.empty((N, K), dtype=torch.bfloat16, device=dev) for _ in range(2)]
    qs = [q, q.clone()]

    def step(i):
        fb.weight_dequant(qs[i % 2], s, out=outs[i % 2])

    for i in range(3):
        step(i)
    stream = torch.cuda.current_stream(dev)
    g_warm = make_runs(step, warmup, 20, torch, args.eager)
    g_main = make_runs(step, steps, 20, torch, args.eager)
    g_soak = make_runs(step, 20, 20, torch, args.eager)
    for g in g_warm:
        g.replay()
    el, _, clocks, _ = timed_runs(dev, stream, torch, g_main, (), g_soak)
    b = dequant_bytes(N, K)
    el_max, units = reduce_over_ranks(el, steps * b, dev)
    achieved = b / (el / steps) / 1e9
    return {
        "value": units / el_max / 1e9, "unit": "GB/s", "ms_per_step": el_max / steps * 1e3,
        "clocks": clocks, "gpu_launches": steps,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm"], "unit": "GB/s",
                     "frac": achieved / peaks["hbm"], "traffic": recorded_traffic(args.workload, "weight_dequant"),
                     "peak_source": f"hbm_gbs ({peaks['src']})", "algorithmic_bytes_per_launch": b},
        "e2e": None,
        "config": {"workload": args.workload, "N": N, "K": K,
                   "l2": "two alternating inputs/outputs of 396 MB each (> L2)"},
        "dtype": "e4m3 -> f32 multiply -> bf16",
    }


def run_mla(args, shape, dev, torch, fb, peaks, steps, warmup, rank, world):
    """The two MLA absorb projections of one layer (q_nope through wkv_b's
    no-positional rows, the attention output through its v rows) with the FP8
    wkv_b of the 671B config (128 heads, kv_lora 512): bf16 tensor-core
    products of the dequantised weight."""
    T, H, C, seed = shape["T"], shape["H"], shape["C"], shape["seed"]
    dn = dv = 128
    props = torch.cuda.get_device_properties(dev)
    l2 = int(getattr(props, "L2_cache_size", 0) or 132 * 2 ** 20)
    w_bytes = H * (dn + dv) * C
    R = min(64, max(2, math.ceil(3 * l2 / w_bytes)))
    w0, s0 = fb.weight_quant(synthetic.device_normal((H * (dn + dv), C), seed + 7, 0.02, dev))
    qs = [w0] + [w0.clone() for _ in range(R - 1)]
    q = synthetic.device_activations(T, H * dn, seed + 8, dev).view(T, H, dn)
    x = synthetic.device_activations(T, H * C, seed + 9, dev).view(T, H, C)
    oq = torch.empty((T, H, C), dtype=torch.bfloat16, device=dev)
    ov = torch.empty((T, H, dv), dtype=torch.bfloat16, device=dev)

    def step(i):
        fb.mla_absorb(q, qs[i % R], s0, "qk", out=oq)
        fb.mla_absorb(x, qs[i % R], s0, "v", out=ov)

    for i in range(3):
        step(i)
    stream = torch.cuda.current_stream(dev)
    g_warm = make_runs(step, warmup, 50, torch, args.eager)
    g_main = make_runs(step, steps, 50, torch, args.eager)
    g_soak = make_runs(step, 50, 50, torch, args.eager)
    for g in g_warm:
        g.replay()
    el, _, clocks, _ = timed_runs(dev, stream, torch, g_main, (), g_soak)
    assert fb.last_device_error(dev) == 0
    b = w_bytes + (H * (dn + dv) // 128) * (C // 128) * 4 + 2 * T * H * (dn + C) * 2
    flops = 2 * 2.0 * T * H * dn * C
    el_max, units = reduce_over_ranks(el, steps * b, dev)
    hbm_bound = flops / b < 300
    per = el / steps
    if hbm_bound:
        value, unit = units / el_max / 1e9, "GB/s"
        roof = {"bound": "hbm", "achieved": b / per / 1e9, "peak": peaks["hbm"], "unit": "GB/s",
                "frac": b / per / 1e9 / peaks["hbm"], "peak_source": f"hbm_gbs ({peaks['src']})"}
    else:
        value, unit = steps * flops * world / el_max / 1e12, "TFLOP/s"
        roof = {"bound": "tensor", "achieved": flops / per / 1e12, "peak": peaks["bf16"], "unit": "TFLOP/s",
                "frac": flops / per / 1e12 / peaks["bf16"],
                "peak_source": f"bf16_tflops ({peaks['src']}): the products are bf16"}
    roof.update({"kernel": "mla_absorb_kernel (qk + v)", "traffic": recorded_traffic(args.workload, "mla"),
                 "algorithmic_bytes_per_launch": b // 2,
                 "kernel_us": per / 2 * 1e6})
    return {
        "value": value, "unit": unit, "ms_per_step": el_max / steps * 1e3, "clocks": clocks,
        "gpu_launches": 2 * steps, "roofline": roof, "e2e": None,
        "config": {"workload": args.workload, "T": T, "heads": H, "kv_lora": C, "qk_nope": dn, "v_head": dv,
                   "l2": f"wkv_b rotates over {R} copies ({R * w_bytes / 1e6:.0f} MB > 3x L2)"},
        "dtype": "bf16 x bf16(dequantised e4m3) -> f32 accumulate, bf16 out",
    }


def run_gate(args, shape, dev, torch, fb, peaks, steps, warmup, rank, world):
    """The 671B gate (sigmoid scores, per-expert bias, 8 groups with 4 kept,
    top-8, route_scale 2.5) on T tokens of fp32 logits together with the
    routing permutation of its output (fp8blk_moe_route: the gate kernel also
    ranks the pairs, one scatter pass): the step that turns gate logits into
    the grouped GEMMs' row order. Also timed: the gate alone, and the gate
    followed by the separate three-pass permutation."""
    T, E, G, TG, k, scale, seed = (shape[n] for n in ("T", "E", "groups", "kept", "k", "route_scale", "seed"))
    props = torch.cuda.get_device_properties(dev)
    l2 = int(getattr(props, "L2_cache_size", 0) or 132 * 2 ** 20)
    R = min(128, max(2, math.ceil(3 * l2 / (T * E * 4))))
    ls = [torch.from_numpy(synthetic.gate_logits(T, E, seed + i)).to(dev) for i in range(R)]
    b = torch.from_numpy(synthetic.gate_bias(E, seed)).to(dev)
    out = (torch.empty((T, k), dtype=torch.int32, device=dev), torch.empty((T, k), dtype=torch.float32, device=dev),
           torch.empty(E, dtype=torch.int32, device=dev), torch.empty(E + 1, dtype=torch.int32, device=dev),
           torch.empty(T * k, dtype=torch.int32, device=dev))

    def gate(i):
        fb.moe_gate(ls[i % R], b, G, TG, k, fb.SCORE_SIGMOID, scale, True, idx=out[0], w=out[1])

    def unfused(i):
        gate(i)
        fb.moe_permute(out[0], E)

    def step(i):
        fb.moe_route(ls[i % R], b, G, TG, k, fb.SCORE_SIGMOID, scale, True, out=out)

    for i in range(3):
        step(i)
        unfused(i)
    stream = torch.cuda.current_stream(dev)
    g_warm = make_runs(step, warmup, 50, torch, args.eager)
    g_main = make_runs(step, steps, 50, torch, args.eager)
    g_gate = make_runs(gate, steps, 50, torch, args.eager)
    g_unf = make_runs(unfused, steps, 50, torch, args.eager)
    g_soak = make_runs(step, 50, 50, torch, args.eager)
    for g in g_warm:
        g.replay()
    el, (el_gate, el_unf), clocks, _ = timed_runs(dev, stream, torch, g_main, (g_gate, g_unf), g_soak)
    assert fb.last_device_error(dev) == 0
    b_gate = T * E * 4 + E * 4 + T * k * 8            # logits, bias in; ids, weights out
    b_step = b_gate + T * k * 4 + (2 * E + 1) * 4      # + perm, counts, offsets out
    el_max, units = reduce_over_ranks(el, steps * b_step, dev)
    achieved = b_step / (el / steps) / 1e9
    return {
        "value": units / el_max / 1e9, "unit": "GB/s", "ms_per_step": el_max / steps * 1e3,
        "clocks": clocks, "gpu_launches": 2 * steps,
        "kernels_us": {"route (gate + permutation, 2 launches)": el / steps * 1e6, "gate_alone": el_gate / steps * 1e6,
                       "gate then three-pass permutation (4 launches)": el_unf / steps * 1e6},
        "roofline": {"bound": "hbm", "kernel": "moe_route (gate + rank kernel, scatter kernel)", "achieved": achieved,
                     "peak": peaks["hbm"], "unit": "GB/s", "frac": achieved / peaks["hbm"], "traffic": None,
                     "peak_source": f"hbm_gbs ({peaks['src']})", "algorithmic_bytes_per_launch": b_step,
                     "kernel_us": el / steps * 1e6},
        "e2e": None,
        "config": {"workload": args.workload, "T": T, "E": E, "groups": G, "kept_groups": TG, "topk": k,
                   "score": "sigmoid + per-expert bias", "route_scale": scale,
                   "logits": "fp32 N(0,1), bias N(0,0.01)",
                   "l2": f"logits rotate over {R} copies ({R * T * E * 4 / 1e6:.0f} MB > 3x L2)"},
        "dtype": "f32",
    }


# ---------------------------------------------------------------------------
# the oracle on the host cores (cpu_baseline leg and the reference arm)
# ---------------------------------------------------------------------------

_SAMPLE_CACHE = {}


def oracle_linear_sample(shape, n_cols: int):
    """One oracle step on a sample of the linear workload: act_quant of all
    of X and the fp64 GEMM for n_cols weight rows. The sampled weight rows are
    quantised once, outside the timed part (input preparation). Returns
    (seconds, algorithmic bytes of the sampled work)."""
    import oracle

    M, N, K = shape["M"], shape["N"], shape["K"]
    n_cols = max(1, min(n_cols, N))
    key = (M, N, K, shape["seed"], n_cols)
    if key not in _SAMPLE_CACHE:
        x = synthetic.activations(M, K, shape["seed"], outlier_frac=shape["frac"])
        w = synthetic.weights(-(-n_cols // 128) * 128, K, shape["seed"] + 1)
        _SAMPLE_CACHE[key] = (x,) + oracle.weight_quant(w)
    x, wq, ws = _SAMPLE_CACHE[key]
    t0 = time.perf_counter()
    xq, xs = oracle.act_quant(x)
    oracle.gemm(xq, xs, wq[:n_cols], ws[: -(-n_cols // 128)])
    dt = time.perf_counter() - t0
    kb = K // 128
    b = M * K * 2 + n_cols * K + (-(-n_cols // 128)) * kb * 4 + M * n_cols * 2
    return dt, b


def cpu_cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def block_row_ranges(N: int, parts: int):
    """Row ranges of whole 128-row weight blocks (the last one ragged), about
    N / parts rows each: the oracle runs one range per host thread."""
    nb = -(-N // 128)
    parts = max(1, min(parts, nb))
    edges = [min(N, (nb * i // parts) * 128) for i in range(parts + 1)]
    return [(edges[i], edges[i + 1]) for i in range(parts) if edges[i + 1] > edges[i]]


def oracle_gemm_threads(xq, xs, wq, ws, cores: int):
    """The oracle's GEMM with the weight rows split over `cores` host threads
    (the C oracle runs outside the interpreter lock), joined by columns."""
    import concurrent.futures as cf

    import oracle

    ranges = block_row_ranges(wq.shape[0], cores)
    with cf.ThreadPoolExecutor(len(ranges)) as ex:
        parts = list(ex.map(lambda r: oracle.gemm(xq, xs, wq[r[0]:r[1]], ws[r[0] // 128:-(-r[1] // 128)]), ranges))
    return np.concatenate(parts, axis=1)


def oracle_dequant_threads(q, s, cores: int):
    import concurrent.futures as cf

    import oracle

    ranges = block_row_ranges(q.shape[0], cores)
    with cf.ThreadPoolExecutor(len(ranges)) as ex:
        parts = list(ex.map(lambda r: oracle.weight_dequant(q[r[0]:r[1]], s[r[0] // 128:-(-r[1] // 128)]), ranges))
    return np.concatenate(parts, axis=0)


def oracle_linear_full(shape, cores: int):
    """One full oracle step of the linear workload on `cores` host threads:
    act_quant of all of X, then the fp64 GEMM over every weight row (the
    weight is quantised once, outside the timed part). Returns (seconds,
    algorithmic bytes)."""
    import oracle

    M, N, K = shape["M"], shape["N"], shape["K"]
    key = ("full", M, N, K, shape["seed"])
    if key not in _SAMPLE_CACHE:
        x = synthetic.activations(M, K, shape["seed"], outlier_frac=shape["frac"])
        w = synthetic.weights(N, K, shape["seed"] + 1)
        _SAMPLE_CACHE[key] = (x,) + oracle.weight_quant(w)
    x, wq, ws = _SAMPLE_CACHE[key]
    t0 = time.perf_counter()
    xq, xs = oracle.act_quant(x)
    oracle_gemm_threads(xq, xs, wq, ws, cores)
    return time.perf_counter() - t0, linear_bytes(M, N, K)


def cpu_baseline(shape, kind, budget_s=5.0):
    """The oracle (plain C, fp64) timed on this host's cores: the full decode
    layer with its weight rows split over every core (the reported value),
    the same layer single-threaded on a sample of rows, and one full run of
    the oracle on the 16x320x256 workload, act_quant of the prefill input and
    weight_dequant of an [18432, 7168] weight."""
    if kind != "linear":
        return None
    import oracle

    M, N, K = shape["M"], shape["N"], shape["K"]
    cores = cpu_cores()
    oracle_linear_full(shape, cores)                       # warm: inputs, library, threads
    tt, tb, reps = 0.0, 0, 0
    while tt < budget_s or reps == 0:
        dt, b = oracle_linear_full(shape, cores)
        tt, tb, reps = tt + dt, tb + b, reps + 1
    allc = tb / tt / 1e9
    # single-threaded, on a sample of weight rows sized to about 1 s per step
    n_cols = max(1, min(N, int(4e7 / (M * K))))
    st_t, st_b, st_reps = 0.0, 0, 0
    while st_t < budget_s or st_reps == 0:
        dt, b = oracle_linear_sample(shape, n_cols)
        st_t, st_b, st_reps = st_t + dt, st_b + b, st_reps + 1
    full = {}
    x = synthetic.activations(16, 256, synthetic.SEED_PR1)
    wq, ws = oracle.weight_quant(synthetic.weights(320, 256, synthetic.SEED_PR1))
    t0 = time.perf_counter()
    xq, xs = oracle.act_quant(x)
    oracle.gemm(xq, xs, wq, ws)
    full["pr1_linear_16x320x256 (1 thread)"] = time.perf_counter() - t0
    x = synthetic.activations(4096, 7168, synthetic.SEED_PREFILL)
    t0 = time.perf_counter()
    oracle.act_quant(x)
    full["act_quant_4096x7168 (1 thread)"] = time.perf_counter() - t0
    del x
    # every finite positive code, one power-of-two scale per block: dequant cost does not depend on values
    q = np.random.default_rng(synthetic.SEED_ATTN).integers(0, 126, size=(18432, 7168), dtype=np.uint8)
    s = np.full((144, 56), 2.0 ** -7, np.float32)
    t0 = time.perf_counter()
    oracle_dequant_threads(q, s, cores)
    full[f"weight_dequant_18432x7168 ({cores} threads)"] = time.perf_counter() - t0
    full[f"decode_linear_{M}x{N}x{K} ({cores} threads)"] = tt / reps
    return {"value": allc, "unit": "GB/s", "cores": cores, "kind": "oracle",
            "sample": f"{reps} x the full layer: act_quant of X[{M},{K}] + fp64 GEMM over all {N} weight rows "
                      f"split over {cores} threads, {tt:.1f} s",
            "single_thread": {"value": st_b / st_t / 1e9, "unit": "GB/s", "cores": 1,
                              "sample": f"{st_reps} x (act_quant of X[{M},{K}] + fp64 GEMM over {n_cols} of {N} "
                                        f"weight rows), {st_t:.1f} s"},
            "full_oracle_seconds": {k: round(v, 4) for k, v in full.items()},
            "threads": "the C oracle unchanged, one call per range of 128-row weight blocks per host thread"}


def run_reference(args, kind, shape, steps, warmup):
    """The reference arm: the oracle on the host cores. Each step is the full
    decode layer with its weight rows split over every core, or, when
    warm-up + steps would take more than about a minute and a half that way,
    a single-threaded sample of weight rows sized to fit."""
    ws, rank, _ = dist_env()
    if rank != 0:
        return 0
    if kind != "linear":
        print(json.dumps({"impl": "reference", "unavailable": "the oracle leg covers the linear workloads only"}))
        return 0
    M, N, K = shape["M"], shape["N"], shape["K"]
    cores = cpu_cores()
    oracle_linear_full(shape, cores)
    probe, _ = oracle_linear_full(shape, cores)
    full = probe * (steps + min(warmup, 3)) <= 90.0
    if full:
        def step():
            return oracle_linear_full(shape, cores)
        used = cores
        sample = f"each step: the full layer, act_quant of X[{M},{K}] + fp64 GEMM over all {N} rows " \
                 f"split over {cores} threads"
    else:
        per_step_s = 60.0 / max(1, steps + warmup)
        n_cols = max(1, min(N, int(4e7 * per_step_s / (M * K))))

        def step():
            return oracle_linear_sample(shape, n_cols)
        used = 1
        sample = f"each step: act_quant of X[{M},{K}] + fp64 GEMM over {n_cols} of {N} rows, 1 thread"
    for _ in range(min(warmup, 3)):
        step()
    tt, tb = 0.0, 0
    for _ in range(steps):
        dt, b = step()
        tt += dt
        tb += b
    val = tb / tt / 1e9
    line = {
        "metric": "block-scaled FP8 GEMM TFLOP/s & decode GB/s, % of GB300 roofline, 1 GPU",
        "value": val, "unit": "GB/s", "impl": "reference", "n_gpus": 1, "steps": steps, "warmup": warmup,
        "ms_per_step": tt / steps * 1e3, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f64 (oracle)", "data": "synthetic",
        "config": {"workload": args.workload, "M": M, "N": N, "K": K,
                   "sample": "full layer" if full else "sampled weight rows"},
        "cpu_baseline": {"value": val, "unit": "GB/s", "kind": "oracle", "cores": used, "sample": sample},
        "e2e": {"value": val, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))
    return 0


# ---------------------------------------------------------------------------

# Measured after the default workload and reported under "other_workloads":
# the TFLOP/s half of the metric (the prefill GEMM, both scale formats) and
# the MoE step (both scale formats), each a short run of its own.
OTHER_WORKLOADS = ("prefill_gemm_w1", "prefill_gemm_w1_ue8m0", "moe_t4096_uniform", "moe_t4096_uniform_ue8m0")


def run_other_workloads(args, dev, torch, fb, peaks, steps=20, warmup=3):
    out = {}
    runners = {"linear": run_linear, "moe": run_moe, "ffn": run_ffn}
    for name in OTHER_WORKLOADS:
        if name == args.workload:
            continue
        kind, shape = WORKLOADS[name]
        sub = argparse.Namespace(**dict(vars(args), workload=name, no_e2e=True))
        r = runners[kind](sub, shape, dev, torch, fb, peaks, steps, warmup, 0, 1)
        roof = r["roofline"]
        out[name] = {"value": r["value"], "unit": r["unit"], "ms_per_step": r["ms_per_step"], "steps": steps,
                     "warmup": warmup, "clocks": r["clocks"],
                     "roofline": {k: roof.get(k) for k in ("bound", "kernel", "achieved", "peak", "unit", "frac",
                                                           "frac_of_burst_peak", "peak_source", "kernel_us",
                                                           "traffic") if k in roof},
                     "config": r["config"]}
        if "tflops" in r:
            out[name]["tflops"] = r["tflops"]
        del r
        torch.cuda.synchronize()
        torch.cuda.empty_cache()
    return out


def reaches_cluster_multicast(kind, shape) -> bool:
    """True if the workload can run a GEMM kernel that loads with TMA
    cluster multicast: the CTA-pair plans of dense GEMMs with M > 128 (and the
    dense SwiGLU GEMM of the FFN). Decode-sized GEMMs (M <= 128, weights as the
    MMA's M operand), the grouped expert GEMMs, dequant, the gate and the MLA
    kernels never do."""
    return (kind == "linear" and shape["M"] > 128) or kind == "ffn"


def main():
    args = parse()
    if args.no_soak:
        _SOAK[0] = 0.0
    kind, shape = WORKLOADS[args.workload]
    world, rank, _ = dist_env()
    if (world > 1 or args.gpus > 1) and args.impl == "ours" and reaches_cluster_multicast(kind, shape):
        # Cluster-multicast kernels run only in single-GPU processes: refuse
        # before the library is loaded or any GPU is touched.
        if rank == 0:
            print(json.dumps({"impl": "ours", "workload": args.workload, "unavailable":
                              "one GPU by design: this workload's GEMMs use cluster-multicast TMA loads, "
                              "which run only in single-GPU calls; multi-GPU replicas are offered for the "
                              "decode-sized, expert, dequant, gate and MLA workloads"}))
        return 0
    big = kind == "linear" and shape["M"] >= 2048 or kind in ("dequant", "ffn", "moe") or \
        kind == "mla" and shape["T"] >= 2048
    steps = args.steps if args.steps is not None else (200 if big else 100000)
    warmup = args.warmup if args.warmup is not None else (10 if big else 1000)
    if warmup < 3:
        raise SystemExit("--warmup must be >= 3")
    if args.impl == "reference":
        return run_reference(args, kind, shape, steps, warmup)

    import torch
    import torch.distributed as dist

    world, rank, local = dist_env()
    if args.gpus != world and world > 1:
        raise SystemExit(f"--gpus {args.gpus} but WORLD_SIZE {world}")
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    if world > 1:
        dist.init_process_group("nccl", device_id=dev)
    import fp8_block_scaled_quant_gb300 as fb

    fb.lib()
    peaks = load_peaks()
    if kind == "linear":
        res = run_linear(args, shape, dev, torch, fb, peaks, steps, warmup, rank, world)
    elif kind == "ffn":
        res = run_ffn(args, shape, dev, torch, fb, peaks, steps, warmup, rank, world)
    elif kind == "moe":
        res = run_moe(args, shape, dev, torch, fb, peaks, steps, warmup, rank, world)
    elif kind == "gate":
        res = run_gate(args, shape, dev, torch, fb, peaks, steps, warmup, rank, world)
    elif kind == "mla":
        res = run_mla(args, shape, dev, torch, fb, peaks, steps, warmup, rank, world)
    else:
        res = run_dequant(args, shape, dev, torch, fb, peaks, steps, warmup, rank, world)
    other = None
    if world == 1 and not args.no_other and args.workload == DEFAULT:
        other = run_other_workloads(args, dev, torch, fb, peaks)
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(shape, kind)
    if rank == 0:
        line = {
            "metric": "block-scaled FP8 GEMM TFLOP/s & decode GB/s, % of GB300 roofline, 1 GPU",
            "value": res["value"], "unit": res["unit"], "n_gpus": world, "steps": steps, "warmup": warmup,
            "ms_per_step": res["ms_per_step"], "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": res["dtype"], "data": "synthetic (seeded; no dataset on the pages)",
            "config": dict(res["config"], parallelism=f"replicas x{world}"),
            "clocks": res["clocks"], "roofline": res["roofline"], "e2e": res["e2e"],
            "gpu_launches": res["gpu_launches"], "cpu_baseline": cpu,
        }
        for extra in ("kernels_us", "tflops"):
            if extra in res:
                line[extra] = res[extra]
        if other is not None:
            line["other_workloads"] = other
        print(json.dumps(line))
    if world > 1:
        dist.barrier()
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
