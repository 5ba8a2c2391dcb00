"""Benchmark of the fused MoE layer (forward + backward) on GB300.

One step = forward + backward of the whole layer (routing, dispatch, gate/up +
SwiGLU, down + combine, and the backward's dgrads, wgrads, router gradient and
un-permute) over one batch of synthetic inputs already resident in HBM.
Prints one JSON line.  ``--impl reference`` times the CPU oracle instead.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
    torchrun --nproc-per-node N bench.py --gpus N ...   (independent replicas)
"""

from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

import synth_inputs as si  # noqa: E402

METRIC = "MoE layer fwd+bwd tokens/s and TFLOP/s on 1×GB300 (% of tensor-core peak)"
DEFAULT_WORKLOAD = "qwen3_235b"

# algorithmic FLOPs per launch of each GEMM kernel (P = T*k rows)
def gemm_flops(sh):
    P, T, H, F, E = sh.P, sh.T, sh.H, sh.F, sh.E
    return {
        "router_gemm_topk": 2 * T * H * E,
        "gate_up_gemm_swiglu": 4 * P * H * F,
        "down_gemm_scatter": 2 * P * F * H,
        "down_dgrad_swiglu_bwd": 2 * P * H * F,
        "down_wgrad": 2 * P * F * H,
        "gate_up_dgrad_scatter": 4 * P * H * F,
        "gate_up_wgrad": 4 * P * H * F,
        "router_wgrad": 2 * T * H * E,
    }


def gemm_flops_all(sh):
    """gemm_flops plus the MXFP8 kernels (same algorithmic work, "_mx" suffix)."""
    f = gemm_flops(sh)
    f.update({name + "_mx": v for name, v in f.items() if not name.startswith("router")})
    return f


# nominal dense fp8 : bf16 tensor-core rate on GB300 (4.5 : 2.25 PFLOP/s)
FP8_OVER_BF16 = 2.0


def bf16_peak(peaks, clk):
    """(TFLOP/s, kind) of the measured bf16 GEMM peak that matches the clocks
    sampled in the timed region: the burst figure when the median SM clock
    under load is within 5% of the maximum, else the sustained (power-capped)
    figure."""
    med, mx = (clk or {}).get("sm_mhz"), (clk or {}).get("sm_max_mhz")
    if med is not None and mx and med >= 0.95 * mx:
        return peaks["bf16_tflops"], "burst"
    return peaks["bf16_tflops_sustained"], "sustained"


def tensor_peak(name, peaks, clk):
    """(peak TFLOP/s, source) for a GEMM kernel: the bf16 peak chosen by the
    clocks, and for MXFP8 kernels that peak times the nominal fp8:bf16 ratio."""
    tf, kind = bf16_peak(peaks, clk)
    if name.endswith("_mx"):
        return tf * FP8_OVER_BF16, (f"{peaks['source']} bf16 {kind} x {FP8_OVER_BF16:g} "
                                    f"(nominal fp8:bf16)")
    return tf, f"{peaks['source']} bf16 {kind}"


# algorithmic bytes per launch of the memory-bound kernels
def kernel_bytes(sh):
    P, T, H, k = sh.P, sh.T, sh.H, sh.top_k
    row = 2 * H
    return {
        "gather_x": T * row + P * row + 4 * P,
        "gather_dy": T * row + P * row + 4 * P,
        "combine": P * row + T * row,
        "unpermute_dx": P * row + T * row + 8 * P,
    }


def gemm_bytes(sh):
    """Algorithmic DRAM bytes per launch of each bf16 expert GEMM: every
    operand read once and every output written once (2 bytes per element).
    With ~256 rows per expert (the 30B shape) the weight bytes alone put these
    GEMMs near the ridge of the roofline, so the bench reports whichever of the
    FLOP time and the byte time is larger."""
    P, H, F, E = sh.P, sh.H, sh.F, sh.E
    W1, W2 = 2 * E * H * F * 2, E * F * H * 2      # [W_gate | W_up], W_down
    return {
        "gate_up_gemm_swiglu": P * H * 2 + W1 + P * 2 * F * 2 + P * F * 2,
        "down_gemm_scatter": P * F * 2 + W2 + P * H * 2,
        "down_dgrad_swiglu_bwd": P * H * 2 + W2 + P * 2 * F * 2 + P * 2 * F * 2 + P * F * 2,
        "down_wgrad": P * F * 2 + P * H * 2 + W2,
        "gate_up_dgrad_scatter": P * 2 * F * 2 + W1 + P * H * 2,
        "gate_up_wgrad": P * H * 2 + P * 2 * F * 2 + W1,
    }


def csrc_hash() -> str:
    """Hash of the kernel sources: a stored ncu traffic figure is only used
    while the kernels it was taken on are unchanged."""
    import hashlib
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "mixture_experts_layer_17_gb300", "csrc")
    for name in sorted(os.listdir(csrc)):
        with open(os.path.join(csrc, name), "rb") as fh:
            h.update(name.encode() + fh.read())
    return h.hexdigest()[:16]


def stored_traffic(kernel: str, workload: str):
    """dram__bytes_read.sum + dram__bytes_write.sum per launch from the
    committed ncu capture (profiles/dram_traffic.json), or None."""
    path = os.path.join(ROOT, "profiles", "dram_traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as fh:
        table = json.load(fh)
    rec = table.get(f"{kernel}@{workload}")
    if rec is None or rec.get("csrc_hash") != csrc_hash():
        return None
    return rec["bytes_per_launch"]


# ncu kernel name (template argument) -> the label the library's profiler uses
NCU_LABELS = [
    ("WgradMXProblem<true>", "gate_up_wgrad_mx"), ("WgradMXProblem<false>", "down_wgrad_mx"),
    ("WgradMXProblem<1>", "gate_up_wgrad_mx"), ("WgradMXProblem<0>", "down_wgrad_mx"),
    ("GateUpFwdMXProblem", "gate_up_gemm_swiglu_mx"), ("DownFwdMXProblem", "down_gemm_scatter_mx"),
    ("DownDgradMXProblem", "down_dgrad_swiglu_bwd_mx"),
    ("GateUpDgradMXProblem", "gate_up_dgrad_scatter_mx"),
    ("WgradMXPairProblem<true>", "gate_up_wgrad_mx"), ("WgradMXPairProblem<false>", "down_wgrad_mx"),
    ("WgradMXPairProblem<1>", "gate_up_wgrad_mx"), ("WgradMXPairProblem<0>", "down_wgrad_mx"),
    ("GateUpFwdMXPairProblem", "gate_up_gemm_swiglu_mx"),
    ("DownFwdMXPairProblem", "down_gemm_scatter_mx"),
    ("DownDgradMXPairProblem", "down_dgrad_swiglu_bwd_mx"),
    ("GateUpDgradMXPairProblem", "gate_up_dgrad_scatter_mx"),
    ("GateUpWgradProblem", "gate_up_wgrad"), ("DownWgradProblem", "down_wgrad"),
    ("GateUpFwdPairProblem", "gate_up_gemm_swiglu"), ("GateUpFwdProblem", "gate_up_gemm_swiglu"),
    ("DownFwdPairProblem", "down_gemm_scatter"), ("DownFwdProblem", "down_gemm_scatter"),
    ("DownDgradPairProblem", "down_dgrad_swiglu_bwd"), ("DownDgradProblem", "down_dgrad_swiglu_bwd"),
    ("GateUpDgradPairProblem", "gate_up_dgrad_scatter"),
    ("GateUpDgradProblem", "gate_up_dgrad_scatter"),
    ("RouterWgradProblem", "router_wgrad"), ("RouterProblem", "router_gemm_topk"),
    ("combine_kernel", "combine"), ("unpermute_kernel", "unpermute_dx"),
]
_BYTE_UNITS = {"byte": 1, "Kbyte": 1e3, "Mbyte": 1e6, "Gbyte": 1e9, "KB": 1e3, "MB": 1e6,
               "GB": 1e9}


def record_traffic(csv_path: str, workload: str, command: str, path: str = None,
                   scale: float = 1.0, captured_on: str = None) -> dict:
    """Fold an ncu CSV (metrics dram__bytes_read.sum and dram__bytes_write.sum,
    one row per launch and metric) into profiles/dram_traffic.json: bytes per
    launch for each library kernel of ``workload``, stamped with the hash of
    the kernel sources they were taken on.  A capture taken on a smaller case
    of the same per-expert shape (``captured_on``) is scaled to ``workload``
    by ``scale``, the ratio of the units the two process (every term of the
    traffic grows with them)."""
    import csv
    rows = []
    with open(csv_path) as fh:
        lines = [ln for ln in fh if ln.startswith('"')]
    for rec in csv.DictReader(lines):
        rows.append(rec)
    per_launch = {}
    for rec in rows:
        metric = rec.get("Metric Name", "")
        if metric not in ("dram__bytes_read.sum", "dram__bytes_write.sum"):
            continue
        label = next((lab for pat, lab in NCU_LABELS if pat in rec["Kernel Name"]), None)
        if label is None:
            continue
        val = float(rec["Metric Value"].replace(",", "")) * _BYTE_UNITS.get(rec["Metric Unit"], 1)
        key = (label, rec["ID"])
        per_launch[key] = per_launch.get(key, 0.0) + val
    table = {}
    path = path or os.path.join(ROOT, "profiles", "dram_traffic.json")
    if os.path.exists(path):
        with open(path) as fh:
            table = json.load(fh)
    labels = sorted({lab for lab, _ in per_launch})
    h = csrc_hash()
    for lab in labels:
        vals = [v for (l2, _), v in per_launch.items() if l2 == lab]
        rec = {"bytes_per_launch": scale * sum(vals) / len(vals), "launches": len(vals),
               "csrc_hash": h, "command": command}
        if captured_on:
            rec["captured_on"] = captured_on
            rec["scale"] = scale
        table[f"{lab}@{workload}"] = rec
    with open(path, "w") as fh:
        json.dump(table, fh, indent=1, sort_keys=True)
        fh.write("\n")
    return {lab: table[f"{lab}@{workload}"]["bytes_per_launch"] for lab in labels}


def layer_flops(sh):
    fwd = 6 * sh.P * sh.H * sh.F + 2 * sh.T * sh.H * sh.E
    bwd = 12 * sh.P * sh.H * sh.F + 4 * sh.T * sh.H * sh.E
    return fwd, bwd


def expert_router_flops(sh):
    """(expert GEMM FLOPs, router GEMM FLOPs) of the forward and of the backward."""
    fe, fr = 6 * sh.P * sh.H * sh.F, 2 * sh.T * sh.H * sh.E
    return (fe, fr), (2 * fe, 2 * fr)


def layer_peak_frac(sh, achieved_ms, peaks, clk):
    """The step against the tensor-core roofline of its precision: the time
    every GEMM would take at the measured peak (bf16 peak chosen by the
    clocks; MXFP8 GEMMs at FP8_OVER_BF16 times it; the router GEMMs are bf16
    in every precision) divided by the measured step time."""
    tf, kind = bf16_peak(peaks, clk)
    (fe, fr), (be, br) = expert_router_flops(sh)
    fwd_rate = tf * (FP8_OVER_BF16 if sh.precision == "mxfp8" else 1.0)
    bwd_rate = tf * (FP8_OVER_BF16 if sh.precision in ("mxfp8", "fp8_bwd") else 1.0)
    ideal_ms = ((fe / fwd_rate + be / bwd_rate) + (fr + br) / tf) / 1e9
    out = {"frac": ideal_ms / achieved_ms, "ideal_ms": ideal_ms,
           "peak": f"{peaks['source']} bf16 {kind} {tf:.1f} TFLOP/s"
                   + (f", MXFP8 GEMMs at x{FP8_OVER_BF16:g}" if sh.precision != "bf16" else "")}
    if sh.precision == "bf16":
        # the step's roofline with both roofs: every expert GEMM at the larger
        # of its FLOP time and its algorithmic-byte time, the router GEMMs at
        # their FLOP time, the memory-bound kernels at their byte time
        fl, gb, kb = gemm_flops(sh), gemm_bytes(sh), kernel_bytes(sh)
        hbm = peaks["hbm_gbs"] * 1e9
        t = sum(max(fl[k] / (tf * 1e12), gb[k] / hbm) for k in gb)
        t += (fl["router_gemm_topk"] + fl["router_wgrad"]) / (tf * 1e12)
        t += sum(kb.values()) / hbm
        out["roofline_ms"] = t * 1e3
        out["frac_of_roofline"] = t * 1e3 / achieved_ms
    return out


def dominant_kernel(prof):
    """The label with the largest total time in a profile."""
    return max(prof, key=lambda n: prof[n][1])


def profile_pass(step, inp, n):
    """n fwd+bwd steps with the library's CUDA events around every launch;
    returns {label: (launches, total ms)}."""
    from mixture_experts_layer_17_gb300 import (moe_profile_enable, moe_profile_read,
                                                moe_profile_select)
    torch.cuda.synchronize()
    moe_profile_read()
    moe_profile_select(None)
    moe_profile_enable(True)
    for _ in range(n):
        step(inp["x"], inp["dY"])
    torch.cuda.synchronize()
    moe_profile_enable(False)
    return moe_profile_read()


def summarize_kernels(prof, sh, peaks, clk, live=None):
    """Per-kernel launches, mean time, share, achieved rate and fraction of
    roofline from the library's CUDA-event records, and the roofline object of
    the kernel with the largest total time.  `live`: that kernel's records from
    the timed region (timed alone there), which then give the roofline."""
    flops = gemm_flops_all(sh)
    byts = kernel_bytes(sh)
    gbyts = gemm_bytes(sh) if sh.precision == "bf16" else {}
    kernels = {name: {"launches": n, "avg_ms": ms / max(n, 1), "share": None}
               for name, (n, ms) in prof.items()}
    ktotal = sum(v["avg_ms"] * v["launches"] for v in kernels.values())
    for v in kernels.values():
        v["share"] = v["avg_ms"] * v["launches"] / ktotal if ktotal else None
    dom = max(kernels, key=lambda n: kernels[n]["avg_ms"] * kernels[n]["launches"])
    timed_live = live is not None and dom in live and live[dom][0] > 0
    if timed_live:
        kernels[dom] = dict(kernels[dom], avg_ms_profiled_pass=kernels[dom]["avg_ms"],
                            avg_ms=live[dom][1] / live[dom][0], launches_timed=live[dom][0])

    def hbm_bound(name):
        # a bf16 expert GEMM whose algorithmic bytes take longer at the HBM
        # peak than its FLOPs at the tensor peak
        if name not in gbyts:
            return False
        return gbyts[name] / (peaks["hbm_gbs"] * 1e9) > \
            flops[name] / (tensor_peak(name, peaks, clk)[0] * 1e12)

    if dom in flops and not hbm_bound(dom):
        ach = flops[dom] / (kernels[dom]["avg_ms"] * 1e-3) / 1e12
        peak, src = tensor_peak(dom, peaks, clk)
        roof = {"kernel": dom, "bound": "tensor", "achieved": ach, "peak": peak,
                "unit": "TFLOP/s", "frac": ach / peak, "traffic": stored_traffic(dom, sh.name),
                "peak_source": src, "sm_mhz_median": clk.get("sm_mhz"),
                "sm_max_mhz": clk.get("sm_max_mhz")}
    elif dom in flops:
        ach = gbyts[dom] / (kernels[dom]["avg_ms"] * 1e-3) / 1e9
        peak = peaks["hbm_gbs"]
        roof = {"kernel": dom, "bound": "hbm", "achieved": ach, "peak": peak, "unit": "GB/s",
                "frac": ach / peak, "traffic": stored_traffic(dom, sh.name),
                "peak_source": f"{peaks['source']} hbm (algorithmic bytes above the tensor "
                               f"time at this shape)",
                "tensor_frac": flops[dom] / (kernels[dom]["avg_ms"] * 1e-3) / 1e12
                / tensor_peak(dom, peaks, clk)[0]}
    else:
        ach = byts.get(dom, 0) / (kernels[dom]["avg_ms"] * 1e-3) / 1e9
        peak = peaks["hbm_gbs"]
        roof = {"kernel": dom, "bound": "hbm", "achieved": ach, "peak": peak, "unit": "GB/s",
                "frac": ach / peak, "traffic": stored_traffic(dom, sh.name),
                "peak_source": f"{peaks['source']} hbm"}
    if timed_live:
        roof["timing"] = (f"{live[dom][0]} launches timed with CUDA events inside the timed "
                          f"region, the only launches timed there")
    per_kernel = {}
    for name, v in sorted(kernels.items(), key=lambda kv: -kv[1]["share"]):
        d = {"launches": v["launches"], "avg_ms": round(v["avg_ms"], 4),
             "share": round(v["share"], 4)}
        if "avg_ms_profiled_pass" in v:
            d["avg_ms_profiled_pass"] = round(v["avg_ms_profiled_pass"], 4)
        if name in flops:
            d["tflops"] = round(flops[name] / (v["avg_ms"] * 1e-3) / 1e12, 1)
            d["frac_of_peak"] = round(d["tflops"] / tensor_peak(name, peaks, clk)[0], 3)
        if name in gbyts:
            d["gbs"] = round(gbyts[name] / (v["avg_ms"] * 1e-3) / 1e9, 1)
            d["frac_hbm"] = round(d["gbs"] / peaks["hbm_gbs"], 3)
            d["bound"] = "hbm" if hbm_bound(name) else "tensor"
        if name in byts:
            d["gbs"] = round(byts[name] / (v["avg_ms"] * 1e-3) / 1e9, 1)
            d["frac_hbm"] = round(d["gbs"] / peaks["hbm_gbs"], 3)
        per_kernel[name] = d
    return per_kernel, roof


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as fh:
            p = json.load(fh)
        return {"hbm_gbs": p["hbm_gbs"], "bf16_tflops": p["bf16_tflops"],
                "bf16_tflops_sustained": p.get("bf16_tflops_sustained", p["bf16_tflops"]),
                "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
            "source": "fallback"}


class ClockSampler:
    """Samples nvidia-smi clocks and throttle reasons while the timed region runs."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.rows = []
        self.proc = None
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) == 7:
                self.rows.append(parts)

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.thread.join(timeout=5)
        sm = [float(r[0]) for r in self.rows if r[0].replace(".", "").isdigit()]
        mx = [float(r[1]) for r in self.rows if r[1].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in self.rows for i in range(4) if r[3 + i] == "Active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "samples": len(self.rows)}


def dist_setup(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if args.impl == "ours" else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
    elif torch.cuda.is_available() and args.impl == "ours":
        torch.cuda.set_device(local)
    return world, rank, local


def max_over_ranks(v: float, world: int) -> float:
    if world == 1:
        return v
    import torch.distributed as dist
    t = torch.tensor([v], dtype=torch.float64,
                     device="cuda" if dist.get_backend() == "nccl" else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


# ------------------------------------------------------------------ CPU oracle

def oracle_sample_time(sh, inp_cpu, n_tokens: int):
    """Times the CPU oracle (as it stands) on the first n_tokens tokens of the
    workload: routing, forward and the full backward (expert weight
    gradients are computed expert by expert and dropped)."""
    from oracle import moe_oracle as mo
    x = inp_cpu["x"][:n_tokens]
    dY = inp_cpu["dY"][:n_tokens]
    t0 = time.perf_counter()
    g = mo.backward(x, inp_cpu["W_r"], inp_cpu["W_gate"], inp_cpu["W_up"], inp_cpu["W_down"],
                    sh.top_k, dY, logit_bias=inp_cpu["logit_bias"], keep_weight_grads=False)
    dt = time.perf_counter() - t0
    assert np.isfinite(g["dx"]).all()
    return dt


def host_copy_for_oracle(inp):
    """fp32 numpy copies of the (bf16) inputs; the oracle widens them to fp64."""
    out = {}
    for k in ("x", "W_r", "W_gate", "W_up", "W_down", "dY"):
        out[k] = inp[k].float().cpu().numpy()
    out["logit_bias"] = None if inp["logit_bias"] is None else inp["logit_bias"].cpu().numpy()
    return out


def blas_threads() -> int:
    for var in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS"):
        if os.environ.get(var):
            return int(os.environ[var])
    return os.cpu_count() or 1


def cpu_baseline(sh, inp, budget_s: float = 20.0):
    """Oracle throughput on a bounded sample of the same workload."""
    inp_cpu = host_copy_for_oracle(inp)
    # grow the sample until one timing takes about budget_s / 2 (the cost is
    # not linear in small samples: every touched expert's weights are widened)
    n = 8
    dt = oracle_sample_time(sh, inp_cpu, n)
    for _ in range(4):
        if dt >= 0.35 * budget_s or n >= sh.T:
            break
        grow = min(8.0, (0.5 * budget_s) / max(dt, 1e-3))
        n = min(sh.T, max(n + 1, int(n * grow)))
        dt = oracle_sample_time(sh, inp_cpu, n)
    return {"value": n / dt, "unit": "tokens/s", "cores": blas_threads(), "kind": "oracle",
            "sample": f"first {n} of {sh.T} tokens of {sh.name}: route + fwd + full bwd in "
                      f"numpy fp64 ({dt:.1f} s)"}


# ------------------------------------------------------------------ our arm

def run_ours(args, sh, world, rank, local):
    from mixture_experts_layer_17_gb300 import (MoeLayer, moe_launch_count, moe_profile_enable,
                                                moe_profile_read, moe_profile_select)
    dev = torch.device("cuda", local)
    shr = si.shape(sh.name) if sh.name in si.WORKLOADS else sh
    import dataclasses
    shr = dataclasses.replace(shr, seed=shr.seed + 1000 * rank) if rank else shr
    inp = si.make_inputs(shr, dev)
    layer = MoeLayer(sh.T, sh.H, sh.F, sh.E, sh.top_k, sh.precision, flags=args.flags, device=dev,
                     max_sms=args.max_sms)
    grads = {"dx": torch.empty_like(inp["x"]), "dW_r": torch.empty_like(inp["W_r"]),
             "dW_gate": torch.empty_like(inp["W_gate"]), "dW_up": torch.empty_like(inp["W_up"]),
             "dW_down": torch.empty_like(inp["W_down"])}
    y = torch.empty_like(inp["x"])
    W = (inp["W_r"], inp["W_gate"], inp["W_up"], inp["W_down"])
    prepare_ms = None
    if args.prepared_weights:
        # MXFP8 weights quantised once (as once per optimizer step), timed apart
        layer.prepare_weights(W[1], W[2], W[3])
        torch.cuda.synchronize()
        p0 = torch.cuda.Event(enable_timing=True)
        p1 = torch.cuda.Event(enable_timing=True)
        p0.record()
        layer.prepare_weights(W[1], W[2], W[3])
        p1.record()
        torch.cuda.synchronize()
        prepare_ms = p0.elapsed_time(p1)
    acc = None
    if args.accumulate:
        # fp32 gradient accumulation buffers (micro-batch training)
        acc = {k: torch.zeros(inp[k[1:]].shape, dtype=torch.float32, device=dev)
               for k in ("dW_r", "dW_gate", "dW_up", "dW_down")}

    def backward(x, dY):
        if acc is None:
            layer.backward(x, W[0], W[1], W[2], W[3], dY, grads=grads)
        else:
            layer.backward_accumulate(x, W[0], W[1], W[2], W[3], dY, acc, dx=grads["dx"])

    def step(x, dY):
        layer.forward(x, W[0], W[1], W[2], W[3], inp["logit_bias"], y=y)
        backward(x, dY)

    for _ in range(args.warmup):
        step(inp["x"], inp["dY"])
    torch.cuda.synchronize()
    assert layer.device_status("fwd") == 0 and layer.device_status("bwd") == 0

    # ---- per-kernel profile: events around every launch, in a pass of a few
    # steps just before the timed region.  Events between all ~20 launches
    # cost up to 5% of a short step (0.07 ms at 30B), so the timed region
    # times only the dominant kernel's launches (the roofline object).
    prof_all = profile_pass(step, inp, min(args.steps, 10))
    dom = dominant_kernel(prof_all)

    # ---- device-resident timed region (the dominant kernel's events live)
    stream = torch.cuda.current_stream()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True),
           torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    clocks = ClockSampler(local)
    moe_profile_read()
    moe_profile_select(dom)
    moe_profile_enable(True)
    launches0 = moe_launch_count()
    barrier(world)
    torch.cuda.synchronize()
    clocks.start()
    time.sleep(1.0)          # let nvidia-smi start sampling before the timed region
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    t_start.record(stream)
    for i in range(args.steps):
        ev[i][0].record(stream)
        layer.forward(inp["x"], W[0], W[1], W[2], W[3], inp["logit_bias"], y=y)
        ev[i][1].record(stream)
        backward(inp["x"], inp["dY"])
        ev[i][2].record(stream)
    t_end.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    clk = clocks.stop()
    launches = moe_launch_count() - launches0
    moe_profile_enable(False)
    moe_profile_select(None)
    prof_live = moe_profile_read()
    total_ms = max_over_ranks(t_start.elapsed_time(t_end), world)
    fwd_ms = statistics.median(e[0].elapsed_time(e[1]) for e in ev)
    bwd_ms = statistics.median(e[1].elapsed_time(e[2]) for e in ev)
    ms_per_step = total_ms / args.steps
    assert layer.device_status("fwd") == 0 and layer.device_status("bwd") == 0

    # ---- end to end through the API with pinned host buffers: every step copies
    # its x and dY in and its y and dx out; the copies run on a side stream,
    # double-buffered, so step i + 1's inputs arrive and step i's results leave
    # while the layer computes (as a data loader would feed it)
    hx = inp["x"].cpu().pin_memory()
    hdY = inp["dY"].cpu().pin_memory()
    hy = torch.empty_like(hx).pin_memory()
    hdx = torch.empty_like(hx).pin_memory()
    xs = [torch.empty_like(inp["x"]) for _ in range(2)]
    dYs = [torch.empty_like(inp["dY"]) for _ in range(2)]
    ys = [torch.empty_like(inp["x"]) for _ in range(2)]
    dxs = [torch.empty_like(inp["x"]) for _ in range(2)]
    cs = torch.cuda.Stream(device=dev)
    in_ready = [torch.cuda.Event() for _ in range(2)]
    done = [torch.cuda.Event() for _ in range(2)]
    out_done = [torch.cuda.Event() for _ in range(2)]
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)

    def backward_into(x, dY, dx):
        if acc is None:
            g = dict(grads)
            g["dx"] = dx
            layer.backward(x, W[0], W[1], W[2], W[3], dY, grads=g)
        else:
            layer.backward_accumulate(x, W[0], W[1], W[2], W[3], dY, acc, dx=dx)

    barrier(world)
    torch.cuda.synchronize()
    e0.record(stream)
    cs.wait_event(e0)
    with torch.cuda.stream(cs):
        xs[0].copy_(hx, non_blocking=True)
        dYs[0].copy_(hdY, non_blocking=True)
        in_ready[0].record(cs)
    for i in range(args.steps):
        b = i % 2
        stream.wait_event(in_ready[b])
        if i >= 2:
            stream.wait_event(out_done[b])        # step i - 2's results have left
        layer.forward(xs[b], W[0], W[1], W[2], W[3], inp["logit_bias"], y=ys[b])
        backward_into(xs[b], dYs[b], dxs[b])
        done[b].record(stream)
        with torch.cuda.stream(cs):
            if i + 1 < args.steps:
                if i >= 1:
                    cs.wait_event(done[1 - b])    # step i - 1 no longer reads its inputs
                xs[1 - b].copy_(hx, non_blocking=True)
                dYs[1 - b].copy_(hdY, non_blocking=True)
                in_ready[1 - b].record(cs)
            cs.wait_event(done[b])
            hy.copy_(ys[b], non_blocking=True)
            hdx.copy_(dxs[b], non_blocking=True)
            out_done[b].record(cs)
    stream.wait_stream(cs)
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(e0.elapsed_time(e1), world) / args.steps

    # ---- the same step captured once into a CUDA graph and replayed (the C ABI
    # only enqueues work on the caller's stream, so a whole step captures)
    side = torch.cuda.Stream(device=dev)
    side.wait_stream(stream)
    with torch.cuda.stream(side):
        step(inp["x"], inp["dY"])
    stream.wait_stream(side)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step(inp["x"], inp["dY"])
    graph.replay()
    torch.cuda.synchronize()
    g0 = torch.cuda.Event(enable_timing=True)
    g1 = torch.cuda.Event(enable_timing=True)
    barrier(world)
    g0.record(stream)
    for _ in range(args.steps):
        graph.replay()
    g1.record(stream)
    torch.cuda.synchronize()
    graph_ms = max_over_ranks(g0.elapsed_time(g1), world) / args.steps
    assert layer.device_status("fwd") == 0 and layer.device_status("bwd") == 0

    fwd_fl, bwd_fl = layer_flops(sh)
    peaks = load_peaks()
    per_kernel, roof = summarize_kernels(prof_all, sh, peaks, clk, live=prof_live)

    tokens_per_s = world * sh.T / (ms_per_step * 1e-3)
    line = {
        "metric": METRIC,
        "value": tokens_per_s,
        "unit": "tokens/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": ms_per_step,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": {"bf16": "bf16", "mxfp8": "mxfp8 (e4m3 + e8m0 scales)",
                  "fp8_bwd": "bf16 fwd, mxfp8 bwd"}[sh.precision],
        "data": "synthetic (seeded N(0,1) activations, N(0,0.02) weights, random init)",
        "config": {"workload": sh.name, "T": sh.T, "H": sh.H, "F": sh.F, "E": sh.E,
                   "top_k": sh.top_k, "precision": sh.precision,
                   "parallelism": "replicas" if world > 1 else "single",
                   "flags": args.flags, "max_sms": args.max_sms,
                   "grad_accumulate_fp32": bool(args.accumulate),
                   "prepared_weights": (f"MXFP8 weights quantised once by moe_prepare_weights "
                                        f"({prepare_ms:.3f} ms, outside the step)"
                                        if prepare_ms is not None else False),
                   "l2": "inputs larger than L2 (no flush): weights and activations exceed 129 MB"},
        "tflops": world * (fwd_fl + bwd_fl) / (ms_per_step * 1e-3) / 1e12,
        "fwd_ms": fwd_ms,
        "bwd_ms": bwd_ms,
        "full_layer_ms": 2 * fwd_ms + bwd_ms,
        "full_layer_tflops": (2 * fwd_fl + bwd_fl) / ((2 * fwd_ms + bwd_ms) * 1e-3) / 1e12,
        "layer_frac_of_peak": layer_peak_frac(sh, ms_per_step, peaks, clk),
        "clocks": clk,
        "e2e": {"value": world * sh.T / (e2e_ms * 1e-3), "unit": "tokens/s",
                "h2d_bytes_per_step": 2 * hx.numel() * 2, "d2h_bytes_per_step": 2 * hx.numel() * 2,
                "copies": "pinned host memory, side stream, double-buffered across steps"},
        "graph": {"ms_per_step": graph_ms, "value": world * sh.T / (graph_ms * 1e-3),
                  "unit": "tokens/s", "note": "one fwd+bwd step captured in a CUDA graph, replayed"},
        "gpu_launches": launches,
        "roofline": roof,
        "kernels": per_kernel,
        "kernels_note": (f"launches, mean times and shares from a pass of {min(args.steps, 10)} "
                         f"steps with events around every launch, just before the timed region; "
                         f"{dom}'s avg_ms from its launches inside the timed region"),
    }
    if world == 1 and not args.no_configs and args.shape is None:
        line["configs"] = run_configs(args, dev, peaks)
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(sh, inp, args.cpu_budget)
    return line


# ------------------------------------------------------------------ the other workloads

# Every Qwen3-shaped workload besides the headline one, timed in the same
# process after it: (workload, weights quantised once by moe_prepare_weights)
CONFIG_RUNS = [("qwen3_30b", False), ("qwen3_30b_skew", False), ("qwen3_235b_mxfp8", False),
               ("qwen3_235b_mxfp8", True), ("qwen3_235b_fp8_bwd", False),
               ("qwen3_235b_mxfp8_skew", False)]


def time_config(name, prepared, dev, steps, warmup, peaks, flags, max_sms):
    """W warm-up steps, then K timed fwd+bwd steps of one workload (inputs
    resident in HBM), the dominant kernel's launches timed live (every launch
    profiled in a short pass before); returns the
    workload's entry of the ``configs`` object."""
    from mixture_experts_layer_17_gb300 import (MoeLayer, moe_profile_enable, moe_profile_read,
                                                moe_profile_select)
    sh = si.shape(name)
    inp = si.make_inputs(sh, dev)
    layer = MoeLayer(sh.T, sh.H, sh.F, sh.E, sh.top_k, sh.precision, flags=flags, device=dev,
                     max_sms=max_sms)
    W = (inp["W_r"], inp["W_gate"], inp["W_up"], inp["W_down"])
    grads = {"dx": torch.empty_like(inp["x"]), "dW_r": torch.empty_like(W[0]),
             "dW_gate": torch.empty_like(W[1]), "dW_up": torch.empty_like(W[2]),
             "dW_down": torch.empty_like(W[3])}
    y = torch.empty_like(inp["x"])
    prepare_ms = None
    if prepared:
        layer.prepare_weights(W[1], W[2], W[3])
        torch.cuda.synchronize()
        p0, p1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        p0.record()
        layer.prepare_weights(W[1], W[2], W[3])
        p1.record()
        torch.cuda.synchronize()
        prepare_ms = p0.elapsed_time(p1)
    def step(x, dY):
        layer.forward(x, *W, inp["logit_bias"], y=y)
        layer.backward(x, *W, dY, grads=grads)

    for _ in range(warmup):
        step(inp["x"], inp["dY"])
    torch.cuda.synchronize()
    # every launch profiled in a short pass; only the dominant kernel's
    # launches timed inside the timed region (as for the headline workload)
    prof_all = profile_pass(step, inp, min(steps, 5))
    dom = dominant_kernel(prof_all)
    stream = torch.cuda.current_stream()
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(steps)]
    clocks = ClockSampler(dev.index or 0)
    moe_profile_read()
    moe_profile_select(dom)
    moe_profile_enable(True)
    clocks.start()
    time.sleep(0.5)
    for i in range(steps):
        ev[i][0].record(stream)
        layer.forward(inp["x"], *W, inp["logit_bias"], y=y)
        ev[i][1].record(stream)
        layer.backward(inp["x"], *W, inp["dY"], grads=grads)
        ev[i][2].record(stream)
    torch.cuda.synchronize()
    clk = clocks.stop()
    moe_profile_enable(False)
    moe_profile_select(None)
    prof_live = moe_profile_read()
    assert layer.device_status("fwd") == 0 and layer.device_status("bwd") == 0
    total = ev[0][0].elapsed_time(ev[-1][2])
    ms = total / steps
    fwd_ms = statistics.median(e[0].elapsed_time(e[1]) for e in ev)
    bwd_ms = statistics.median(e[1].elapsed_time(e[2]) for e in ev)
    fwd_fl, bwd_fl = layer_flops(sh)
    per_kernel, roof = summarize_kernels(prof_all, sh, peaks, clk, live=prof_live)
    out = {"workload": name, "precision": sh.precision, "T": sh.T, "H": sh.H, "F": sh.F,
           "E": sh.E, "top_k": sh.top_k, "steps": steps, "warmup": warmup,
           "ms_per_step": ms, "tokens_per_s": sh.T / (ms * 1e-3),
           "tflops": (fwd_fl + bwd_fl) / (ms * 1e-3) / 1e12,
           "fwd_ms": fwd_ms, "bwd_ms": bwd_ms, "full_layer_ms": 2 * fwd_ms + bwd_ms,
           "full_layer_tflops": (2 * fwd_fl + bwd_fl) / ((2 * fwd_ms + bwd_ms) * 1e-3) / 1e12,
           "layer_frac_of_peak": layer_peak_frac(sh, ms, peaks, clk),
           "dominant_kernel": {k: roof[k] for k in ("kernel", "bound", "achieved", "peak",
                                                     "unit", "frac", "peak_source")},
           "clocks": clk,
           "kernels": {k: {"avg_ms": v["avg_ms"], "share": v["share"],
                           **({"frac_of_peak": v["frac_of_peak"]} if "frac_of_peak" in v else {}),
                           **({"frac_hbm": v["frac_hbm"]} if "frac_hbm" in v else {})}
                       for k, v in per_kernel.items()}}
    if prepared:
        out["prepared_weights"] = (f"MXFP8 weights quantised once by moe_prepare_weights "
                                   f"({prepare_ms:.3f} ms, outside the step)")
    if sh.skew:
        c = layer.route(inp["x"], W[0], inp["logit_bias"], with_logits=False)["counts"]
        c = c.double().cpu()
        out["expert_load"] = {"zero_experts": int((c == 0).sum()),
                              "max_over_mean": float(c.max() / c.mean()),
                              "min_over_mean": float(c.min() / c.mean())}
    del layer, inp, grads, y
    torch.cuda.empty_cache()
    return out


def run_configs(args, dev, peaks):
    """The ``configs`` object: every other Qwen3-shaped workload."""
    out = {"tiny": "parity case only (T=128, H=256, F=128, E=8, top-2): its fp32 draws are "
                   "rounded to bf16 for the GPU, and it is compared with the oracle element by "
                   "element in the tests, not timed"}
    for name, prepared in CONFIG_RUNS:
        key = name + ("_prepared" if prepared else "")
        out[key] = time_config(name, prepared, dev, args.config_steps, 3, peaks, args.flags,
                               args.max_sms)
    return out


# ------------------------------------------------------------------ reference arm

# seconds of oracle work the K timed steps of the reference arm share
REF_BUDGET_S = 150.0


def run_reference(args, sh, world, rank):
    """The CPU oracle timed on the host cores, each step a bounded sample.

    The oracle's cost per call is a fixed part (every expert a sample touches
    has its weights widened to fp64 and its weight-gradient blocks formed)
    plus a part linear in the tokens.  Two probe calls fit that cost, and each
    timed step then runs the largest sample whose predicted time is its share
    of REF_BUDGET_S (4 to 30 s), so the fixed part is amortised as it is in
    the cpu_baseline leg.  The W warm-up steps (untimed) run 8 tokens."""
    if rank != 0:
        return None
    inp = si.make_inputs(sh, "cpu")
    inp_cpu = host_copy_for_oracle(inp)
    n1, n2 = min(64, sh.T), min(256, sh.T)
    t1 = oracle_sample_time(sh, inp_cpu, n1)
    t2 = oracle_sample_time(sh, inp_cpu, n2)
    per_tok = max((t2 - t1) / (n2 - n1), 1e-6) if n2 > n1 else t2 / n2
    fixed = max(t1 - n1 * per_tok, 0.0)
    per_step = min(30.0, max(4.0, REF_BUDGET_S / max(1, args.steps)))
    n = max(8, min(sh.T, int((per_step - fixed) / per_tok)))
    for _ in range(args.warmup):
        oracle_sample_time(sh, inp_cpu, min(8, sh.T))
    times = [oracle_sample_time(sh, inp_cpu, n) for _ in range(args.steps)]
    sec = sum(times) / len(times)
    value = n / sec
    sample = (f"first {n} of {sh.T} tokens of {sh.name} per timed step: route + fwd + full "
              f"bwd, numpy fp64 (sample sized from probe calls on {n1} and {n2} tokens: "
              f"{fixed:.2f} s fixed + {per_tok * 1e3:.2f} ms per token)")
    return {
        "impl": "reference",
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": sec * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": {"workload": sh.name, "T": sh.T, "H": sh.H, "F": sh.F,
                                        "E": sh.E, "top_k": sh.top_k, "precision": sh.precision},
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": blas_threads(),
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=60)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(si.WORKLOADS))
    ap.add_argument("--flags", type=lambda v: int(v, 0), default=0,
                    help="moe_config_t flags (e.g. 0x4: single-CTA tiles only; 0x8: CTA pairs)")
    ap.add_argument("--shape", default=None,
                    help="T,H,F,E,top_k: a custom shape (profiling aid) instead of --workload")
    ap.add_argument("--precision", default="bf16", choices=["bf16", "mxfp8", "fp8_bwd"],
                    help="precision of a --shape layer")
    ap.add_argument("--accumulate", action="store_true",
                    help="backward adds the weight gradients into fp32 buffers")
    ap.add_argument("--max-sms", type=int, default=0, help="SM budget (0: every SM)")
    ap.add_argument("--prepared-weights", action="store_true",
                    help="MXFP8: quantise the weights once before the timed steps")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-configs", action="store_true",
                    help="skip the other Qwen3-shaped workloads (the configs object)")
    ap.add_argument("--config-steps", type=int, default=10,
                    help="timed steps of each workload in the configs object")
    ap.add_argument("--cpu-budget", type=float, default=30.0)
    ap.add_argument("--record-traffic", default=None, metavar="NCU_CSV",
                    help="store per-launch DRAM bytes from an ncu CSV for --workload and exit")
    ap.add_argument("--traffic-command", default="",
                    help="the ncu command line the CSV came from (stored beside the figures)")
    ap.add_argument("--traffic-scale", type=float, default=1.0,
                    help="scale a smaller capture's bytes to --workload (ratio of the units)")
    ap.add_argument("--traffic-captured-on", default=None,
                    help="the shape the capture was taken on, when it is not --workload")
    args = ap.parse_args()
    if args.record_traffic:
        print(json.dumps(record_traffic(args.record_traffic, args.workload, args.traffic_command,
                                        scale=args.traffic_scale,
                                        captured_on=args.traffic_captured_on)))
        return
    args.warmup = max(args.warmup, 3)
    if args.shape:
        T, H, F, E, k = (int(v) for v in args.shape.split(","))
        sh = si.custom_shape(T, H, F, E, k, seed=5, precision=args.precision,
                             name=f"custom_{T}x{H}x{F}x{E}x{k}_{args.precision}")
    else:
        sh = si.shape(args.workload)
    world, rank, local = dist_setup(args)
    if args.impl == "reference":
        line = run_reference(args, sh, world, rank)
    else:
        line = run_ours(args, sh, world, rank, local)
    if rank == 0 and line is not None:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
