#!/usr/bin/env python
"""Benchmark of one Beam MoE block forward pass on B300 (tokens/s and roofline fraction).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload decode|prefill|skewed]
                    [--impl ours|reference]

A step is one moe_forward call (router -> permute -> expert GEMM1+SwiGLU ->
expert GEMM2 -> combine) over one batch of seeded synthetic inputs with the
Beam layer's shapes (release article, section "Mixture of Experts": 256
experts in 8 groups of 32, top-4 groups, top-8 experts, SwiGLU 5120 -> 2560 ->
5120, combine x2.5). Random-init weights (no checkpoint). Prints one JSON line.

Under torchrun (N > 1) every rank runs an independent replica of the layer on
its own batch (the block has no cross-token exchange on one GPU's data), so
the work per GPU is fixed: weak scaling, no data-path collective.

--impl reference times the CPU oracle (plain C, fp64) on the host cores on a
bounded sample of the same workload; it exists to be compared against.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workload as W  # noqa: E402  (seeded input generators only)

METRIC = "MoE-layer tokens/s at Beam shape (T=64 decode, T=4096 prefill); % of roofline"


ROUTE_TICKETS = 192  # groups of 8 tokens whose selection the SIMT logits kernel can run itself


def simt_router_kernels(T, E):
    """Kernels of the library's SIMT router (router.cu): the logits kernel (which also selects
    while ceil(T/64) * 8 <= ROUTE_TICKETS), a selection kernel otherwise, and a W_r padding copy
    when E is not a multiple of 4."""
    return 1 + (0 if -(-T // 64) * 8 <= ROUTE_TICKETS else 1) + (1 if E % 4 else 0)


ROUTER_TC_MIN_TOKENS = 1024  # the library routes batches this large on the tensor cores


def permute_uses_plan_kernel(T, E):
    """The library's small-batch permutation rule (permute.cu): one plan kernel when the token x
    expert bitmap (E * ceil(T/32) words) fits in 8192 words of shared memory."""
    return E <= 256 and E * ((T + 31) // 32) <= 8192


def kernels_per_step(cfg, num_sms):
    """Kernels one moe_forward launches: router (tensor-core: W_r split, tensor-core logits,
    selection, narrow-margin recompute (logits + selection); SIMT: logits with the selection,
    see simt_router_kernels), permutation (small batches: plan kernel, which also builds the GEMM
    schedule, + gather; otherwise bitmap, column scan, offsets (which also builds the schedule),
    gather), GEMM1, GEMM2, combine."""
    if cfg.T >= ROUTER_TC_MIN_TOKENS:
        router = 5
    else:
        router = simt_router_kernels(cfg.T, cfg.E)
    permute_and_schedule = 2 if permute_uses_plan_kernel(cfg.T, cfg.E) else 4
    return router + permute_and_schedule + 2 + 1


def max_over_ranks(value, world, device):
    """Max of a float over all ranks (the job is as slow as its slowest rank)."""
    if world <= 1:
        return float(value)
    import torch
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())

# small cases of the same kernels, sized for ncu captures (a few GB on the device)
PROFILE_CASES = {
    "profile_decode": W.MoEConfig("profile_decode", T=8, d=5120, E=32, n_groups=8, topk_groups=4, top_k=8, inter=2560),
    "profile_prefill": W.MoEConfig("profile_prefill", T=512, d=5120, E=32, n_groups=8, topk_groups=4, top_k=8,
                                   inter=2560),
    # ~1024 tokens per expert, like the skewed workload's compute-bound tiles
    "profile_dense": W.MoEConfig("profile_dense", T=2048, d=5120, E=16, n_groups=4, topk_groups=4, top_k=8,
                                 inter=2560),
    # the NVFP4 prefill shape with 32 experts (0.7 GB of NVFP4 weights)
    "profile_nvfp4": W.MoEConfig("profile_nvfp4", T=512, d=5120, E=32, n_groups=8, topk_groups=4, top_k=8,
                                 inter=2560, wfmt="nvfp4"),
    # the FP8 prefill shape with 32 experts (1.3 GB of FP8 weights)
    "profile_fp8": W.MoEConfig("profile_fp8", T=512, d=5120, E=32, n_groups=8, topk_groups=4, top_k=8,
                               inter=2560, wfmt="fp8"),
    # the router, permutation and combine of the decode and prefill workloads exactly (d = 5120, 256
    # experts in 8 groups of 32, top-4 groups, top-8) with a 64-wide intermediate, so the experts
    # hold 0.5 GB instead of 20 GB: for captures of the small stages
    "profile_stages_decode": W.MoEConfig("profile_stages_decode", T=64, d=5120, E=256, n_groups=8, topk_groups=4,
                                         top_k=8, inter=64),
    "profile_stages_prefill": W.MoEConfig("profile_stages_prefill", T=4096, d=5120, E=256, n_groups=8,
                                          topk_groups=4, top_k=8, inter=64),
}

# Dense SwiGLU MLP of the first decoder layers. The pages give no intermediate size for them;
# 20480 = 8 x 2560 gives the dense FFN the per-token work of the 8 routed experts.
DENSE_CASES = {
    "dense_prefill": W.MoEConfig("dense_prefill", T=4096, d=5120, E=1, n_groups=1, topk_groups=1, top_k=1,
                                 inter=20480),
}

RESIDUAL_STEP = 10  # the residual-addition index k used with --residual (weights sqrt(9/10), 1/sqrt(10))

DEFAULT_STEPS = {"dense_prefill": 100, "decode": 300, "prefill": 200, "skewed": 40, "nvfp4": 200, "fp8": 200,
                 "profile_decode": 20, "profile_prefill": 20, "profile_dense": 20, "profile_nvfp4": 20,
                 "profile_fp8": 20, "profile_stages_decode": 20, "profile_stages_prefill": 20}


def workload_cfg(name):
    if name in W.CONFIGS:
        return W.CONFIGS[name]
    return PROFILE_CASES[name] if name in PROFILE_CASES else DENSE_CASES[name]


def describe(cfg):
    s = (f"{cfg.name}: T={cfg.T} tokens, d={cfg.d}, E={cfg.E} experts in {cfg.n_groups} groups of "
         f"{cfg.E // cfg.n_groups}, top-{cfg.topk_groups} groups, top-{cfg.top_k} experts, SwiGLU inter={cfg.inter}, "
         f"{cfg.wfmt} expert weights, fp32 router, combine x{cfg.routed_scale}")
    if cfg.skew:
        s += ", 16 hot experts at ~4x mean load"
    return s


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return {"hbm_gbs": d["hbm_gbs"], "bf16_tflops": d["bf16_tflops"],
                "bf16_tflops_sustained": d.get("bf16_tflops_sustained"), "source": "measured"}
    return {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0, "source": "fallback"}


def profiled_traffic(workload, kernel, algorithmic_bytes):
    """DRAM bytes of one launch of `kernel`, from the committed ncu capture of the small case that
    stands for `workload`, scaled by algorithmic bytes (weights of touched experts + activations);
    None when the kernel's sources changed since the capture."""
    import hashlib
    p = os.path.join(ROOT, "profiles", "dram_traffic.json")
    if not os.path.exists(p):
        return None, "no capture"
    rec = json.load(open(p))
    cap_name = rec.get("capture_for_workload", {}).get(workload)
    cap = rec.get("captures", {}).get(cap_name) if cap_name else None
    k = cap["kernels"].get(kernel) if cap else None
    if not k:
        return None, "no capture"
    h = hashlib.sha256()
    for src in rec["sources"]:
        h.update(open(os.path.join(ROOT, src), "rb").read())
    if h.hexdigest() != rec["source_sha256"]:
        return None, "kernel changed since the capture"
    measured = k["dram_bytes_read"] + k["dram_bytes_write"]
    return int(round(measured * algorithmic_bytes / k["algorithmic_bytes"])), (
        f"ncu dram__bytes_read+write of {cap_name} ({cap['workload']}), scaled by algorithmic bytes")


# kernel names in ncu's launch list -> the names bench.py reports (template <GLU, format>)
NCU_GEMM_NAMES = {"<1, 0>": "expert_gemm_kernel<GLU>", "<0, 0>": "expert_gemm_kernel<plain>",
                  "<1, 1>": "expert_gemm_kernel<GLU, NVFP4>", "<0, 1>": "expert_gemm_kernel<plain, NVFP4>",
                  "<1, 2>": "expert_gemm_kernel<GLU, FP8>", "<0, 2>": "expert_gemm_kernel<plain, FP8>"}
TRAFFIC_SOURCES = ["sparse_moe_layer_14_b300/csrc/expert_gemm.cu", "sparse_moe_layer_14_b300/csrc/common.cuh",
                   "sparse_moe_layer_14_b300/csrc/schedule.cuh"]
TRAFFIC_CAPTURES = {"decode": "profile_decode", "prefill": "profile_prefill", "skewed": "profile_dense",
                    "nvfp4": "profile_nvfp4", "fp8": "profile_fp8"}


def parse_ncu_csv(path):
    """ncu --csv --log-file output -> list of (kernel name, {metric: value in base units}) per launch."""
    import csv
    rows = [r for r in csv.reader(open(path)) if r]
    hi = next(i for i, r in enumerate(rows) if r[0] == "ID")
    hdr = rows[hi]
    ki, mi, ni, ui = (hdr.index(c) for c in ("Kernel Name", "Metric Value", "Metric Name", "Metric Unit"))
    scale = {"byte": 1, "Kbyte": 1e3, "Mbyte": 1e6, "Gbyte": 1e9, "ns": 1, "us": 1e3, "usecond": 1e3, "ms": 1e6,
             "msecond": 1e6, "nsecond": 1}
    launches = {}
    for r in rows[hi + 1:]:
        if len(r) <= mi:
            continue
        d = launches.setdefault(r[0], [r[ki], {}])
        d[1][r[ni]] = float(r[mi].replace(",", "")) * scale.get(r[ui], 1)
    return [tuple(v) for _, v in sorted(launches.items(), key=lambda kv: int(kv[0]))]


def record_traffic(directory, out=None):
    """Write profiles/dram_traffic.json from captures in `directory`: for every small case named in
    TRAFFIC_CAPTURES, <case>.json (its plain bench line: experts touched) and <case>.csv (ncu
    --metrics dram__bytes_read.sum,dram__bytes_write.sum,gpu__time_duration.sum over its GEMM1 and
    GEMM2 launches). Algorithmic bytes per launch are this file's roofline_numbers for the case."""
    import hashlib
    peaks = load_peaks()
    rec = {"sources": TRAFFIC_SOURCES, "note": "DRAM bytes of one launch from ncu on one B300; bench.py scales "
           "them to its workload by algorithmic bytes", "capture_for_workload": {}, "captures": {}}
    h = hashlib.sha256()
    for src in TRAFFIC_SOURCES:
        h.update(open(os.path.join(ROOT, src), "rb").read())
    rec["source_sha256"] = h.hexdigest()
    for workload, case in TRAFFIC_CAPTURES.items():
        jpath, cpath = os.path.join(directory, case + ".json"), os.path.join(directory, case + ".csv")
        if not (os.path.exists(jpath) and os.path.exists(cpath)):
            continue
        line = json.loads(open(jpath).read().strip().splitlines()[-1])
        cfg = workload_cfg(case)
        touched = line["layer_roofline"]["experts_touched"]
        g1, g2, _ = roofline_numbers(cfg, touched, peaks)
        kernels = {}
        for name, m in parse_ncu_csv(cpath):
            tmpl = (name[name.index("<", name.index("expert_gemm_kernel")):name.index(">", name.index("expert_gemm_kernel")) + 1]
                    if "expert_gemm_kernel" in name else None)
            if tmpl not in NCU_GEMM_NAMES:
                continue
            kname = NCU_GEMM_NAMES[tmpl]
            kernels[kname] = {"dram_bytes_read": int(m["dram__bytes_read.sum"]),
                              "dram_bytes_write": int(m["dram__bytes_write.sum"]),
                              "algorithmic_bytes": int((g1 if "GLU" in kname else g2)["bytes"]),
                              "gpu_time_ns_serialised": int(m["gpu__time_duration.sum"])}
        rec["captures"][case] = {"workload": describe(cfg), "experts_touched": touched, "kernels": kernels,
                                 "command": f"ncu --metrics dram__bytes_read.sum,dram__bytes_write.sum,"
                                            f"gpu__time_duration.sum --clock-control none -k regex:expert_gemm_kernel "
                                            f"-s 6 -c 2 --csv python bench.py --workload {case} --steps 2 --warmup 3 "
                                            f"--no-cpu-baseline"}
        rec["capture_for_workload"][workload] = case
        rec["capture_for_workload"][case] = case
    out = out or os.path.join(ROOT, "profiles", "dram_traffic.json")
    json.dump(rec, open(out, "w"), indent=1)
    return out


# ----------------------------------------------------------------------------- clocks

class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons, kept with timestamps."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, index=0, period_ms=50):
        self.samples = []
        self.proc = None
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(index), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", f"-lms={period_ms}"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except (OSError, FileNotFoundError):
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) >= 7:
                self.samples.append((time.time(), parts))

    def stop(self):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self, t0, t1):
        inside = [p for (t, p) in self.samples if t0 <= t <= t1]
        window = "timed region"
        if not inside:  # region shorter than the sampling period: take the nearest samples
            near = sorted(self.samples, key=lambda s: min(abs(s[0] - t0), abs(s[0] - t1)))[:3]
            inside = [p for (_, p) in near]
            window = "nearest samples (timed region shorter than the sampling period)"
        if not inside:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        sm = [num(p[0]) for p in inside if num(p[0]) is not None]
        reasons = set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for p in inside:
            for name, v in zip(names, p[3:7]):
                if v.strip().lower() in ("active", "1", "yes"):
                    reasons.add(name)
        return {"sm_mhz": float(np.median(sm)) if sm else None, "sm_max_mhz": num(inside[0][1]),
                "power_w_max": max((num(p[2]) or 0.0) for p in inside), "reasons": sorted(reasons),
                "samples": len(inside), "window": window}


# ----------------------------------------------------------------------------- ours

def make_device_weights(cfg, seed, torch, keep_host):
    """Seeded expert weights generated expert by expert on the host and copied to the device
    (NVFP4, FP8: quantised from the same seeded bf16 draws)."""
    import sparse_moe_layer_14_b300 as bm
    host = {}
    tens = {}
    if cfg.wfmt == "fp8":
        for which in ("gate", "up", "down"):
            codes, scales = W.gen_expert_fp8(cfg, seed, which, 0, cfg.E)
            tens[which] = torch.from_numpy(codes).cuda()
            tens[which + "_sf"] = torch.from_numpy(scales).cuda()
            if keep_host:
                host[which], host[which + "_sf"] = codes, scales
        return bm.ExpertWeights(**tens), host
    if cfg.wfmt == "nvfp4":
        for which in ("gate", "up", "down"):
            p, s, ts = W.gen_expert_nvfp4(cfg, seed, which, 0, cfg.E)
            tens[which] = torch.from_numpy(p).cuda()
            tens[which + "_sf"] = torch.from_numpy(s).cuda()
            tens[which + "_ts"] = torch.from_numpy(ts).cuda()
            if keep_host:
                host[which], host[which + "_sf"], host[which + "_ts"] = p, s, ts
        return bm.ExpertWeights(**tens), host
    for which in ("gate", "up", "down"):
        N_, K_ = W.weight_shape(cfg, which)
        t = torch.empty((cfg.E, N_, K_), dtype=torch.bfloat16, device="cuda")
        h = np.empty((cfg.E, N_, K_), np.uint16) if keep_host else None
        step = max(1, (1 << 28) // (N_ * K_))
        buf = torch.empty((step, N_, K_), dtype=torch.int16).pin_memory()
        for e0 in range(0, cfg.E, step):
            e1 = min(cfg.E, e0 + step)
            chunk = buf[: e1 - e0].numpy().view(np.uint16)
            W.gen_expert_bf16(cfg, seed, which, e0, e1, out=chunk)
            t[e0:e1].copy_(buf[: e1 - e0].view(torch.bfloat16))
            if keep_host:
                h[e0:e1] = chunk
        tens[which] = t
        if keep_host:
            host[which] = h
    return bm.ExpertWeights(tens["gate"], tens["up"], tens["down"]), host


def weight_bytes_per_param(cfg):
    """bf16: 2 B; NVFP4: 0.5 B of e2m1 code + 1/16 B of e4m3 block scale; FP8: 1 B of e4m3
    code + 4 B of fp32 scale per 128 x 128 block."""
    return {"bf16": 2.0, "nvfp4": 0.5 + 1.0 / 16, "fp8": 1.0 + 4.0 / (128 * 128)}[cfg.wfmt]


def roofline_numbers(cfg, touched, peaks):
    """Algorithmic bytes and FLOPs of the layer and of each expert GEMM launch."""
    R = cfg.T * cfg.top_k
    d, I, E = cfg.d, cfg.inter, cfg.E
    bpp = weight_bytes_per_param(cfg)
    w_bytes_expert = 3 * d * I * bpp
    gemm1 = {"bytes": touched * 2 * I * d * bpp + R * d * 2 + R * I * 2, "flops": 2.0 * R * d * 2 * I}
    gemm2 = {"bytes": touched * d * I * bpp + R * I * 2 + R * d * 4, "flops": 2.0 * R * I * d}
    layer = {"bytes": touched * w_bytes_expert + d * E * 4 + cfg.T * d * 2 * 2,
             "flops": 2.0 * R * 3 * d * I + 2.0 * cfg.T * d * E}
    for x in (gemm1, gemm2, layer):
        t_mem = x["bytes"] / (peaks["hbm_gbs"] * 1e9)
        t_flop = x["flops"] / (peaks["bf16_tflops"] * 1e12)
        x["bound"] = "hbm" if t_mem >= t_flop else "tensor"
        x["t_roof_s"] = max(t_mem, t_flop)
    return gemm1, gemm2, layer


# FP32 FFMA peak of the SIMT router: 148 SMs x 128 FP32 lanes x 2 FLOP x 2.032 GHz (maximum SM clock)
FP32_ALU_TFLOPS = 148 * 128 * 2 * 2.032e9 / 1e12


def stage_rooflines(cfg, stage_ms, peaks, residual=False):
    """Achieved HBM bandwidth of the router, permute and combine stages from their algorithmic bytes
    and live durations (ms), and the router's FP32 rate against the FFMA peak.
    router: x read, W_r read once, indices and weights written;
    permute: indices read, x read once, x_perm and the two row maps written, counts and offsets;
    combine: the K FP32 expert rows of every token, its weights and rows read, out written (with
    the residual update also the stream read and the gain)."""
    T, d, E, K = cfg.T, cfg.d, cfg.E, cfg.top_k
    R = T * K
    by = {"router": T * d * 2 + d * E * 4 + R * 8,
          "permute": R * 4 + T * d * 2 + R * d * 2 + R * 8 + (2 * E + 1) * 4,
          "combine": R * d * 4 + R * 8 + T * d * 2 + ((T * d * 2 + d * 2) if residual else 0)}
    ms = {"router": stage_ms[0], "permute": stage_ms[1], "combine": stage_ms[4]}
    out = {}
    for k in by:
        gbs = by[k] / (ms[k] / 1e3) / 1e9 if ms[k] > 0 else None
        out[k] = {"bytes": int(by[k]), "ms": round(float(ms[k]), 4),
                  "achieved_gbs": None if gbs is None else round(gbs, 1),
                  "frac_hbm": None if gbs is None else round(gbs / peaks["hbm_gbs"], 4)}
    if ms["router"] <= 0:
        return out
    tf = 2.0 * T * d * E / (ms["router"] / 1e3) / 1e12
    out["router"]["achieved_fp32_tflops"] = round(tf, 2)
    if T >= ROUTER_TC_MIN_TOKENS:  # logits on the tensor cores (three exact bf16 terms of W_r)
        out["router"]["path"] = "tensor cores + fp32 recompute of narrow-margin tokens"
    else:
        out["router"]["path"] = "fp32 simt"
        out["router"]["frac_fp32_alu"] = round(tf / FP32_ALU_TFLOPS, 4)
    return out


def measure_block(args, cfg, weights, host_w, rank, world, local_rank, peaks, want_cpu, x_h, wr_h):
    """Time moe_forward (or the residual / sublayer variants) on one batch of `cfg` with the
    expert weights already resident: W warm-up steps, K timed steps between barriers, stage
    events, clocks, the end-to-end run with host copies, and (rank 0, one GPU) the oracle on a
    token sample with its parity against this run's output. Returns the JSON record (rank 0)."""
    import torch
    import sparse_moe_layer_14_b300 as bm

    dims = bm.Dims.from_config(cfg)
    x = torch.from_numpy(x_h).view(torch.int16).view(torch.bfloat16).cuda()
    w_r = torch.from_numpy(wr_h).cuda()
    out = torch.empty((cfg.T, cfg.d), dtype=torch.bfloat16, device="cuda")
    counts = torch.empty(cfg.E, dtype=torch.int32, device="cuda")
    ws = bm.allocate_workspace(dims)
    stream = torch.cuda.current_stream()

    gain = pre_gain = None
    if args.sublayer:
        args.residual = True
        pre_gain = (1.0 + 0.05 * torch.randn(cfg.d, generator=torch.Generator().manual_seed(args.seed + 2))).to(
            torch.bfloat16).cuda()
    if args.residual:  # post-norm gain ~ 1 and a unit-RMS residual stream, updated in place each step
        gain = (1.0 + 0.05 * torch.randn(cfg.d, generator=torch.Generator().manual_seed(args.seed))).to(
            torch.bfloat16).cuda()
        out.copy_(torch.randn((cfg.T, cfg.d), generator=torch.Generator().manual_seed(args.seed + 1)).to(
            torch.bfloat16))

    def forward(x_, out_, counts_=None, idx_=None):
        if args.sublayer:  # x_ is the residual stream (updated in place), out_ the pre-norm output
            bm.moe_sublayer(dims, x_, pre_gain, gain, 1e-6, RESIDUAL_STEP, w_r, weights, out_, ws, counts=counts_)
        elif args.residual:
            bm.moe_forward_residual(dims, x_, w_r, weights, gain, 1e-6, RESIDUAL_STEP, out_, ws, counts=counts_)
        else:
            bm.moe_forward(dims, x_, w_r, weights, out_, ws, counts=counts_, topk_idx=idx_)

    def step():
        forward(x, out, counts)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    if bm.moe_get_device_status(ws) != bm.MOE_DEV_OK:
        raise RuntimeError("device status set during warm-up")

    K = args.steps
    ev_sets = [[torch.cuda.Event(enable_timing=True) for _ in range(6)] for _ in range(K)]
    for evs in ev_sets:  # create the CUDA handles before the timed region
        for ev in evs:
            ev.record(stream)
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    clocks = ClockSampler(local_rank) if rank == 0 else None
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    # timed region: K steps back to back (the block's kernels launch with programmatic
    # dependencies, so nothing is recorded between them here)
    wall0 = time.time()
    start.record(stream)
    for i in range(K):
        step()
    end.record(stream)
    torch.cuda.synchronize()
    wall1 = time.time()
    if world > 1:
        torch.distributed.barrier()
    elapsed_ms = max_over_ranks(start.elapsed_time(end), world, "cuda")
    # stage-timed region: K more steps with a CUDA event recorded on the stream between stages
    # (router, permutation with the GEMM schedule, GEMM1, GEMM2, combine); the events serialise the launches
    # at the stage boundaries, so these times are an upper bound on each stage's share
    for i in range(K):
        bm.moe_set_stage_events(ev_sets[i])
        step()
    torch.cuda.synchronize()
    wall2 = time.time()
    bm.moe_set_stage_events(None)
    stage_ms = np.zeros(5)
    for evs in ev_sets:
        stage_ms += np.array([evs[j].elapsed_time(evs[j + 1]) for j in range(5)])
    stage_ms /= K
    staged_step_ms = float(np.mean([evs[0].elapsed_time(evs[5]) for evs in ev_sets]))
    if bm.moe_get_device_status(ws) != bm.MOE_DEV_OK:
        raise RuntimeError("device status set during the timed region")
    clk = clocks.summary(wall0, wall1) if clocks else None
    clk_staged = clocks.summary(wall1, wall2) if clocks else None
    recomputed = int(ws[16:20].view(torch.int32).item()) if cfg.T >= ROUTER_TC_MIN_TOKENS else None

    # end to end through the public API: every step copies its x from pinned host memory to the
    # device, runs moe_forward and copies its output back to pinned host memory. The copies run on
    # a second stream, double-buffered, so step i+1's input and step i-1's output move while step
    # i computes (as a serving loop would); the timed region spans the first copy to the last.
    x_pin = torch.from_numpy(x_h).view(torch.int16).pin_memory()
    out_pin = [torch.empty((cfg.T, cfg.d), dtype=torch.int16).pin_memory() for _ in range(2)]
    x_dev = [torch.empty((cfg.T, cfg.d), dtype=torch.bfloat16, device="cuda") for _ in range(2)]
    out_dev = [out.clone() for _ in range(2)]  # (with --residual: the residual stream, updated in place)
    copy_stream = torch.cuda.Stream()

    def e2e_run(n):
        h2d = [torch.cuda.Event() for _ in range(2)]
        fwd = [torch.cuda.Event() for _ in range(2)]
        d2h = [torch.cuda.Event() for _ in range(2)]
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(copy_stream):
            t0.record(copy_stream)
            x_dev[0].view(torch.int16).copy_(x_pin, non_blocking=True)
            h2d[0].record(copy_stream)
        for i in range(n):
            b = i % 2
            stream.wait_event(h2d[b])
            if i >= 2:
                stream.wait_event(d2h[b])  # out_dev[b] was read back
            forward(x_dev[b], out_dev[b])
            fwd[b].record(stream)
            with torch.cuda.stream(copy_stream):
                if i + 1 < n:
                    if i >= 1:
                        copy_stream.wait_event(fwd[1 - b])  # x_dev[1-b] was read by step i-1
                    x_dev[1 - b].view(torch.int16).copy_(x_pin, non_blocking=True)
                    h2d[1 - b].record(copy_stream)
                copy_stream.wait_event(fwd[b])
                res_b = x_dev[b] if args.sublayer else out_dev[b]  # the step's result
                out_pin[b].copy_(res_b.view(torch.int16), non_blocking=True)
                d2h[b].record(copy_stream)
        with torch.cuda.stream(copy_stream):
            t1.record(copy_stream)
        return t0, t1

    e2e_run(max(2, args.warmup))
    torch.cuda.synchronize()
    e0, e1 = e2e_run(K)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(e0.elapsed_time(e1), world, "cuda")
    if clocks:
        clocks.stop()

    c = counts.cpu().numpy()
    touched = int((c > 0).sum())
    g1, g2, layer = roofline_numbers(cfg, touched, peaks)
    ms_per_step = elapsed_ms / K
    tokens_per_s = world * cfg.T / (ms_per_step / 1e3)
    if rank != 0:
        return None

    gemm1_s = stage_ms[2] / 1e3
    bound = g1["bound"]
    if bound == "hbm":
        achieved, peak, unit = g1["bytes"] / gemm1_s / 1e9, peaks["hbm_gbs"], "GB/s"
    else:
        achieved, peak, unit = g1["flops"] / gemm1_s / 1e12, peaks["bf16_tflops"], "TFLOP/s"
    kname = {"bf16": "expert_gemm_kernel<GLU>", "nvfp4": "expert_gemm_kernel<GLU, NVFP4>",
             "fp8": "expert_gemm_kernel<GLU, FP8>"}[cfg.wfmt]
    traffic, traffic_src = profiled_traffic(cfg.name, kname, g1["bytes"])
    rec = {
        "metric": METRIC, "value": round(tokens_per_s, 1), "unit": "tokens/s", "n_gpus": world, "steps": K,
        "warmup": args.warmup, "ms_per_step": round(ms_per_step, 4), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16" if cfg.wfmt == "bf16" else f"bf16 ({cfg.wfmt.upper()} weights decoded to bf16)",
        "data": "synthetic (seeded N(0,1) activations, N(0,1/fan_in) weights)",
        "impl": "ours",
        "config": {"workload": describe(cfg), "T": cfg.T, "d": cfg.d, "E": cfg.E, "inter": cfg.inter,
                   "top_k": cfg.top_k, "parallelism": f"replicas x{world}",
                   "last_stage": (f"combine fused with post-norm (RMSNorm) and residual update, step k={RESIDUAL_STEP}"
                                  if args.residual else "combine to out"),
                   "first_stage": ("pre-norm (RMSNorm) of the residual stream" if args.sublayer else "router on x"),
                   "l2": f"no flush: {touched} experts x {3 * cfg.d * cfg.inter * weight_bytes_per_param(cfg) / 1e6:.1f} MB "
                         f"of weights streamed per step exceed the 126 MB L2"},
        "roofline": {"kernel": f"{kname} (GEMM1 + SwiGLU)", "bound": bound,
                     "achieved": round(achieved, 1), "peak": peak, "unit": unit, "frac": round(achieved / peak, 4),
                     "peak_source": f"{peaks['source']} ({'hbm_gbs' if bound == 'hbm' else 'bf16_tflops'})",
                     "traffic": traffic, "traffic_source": traffic_src, "algorithmic_bytes": g1["bytes"],
                     "algorithmic_flops": g1["flops"], "avg_launch_ms": round(stage_ms[2], 4),
                     "duration_from": "CUDA events on the launching stream around GEMM1 (the permutation builds "
                                      "the GEMM schedule), stage-timed pass"},
        "layer_roofline": {"bound": layer["bound"], "roofline_ms": round(layer["t_roof_s"] * 1e3, 4),
                           "frac": round(layer["t_roof_s"] * 1e3 / ms_per_step, 4),
                           "algorithmic_bytes": layer["bytes"], "algorithmic_flops": layer["flops"],
                           "experts_touched": touched},
        "stages_ms": {"router": round(stage_ms[0], 4), "permute": round(stage_ms[1], 4),
                      "gemm1": round(stage_ms[2], 4), "gemm2": round(stage_ms[3], 4),
                      "combine": round(stage_ms[4], 4), "step_with_stage_events": round(staged_step_ms, 4),
                      "how": "CUDA events between stages in a second timed pass of the same K steps (the "
                             "events serialise the launches at stage boundaries); clocks of that pass: "
                             + ("n/a" if not clk_staged else f"{clk_staged.get('sm_mhz')} MHz median, "
                                f"reasons {clk_staged.get('reasons')}")},
        "gemm2_roofline": {"bound": g2["bound"], "frac": round(g2["t_roof_s"] / (stage_ms[3] / 1e3), 4)},
        "stage_rooflines": stage_rooflines(cfg, stage_ms, peaks, residual=args.residual),
        "e2e": {"value": round(world * cfg.T / (e2e_ms / K / 1e3), 1), "unit": "tokens/s",
                "h2d_bytes_per_step": cfg.T * cfg.d * 2, "d2h_bytes_per_step": cfg.T * cfg.d * 2,
                "ms_per_step": round(e2e_ms / K, 4),
                "pipelining": "copies on a second stream, double-buffered: step i+1's input and step i-1's "
                              "output move while step i computes"},
        "router_fp32_recomputed_tokens": recomputed,
        "gpu_launches": (kernels_per_step(cfg, torch.cuda.get_device_properties(local_rank).multi_processor_count)
                         + (1 if args.sublayer else 0)) * K,
        "clocks": clk,
    }
    if want_cpu:
        idx = None
        if not args.residual:  # the routing of this batch, for the parity report (after the timed region)
            idx = torch.empty((cfg.T, cfg.top_k), dtype=torch.int32, device="cuda")
            forward(x, out, None, idx)
            torch.cuda.synchronize()
        got = out.view(torch.int16).cpu().numpy().view(np.uint16)
        rec["cpu_baseline"] = cpu_baseline(cfg, args, x_h, wr_h, host_w,
                                           gpu=None if idx is None else (idx.cpu().numpy(), got))
    del ws
    torch.cuda.empty_cache()
    return rec


def run_ours(args, rank, world, local_rank):
    """The --workload batch; with the default decode workload, also the prefill batch (T=4096)
    on the same resident weights, reported as the `prefill` sub-record of the same line."""
    import torch

    torch.cuda.set_device(local_rank)
    cfg = workload_cfg(args.workload)
    peaks = load_peaks()
    want_cpu = (rank == 0 and world == 1 and not args.no_cpu_baseline)
    t_setup = time.time()
    weights, host_w = make_device_weights(cfg, args.seed, torch, keep_host=want_cpu)
    wr_h = W.gen_wr(cfg, args.seed)
    setup_s = time.time() - t_setup
    line = measure_block(args, cfg, weights, host_w, rank, world, local_rank, peaks, want_cpu,
                         W.gen_x(cfg, args.seed + 1000 * rank), wr_h)
    if args.workload == "decode" and not args.no_prefill:
        pcfg = W.CONFIGS["prefill"]  # the same layer (weights, router) with T = 4096
        sub = measure_block(args, pcfg, weights, host_w, rank, world, local_rank, peaks, want_cpu,
                            W.gen_x(pcfg, args.seed + 1000 * rank), W.gen_wr(pcfg, args.seed))
        if line is not None:
            for k in ("metric", "n_gpus", "steps", "warmup", "higher_is_better", "scaling", "vs_baseline", "dtype",
                      "data", "impl"):
                sub.pop(k, None)
            line["prefill"] = sub
    if line is not None:
        line["setup_s"] = round(setup_s, 1)
    return line


# ----------------------------------------------------------------------------- oracle legs

def run_dense(args, rank, world, local_rank):
    """The dense SwiGLU MLP (moe_dense_mlp) on one batch, timed like the MoE forward."""
    import torch
    import sparse_moe_layer_14_b300 as bm

    torch.cuda.set_device(local_rank)
    cfg = workload_cfg(args.workload)
    peaks = load_peaks()
    want_cpu = rank == 0 and world == 1 and not args.no_cpu_baseline
    dims = bm.Dims.from_config(cfg)
    weights, host_w = make_device_weights(cfg, args.seed, torch, keep_host=want_cpu)
    x_h = W.gen_x(cfg, args.seed + 1000 * rank)
    x = torch.from_numpy(x_h).view(torch.int16).view(torch.bfloat16).cuda()
    out = torch.empty((cfg.T, cfg.d), dtype=torch.bfloat16, device="cuda")
    ws = bm.allocate_dense_workspace(dims)
    stream = torch.cuda.current_stream()
    for _ in range(args.warmup):
        bm.moe_dense_mlp(dims, x, weights, out, ws)
    torch.cuda.synchronize()
    K = args.steps
    ev_sets = [[torch.cuda.Event(enable_timing=True) for _ in range(6)] for _ in range(K)]
    for evs in ev_sets:
        for ev in evs:
            ev.record(stream)
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    clocks = ClockSampler(local_rank) if rank == 0 else None
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    wall0 = time.time()
    start.record(stream)
    for i in range(K):
        bm.moe_dense_mlp(dims, x, weights, out, ws)
    end.record(stream)
    torch.cuda.synchronize()
    wall1 = time.time()
    if world > 1:
        torch.distributed.barrier()
    for i in range(K):  # stage-timed pass: events around GEMM1 and GEMM2
        bm.moe_set_stage_events(ev_sets[i])
        bm.moe_dense_mlp(dims, x, weights, out, ws)
    torch.cuda.synchronize()
    bm.moe_set_stage_events(None)
    if bm.moe_get_device_status(ws) != bm.MOE_DEV_OK:
        raise RuntimeError("device status set during the timed region")
    elapsed_ms = max_over_ranks(start.elapsed_time(end), world, "cuda")
    g1_ms = float(np.mean([e[0].elapsed_time(e[3]) for e in ev_sets]))
    g2_ms = float(np.mean([e[3].elapsed_time(e[4]) for e in ev_sets]))
    clk = clocks.summary(wall0, wall1) if clocks else None
    if clocks:
        clocks.stop()

    # end to end: pinned-host copies on a second stream, double-buffered (as for the MoE block)
    x_pin = torch.from_numpy(x_h).view(torch.int16).pin_memory()
    out_pin = [torch.empty((cfg.T, cfg.d), dtype=torch.int16).pin_memory() for _ in range(2)]
    x_dev = [torch.empty_like(x) for _ in range(2)]
    out_dev = [torch.empty_like(out) for _ in range(2)]
    copy_stream = torch.cuda.Stream()

    def e2e_run(n):
        h2d = [torch.cuda.Event() for _ in range(2)]
        fwd = [torch.cuda.Event() for _ in range(2)]
        d2h = [torch.cuda.Event() for _ in range(2)]
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(copy_stream):
            t0.record(copy_stream)
            x_dev[0].view(torch.int16).copy_(x_pin, non_blocking=True)
            h2d[0].record(copy_stream)
        for i in range(n):
            b = i % 2
            stream.wait_event(h2d[b])
            if i >= 2:
                stream.wait_event(d2h[b])
            bm.moe_dense_mlp(dims, x_dev[b], weights, out_dev[b], ws)
            fwd[b].record(stream)
            with torch.cuda.stream(copy_stream):
                if i + 1 < n:
                    if i >= 1:
                        copy_stream.wait_event(fwd[1 - b])
                    x_dev[1 - b].view(torch.int16).copy_(x_pin, non_blocking=True)
                    h2d[1 - b].record(copy_stream)
                copy_stream.wait_event(fwd[b])
                out_pin[b].copy_(out_dev[b].view(torch.int16), non_blocking=True)
                d2h[b].record(copy_stream)
        with torch.cuda.stream(copy_stream):
            t1.record(copy_stream)
        return t0, t1

    e2e_run(max(2, args.warmup))
    torch.cuda.synchronize()
    e0, e1 = e2e_run(K)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(e0.elapsed_time(e1), world, "cuda")
    if rank != 0:
        return None

    d, I, T = cfg.d, cfg.inter, cfg.T
    flops1, flops2 = 2.0 * T * d * 2 * I, 2.0 * T * I * d
    bytes1 = 2 * I * d * 2 + T * d * 2 + T * I * 2
    bytes2 = d * I * 2 + T * I * 2 + T * d * 2
    ms_per_step = elapsed_ms / K

    def roof(fl, by, ms):
        t_f, t_b = fl / (peaks["bf16_tflops"] * 1e12), by / (peaks["hbm_gbs"] * 1e9)
        bound = "tensor" if t_f >= t_b else "hbm"
        ach = fl / (ms / 1e3) / 1e12 if bound == "tensor" else by / (ms / 1e3) / 1e9
        pk = peaks["bf16_tflops"] if bound == "tensor" else peaks["hbm_gbs"]
        return bound, ach, pk, max(t_f, t_b) * 1e3

    b1, a1, p1, r1 = roof(flops1, bytes1, g1_ms)
    _, _, _, r2 = roof(flops2, bytes2, g2_ms)
    line = {
        "metric": "dense SwiGLU MLP tokens/s (first decoder layers)", "value": round(world * T / (ms_per_step / 1e3), 1),
        "unit": "tokens/s", "n_gpus": world, "steps": K, "warmup": args.warmup, "ms_per_step": round(ms_per_step, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded N(0,1) activations, N(0,1/fan_in) weights)", "impl": "ours",
        "config": {"workload": f"{cfg.name}: dense SwiGLU MLP, T={T} tokens, d={d}, intermediate {I} (a reading: "
                               f"8 x 2560, the routed experts' per-token width), bf16 weights",
                   "T": T, "d": d, "inter": I, "parallelism": f"replicas x{world}",
                   "l2": f"no flush: {3 * d * I * 2 / 1e6:.0f} MB of weights and {T * I * 2 / 1e6:.0f} MB of h "
                         f"per step exceed the 126 MB L2"},
        "roofline": {"kernel": "expert_gemm_kernel<GLU> (GEMM1 + SwiGLU, one expert)", "bound": b1,
                     "achieved": round(a1, 1), "peak": p1, "unit": "TFLOP/s" if b1 == "tensor" else "GB/s",
                     "frac": round(a1 / p1, 4), "peak_source": f"{peaks['source']} "
                     f"({'bf16_tflops' if b1 == 'tensor' else 'hbm_gbs'})", "traffic": None,
                     "traffic_source": "no capture of this case", "algorithmic_bytes": bytes1,
                     "algorithmic_flops": flops1, "avg_launch_ms": round(g1_ms, 4)},
        "layer_roofline": {"roofline_ms": round(r1 + r2, 4), "frac": round((r1 + r2) / ms_per_step, 4),
                           "algorithmic_flops": flops1 + flops2},
        "stages_ms": {"offsets+schedule+gemm1": round(g1_ms, 4), "gemm2": round(g2_ms, 4)},
        "gemm2_roofline": {"frac": round(r2 / g2_ms, 4)},
        "e2e": {"value": round(world * T / (e2e_ms / K / 1e3), 1), "unit": "tokens/s",
                "h2d_bytes_per_step": T * d * 2, "d2h_bytes_per_step": T * d * 2, "ms_per_step": round(e2e_ms / K, 4),
                "pipelining": "copies on a second stream, double-buffered: step i+1's input and step i-1's "
                              "output move while step i computes"},
        "gpu_launches": 4 * K,
        "clocks": clk,
    }
    if want_cpu:
        import oracle as O
        n = 16
        t0 = time.time()
        O.ffn_rows(np.zeros(n, np.int32), x_h[:n], host_w, d, I, cfg.wfmt)
        dt = time.time() - t0
        line["cpu_baseline"] = {"value": round(n / dt, 3), "unit": "tokens/s", "cores": O.num_threads(),
                                "kind": "oracle", "sample": f"first {n} of the {T} tokens (fp64 SwiGLU MLP rows)",
                                "seconds": round(dt, 2)}
    return line


def cpu_sample_tokens(cfg):
    return min(cfg.T, 64)


def cpu_baseline(cfg, args, x_h, wr_h, host_w, n_tok=None, gpu=None):
    """The CPU oracle, as it stands, on a bounded token sample of the same workload (timed), then
    its parity against the GPU run on those tokens: gpu = (topk_idx [T, K], out [T, d] bf16 bits)
    of the timed batch. Routing must match outside near-ties (margins below 1e-6, counted and
    excluded); the output error is reported against the bar of the weight format."""
    import oracle as O
    n = n_tok or cpu_sample_tokens(cfg)
    sub = cfg.with_tokens(n)
    toks = np.linspace(0, cfg.T - 1, n).astype(np.int64) if n < cfg.T else np.arange(cfg.T)
    xs = np.ascontiguousarray(x_h[toks])
    t0 = time.time()
    r = O.route(sub, xs, wr_h)
    ref = O.forward_tokens(sub, xs, r["idx"], r["w"], np.arange(n), host_w)
    dt = time.time() - t0
    rec = {"value": round(n / dt, 3), "unit": "tokens/s", "cores": O.num_threads(), "kind": "oracle",
           "sample": f"{n} of the {cfg.T} tokens of the same seeded batch, evenly spaced (routing + all "
                     f"{cfg.top_k} experts per token + combine, fp64 accumulation)", "seconds": round(dt, 2)}
    if gpu is not None:
        gi, got = gpu[0][toks], gpu[1][toks]
        near = (r["margin_group"] < 1e-6) | (r["margin_expert"] < 1e-6)
        mism = int(np.sum(np.any(np.sort(gi[~near], 1) != np.sort(r["idx"][~near], 1), axis=1)))
        # near-tie tokens: the reference output under the GPU's choice (checked only for validity in the tests)
        idx_ref, w_ref = r["idx"].copy(), r["w"].copy()
        s = r["scores"].astype(np.float64)
        for t in np.nonzero(near)[0]:
            idx_ref[t] = gi[t]
            w_ref[t] = cfg.routed_scale * s[t, gi[t]] / s[t, gi[t]].sum()
        if near.any():
            ref = O.forward_tokens(sub, xs, idx_ref, w_ref, np.arange(n), host_w)
        g = W.bf16_to_f32(got).astype(np.float64)
        rms = float(np.sqrt(np.mean(ref ** 2)))
        e = np.abs(g - ref)
        bar = {"bf16": 2e-2, "nvfp4": 5e-2, "fp8": 3.5e-2}[cfg.wfmt]
        rec["parity"] = {"tokens": int(n), "routing_mismatches": mism, "excluded_near_ties": int(near.sum()),
                         "max_err_over_rms": round(float(e.max()) / rms, 6),
                         "rms_err_over_rms": round(float(np.sqrt(np.mean(e ** 2))) / rms, 6), "bar": bar,
                         "ok": bool(mism == 0 and e.max() <= bar * rms)}
    return rec


def run_reference(args):
    import oracle as O
    cfg = workload_cfg(args.workload)
    host = {}
    for which in ("gate", "up", "down"):
        host[which] = W.gen_expert_bf16(cfg, args.seed, which, 0, cfg.E)
    x_h = W.gen_x(cfg, args.seed)
    wr_h = W.gen_wr(cfg, args.seed)
    n = min(cfg.T, args.ref_tokens)

    def step(i):
        t0 = (i * n) % max(1, cfg.T - n + 1)
        sub = cfg.with_tokens(n)
        xs = np.ascontiguousarray(x_h[t0:t0 + n])
        r = O.route(sub, xs, wr_h)
        O.forward_tokens(sub, xs, r["idx"], r["w"], np.arange(n), host)

    for i in range(args.warmup):
        step(i)
    t0 = time.time()
    for i in range(args.steps):
        step(args.warmup + i)
    dt = time.time() - t0
    value = n * args.steps / dt
    return {"metric": METRIC, "value": round(value, 3), "unit": "tokens/s", "n_gpus": 1, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(dt / args.steps * 1e3, 2), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic", "impl": "reference",
            "config": {"workload": describe(cfg), "T": cfg.T, "d": cfg.d, "E": cfg.E, "inter": cfg.inter,
                       "top_k": cfg.top_k, "parallelism": "host cores"},
            "cpu_baseline": {"value": round(value, 3), "unit": "tokens/s", "cores": O.num_threads(), "kind": "oracle",
                             "sample": f"{n} tokens of the {cfg.T}-token batch per step (routing + experts + combine)"},
            "e2e": {"value": round(value, 3), "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=None)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default="decode",
                    choices=sorted(list(W.CONFIGS) + list(PROFILE_CASES) + list(DENSE_CASES)))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-prefill", action="store_true",
                    help="with the default decode workload, skip the prefill (T=4096) sub-record")
    ap.add_argument("--ref-tokens", type=int, default=16, help="tokens per reference-arm step")
    ap.add_argument("--sublayer", action="store_true",
                    help="run the whole MoE sublayer (moe_sublayer): pre-norm of the residual stream, the block, "
                         "post-norm and residual update in place")
    ap.add_argument("--residual", action="store_true",
                    help="end the block with the fused post-norm and depth-scaled residual update "
                         "(moe_forward_residual) instead of writing the output")
    ap.add_argument("--record-traffic", metavar="DIR",
                    help="write profiles/dram_traffic.json from the ncu captures and bench lines in DIR, then exit")
    args = ap.parse_args()
    if args.record_traffic:
        print(record_traffic(args.record_traffic))
        return
    if args.warmup < 3:
        args.warmup = 3
    if args.steps is None:
        args.steps = DEFAULT_STEPS.get(args.workload, 50) if args.impl == "ours" else 5

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.gpus != world:
        # one process per GPU: N GPUs need N ranks (torchrun --nproc-per-node N)
        sys.exit(f"bench.py: --gpus {args.gpus} but WORLD_SIZE={world}; launch one rank per GPU, e.g. "
                 f"python -m torch.distributed.run --nproc-per-node {args.gpus} bench.py --gpus {args.gpus}")
    if args.impl == "reference":
        if rank != 0:
            return
        print(json.dumps(run_reference(args)), flush=True)
        return
    if world > 1:
        import torch
        torch.cuda.set_device(local_rank)
        torch.distributed.init_process_group("nccl")
    line = (run_dense if args.workload in DENSE_CASES else run_ours)(args, rank, world, local_rank)
    if line is not None:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
