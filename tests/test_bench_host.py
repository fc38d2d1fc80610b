"""Host logic of bench.py that needs no GPU: the multi-rank aggregation (world size 2,
gloo on CPU), the reference arm's rank handling, clock-sample parsing and the
roofline arithmetic."""
import os
import socket
import subprocess
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench
import workload as W

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        got = bench.max_over_ranks(10.0 + 5.0 * rank, world, "cpu")
        q.put((rank, got))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_world2_gloo():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    res = dict(q.get(timeout=10) for _ in range(2))
    assert res == {0: 15.0, 1: 15.0}
    assert bench.max_over_ranks(3.5, 1, "cpu") == 3.5


def test_reference_arm_only_rank0_runs():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                        "--gpus", "2"], env=env, capture_output=True, text=True, timeout=120)
    assert r.returncode == 0 and r.stdout.strip() == ""


def test_gpus_flag_must_match_world_size():
    """--gpus N without N ranks is refused (it would otherwise measure one GPU and call it N)."""
    env = {k: v for k, v in os.environ.items() if k not in ("RANK", "WORLD_SIZE", "LOCAL_RANK")}
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--gpus", "8", "--steps", "1"],
                       env=env, capture_output=True, text=True, timeout=120)
    assert r.returncode != 0 and "WORLD_SIZE=1" in r.stderr and r.stdout.strip() == ""


def test_clock_summary_flags_throttle():
    cs = bench.ClockSampler.__new__(bench.ClockSampler)
    cs.samples = [(1.0, ["1900", "2032", "700.5", "Not Active", "Not Active", "Not Active", "Active"]),
                  (1.1, ["1950", "2032", "710.0", "Not Active", "Active", "Not Active", "Not Active"]),
                  (5.0, ["300", "2032", "100.0", "Not Active", "Not Active", "Not Active", "Not Active"])]
    s = cs.summary(0.5, 2.0)
    assert s["samples"] == 2 and s["sm_mhz"] == 1925.0 and s["sm_max_mhz"] == 2032.0
    assert s["reasons"] == ["hw_thermal_slowdown", "sw_power_cap"]
    s2 = cs.summary(4.0, 4.01)  # shorter than the sampling period: nearest samples
    assert s2["samples"] == 3 and "nearest" in s2["window"]


def test_roofline_arithmetic():
    cfg = W.CONFIGS["decode"]
    peaks = {"hbm_gbs": 6500.0, "bf16_tflops": 1800.0}
    g1, g2, layer = bench.roofline_numbers(cfg, 222, peaks)
    R = 64 * 8
    assert layer["flops"] == 2.0 * R * 3 * 5120 * 2560 + 2.0 * 64 * 5120 * 256
    assert layer["bytes"] == 222 * 3 * 5120 * 2560 * 2 + 5120 * 256 * 4 + 64 * 5120 * 2 * 2
    assert g1["bound"] == g2["bound"] == layer["bound"] == "hbm"
    big = bench.roofline_numbers(W.CONFIGS["skewed"], 256, peaks)
    assert big[0]["bound"] == "tensor"


def test_kernel_counts():
    assert bench.simt_router_kernels(64, 256) == 1       # logits kernel selects itself
    assert bench.simt_router_kernels(1536, 256) == 1     # 24 tiles x 8 tickets = 192
    assert bench.simt_router_kernels(1537, 256) == 2     # + a selection kernel
    assert bench.simt_router_kernels(64, 18) == 2        # + the W_r padding copy
    assert bench.kernels_per_step(W.CONFIGS["skewed"], 148) == 12   # tensor-core router: 5 kernels
    # SIMT router; plan kernel (with the GEMM schedule) + gather; GEMM1, GEMM2, combine
    assert bench.kernels_per_step(W.CONFIGS["decode"], 148) == 6
    assert bench.permute_uses_plan_kernel(1024, 256) and not bench.permute_uses_plan_kernel(1025, 256)


def test_stage_roofline_arithmetic():
    """Prefill shape: the combine reads 8 FP32 rows of 5120 per token plus its 8 weights and rows and
    writes one bf16 row; at 0.12 ms that is 5.95 TB/s."""
    cfg = W.CONFIGS["prefill"]
    peaks = {"hbm_gbs": 6497.4}
    st = bench.stage_rooflines(cfg, [0.161, 0.093, 2.255, 1.165, 0.12], peaks)
    R = 4096 * 8
    assert st["combine"]["bytes"] == R * 5120 * 4 + R * 8 + 4096 * 5120 * 2
    assert abs(st["combine"]["achieved_gbs"] - st["combine"]["bytes"] / 0.12e-3 / 1e9) < 0.1
    assert 0.85 < st["combine"]["frac_hbm"] < 0.95
    res = bench.stage_rooflines(cfg, [0.161, 0.093, 2.255, 1.165, 0.141], peaks, residual=True)
    assert res["combine"]["bytes"] == st["combine"]["bytes"] + 4096 * 5120 * 2 + 5120 * 2
    assert abs(st["router"]["achieved_fp32_tflops"] - 2 * 4096 * 5120 * 256 / 0.161e-3 / 1e12) < 0.01
    assert "frac_fp32_alu" not in st["router"]  # T = 4096 routes on the tensor cores
    dec = bench.stage_rooflines(W.CONFIGS["decode"], [0.0474, 0.0213, 1.68, 0.83, 0.0079], peaks)
    assert 0.04 < dec["router"]["frac_fp32_alu"] < 0.05


def test_cpu_baseline_parity_report():
    """The bench's CPU-baseline leg times the oracle on a token sample and reports parity against
    the GPU run's routing and output: fed the oracle's own routing and its output rounded to bf16,
    it must report no mismatch and an error within the bf16 rounding; a routing with one token's
    experts changed must count one mismatch."""
    import numpy as np
    import oracle as O
    cfg = W.CONFIGS["tiny"]
    inp = W.make_host_inputs(cfg, 3)
    r = O.route(cfg, inp["x"], inp["w_r"])
    out = O.forward_tokens(cfg, inp["x"], r["idx"], r["w"], np.arange(cfg.T), inp)
    bits = torch.from_numpy(out.astype(np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)

    class A:
        pass
    rec = bench.cpu_baseline(cfg, A(), inp["x"], inp["w_r"], inp, n_tok=16, gpu=(r["idx"], bits))
    p = rec["parity"]
    assert p["tokens"] == 16 and p["routing_mismatches"] == 0 and p["ok"]
    assert p["max_err_over_rms"] <= 2.0 ** -8 * np.abs(out).max() / np.sqrt(np.mean(out ** 2))
    decided = np.nonzero((r["margin_group"] >= 1e-6) & (r["margin_expert"] >= 1e-6))[0]
    bad = r["idx"].copy()
    t = int(decided[0])
    bad[t] = (bad[t] + 1) % cfg.E  # a different expert set for one sampled token (token 0 is sampled)
    assert t == 0
    rec2 = bench.cpu_baseline(cfg, A(), inp["x"], inp["w_r"], inp, n_tok=16, gpu=(bad, bits))
    assert rec2["parity"]["routing_mismatches"] == 1 and not rec2["parity"]["ok"]


def test_record_traffic_from_ncu_csv(tmp_path):
    """bench.py --record-traffic: ncu's CSV launch list and the plain bench line of a small case
    become the DRAM-traffic record the roofline's `traffic` reads (scaled by algorithmic bytes)."""
    import json
    hdr = '"ID","Process ID","Process Name","Host Name","Kernel Name","Context","Stream","Block Size",' \
          '"Grid Size","Device","CC","Section Name","Metric Name","Metric Unit","Metric Value"'
    rows = []
    # both spellings ncu uses for the anonymous namespace (its '>' must not end the template match)
    for i, (name, rd, wr, t) in enumerate([("void unnamed>::expert_gemm_kernel<1, 1>(CUtensorMap_st)", "525.5",
                                            "17.8", "285.3"),
                                           ("void (anonymous namespace)::expert_gemm_kernel<0, 1>(CUtensorMap_st)",
                                            "257.6", "27.4", "142.2")]):
        for m, u, v in (("dram__bytes_read.sum", "Mbyte", rd), ("dram__bytes_write.sum", "Mbyte", wr),
                        ("gpu__time_duration.sum", "usecond", t)):
            rows.append(f'"{i}","1","python","h","{name}","1","7","(576, 1, 1)","(148, 1, 1)","0","10.3","",'
                        f'"{m}","{u}","{v}"')
    (tmp_path / "profile_nvfp4.csv").write_text("==PROF== note\n" + hdr + "\n" + "\n".join(rows) + "\n")
    (tmp_path / "profile_nvfp4.json").write_text(json.dumps({"layer_roofline": {"experts_touched": 32}}) + "\n")
    out = bench.record_traffic(str(tmp_path), out=str(tmp_path / "traffic.json"))
    rec = json.load(open(out))
    assert rec["capture_for_workload"]["nvfp4"] == "profile_nvfp4"
    k = rec["captures"]["profile_nvfp4"]["kernels"]
    assert k["expert_gemm_kernel<GLU, NVFP4>"]["dram_bytes_read"] == 525_500_000
    assert k["expert_gemm_kernel<plain, NVFP4>"]["gpu_time_ns_serialised"] == 142_200
    g1, _, _ = bench.roofline_numbers(W.CONFIGS["nvfp4"].__class__(**{**W.CONFIGS["nvfp4"].__dict__, "name": "x",
                                                                      "T": 512, "E": 32, "n_groups": 8}), 32,
                                      {"hbm_gbs": 6497.4, "bf16_tflops": 1811.4})
    assert k["expert_gemm_kernel<GLU, NVFP4>"]["algorithmic_bytes"] == int(g1["bytes"])
