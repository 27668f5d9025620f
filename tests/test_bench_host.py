"""Host logic of bench.py: the byte/FLOP model, the roofline arithmetic, the
clock summary, the max-over-ranks reduction across two gloo ranks and the
--gpus N replica launcher (no GPU)."""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench
from router_experts_gb300 import workloads as W


def test_work_model_matches_page_figures():
    # "Mixture of Experts": one DeepSeek-V3 expert is 3 * 7168 * 2048 = 44.04 M
    # parameters and 6 * 7168 * 2048 = 88.08 MFLOP per token-expert
    w = W.WORKLOADS["dsv3"]
    st, layer = bench.work_model(w, 1, touched=8, block_m=16)
    assert layer["flops"] - st["router"]["flops"] == 8 * 6 * 7168 * 2048
    per_expert = (st["gemm1"]["bytes"] - 7168 * 2 - 8 * 2048 * 2) / 8 + \
        (st["gemm2"]["bytes"] - 8 * 2048 * 2 - 8 * 7168 * 2) / 8
    assert per_expert == 3 * 7168 * 2048 * 2
    # worst-case capacity T*k + E*(BM-1) at T=64, BM=16: 4,352 rows, 272 blocks
    st, _ = bench.work_model(w, 64, touched=222, block_m=16)
    assert st["align"]["bytes"] == 4 * 512 + 4 * 4352 + 4 * 272


def test_roofline_picks_binding_resource():
    peaks = {"hbm_gbs": 1000.0, "bf16_tflops": 1000.0}
    r = bench.roofline_of(1e9, 1e9, 2e-3, peaks)  # 1 ms of bytes vs 1 us of flops
    assert r["bound"] == "hbm" and r["achieved"] == pytest.approx(500.0)
    assert r["frac"] == pytest.approx(0.5)
    r = bench.roofline_of(1e3, 1e15, 2.0, peaks)
    assert r["bound"] == "tensor" and r["frac"] == pytest.approx(0.5)
    # block-scaled fp8 contractions: twice the bf16 rate
    r = bench.roofline_of(1e3, 1e15, 2.0, peaks, fp8=True)
    assert r["bound"] == "tensor" and r["peak"] == 2000.0 and r["frac"] == pytest.approx(0.25)
    # the binding resource moves with the faster tensor rate
    r = bench.roofline_of(1.5e9, 2e12, 1.0, peaks, fp8=True)
    assert r["bound"] == "hbm"
    # an fp8 rate measured in the run replaces the nominal ratio
    r = bench.roofline_of(1e3, 1e15, 2.0, dict(peaks, fp8_tflops=1600.0), fp8=True)
    assert r["peak"] == 1600.0 and r["frac"] == pytest.approx(500.0 / 1600.0)
    assert "measured" in r["tensor_dtype"]


def test_clock_summary_window_and_reasons():
    c = bench.ClockSampler("0")
    c.max_mhz = 2070.0
    # (host time, SM MHz, NVML clocks-event reasons, W): power cap at t = 2
    c.samples = [(1.0, 2070.0, 0, 500.0), (2.0, 1900.0, 0x4, 1390.0), (3.0, 1950.0, 0, 1200.0),
                 (9.0, 600.0, 0x8, 100.0)]
    s = c.summary(1.5, 3.5)
    assert s["samples"] == 2 and s["sm_mhz"] == pytest.approx(1925.0)
    assert s["reasons"] == ["sw_power_cap"] and s["sm_max_mhz"] == 2070.0
    assert c.summary()["reasons"] == ["hw_slowdown", "sw_power_cap"]
    assert c.summary(10.0, 11.0)["samples"] == 0


def test_lowbit_work_model_bytes():
    # V4-Flash low-bit: e2m1 weights with a UE8M0 byte per 32 (0.5 + 1/32 bytes
    # per weight), e4m3 activations with a byte per 32, fp32 gate
    w = W.WORKLOADS["v4lo"]
    st, layer = bench.work_model(w, 1, touched=6, block_m=16)
    w13 = 2 * w.F * w.H * (0.5 + 1 / 32)
    assert st["gemm1"]["bytes"] == pytest.approx(6 * w13 + w.H * (1 + 1 / 32) + 6 * w.F * (1 + 1 / 32))
    assert st["router"]["bytes"] == pytest.approx(w.E * w.H * 4 + w.H * (1 + 1 / 32) + 8 * 6)


def test_touched_expert_model():
    # "Mixture of Experts": half-way batch 21.8 tokens for DeepSeek-V3
    assert W.touched_experts_model(1, 8, 256) == pytest.approx(8.0)
    assert W.touched_experts_model(22, 8, 256) == pytest.approx(128, rel=0.02)


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    v = bench.reduce_max(float(rank + 1) * 1.5, world)
    bench.barrier(world)
    q.put((rank, v, bench.dist_env()))
    dist.destroy_process_group()


def test_reduce_max_over_two_gloo_ranks():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        port = s.getsockname()[1]
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
    assert [r[1] for r in res] == [3.0, 3.0]
    assert [r[2] for r in res] == [(2, 0, 0), (2, 1, 1)]


def test_smi_index_honours_visible_devices(monkeypatch):
    monkeypatch.setenv("CUDA_VISIBLE_DEVICES", "5,7")
    assert bench.smi_index(1) == "7"
    monkeypatch.delenv("CUDA_VISIBLE_DEVICES")
    assert bench.smi_index(2) == "2"


def test_gpus_flag_launches_replicas_without_torchrun():
    # bench.py --gpus 2 outside torchrun starts two replica processes itself;
    # --dry-run keeps them off the GPU (gloo), each reporting rank + 1 ms, and
    # rank 0 prints the maximum over ranks
    env = {k: v for k, v in os.environ.items()
           if k not in ("WORLD_SIZE", "RANK", "LOCAL_RANK", "MASTER_ADDR", "MASTER_PORT")}
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    r = subprocess.run([sys.executable, os.path.join(root, "bench.py"), "--gpus", "2",
                        "--dry-run", "--steps", "3", "--warmup", "3"],
                       capture_output=True, text=True, timeout=300, env=env)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, r.stdout
    out = json.loads(lines[0])
    assert out["n_gpus"] == 2 and out["ms_per_step"] == 2.0 and out["scaling"] == "weak"
