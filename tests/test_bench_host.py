"""Host logic of bench.py: the byte/FLOP model, the roofline arithmetic and
the max-over-ranks reduction across two gloo ranks (no GPU)."""
import os
import socket

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
