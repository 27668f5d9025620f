"""Seeded synthetic inputs of the layer's workloads.

This module only draws random numbers and lays them out in the formats the
library takes; it holds none of the method's arithmetic (no routing, no
alignment, no GEMM).  Both the CUDA path and the CPU oracle are fed from it.

Workloads (shapes from "Mixture of Experts" -- Qwen3-30B-A3B d=2048, E=128,
k=8, d_ff=768; DeepSeek-V3 d=7168, E=256, k=8, d_ff=2048, n_group=8,
topk_group=4 -- "How an MoE Model Picks Its Experts During LLM Inference" --
GLM-5.3-Flash 288 x 4,096 gate, k=8 -- and "How GPUs Fuse Communication and
Computation During LLM Inference" -- DeepSeek-V4-Flash 256 experts, k=6,
4,096 -> 2 x 2,048, FP8 activations x FP4 weights with a scale per 32 values):

  toy     T=16, H=64, E=8, k=2, F=32, softmax + renormalise, BLOCK_M 16
  qwen3   H=2048, E=128, k=8, F=768, softmax + renormalise, T in {1,64,512,4096}
  dsv3    H=7168, E=256, k=8, F=2048, sigmoid + bias, 8 groups keep 4,
          routed scaling 2.5, per-expert Zipf(1.1) logit offset
  glm     H=4096, E=288, k=8, sigmoid + bias, router + align only
  v4lo    H=4096, E=256, k=6, F=2048, sigmoid + bias; e4m3 activations and
          e2m1 weights, one UE8M0 scale per 32 values, scale exponents
          uniform in {-4..0}; the router reads the dequantised fp32 hidden
          rows and an fp32 gate
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np
import torch


@dataclass(frozen=True)
class Workload:
    name: str
    H: int
    E: int
    k: int
    F: int                  # 0: router + align only
    scoring: str            # "softmax" | "sigmoid"
    n_group: int = 1
    topk_group: int = 1
    renormalize: bool = True
    scaling: float = 1.0
    bias: bool = False
    lowbit: bool = False
    zipf: float = 0.0
    Ts: tuple = ()
    block_ms: tuple = ()


WORKLOADS = {
    "toy": Workload("toy", H=64, E=8, k=2, F=32, scoring="softmax", Ts=(16,), block_ms=(16,)),
    "qwen3": Workload("qwen3", H=2048, E=128, k=8, F=768, scoring="softmax",
                      Ts=(1, 64, 512, 4096)),
    "dsv3": Workload("dsv3", H=7168, E=256, k=8, F=2048, scoring="sigmoid", n_group=8,
                     topk_group=4, scaling=2.5, bias=True, zipf=1.1, Ts=(1, 256, 4096)),
    "glm": Workload("glm", H=4096, E=288, k=8, F=0, scoring="sigmoid", bias=True,
                    Ts=(1, 8, 64, 512, 4096), block_ms=(16, 64, 128)),
    "v4lo": Workload("v4lo", H=4096, E=256, k=6, F=2048, scoring="sigmoid", bias=True,
                     lowbit=True, Ts=(512, 4096)),
}


def block_m_for(T: int, k: int, E: int) -> int:
    """Tile height by mean rows per expert: 16 below 8, 64 below 64, else 128
    ("MoE Kernels, in depth": tile shape depends on tokens per expert)."""
    mean = T * k / E
    return 16 if mean < 8 else (64 if mean < 64 else 128)


def cap_rows(T: int, k: int, E: int, block_m: int) -> int:
    """Worst-case padded rows T*k + E*(BLOCK_M-1)."""
    return T * k + E * (block_m - 1)


def _gen(device, seed: int, idx: int) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed) * 1009 + idx)
    return g


def _bf16_normal(shape, std, g, device, chunk_rows=None):
    out = torch.empty(shape, dtype=torch.bfloat16, device=device)
    flat = out.view(shape[0], -1)
    step = chunk_rows or shape[0]
    for r0 in range(0, shape[0], step):
        r1 = min(shape[0], r0 + step)
        flat[r0:r1] = (torch.randn((r1 - r0, flat.shape[1]), generator=g, device=device,
                                   dtype=torch.float32) * std).to(torch.bfloat16)
    return out


_E2M1_EDGES = torch.tensor([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0])


def _fp4_codes(rows, cols, g, device):
    """e2m1 nibbles nearest to 2*N(0,1) (magnitude saturating at 6), packed two
    per byte, low nibble first: [rows, cols/2] uint8."""
    v = torch.randn((rows, cols), generator=g, device=device, dtype=torch.float32) * 2.0
    mag = torch.bucketize(v.abs(), _E2M1_EDGES.to(device)).to(torch.uint8)
    nib = mag | ((v < 0).to(torch.uint8) << 3)
    return nib[:, 0::2] | (nib[:, 1::2] << 4)


def _scales(rows, groups, g, device):
    """UE8M0 exponents 127 + u with u uniform in {-4, ..., 0}."""
    u = torch.randint(-4, 1, (rows, groups), generator=g, device=device, dtype=torch.int32)
    return (u + 127).to(torch.uint8)


def make_inputs(w: Workload, T: int, seed: int = 0, device="cpu", experts: bool = True) -> dict:
    """Synthetic inputs for T tokens, one torch.Generator per tensor, in order:
    hidden, gate, bias, w13, w2 (and their scales for the low-bit workload)."""
    H, E, F = w.H, w.E, w.F
    d = {}
    if w.lowbit:
        # activations: e4m3 codes of N(0,1) / 2^u, scale 2^u per 32 values
        gx = _gen(device, seed, 0)
        sc = _scales(T, H // 32, gx, device)
        u = sc.to(torch.float32) - 127.0
        v = torch.randn((T, H), generator=gx, device=device, dtype=torch.float32)
        v = v / torch.exp2(u).repeat_interleave(32, dim=1)
        d["hidden"] = v.to(torch.float8_e4m3fn).view(torch.uint8)
        d["hidden_scale"] = sc
        gg = _gen(device, seed, 1)
        d["gate"] = torch.randn((E, H), generator=gg, device=device,
                                dtype=torch.float32) / math.sqrt(H)
    else:
        d["hidden"] = _bf16_normal((T, H), 1.0, _gen(device, seed, 0), device)
        d["gate"] = _bf16_normal((E, H), 1.0 / math.sqrt(H), _gen(device, seed, 1), device)
    if w.bias:
        gb = _gen(device, seed, 2)
        d["bias"] = torch.rand((E,), generator=gb, device=device, dtype=torch.float32) * 0.2 - 0.1
    if w.zipf > 0:
        # a seeded permutation ranks the experts; rank r gets logit offset
        # zipf * (mean_r ln r - ln r), carried by hidden column H-1 (= 1.0)
        gz = _gen(device, seed, 3)
        perm = torch.randperm(E, generator=gz, device=device)
        lnr = torch.log(torch.arange(1, E + 1, dtype=torch.float64, device=device))
        off = w.zipf * (lnr.mean() - lnr[perm])
        d["hidden"][:, H - 1] = 1.0
        d["gate"][:, H - 1] = off.to(d["gate"].dtype)
    if experts and F > 0:
        if w.lowbit:
            g13, g2 = _gen(device, seed, 4), _gen(device, seed, 5)
            d["w13"] = torch.empty((E, 2 * F, H // 2), dtype=torch.uint8, device=device)
            d["w13_scale"] = torch.empty((E, 2 * F, H // 32), dtype=torch.uint8, device=device)
            d["w2"] = torch.empty((E, H, F // 2), dtype=torch.uint8, device=device)
            d["w2_scale"] = torch.empty((E, H, F // 32), dtype=torch.uint8, device=device)
            for e in range(E):
                d["w13"][e] = _fp4_codes(2 * F, H, g13, device)
                d["w13_scale"][e] = _scales(2 * F, H // 32, g13, device)
                d["w2"][e] = _fp4_codes(H, F, g2, device)
                d["w2_scale"][e] = _scales(H, F // 32, g2, device)
        else:
            per = max(1, (1 << 26) // (2 * F * H))  # experts per fp32 temporary
            d["w13"] = _bf16_normal((E, 2 * F, H), 0.02, _gen(device, seed, 4), device,
                                    chunk_rows=per)
            d["w2"] = _bf16_normal((E, H, F), 0.02, _gen(device, seed, 5), device,
                                   chunk_rows=per)
    return d


def random_routing(T: int, k: int, E: int, seed: int = 0, skew: float = 0.0,
                   device="cpu"):
    """Synthetic (topk_ids [T,k] int32, topk_weights [T,k] f32) for testing the
    steps after the router: k distinct experts per token, drawn with
    probabilities proportional to rank^-skew over a seeded permutation, and
    positive weights."""
    g = _gen("cpu", seed, 7)
    perm = torch.randperm(E, generator=g)
    p = torch.arange(1, E + 1, dtype=torch.float64) ** (-skew)
    p = p[torch.argsort(perm)]
    if T == 0:
        ids = torch.zeros((0, k), dtype=torch.int32)
    else:
        ids = torch.multinomial(p.expand(T, E).contiguous(), k, replacement=False,
                                generator=g).to(torch.int32)
    wts = torch.rand((T, k), generator=g, dtype=torch.float32) * 0.9 + 0.1
    return ids.to(device), wts.to(device)


def to_host_raw(t: torch.Tensor) -> np.ndarray:
    """Host numpy view of a tensor's raw storage (bf16 -> uint16 bits)."""
    t = t.detach().contiguous().cpu()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    if t.dtype == torch.float8_e4m3fn:
        return t.view(torch.uint8).numpy()
    return t.numpy()


def touched_experts_model(T: int, k: int, E: int) -> float:
    """Expected experts touched by T uniform tokens, E (1 - (1 - k/E)^T)
    ("Mixture of Experts", How many experts does a batch touch?)."""
    return E * (1.0 - (1.0 - k / E) ** T)
