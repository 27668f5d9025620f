"""The fused router on the GPU against the oracle router on the same seeded
inputs: ids identical (in selection order) for every token whose margin at
the cut exceeds 1e-4, weights within 1e-5 absolute; the residual mismatch
fraction is reported."""
import dataclasses

import numpy as np
import pytest
import torch

import oracle
from router_experts_gb300 import moe
from router_experts_gb300 import workloads as W

from _gpu import GAP_MIN, WEIGHT_ATOL, oracle_router, sample_tokens

pytestmark = pytest.mark.gpu

# (T <= 4 with a bf16 gate: the tensor-core router selects in its last CTA)
CASES = [("toy", 16), ("toy", 5), ("qwen3", 1), ("qwen3", 4), ("qwen3", 5), ("qwen3", 12),
         ("qwen3", 64), ("qwen3", 512), ("dsv3", 3), ("glm", 2),
         ("qwen3", 4096), ("dsv3", 1), ("dsv3", 256), ("dsv3", 4096), ("glm", 1), ("glm", 8),
         ("glm", 13), ("glm", 64), ("glm", 512), ("glm", 4096), ("v4lo", 8), ("v4lo", 512),
         ("v4lo", 4096)]


def check_router(w, T):
    d = W.make_inputs(w, T, seed=T, device="cuda", experts=False)
    ids, wts = moe.router(d["hidden"], d["gate"], d.get("bias"), w.k, w.scoring, w.n_group,
                          w.topk_group, w.renormalize, w.scaling,
                          hidden_scale=d.get("hidden_scale"))
    torch.cuda.synchronize()
    tokens = sample_tokens(T, 384 if w.H <= 4096 else 128, seed=T)
    ids_o, w_o, gap = oracle_router(oracle, w, d, T, tokens)
    ids_g = ids.cpu().numpy()[tokens]
    w_g = wts.cpu().numpy()[tokens]
    clear = gap > GAP_MIN
    same = (ids_g == ids_o).all(axis=1)
    mismatch = 1.0 - same.mean()
    print(f"{w.name} {w.scoring} T={T}: {len(tokens)} tokens, {clear.mean():.3f} clear of the 1e-4 cut, "
          f"mismatch fraction {mismatch:.4f}")
    assert same[clear].all(), np.nonzero(clear & ~same)
    assert np.abs(w_g[same] - w_o[same]).max() <= WEIGHT_ATOL
    assert clear.mean() > 0.5  # the comparison is not vacuous


@pytest.mark.parametrize("name,T", CASES)
def test_router_matches_oracle(name, T):
    check_router(W.WORKLOADS[name], T)


# DeepSeek-V4's score, the square root of a softplus, through both router
# paths (tensor-core pair; one launch for the fp32 gate below 8 tokens) and
# the grouped selection.
@pytest.mark.parametrize("name,T", [("qwen3", 1), ("qwen3", 64), ("qwen3", 4096), ("dsv3", 1),
                                    ("dsv3", 256), ("glm", 8), ("v4lo", 1), ("v4lo", 512)])
def test_router_sqrt_softplus(name, T):
    check_router(dataclasses.replace(W.WORKLOADS[name], scoring="sqrt_softplus"), T)


def test_router_ties_lowest_id_and_renorm():
    # all logits equal -> experts 0..k-1 in order, equal weights
    H, E, k = 64, 16, 4
    x = torch.zeros((3, H), dtype=torch.bfloat16, device="cuda")
    g = torch.randn((E, H), dtype=torch.float32, device="cuda").to(torch.bfloat16)
    for scoring in ("softmax", "sigmoid"):
        ids, wts = moe.router(x, g, None, k, scoring)
        torch.cuda.synchronize()
        assert (ids.cpu() == torch.arange(k, dtype=torch.int32)).all()
        assert torch.allclose(wts.cpu(), torch.full((3, k), 1.0 / k), atol=1e-7)


def test_router_zero_tokens_is_noop():
    g = torch.zeros((8, 64), dtype=torch.bfloat16, device="cuda")
    x = torch.zeros((0, 64), dtype=torch.bfloat16, device="cuda")
    ids, wts = moe.router(x, g, None, 2)
    assert ids.shape == (0, 2)


# Shapes around the tensor-core (tiled) router: the first tiled T, ragged
# 128-token tiles, one or two K splits, E from 16 to 512 (two MMAs of E/2
# above 256), bf16 and e4m3/fp32 operands.  Oracle on every token.
SMALL = [
    W.Workload("t1", H=128, E=64, k=4, F=0, scoring="softmax"),
    W.Workload("t2", H=256, E=288, k=8, F=0, scoring="sigmoid", bias=True),
    W.Workload("t3", H=192, E=16, k=2, F=0, scoring="softmax", renormalize=False, scaling=1.5),
    W.Workload("t4", H=256, E=512, k=16, F=0, scoring="sigmoid", bias=True, n_group=8,
               topk_group=4),
    W.Workload("t5", H=256, E=32, k=4, F=0, scoring="sigmoid", bias=True, lowbit=True),
]


@pytest.mark.parametrize("wi", range(len(SMALL)))
@pytest.mark.parametrize("T", [255, 256, 257, 300, 1000])
def test_tiled_router_shapes(wi, T):
    w = SMALL[wi]
    d = W.make_inputs(w, T, seed=T + wi, device="cuda", experts=False)
    ids, wts = moe.router(d["hidden"], d["gate"], d.get("bias"), w.k, w.scoring, w.n_group,
                          w.topk_group, w.renormalize, w.scaling,
                          hidden_scale=d.get("hidden_scale"))
    torch.cuda.synchronize()
    tokens = np.arange(T, dtype=np.int32)
    ids_o, w_o, gap = oracle_router(oracle, w, d, T, tokens)
    ids_g = ids.cpu().numpy()
    w_g = wts.cpu().numpy()
    clear = gap > GAP_MIN
    same = (ids_g == ids_o).all(axis=1)
    assert same[clear].all(), np.nonzero(clear & ~same)
    assert np.abs(w_g[same] - w_o[same]).max() <= WEIGHT_ATOL
    assert clear.mean() > 0.5
    x_dt = "e4m3" if w.lowbit else "bf16"
    g_dt = "f32" if w.lowbit else "bf16"
    assert moe.router_kernel_count(T, w.H, w.E, x_dt, g_dt) == (3 if w.lowbit else 2)


# The one-launch kernel: fp32 hidden rows, E not a multiple of 16, and fp32
# gates below 8 tokens.
@pytest.mark.parametrize("name,T,f32_hidden", [("qwen3", 1, True), ("qwen3", 64, True),
                                               ("dsv3", 200, True), ("glm", 9, True),
                                               ("v4lo", 1, False), ("v4lo", 7, False)])
def test_one_launch_router(name, T, f32_hidden):
    w = W.WORKLOADS[name]
    d = W.make_inputs(w, T, seed=T, device="cuda", experts=False)
    x = d["hidden"].float() if f32_hidden else d["hidden"]
    g_dt = "f32" if w.lowbit else "bf16"
    x_dt = "f32" if f32_hidden else ("e4m3" if w.lowbit else "bf16")
    assert moe.router_kernel_count(T, w.H, w.E, x_dt, g_dt) == 1
    ids, wts = moe.router(x, d["gate"], d.get("bias"), w.k, w.scoring, w.n_group,
                          w.topk_group, w.renormalize, w.scaling,
                          hidden_scale=d.get("hidden_scale"))
    torch.cuda.synchronize()
    tokens = np.arange(T, dtype=np.int32)
    ids_o, w_o, gap = oracle_router(oracle, w, d, T, tokens)
    ids_g, w_g = ids.cpu().numpy(), wts.cpu().numpy()
    clear = gap > GAP_MIN
    same = (ids_g == ids_o).all(axis=1)
    assert same[clear].all(), np.nonzero(clear & ~same)
    assert np.abs(w_g[same] - w_o[same]).max() <= WEIGHT_ATOL
    assert clear.any()
