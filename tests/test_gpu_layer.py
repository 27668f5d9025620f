"""The fused layer (router -> align -> GEMM1+SwiGLU -> GEMM2 -> finalize in one
call) against the oracle layer (which routes on its own, in fp64) on the same
seeded inputs, over sampled tokens whose routing margin exceeds 1e-4."""
import numpy as np
import pytest
import torch

import oracle
from router_experts_gb300 import moe
from router_experts_gb300 import workloads as W

from _gpu import GAP_MIN, LAYER_RTOL_BF16, compact_experts, host, oracle_router, rel_err, \
    sample_tokens

pytestmark = pytest.mark.gpu


def layer_case(name, T, ntok, block_m=0, seed=0):
    w = W.WORKLOADS[name]
    # small batches may have no token clear of the 1e-4 cut: try further seeds
    for seed in range(seed, seed + 10):
        d = W.make_inputs(w, T, seed=seed, device="cuda")
        tokens = sample_tokens(T, ntok, seed=seed)
        ids_o, w_o, gap = oracle_router(oracle, w, d, T, tokens)
        keep = gap > GAP_MIN
        if keep.any():
            break
    y = moe.layer(d["hidden"], d["gate"], d.get("bias"), d["w13"], d["w2"], w.k, w.scoring,
                  w.n_group, w.topk_group, w.renormalize, w.scaling, block_m=block_m)
    torch.cuda.synchronize()
    tokens, ids_o, w_o = tokens[keep], ids_o[keep], w_o[keep]
    w13h, w2h, rid, En = compact_experts(d["w13"], d["w2"], ids_o)
    ref = oracle.moe_ffn(host(d["hidden"])[tokens], "bf16", w13h, w2h, "bf16", len(tokens), w.H,
                         w.F, En, w.k, rid, w_o)
    got = y.float().cpu().numpy()[tokens]
    err = rel_err(got, ref)
    print(f"layer {name} T={T}: {len(tokens)} tokens compared, rel max err {err:.2e}")
    assert len(tokens) > 0 and np.isfinite(got).all()
    assert err <= LAYER_RTOL_BF16


@pytest.mark.parametrize("name,T,ntok", [("toy", 16, 16), ("qwen3", 1, 1), ("qwen3", 64, 32),
                                         ("qwen3", 512, 32), ("qwen3", 4096, 32),
                                         ("dsv3", 1, 1), ("dsv3", 256, 12), ("dsv3", 4096, 12)])
def test_layer_matches_oracle(name, T, ntok):
    layer_case(name, T, ntok)


def test_layer_zero_tokens():
    w = W.WORKLOADS["toy"]
    d = W.make_inputs(w, 1, device="cuda")
    y = moe.layer(d["hidden"][:0], d["gate"], None, d["w13"], d["w2"], w.k)
    assert y.shape == (0, w.H)


def test_layer_is_deterministic():
    w = W.WORKLOADS["qwen3"]
    d = W.make_inputs(w, 512, seed=5, device="cuda")
    a = moe.layer(d["hidden"], d["gate"], None, d["w13"], d["w2"], w.k)
    b = moe.layer(d["hidden"], d["gate"], None, d["w13"], d["w2"], w.k)
    torch.cuda.synchronize()
    assert torch.equal(a, b)
    ws = moe.default_workspace("cuda")
    assert moe.read_device_error(ws.buf) == 0


# The layer must equal the separate public calls (router, align, grouped FFN,
# finalize) bit for bit: across the align kernel's one-CTA / many-CTA switch at
# T*k = 512, and at one token, where the layer skips the align launch and
# uses single-assignment blocks (a token's experts are distinct, so these are
# align's blocks).
@pytest.mark.parametrize("name,T", [("qwen3", 1), ("qwen3", 2), ("qwen3", 3), ("qwen3", 13),
                                    ("qwen3", 64), ("qwen3", 65), ("qwen3", 255), ("qwen3", 256),
                                    ("qwen3", 257), ("dsv3", 1), ("dsv3", 2), ("dsv3", 256)])
def test_layer_equals_separate_calls(name, T):
    w = W.WORKLOADS[name]
    d = W.make_inputs(w, T, seed=11, device="cuda")
    bm = moe.pick_block_m(T, w.k, w.E)
    y = moe.layer(d["hidden"], d["gate"], d.get("bias"), d["w13"], d["w2"], w.k, w.scoring,
                  w.n_group, w.topk_group, w.renormalize, w.scaling)
    ids, wts = moe.router(d["hidden"], d["gate"], d.get("bias"), w.k, w.scoring, w.n_group,
                          w.topk_group, w.renormalize, w.scaling)
    s, b, n = moe.align(ids, w.E, bm)
    st = moe.grouped_ffn(d["hidden"], d["w13"], d["w2"], w.k, bm, s, b, n, wts)
    y2 = moe.finalize(st, T, w.k)
    torch.cuda.synchronize()
    print(f"layer {name} T={T}: equal to the separate calls")
    assert moe.layer_kernel_count(T, w.H, w.F, w.E, w.k) == (5 if T == 1 else 6)
    assert torch.equal(y, y2)
    assert moe.read_device_error(moe.default_workspace("cuda").buf) == 0


def test_layer_refuses_strided_tensors():
    # the kernels read dense row-major buffers: a transposed view is refused
    # before anything is launched
    w = W.WORKLOADS["toy"]
    d = W.make_inputs(w, 64, seed=3, device="cuda")
    xt = d["hidden"].reshape(w.H, 64).t()  # [64, H] view, not contiguous
    with pytest.raises(ValueError, match="contiguous"):
        moe.layer(xt, d["gate"], None, d["w13"], d["w2"], w.k)
