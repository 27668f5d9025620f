"""The whole layer in one persistent kernel (moe_layer_persistent, small
batches) against the oracle, and against the separate entry points fed the
kernel's own routing.

"How GPUs Fuse Communication and Computation During LLM Inference" §3.3 -
§3.6: one kernel routes, aligns, runs GEMM1 and GEMM2 with readiness counters
between them and combines.  Parity: every token whose routing margin exceeds
1e-4 is compared with the oracle's layer (its own fp64 routing); the kernel's
ids must equal the oracle's there and its weights be within 1e-5; every other
token is compared with the oracle's experts fed the kernel's routing.  The
separate entry points (align with BLOCK_M 16, grouped FFN, finalize) fed the
kernel's routing give the same output bit for bit: the same blocks, split
counts, MMA order and slot-order combine."""
import numpy as np
import pytest
import torch

import oracle
from router_experts_gb300 import moe
from router_experts_gb300 import workloads as W

from _gpu import GAP_MIN, LAYER_RTOL_BF16, WEIGHT_ATOL, blocks_covered, compact_experts, host, \
    oracle_router, rel_err

pytestmark = pytest.mark.gpu

_CACHE = {}


def inputs(name, T, seed):
    key = (name, T, seed)
    if key not in _CACHE:
        _CACHE.clear()
        torch.cuda.empty_cache()
        _CACHE[key] = W.make_inputs(W.WORKLOADS[name], T, seed=seed, device="cuda")
    return _CACHE[key]


def run_persistent(w, d, T, ws=None):
    ids = torch.full((T, w.k), -1, dtype=torch.int32, device="cuda")
    wts = torch.zeros((T, w.k), dtype=torch.float32, device="cuda")
    y = moe.layer_persistent(d["hidden"], d["gate"], d.get("bias"), d["w13"], d["w2"], w.k,
                             w.scoring, w.n_group, w.topk_group, w.renormalize, w.scaling,
                             ws=ws, routing=(ids, wts))
    return y, ids, wts


@pytest.mark.parametrize("name,T", [("qwen3", 1), ("qwen3", 4), ("qwen3", 16), ("qwen3", 64),
                                    ("qwen3", 3), ("dsv3", 1), ("dsv3", 4), ("dsv3", 16),
                                    ("dsv3", 64)])
def test_persistent_layer_matches_oracle(name, T):
    w = W.WORKLOADS[name]
    d = inputs(name, T, seed=7)
    ws = moe.Workspace("cuda")
    y, ids_d, wts_d = run_persistent(w, d, T, ws)
    torch.cuda.synchronize()
    assert moe.read_device_error(ws.buf) == 0
    ids_g, wts_g = ids_d.cpu().numpy(), wts_d.cpu().numpy().astype(np.float64)
    tokens = np.arange(T, dtype=np.int32)
    ids_o, w_o, gap = oracle_router(oracle, w, d, T, tokens)
    clear = gap > GAP_MIN
    assert (ids_g[clear] == ids_o[clear]).all()
    same = (ids_g == ids_o).all(axis=1)
    assert np.abs(wts_g[same] - w_o[same]).max() <= WEIGHT_ATOL
    c = clear[:, None]
    ids_t = np.where(c, ids_o, ids_g)
    w_t = np.where(c, w_o, wts_g)
    w13h, w2h, rid, En = compact_experts(d["w13"], d["w2"], ids_t)
    ref = oracle.moe_ffn(host(d["hidden"]), "bf16", w13h, w2h, "bf16", T, w.H, w.F, En, w.k, rid,
                         w_t)
    got = y.float().cpu().numpy()
    err = rel_err(got, ref)
    s, _, npp = moe.align(ids_d, w.E, 16)
    npp_h = int(npp.item())
    ncov = blocks_covered(s.cpu().numpy(), npp_h, 16, T, w.k, tokens)
    print(f"persistent layer {name} T={T}: {T} tokens ({int(clear.sum())} on the oracle's "
          f"routing), {ncov} of {npp_h // 16} row blocks, rel max err {err:.2e}")
    assert np.isfinite(got).all()
    assert err <= LAYER_RTOL_BF16
    assert ncov == npp_h // 16


@pytest.mark.parametrize("name,T", [("qwen3", 1), ("qwen3", 7), ("qwen3", 64), ("dsv3", 1),
                                    ("dsv3", 33), ("dsv3", 64)])
def test_persistent_equals_separate_calls_on_its_routing(name, T):
    w = W.WORKLOADS[name]
    d = inputs(name, T, seed=3)
    y, ids, wts = run_persistent(w, d, T)
    s, b, npp = moe.align(ids, w.E, 16)
    st = moe.grouped_ffn(d["hidden"], d["w13"], d["w2"], w.k, 16, s, b, npp, wts)
    y2 = moe.finalize(st, T, w.k)
    torch.cuda.synchronize()
    print(f"persistent {name} T={T}: equal to align + grouped FFN + finalize on its routing")
    assert torch.equal(y, y2)


def test_persistent_repeats_and_replays_in_a_graph():
    # the counters the last CTA resets must leave the workspace ready for the
    # next launch: eager calls in a row and graph replays give the same bits
    w = W.WORKLOADS["qwen3"]
    T = 16
    d = inputs("qwen3", T, seed=5)
    ws = moe.Workspace("cuda")
    out = torch.empty((T, w.H), dtype=torch.bfloat16, device="cuda")
    a = moe.layer_persistent(d["hidden"], d["gate"], None, d["w13"], d["w2"], w.k, ws=ws).clone()
    b = moe.layer_persistent(d["hidden"], d["gate"], None, d["w13"], d["w2"], w.k, ws=ws).clone()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        moe.layer_persistent(d["hidden"], d["gate"], None, d["w13"], d["w2"], w.k, ws=ws, out=out)
    for _ in range(5):
        out.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(out, a)
    torch.cuda.synchronize()
    assert torch.equal(a, b)
    assert moe.read_device_error(ws.buf) == 0


def test_persistent_zero_tokens_and_limits():
    w = W.WORKLOADS["qwen3"]
    d = inputs("qwen3", 64, seed=1)
    y = moe.layer_persistent(d["hidden"][:0], d["gate"], None, d["w13"], d["w2"], w.k)
    assert y.shape == (0, w.H)
    # T*k above 512 is outside the persistent kernel's limits
    assert moe.layer_persistent_workspace_bytes(65, w.H, w.F, w.E, w.k) == 0
    assert moe.layer_persistent_workspace_bytes(64, w.H, w.F, w.E, w.k) > 0
