"""The fused layer (router -> align -> GEMM1+SwiGLU -> GEMM2 -> finalize in one
call) against the oracle on the same seeded inputs.

Routing: the oracle routes every token in fp64; the GPU's ids must equal the
oracle's wherever the margin at the cut exceeds 1e-4 and its weights must be
within 1e-5 wherever the ids agree.  Output: the compared tokens are all
tokens (up to Qwen3 T = 4096), or, at the DeepSeek-V3 sizes, at least 256
tokens chosen so that every row block of the align output holds one of their
assignments (the ragged last block of every touched expert included).  Each
compared token's output is checked against the oracle's naive per-expert loop
fed the oracle's own routing, or, for a token whose margin is within 1e-4
(a near-tie that fp32 summation order may flip), the GPU's routing."""
import numpy as np
import pytest
import torch

import oracle
from router_experts_gb300 import moe
from router_experts_gb300 import workloads as W

from _gpu import GAP_MIN, LAYER_RTOL_BF16, WEIGHT_ATOL, blocks_covered, compact_experts, \
    covering_tokens, host, oracle_router, rel_err, sample_tokens

pytestmark = pytest.mark.gpu


def check_routing(w, d, T, ids_g, wts_g):
    """Oracle routing of every token; the GPU's ids and weights against it.
    Returns (oracle ids, oracle weights, clear-margin mask)."""
    ids_o, w_o, gap = oracle_router(oracle, w, d, T, np.arange(T, dtype=np.int32))
    clear = gap > GAP_MIN
    assert (ids_g[clear] == ids_o[clear]).all(), np.nonzero((ids_g != ids_o).any(1) & clear)[0]
    same = (ids_g == ids_o).all(axis=1)
    assert same.any() and np.abs(wts_g[same] - w_o[same]).max() <= WEIGHT_ATOL
    return ids_o, w_o, clear


def layer_case(name, T, ntok, cover=False, seed=0):
    w = W.WORKLOADS[name]
    d = W.make_inputs(w, T, seed=seed, device="cuda")
    y = moe.layer(d["hidden"], d["gate"], d.get("bias"), d["w13"], d["w2"], w.k, w.scoring,
                  w.n_group, w.topk_group, w.renormalize, w.scaling)
    # the layer's own routing and blocks (the same kernels; the layer equals
    # these separate calls bit for bit, test_layer_equals_separate_calls)
    ids_d, wts_d = moe.router(d["hidden"], d["gate"], d.get("bias"), w.k, w.scoring, w.n_group,
                              w.topk_group, w.renormalize, w.scaling)
    bm = moe.pick_block_m(T, w.k, w.E)
    s, _, npp = moe.align(ids_d, w.E, bm)
    torch.cuda.synchronize()
    ids_g = ids_d.cpu().numpy()
    wts_g = wts_d.cpu().numpy().astype(np.float64)
    s_h, npp_h = s.cpu().numpy(), int(npp.item())
    ids_o, w_o, clear = check_routing(w, d, T, ids_g, wts_g)
    nblk = npp_h // bm
    if ntok >= T:
        tokens = np.arange(T, dtype=np.int32)
    elif cover:
        tokens, nblk = covering_tokens(s_h, npp_h, bm, T, w.k, clear, ntok, seed=seed)
    else:
        tokens = sample_tokens(T, ntok, seed=seed)
    # the oracle's routing where the margin is clear, the GPU's on near-ties
    c = clear[tokens][:, None]
    ids_t = np.where(c, ids_o[tokens], ids_g[tokens])
    w_t = np.where(c, w_o[tokens], wts_g[tokens])
    w13h, w2h, rid, En = compact_experts(d["w13"], d["w2"], ids_t)
    ref = oracle.moe_ffn(host(d["hidden"])[tokens], "bf16", w13h, w2h, "bf16", len(tokens), w.H,
                         w.F, En, w.k, rid, w_t)
    got = y.float().cpu().numpy()[tokens]
    err = rel_err(got, ref)
    ncov = blocks_covered(s_h, npp_h, bm, T, w.k, tokens)
    print(f"layer {name} T={T}: {len(tokens)} tokens compared ({int(c.sum())} on the oracle's "
          f"routing, {int((~c).sum())} near-ties on the GPU's), {ncov} of {nblk} row blocks "
          f"(BLOCK_M {bm}), {int(clear.sum())} of {T} tokens clear of the cut, "
          f"rel max err {err:.2e}")
    assert np.isfinite(got).all()
    assert err <= LAYER_RTOL_BF16
    if cover or ntok >= T:
        assert ncov == nblk


@pytest.mark.parametrize("name,T,ntok,cover", [
    ("toy", 16, 16, False), ("qwen3", 1, 1, False), ("qwen3", 64, 64, False),
    ("qwen3", 512, 512, False), ("qwen3", 4096, 4096, False),
    ("dsv3", 1, 1, False), ("dsv3", 256, 64, True), ("dsv3", 4096, 256, True)])
def test_layer_matches_oracle(name, T, ntok, cover):
    layer_case(name, T, ntok, cover)


# 64-bit offsets ("MoE Kernels, in depth", Failure modes: row offsets ids*H in
# 32-bit arithmetic overflow for large prefill batches).  40,000 tokens x k 8
# x H 7,168: the staged rows hold 2.29e9 elements (4.6 GB), past 2^31 both in
# bytes and in elements; a few compact experts keep the work small.  The
# compared tokens include the last ones, whose staged rows lie beyond 2^31
# elements.
BIG = W.Workload("big_offsets", H=7168, E=16, k=8, F=256, scoring="softmax")


def test_layer_64bit_offsets():
    w, T = BIG, 40000
    assert T * w.k * w.H > 2 ** 31
    d = W.make_inputs(w, T, seed=4, device="cuda")
    ws = moe.Workspace("cuda")
    y = moe.layer(d["hidden"], d["gate"], None, d["w13"], d["w2"], w.k, w.scoring, ws=ws)
    torch.cuda.synchronize()
    assert moe.read_device_error(ws.buf) == 0
    first_beyond = -(-(2 ** 31) // (w.k * w.H))  # first token with a row past 2^31 elements
    tokens = np.unique(np.concatenate([np.arange(0, 8), np.arange(first_beyond - 4, first_beyond + 4),
                                       np.arange(T - 16, T)])).astype(np.int32)
    ids_o, w_o, gap = oracle_router(oracle, w, d, T, tokens)
    keep = gap > GAP_MIN
    tokens, ids_o, w_o = tokens[keep], ids_o[keep], w_o[keep]
    assert (tokens >= first_beyond).sum() >= 8
    w13h, w2h, rid, En = compact_experts(d["w13"], d["w2"], ids_o)
    ref = oracle.moe_ffn(host(d["hidden"])[tokens], "bf16", w13h, w2h, "bf16", len(tokens), w.H,
                         w.F, En, w.k, rid, w_o)
    got = y.float().cpu().numpy()[tokens]
    err = rel_err(got, ref)
    print(f"64-bit offsets: T={T}, {len(tokens)} tokens ({int((tokens >= first_beyond).sum())} "
          f"past 2^31 staged elements), rel max err {err:.2e}")
    assert np.isfinite(got).all()
    assert err <= LAYER_RTOL_BF16
    del ws, y, d
    torch.cuda.empty_cache()


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
    # router (one launch up to 4 tokens), align (none at one token), GEMM1,
    # GEMM2, finalize
    router = 1 if T <= 4 else 2
    assert moe.router_kernel_count(T, w.H, w.E) == router
    assert moe.layer_kernel_count(T, w.H, w.F, w.E, w.k) == router + (0 if T == 1 else 1) + 3
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


def test_layer_workspace_reused_across_shapes():
    # One workspace through calls of several shapes (16-, 64- and one-token
    # blocks): the layout of each call puts its regions where earlier calls
    # left other data, and whatever must start at zero lives in the header
    # or is reset by its last user, so every call still gives the separate
    # calls' bits.
    w = W.WORKLOADS["qwen3"]
    ws = moe.Workspace("cuda")
    for T in (300, 64, 7, 33, 1, 64):
        d = W.make_inputs(w, T, seed=T, device="cuda")
        y = moe.layer(d["hidden"], d["gate"], d.get("bias"), d["w13"], d["w2"], w.k, w.scoring,
                      ws=ws)
        ids, wts = moe.router(d["hidden"], d["gate"], d.get("bias"), w.k, w.scoring)
        bm = moe.pick_block_m(T, w.k, w.E)
        s, b, n = moe.align(ids, w.E, bm)
        st = moe.grouped_ffn(d["hidden"], d["w13"], d["w2"], w.k, bm, s, b, n, wts)
        y2 = moe.finalize(st, T, w.k)
        torch.cuda.synchronize()
        print(f"layer qwen3 T={T} (BLOCK_M {bm}) on a reused workspace: equal to the separate calls")
        assert torch.equal(y, y2)
        assert moe.read_device_error(ws.buf) == 0
