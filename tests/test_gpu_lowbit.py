"""Low-bit expert path (FP8 e4m3 activations x FP4 e2m1 weights, one UE8M0
scale per 32 values; "How GPUs Fuse Communication and Computation During LLM
Inference" §1.1, §3.5) against the oracle fed the same dequantised values:
max|err| <= 6e-2 * max|ref| for the layer.  Also checked against the oracle's
emulation of the e4m3 re-quantisation of the intermediate, which the GPU path
performs, with a tighter bound."""
import numpy as np
import pytest
import torch

import oracle
from router_experts_gb300 import moe
from router_experts_gb300 import workloads as W

from _gpu import GAP_MIN, LAYER_RTOL_LOWBIT, WEIGHT_ATOL, blocks_covered, compact_experts, \
    covering_tokens, host, oracle_router, rel_err, sample_tokens

pytestmark = pytest.mark.gpu

_CACHE = {}


def v4lo_inputs(T, seed):
    key = (T, seed)
    if key not in _CACHE:
        _CACHE.clear()
        torch.cuda.empty_cache()
        _CACHE[key] = W.make_inputs(W.WORKLOADS["v4lo"], T, seed=seed, device="cuda")
    return _CACHE[key]


def oracle_ffn_lowbit(d, tokens, ids_rows, w_rows, w, emulate=0):
    w13h, w2h, rid, En, s13, s2 = compact_experts(d["w13"], d["w2"], ids_rows, d["w13_scale"],
                                                  d["w2_scale"])
    xh = host(d["hidden"])[tokens]
    xs = host(d["hidden_scale"])[tokens]
    return oracle.moe_ffn(xh, "e4m3", w13h, w2h, "e2m1", len(tokens), w.H, w.F, En, w.k, rid,
                          np.asarray(w_rows, np.float64), x_scale=xs, w13_scale=s13,
                          w2_scale=s2, emulate=emulate)


# T = 4096: at least 256 tokens covering every row block of the align output
@pytest.mark.parametrize("T,ntok", [(64, 12), (512, 12), (4096, 256)])
def test_lowbit_ffn_matches_oracle(T, ntok):
    w = W.WORKLOADS["v4lo"]
    d = v4lo_inputs(T, seed=2)
    ids, wts = W.random_routing(T, w.k, w.E, seed=T)
    BM = moe.pick_block_m(T, w.k, w.E)
    s, b, npp = moe.align(ids.cuda(), w.E, BM)
    stage = moe.grouped_ffn(d["hidden"], d["w13"], d["w2"], w.k, BM, s, b, npp, wts.cuda(),
                            x_scale=d["hidden_scale"], w13_scale=d["w13_scale"],
                            w2_scale=d["w2_scale"])
    y = moe.finalize(stage, T, w.k)
    torch.cuda.synchronize()
    s_h, npp_h = s.cpu().numpy(), int(npp.item())
    cover = ntok >= 256
    if cover:
        tokens, nblk = covering_tokens(s_h, npp_h, BM, T, w.k, np.ones(T, dtype=bool), ntok,
                                       seed=T)
    else:
        tokens, nblk = sample_tokens(T, ntok, seed=T), npp_h // BM
    got = y.float().cpu().numpy()[tokens]
    ref = oracle_ffn_lowbit(d, tokens, ids.numpy()[tokens], wts.numpy()[tokens], w)
    err = rel_err(got, ref)
    emu = oracle_ffn_lowbit(d, tokens, ids.numpy()[tokens], wts.numpy()[tokens], w, emulate=2)
    err_emu = rel_err(got, emu)
    ncov = blocks_covered(s_h, npp_h, BM, T, w.k, tokens)
    print(f"low-bit ffn T={T} BM={BM}: {len(tokens)} tokens, {ncov} of {nblk} row blocks, "
          f"rel err {err:.2e} (vs exact), {err_emu:.2e} (vs emulated re-quantisation)")
    assert np.isfinite(got).all()
    assert err <= LAYER_RTOL_LOWBIT
    assert err_emu <= 2e-2
    if cover:
        assert ncov == nblk


def test_lowbit_gemm_entry_points_compose():
    w = W.WORKLOADS["v4lo"]
    T = 64
    d = v4lo_inputs(T, seed=3)
    ids, wts = W.random_routing(T, w.k, w.E, seed=5)
    BM = moe.pick_block_m(T, w.k, w.E)
    s, b, npp = moe.align(ids.cuda(), w.E, BM)
    iq, isc = moe.expert_gemm1(d["hidden"], d["w13"], BM, s, b, npp, w.k,
                               x_scale=d["hidden_scale"], w13_scale=d["w13_scale"])
    st1 = moe.expert_gemm2(iq, d["w2"], T, w.k, BM, s, b, npp, wts.cuda(), inter_scale=isc,
                           w2_scale=d["w2_scale"])
    st2 = moe.grouped_ffn(d["hidden"], d["w13"], d["w2"], w.k, BM, s, b, npp, wts.cuda(),
                          x_scale=d["hidden_scale"], w13_scale=d["w13_scale"],
                          w2_scale=d["w2_scale"])
    torch.cuda.synchronize()
    assert torch.equal(st1, st2)
    # the intermediate scales are powers of two bounding every 32-block
    codes = iq[: int(npp.item())].cpu()
    assert codes.dtype == torch.uint8 and isc.dtype == torch.uint8



# GEMM1 reads its token rows permuted into the blocks' padded order when the
# workspace has room for the copy, and gathers them from x otherwise: the
# same tile contents and MMA order, so the same codes and scale bytes.  Pad
# rows are zero codes with scale byte 127 (2^0) in both, also after an
# earlier call left other token rows at those positions of the permuted copy.
@pytest.mark.parametrize("T,BM", [(64, 16), (512, 64), (1024, 128)])
def test_lowbit_gemm1_permuted_equals_gathered(T, BM):
    w = W.WORKLOADS["v4lo"]
    d = v4lo_inputs(T, seed=6)
    lib = moe.load()
    ws = moe.Workspace("cuda")
    small = moe.Workspace("cuda")
    for seed in (6, 8):
        ids, _ = W.random_routing(T, w.k, w.E, seed=seed, skew=1.1)
        s, b, npp = moe.align(ids.cuda(), w.E, BM)
        cap = s.numel()
        pq, ps = moe.expert_gemm1(d["hidden"], d["w13"], BM, s, b, npp, w.k, ws=ws,
                                  x_scale=d["hidden_scale"], w13_scale=d["w13_scale"])
        # a workspace of the header alone: the GEMM gathers the rows
        hdr = lib.moe_align_workspace_bytes()
        buf = small.get(hdr)
        gq = torch.empty((cap, w.F), dtype=torch.uint8, device="cuda")
        gs = torch.empty((cap, w.F // 32), dtype=torch.uint8, device="cuda")
        rc = lib.moe_expert_gemm1(moe._p(d["hidden"]), moe.DT_E4M3, moe._p(d["hidden_scale"]),
                                  moe._p(d["w13"]), moe._p(d["w13_scale"]), moe.DT_E2M1, T, w.H,
                                  w.F, w.E, w.k, BM, moe._p(s), moe._p(b), moe._p(npp), cap,
                                  moe._p(gq), moe._p(gs), moe._p(buf), hdr, moe._stream())
        assert rc == 0
        torch.cuda.synchronize()
        n = int(npp.item())
        pad = (s[:n] >= T * w.k)
        print(f"v4lo T={T} BM={BM} routing {seed}: {n // BM} row blocks, "
              f"{int(pad.sum())} pad rows")
        assert torch.equal(pq[:n], gq[:n]) and torch.equal(ps[:n], gs[:n])
        assert int(pad.sum()) > 0
        assert (pq[:n][pad] == 0).all() and (ps[:n][pad] == 127).all()
        assert moe.read_device_error(ws.buf) == 0

# T = 1 runs with single-assignment blocks (no align launch).  The oracle
# routes every token (fp32 router inputs: the dequantised hidden rows and the
# fp32 gate); at T = 4096 at least 256 tokens covering every row block are
# compared, on the oracle's routing where the margin is clear and on the
# GPU's for near-ties.
@pytest.mark.parametrize("T,ntok", [(1, 1), (8, 8), (512, 12), (4096, 256)])
def test_lowbit_layer_matches_oracle(T, ntok):
    w = W.WORKLOADS["v4lo"]
    d = v4lo_inputs(T, seed=0)
    y = moe.layer(d["hidden"], d["gate"], d["bias"], d["w13"], d["w2"], w.k, w.scoring,
                  renormalize=w.renormalize, scaling=w.scaling, hidden_scale=d["hidden_scale"],
                  w13_scale=d["w13_scale"], w2_scale=d["w2_scale"])
    ids_d, wts_d = moe.router(d["hidden"], d["gate"], d["bias"], w.k, w.scoring,
                              renormalize=w.renormalize, scaling=w.scaling,
                              hidden_scale=d["hidden_scale"])
    BM = moe.pick_block_m(T, w.k, w.E)
    s, _, npp = moe.align(ids_d, w.E, BM)
    torch.cuda.synchronize()
    ids_g, wts_g = ids_d.cpu().numpy(), wts_d.cpu().numpy().astype(np.float64)
    s_h, npp_h = s.cpu().numpy(), int(npp.item())
    ids_o, w_o, gap = oracle_router(oracle, w, d, T, np.arange(T, dtype=np.int32))
    clear = gap > GAP_MIN
    assert (ids_g[clear] == ids_o[clear]).all()
    same = (ids_g == ids_o).all(axis=1)
    assert np.abs(wts_g[same] - w_o[same]).max() <= WEIGHT_ATOL
    cover = ntok >= 256
    if cover:
        tokens, nblk = covering_tokens(s_h, npp_h, BM, T, w.k, clear, ntok, seed=T)
    else:
        tokens, nblk = sample_tokens(T, ntok, seed=T), npp_h // BM
    c = clear[tokens][:, None]
    ids_t = np.where(c, ids_o[tokens], ids_g[tokens])
    w_t = np.where(c, w_o[tokens], wts_g[tokens])
    ref = oracle_ffn_lowbit(d, tokens, ids_t, w_t, w)
    got = y.float().cpu().numpy()[tokens]
    err = rel_err(got, ref)
    ncov = blocks_covered(s_h, npp_h, BM, T, w.k, tokens)
    print(f"low-bit layer T={T}: {len(tokens)} tokens ({int(c.sum())} on the oracle's routing), "
          f"{ncov} of {nblk} row blocks, rel err {err:.2e}")
    assert np.isfinite(got).all()
    assert err <= LAYER_RTOL_LOWBIT
    if cover:
        assert ncov == nblk


def _shifted(t, off):
    """A copy of t whose data starts `off` bytes past a 16-byte boundary."""
    flat = t.reshape(-1)
    buf = torch.empty(flat.numel() + 16, dtype=t.dtype, device=t.device)
    view = buf[off:off + flat.numel()]
    view.copy_(flat)
    return view.view(t.shape)


# Small low-bit shapes: one 64-feature GEMM1 tile and one 128-column GEMM2 tile
# (H = 128, F = 128), several tiles with a ragged last block, BLOCK_M 16/64/128;
# scale rows of 16 bytes (H = F = 512: one group of 4 K steps copied whole) and
# the same with the scale arrays 4 bytes off a 16-byte boundary (word copies).
@pytest.mark.parametrize("T,E,k,H,F,BM,off", [(5, 8, 2, 128, 128, 16, 0),
                                              (40, 8, 2, 256, 128, 16, 0),
                                              (300, 16, 4, 256, 256, 64, 0),
                                              (700, 8, 2, 384, 128, 128, 0),
                                              (200, 8, 2, 512, 512, 64, 0),
                                              (200, 8, 2, 512, 512, 64, 4)])
def test_lowbit_small_shapes(T, E, k, H, F, BM, off):
    w = W.Workload("lb", H=H, E=E, k=k, F=F, scoring="sigmoid", bias=True, lowbit=True)
    d = W.make_inputs(w, T, seed=T, device="cuda")
    if off:
        for key in ("hidden_scale", "w13_scale", "w2_scale"):
            d[key] = _shifted(d[key], off)
    ids, wts = W.random_routing(T, k, E, seed=T)
    s, b, n = moe.align(ids.cuda(), E, BM)
    out = moe.grouped_ffn(d["hidden"], d["w13"], d["w2"], k, BM, s, b, n, wts.cuda(),
                          x_scale=d["hidden_scale"], w13_scale=d["w13_scale"],
                          w2_scale=d["w2_scale"])
    y = moe.finalize(out, T, k)
    torch.cuda.synchronize()
    tokens = np.arange(T, dtype=np.int32)
    ref = oracle_ffn_lowbit(d, tokens, ids.numpy(), wts.numpy(), w)
    err = rel_err(y.float().cpu().numpy(), ref)
    print(f"low-bit T={T} E={E} k={k} H={H} F={F} BM={BM} scale offset {off}: rel err {err:.2e}")
    assert err <= LAYER_RTOL_LOWBIT


# ---- FP8 cast of a bf16 layer input ("How GPUs Fuse ..." §1.1, §3.5) ---------

def test_cast_is_bit_exact_against_the_oracle():
    T, H = 300, 512
    g = torch.Generator(device="cpu").manual_seed(9)
    x = torch.randn((T, H), generator=g, dtype=torch.float32)
    # per-group magnitudes from 2^-140 (bf16 subnormals: the scale clamps at
    # 2^-127) to 2^60, an all-zero group, negative zeros, exact 448 multiples
    mag = torch.exp2(torch.randint(-140, 61, (T, H // 32), generator=g).float())
    x = x * mag.repeat_interleave(32, dim=1)
    x[0, :32] = 0.0
    x[1, :32] = -0.0
    x[2, :32] = 448.0 * 2.0 ** 5
    x[3, 5] = -0.0
    xb = x.to(torch.bfloat16)
    codes, scales = moe.cast_e4m3(xb.cuda())
    torch.cuda.synchronize()
    co, so = oracle.quantize_e4m3(host(xb), "bf16", T, H)
    assert np.array_equal(scales.cpu().numpy(), so)
    assert np.array_equal(codes.cpu().numpy(), co)
    assert scales[2, 0].item() == 127 + 5 and scales[0, 0].item() == 127


# The router's selection launch writes the FP8 cast next to the ids and
# weights ("How GPUs Fuse ..." §1.1): codes and scales bit-exact against the
# oracle's cast, ids and weights against the oracle's routing of the bf16 rows,
# on both router paths (one launch below 8 tokens with an fp32 gate, tensor
# cores from 8) and a bf16 gate.
@pytest.mark.parametrize("T,gate_f32", [(1, True), (7, True), (8, True), (300, True),
                                        (4096, True), (64, False)])
def test_router_writes_the_fp8_cast(T, gate_f32):
    w = W.WORKLOADS["v4lo"]
    d = W.make_inputs(w, T, seed=6, device="cuda", experts=False)
    g = torch.Generator(device="cuda").manual_seed(T + 1)
    xb = torch.randn((T, w.H), generator=g, device="cuda", dtype=torch.float32).to(torch.bfloat16)
    gate = d["gate"] if gate_f32 else d["gate"].to(torch.bfloat16)
    ids, wts, codes, scales = moe.router_cast_e4m3(xb, gate, d["bias"], w.k, w.scoring,
                                                   renormalize=w.renormalize, scaling=w.scaling)
    torch.cuda.synchronize()
    co, so = oracle.quantize_e4m3(host(xb), "bf16", T, w.H)
    assert np.array_equal(codes.cpu().numpy(), co)
    assert np.array_equal(scales.cpu().numpy(), so)
    ids_o, w_o, gap = oracle.router(host(xb), "bf16", host(gate), "f32" if gate_f32 else "bf16",
                                    d["bias"].cpu().numpy(), T, w.H, w.E, w.k, w.scoring,
                                    renormalize=w.renormalize, scaling=w.scaling)
    clear = gap > GAP_MIN
    ids_h, wts_h = ids.cpu().numpy(), wts.cpu().numpy()
    assert (ids_h[clear] == ids_o[clear]).all()
    same = (ids_h == ids_o).all(axis=1)
    assert np.abs(wts_h[same] - w_o[same]).max() <= WEIGHT_ATOL
    print(f"router + FP8 cast T={T}: codes and scales bit-exact, {int(clear.sum())} tokens "
          f"clear of the cut")


@pytest.mark.parametrize("T,ntok", [(1, 1), (64, 16), (512, 12)])
def test_bf16_input_lowbit_layer_matches_oracle(T, ntok):
    w = W.WORKLOADS["v4lo"]
    d = v4lo_inputs(T, seed=4)
    g = torch.Generator(device="cuda").manual_seed(T)
    xb = torch.randn((T, w.H), generator=g, device="cuda", dtype=torch.float32).to(torch.bfloat16)
    y = moe.layer(xb, d["gate"], d["bias"], d["w13"], d["w2"], w.k, w.scoring,
                  renormalize=w.renormalize, scaling=w.scaling, w13_scale=d["w13_scale"],
                  w2_scale=d["w2_scale"])
    torch.cuda.synchronize()
    align = 0 if T == 1 else 1
    # router (+ the cast in its selection launch), align, GEMM1, GEMM2, finalize
    assert moe.layer_kernel_count(T, w.H, w.F, w.E, w.k, "bf16", "f32", "e2m1") == \
        moe.router_kernel_count(T, w.H, w.E, "bf16", "f32") + 3 + align
    tokens = sample_tokens(T, ntok, seed=T)
    # the router reads the bf16 rows; the experts read the oracle's own cast
    ids_o, w_o, gap = oracle.router(host(xb), "bf16", host(d["gate"]), "f32",
                                    d["bias"].cpu().numpy(), T, w.H, w.E, w.k, w.scoring,
                                    renormalize=w.renormalize, scaling=w.scaling, tokens=tokens)
    keep = gap > GAP_MIN
    tokens, ids_o, w_o = tokens[keep], ids_o[keep], w_o[keep]
    codes, scales = oracle.quantize_e4m3(host(xb), "bf16", T, w.H)
    w13h, w2h, rid, En, s13, s2 = compact_experts(d["w13"], d["w2"], ids_o, d["w13_scale"],
                                                  d["w2_scale"])
    ref = oracle.moe_ffn(codes[tokens], "e4m3", w13h, w2h, "e2m1", len(tokens), w.H, w.F, En,
                         w.k, rid, np.asarray(w_o, np.float64), x_scale=scales[tokens],
                         w13_scale=s13, w2_scale=s2)
    got = y.float().cpu().numpy()[tokens]
    err = rel_err(got, ref)
    print(f"bf16-input low-bit layer T={T}: {len(tokens)} tokens, rel err {err:.2e}")
    assert len(tokens) > 0 and np.isfinite(got).all()
    assert err <= LAYER_RTOL_LOWBIT
