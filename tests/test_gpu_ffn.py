"""Grouped expert GEMMs (tcgen05) + finalize on the GPU against the oracle's
naive per-expert loop on the same seeded inputs and the same (synthetic)
routing: max|err| <= 2e-2 * max|ref| over the compared tokens.  Every tile
variant is exercised (BLOCK_M 16 / 64 swap tiles with and without split-K,
BLOCK_M 128 tiles), plus skewed and single-expert routings."""
import numpy as np
import pytest
import torch

import oracle
from router_experts_gb300 import moe
from router_experts_gb300 import workloads as W

from _gpu import LAYER_RTOL_BF16, blocks_covered, compact_experts, covering_tokens, host, \
    rel_err, sample_tokens

pytestmark = pytest.mark.gpu


def ffn_case(name, T, BM, skew=0.0, ntok=64, seed=1, ids=None, cover=False):
    """ntok >= T compares every token; cover=True picks at least ntok tokens
    so that every row block of the align output holds one of their
    assignments."""
    w = W.WORKLOADS[name] if isinstance(name, str) else name
    name = w.name
    d = W.make_inputs(w, T, seed=seed, device="cuda")
    if ids is None:
        ids, wts = W.random_routing(T, w.k, w.E, seed=seed, skew=skew)
    else:
        wts = torch.rand(ids.shape, dtype=torch.float32) * 0.9 + 0.1
    ids_d, wts_d = ids.cuda(), wts.cuda()
    s, b, npp = moe.align(ids_d, w.E, BM)
    stage = moe.grouped_ffn(d["hidden"], d["w13"], d["w2"], w.k, BM, s, b, npp, wts_d)
    y = moe.finalize(stage, T, w.k)
    torch.cuda.synchronize()
    s_h, npp_h = s.cpu().numpy(), int(npp.item())
    nblk = npp_h // BM
    if ntok >= T:
        tokens = np.arange(T, dtype=np.int32)
    elif cover:
        tokens, nblk = covering_tokens(s_h, npp_h, BM, T, w.k, np.ones(T, dtype=bool), ntok,
                                       seed=seed)
    else:
        tokens = sample_tokens(T, ntok, seed=seed)
    rows = ids.numpy()[tokens]
    w13h, w2h, rid, En = compact_experts(d["w13"], d["w2"], rows)
    xh = host(d["hidden"])[tokens]
    ref = oracle.moe_ffn(xh, "bf16", w13h, w2h, "bf16", len(tokens), w.H, w.F, En, w.k, rid,
                         wts.numpy()[tokens].astype(np.float64))
    got = y.float().cpu().numpy()[tokens]
    err = rel_err(got, ref)
    ncov = blocks_covered(s_h, npp_h, BM, T, w.k, tokens)
    print(f"{name} T={T} BM={BM} skew={skew}: {len(tokens)} tokens, {ncov} of {nblk} row "
          f"blocks, rel max err {err:.2e}")
    assert np.isfinite(got).all()
    assert err <= LAYER_RTOL_BF16
    if cover or ntok >= T:
        assert ncov == nblk
    return err


# every token is compared (Qwen3 T = 4096 included: all 32,768 assignments)
@pytest.mark.parametrize("name,T,BM", [("toy", 16, 16), ("toy", 16, 64), ("toy", 16, 128),
                                       ("qwen3", 1, 16), ("qwen3", 64, 16), ("qwen3", 64, 64),
                                       ("qwen3", 64, 128), ("qwen3", 512, 64),
                                       ("qwen3", 4096, 128), ("qwen3", 4096, 64)])
def test_ffn_matches_oracle(name, T, BM):
    ffn_case(name, T, BM, ntok=T)


# skewed routing on the 22.5 GB workload: tokens covering every row block
@pytest.mark.parametrize("name,T,BM,ntok", [("dsv3", 1, 16, 1), ("dsv3", 256, 64, 64),
                                            ("dsv3", 4096, 128, 256)])
def test_ffn_dsv3(name, T, BM, ntok):
    ffn_case(name, T, BM, skew=1.1, ntok=ntok, cover=True)


@pytest.mark.parametrize("BM", [16, 128])
def test_ffn_all_tokens_one_expert(BM):
    T = 300
    ids = torch.full((T, 2), 0, dtype=torch.int32)
    ids[:, 1] = 5
    ffn_case("toy", T, BM, ids=ids, ntok=40)


# 128-row tiles at sizes off the tile grid: F % 64 == 32 (GEMM2 ends on a
# half K step, zero-filled by the copy), F below one 128-column tile, H below
# and above 4096 (four and two gather warps), every expert with a pair of
# blocks and an odd last block
@pytest.mark.parametrize("H,F", [(128, 96), (4160, 96), (4160, 160)])
def test_ffn_row_tiles_off_grid(H, F):
    w = W.Workload("offgrid", H=H, E=4, k=2, F=F, scoring="softmax")
    ffn_case(w, 600, 128, ntok=600)


@pytest.mark.parametrize("BM", [16, 64])
def test_ffn_heavy_skew(BM):
    ffn_case("qwen3", 200, BM, skew=3.0, ntok=48)


def test_gemm_entry_points_compose_like_grouped_ffn():
    w = W.WORKLOADS["qwen3"]
    T, BM = 64, 16
    d = W.make_inputs(w, T, seed=3, device="cuda")
    ids, wts = W.random_routing(T, w.k, w.E, seed=3)
    s, b, npp = moe.align(ids.cuda(), w.E, BM)
    inter = moe.expert_gemm1(d["hidden"], d["w13"], BM, s, b, npp, w.k)
    st1 = moe.expert_gemm2(inter, d["w2"], T, w.k, BM, s, b, npp, wts.cuda())
    st2 = moe.grouped_ffn(d["hidden"], d["w13"], d["w2"], w.k, BM, s, b, npp, wts.cuda())
    torch.cuda.synchronize()
    assert torch.equal(st1, st2)
