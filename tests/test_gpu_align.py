"""moe_align on the GPU is bit-exact against the oracle align given the same
topk_ids (seeded synthetic routings), including skewed, empty, single-token
and maximum-size cases ("MoE Kernels, in depth", Failure modes: counts of 0,
1 and exactly BLOCK_M per expert)."""
import numpy as np
import pytest
import torch

import oracle
from router_experts_gb300 import moe
from router_experts_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def run_both(ids, E, BM):
    T, k = ids.shape
    s, b, npp = moe.align(ids.cuda(), E, BM)
    so, bo, nppo = oracle.align(ids.numpy(), T, k, E, BM)
    torch.cuda.synchronize()
    assert int(npp.item()) == nppo
    assert np.array_equal(s.cpu().numpy(), so)
    assert np.array_equal(b.cpu().numpy(), bo)


@pytest.mark.parametrize("BM", [16, 64, 128])
@pytest.mark.parametrize("T", [1, 8, 64, 65, 512, 4096])
def test_glm_shapes(T, BM):
    ids, _ = W.random_routing(T, 8, 288, seed=T + BM)
    run_both(ids, 288, BM)


@pytest.mark.parametrize("T,k,E,BM,skew", [(16, 2, 8, 16, 0.0), (4096, 8, 128, 128, 0.0),
                                           (4096, 8, 256, 128, 1.1), (256, 8, 256, 64, 3.0),
                                           (1000, 6, 256, 64, 1.1), (4096, 8, 1024, 16, 0.5),
                                           (3, 1, 4, 16, 0.0), (20000, 8, 64, 128, 2.0),
                                           (100, 6, 256, 64, 1.1), (2049, 8, 128, 64, 0.5)])
def test_mixed(T, k, E, BM, skew):
    ids, _ = W.random_routing(T, k, E, seed=7, skew=skew)
    run_both(ids, E, BM)


def test_all_tokens_one_expert_and_block_boundaries():
    for n in [1, 15, 16, 17, 64, 128, 129]:
        ids = torch.full((n, 1), 3, dtype=torch.int32)
        run_both(ids, 8, 16)
        run_both(ids, 8, 128)


def test_zero_tokens_writes_empty_tables():
    ids = torch.zeros((0, 4), dtype=torch.int32)
    s, b, npp = moe.align(ids.cuda(), 8, 16)
    torch.cuda.synchronize()
    assert int(npp.item()) == 0
    assert (s.cpu() == 0).all() and (b.cpu() == -1).all()


def test_bad_ids_are_flagged_not_written():
    ws = moe.Workspace("cuda")
    ids = torch.tensor([[0, 1], [2, 9], [-1, 3]], dtype=torch.int32).cuda()
    s, b, npp = moe.align(ids, 4, 16, ws=ws)
    code = moe.read_device_error(ws.buf)
    assert code & moe.DEVERR_BAD_EXPERT_ID
    so = s.cpu().numpy()
    # the 4 valid assignments are placed, the bad ones are not
    real = sorted(int(a) for a in so if a < 6)
    assert real == [0, 1, 2, 5]
    assert moe.read_device_error(ws.buf) == 0  # cleared


# At most 32 assignments (decode) take a one-warp path; 33 the general one.
@pytest.mark.parametrize("T,k,E,BM", [(1, 1, 1, 16), (2, 1, 2, 16), (3, 1, 3, 64),
                                      (4, 8, 16, 16), (4, 8, 128, 128), (31, 1, 5, 16),
                                      (32, 1, 5, 64), (33, 1, 5, 16), (1, 8, 1024, 16),
                                      (2, 8, 256, 128)])
def test_few_assignments(T, k, E, BM):
    ids, _ = W.random_routing(T, k, E, seed=T * 31 + E)
    run_both(ids, E, BM)
