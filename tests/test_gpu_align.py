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


def test_align_barrier_wait_expires_and_reports():
    """The bounded-wait expiry path, made to run out on purpose without
    faulting anything.  The align kernel's CTAs (a cooperative launch) meet at
    one grid barrier in the workspace header.  Presetting its arrival counter
    to a huge value means no CTA ever draws the last ticket, so the generation
    never advances and every CTA's wait runs out.  The header's wait-limit
    test hook shortens that wait to 2^21 SM cycles (about a millisecond).
    Expected: MOE_DEVERR_WAIT_TIMEOUT in the error word, no output written
    (the CTAs return before placing anything), and a correct align once the
    header is zeroed again."""
    lib = moe.load()
    T, k, E, BM = 512, 8, 128, 64  # 4,096 assignments: 8 CTAs, so the barrier is used
    ids, _ = W.random_routing(T, k, E, seed=21)
    ids_d = ids.cuda()
    cap = T * k + E * (BM - 1)
    nbc = (cap + BM - 1) // BM
    guard = 64
    ws = moe.Workspace("cuda")
    buf = ws.get(lib.moe_align_workspace_bytes())
    marker = -7
    sorted_all = torch.full((cap + 2 * guard,), marker, dtype=torch.int32, device="cuda")
    blk_all = torch.full((nbc + 2 * guard,), marker, dtype=torch.int32, device="cuda")
    npp_all = torch.full((1 + 2 * guard,), marker, dtype=torch.int32, device="cuda")
    sorted_ids, blk, npp = sorted_all[guard:guard + cap], blk_all[guard:guard + nbc], \
        npp_all[guard:guard + 1]
    stream = moe._stream(ids_d.device)

    def call():
        return lib.moe_align(moe._p(ids_d), T, k, E, BM, moe._p(sorted_ids), cap, moe._p(blk),
                             moe._p(npp), moe._p(buf), buf.numel(), stream)

    bar = buf[moe.WS_ALIGN_BARRIER_OFFSET:moe.WS_ALIGN_BARRIER_OFFSET + 8].view(torch.int32)
    limit = buf[moe.WS_WAIT_LIMIT_OFFSET:moe.WS_WAIT_LIMIT_OFFSET + 8].view(torch.int64)
    bar[0] = 1 << 30
    limit[0] = 1 << 21
    assert call() == moe.MOE_OK
    code = moe.read_device_error(buf)
    print(f"align with a barrier that never opens: error word {code}")
    assert code & moe.DEVERR_WAIT_TIMEOUT
    assert (sorted_all == marker).all() and (blk_all == marker).all() and (npp_all == marker).all()
    # the header zeroed again: a normal, correct align on the same workspace
    assert lib.moe_workspace_init(moe._p(buf), buf.numel(), stream) == moe.MOE_OK
    assert call() == moe.MOE_OK
    so, bo, nppo = oracle.align(ids.numpy(), T, k, E, BM)
    torch.cuda.synchronize()
    assert moe.read_device_error(buf) == 0
    assert int(npp.item()) == nppo
    assert np.array_equal(sorted_ids.cpu().numpy(), so)
    assert np.array_equal(blk.cpu().numpy(), bo)
    assert (sorted_all[:guard] == marker).all() and (sorted_all[guard + cap:] == marker).all()
    assert (blk_all[:guard] == marker).all() and (blk_all[guard + nbc:] == marker).all()
