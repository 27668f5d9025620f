"""moe_router_noalloc: the router for callers that cannot allocate device memory.

Callers embedded in a framework that owns all device memory (or forbidden to
allocate after start-up) cannot hand the router a workspace.  This entry point
keeps its scratch in a fixed array inside the library instead.  These tests
call it through the C ABI on several calls in a row (other shapes in between,
so the array always holds the previous call's leftovers) and check every call
against the oracle (ids bit-exact where the routing margin exceeds 1e-4,
weights within 1e-5) and against moe_router, the entry point with a caller
workspace.  They also run a call whose partial logits fill the array exactly
(accepted) and calls one size beyond it (refused).  The file is collected last
on purpose: if it fails, a run that stops at the first failure has already
run every other test."""
import ctypes
import dataclasses

import numpy as np
import pytest
import torch

import oracle
from router_experts_gb300 import moe
from router_experts_gb300 import workloads as W

from _gpu import GAP_MIN, WEIGHT_ATOL, oracle_router

pytestmark = pytest.mark.gpu


def noalloc_fn():
    lib = moe.load()
    fn = lib.moe_router_noalloc
    P, I = ctypes.c_void_p, ctypes.c_int
    fn.restype = I
    fn.argtypes = [P, I, P, P, I, P, I, I, I, I, I, I, I, I, ctypes.c_float, P, P, P]
    return fn


def ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def call_noalloc(fn, w, d, T):
    ids = torch.full((T, w.k), -1, dtype=torch.int32, device="cuda")
    wts = torch.full((T, w.k), -1.0, dtype=torch.float32, device="cuda")
    x_dt = moe.DT_E4M3 if w.lowbit else moe.DT_BF16
    g_dt = moe.DT_F32 if w.lowbit else moe.DT_BF16
    rc = fn(ptr(d["hidden"]), x_dt, ptr(d.get("hidden_scale")), ptr(d["gate"]), g_dt,
            ptr(d.get("bias")), T, w.H, w.E, w.k, moe.SCORING[w.scoring], w.n_group,
            w.topk_group, int(w.renormalize), w.scaling, ptr(ids), ptr(wts),
            ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == moe.MOE_OK, rc
    return ids, wts


def with_workspace(w, d):
    ws = moe.Workspace("cuda")
    return moe.router(d["hidden"], d["gate"], d.get("bias"), w.k, w.scoring, w.n_group,
                      w.topk_group, w.renormalize, w.scaling, hidden_scale=d.get("hidden_scale"),
                      ws=ws)


def check_call(fn, w, T, seed=11):
    d = W.make_inputs(w, T, seed=seed, device="cuda", experts=False)
    ids, wts = call_noalloc(fn, w, d, T)
    ref_ids, ref_w = with_workspace(w, d)
    torch.cuda.synchronize()
    ids_h, wts_h = ids.cpu().numpy(), wts.cpu().numpy().astype(np.float64)
    # against the oracle, every token: ids bit-exact where the margin at the
    # cut exceeds 1e-4, weights within 1e-5 wherever the ids agree
    ids_o, w_o, gap = oracle_router(oracle, w, d, T, np.arange(T, dtype=np.int32))
    clear = gap > GAP_MIN
    assert clear.sum() >= T // 2, (w.name, int(clear.sum()))
    assert (ids_h[clear] == ids_o[clear]).all(), (w.name, T)
    same_o = (ids_h == ids_o).all(axis=1)
    assert np.abs(wts_h[same_o] - w_o[same_o]).max() <= WEIGHT_ATOL
    # against moe_router: its tiled path sums the logits in another order,
    # so the ids may differ only on tokens the oracle shows to be near-ties
    same = (ids == ref_ids).all(dim=1).cpu().numpy()
    assert (gap[~same] <= GAP_MIN).all(), (w.name, np.nonzero(~same & clear)[0])
    assert np.abs(wts_h[same] - ref_w.cpu().numpy()[same]).max() <= WEIGHT_ATOL
    print(f"noalloc {w.name} T={T} {w.scoring}: {int(clear.sum())} of {T} tokens clear of "
          f"the cut, {int((~same).sum())} near-tie tokens differ from moe_router")


def variant(name, **kw):
    return dataclasses.replace(W.WORKLOADS[name], **kw)


# 4,096 tokens x 512 experts x 4 bytes: the partial logits fill the 8 MiB
# array exactly (one K split at this many tokens)
EDGE = W.Workload("edge512", H=256, E=512, k=8, F=0, scoring="softmax")


@pytest.mark.parametrize("seq", [
    [(W.WORKLOADS["glm"], 64), (W.WORKLOADS["glm"], 64)],
    [(W.WORKLOADS["qwen3"], 1), (W.WORKLOADS["dsv3"], 4096), (W.WORKLOADS["qwen3"], 1)],
    [(W.WORKLOADS["v4lo"], 512), (W.WORKLOADS["toy"], 16), (W.WORKLOADS["v4lo"], 512)],
    [(variant("dsv3", scoring="sqrt_softplus"), 64), (variant("v4lo", scoring="sqrt_softplus"), 512),
     (variant("dsv3", scoring="sqrt_softplus"), 64)],
    [(EDGE, 4096), (W.WORKLOADS["toy"], 16), (EDGE, 4096)],
])
def test_noalloc_matches_oracle_on_consecutive_calls(seq):
    fn = noalloc_fn()
    for w, T in seq:
        check_call(fn, w, T)


def test_noalloc_rejects_sizes_beyond_its_array():
    fn = noalloc_fn()
    # one token more than the exact fit above, and twice as many: the partial
    # logits exceed the 8 MiB array.  Every buffer has its full size, so even a
    # wrongly accepted call would only run a correct router.
    E, H, k = 512, 256, 8
    for T in (4097, 8192):
        x = torch.zeros((T, H), dtype=torch.bfloat16, device="cuda")
        g = torch.zeros((E, H), dtype=torch.bfloat16, device="cuda")
        ids = torch.zeros((T, k), dtype=torch.int32, device="cuda")
        wts = torch.zeros((T, k), dtype=torch.float32, device="cuda")
        rc = fn(ptr(x), moe.DT_BF16, None, ptr(g), moe.DT_BF16, None, T, H, E, k, moe.SOFTMAX,
                1, 1, 1, 1.0, ptr(ids), ptr(wts), None)
        torch.cuda.synchronize()
        assert rc == moe.MOE_ERR_ARG, (T, rc)
