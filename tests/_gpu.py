"""Helpers of the GPU parity tests: host copies of the seeded inputs for the
oracle, token sampling, and the comparison rules."""
import numpy as np
import torch

from router_experts_gb300 import workloads as W

GAP_MIN = 1e-4          # router ids must agree where the cut margin exceeds this
WEIGHT_ATOL = 1e-5      # router weights
LAYER_RTOL_BF16 = 2e-2  # max|err| <= 2e-2 * max|ref|
LAYER_RTOL_LOWBIT = 6e-2


def host(t):
    return None if t is None else W.to_host_raw(t)


def sample_tokens(T, n, seed=0):
    if T <= n:
        return np.arange(T, dtype=np.int32)
    rng = np.random.default_rng(seed)
    return np.sort(rng.choice(T, n, replace=False)).astype(np.int32)


def oracle_router(oracle, w, d, T, tokens):
    x_dt = "e4m3" if w.lowbit else "bf16"
    g_dt = "f32" if w.lowbit else "bf16"
    bias = None if "bias" not in d else d["bias"].cpu().numpy()
    return oracle.router(host(d["hidden"]), x_dt, host(d["gate"]), g_dt, bias, T, w.H, w.E, w.k,
                         w.scoring, w.n_group, w.topk_group, w.renormalize, w.scaling,
                         x_scale=host(d.get("hidden_scale")), tokens=tokens)


def compact_experts(w13, w2, ids_rows, w13_scale=None, w2_scale=None):
    """Host copies of only the experts the sampled rows use, with ids remapped
    (keeps the oracle's input small for the 22.5 GB workload).  With scales
    (low-bit weights) returns (w13, w2, ids, n, w13_scale, w2_scale)."""
    used = np.unique(ids_rows.reshape(-1))
    remap = {int(e): i for i, e in enumerate(used)}
    idx = torch.as_tensor(used, dtype=torch.long, device=w13.device)
    w13h = host(w13.index_select(0, idx))
    w2h = host(w2.index_select(0, idx))
    new_ids = np.array([[remap[int(e)] for e in r] for r in ids_rows], dtype=np.int32).reshape(ids_rows.shape)
    if w13_scale is None:
        return w13h, w2h, new_ids, len(used)
    return (w13h, w2h, new_ids, len(used), host(w13_scale.index_select(0, idx)),
            host(w2_scale.index_select(0, idx)))


def rel_err(got, ref):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    scale = np.abs(ref).max()
    return float(np.abs(got - ref).max() / (scale if scale > 0 else 1.0))
