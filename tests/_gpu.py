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


def block_of_assignment(sorted_ids, npp, T, k):
    """Row block (position // BLOCK_M is taken by the caller) of every
    assignment: position of assignment a in sorted_ids, -1 if absent."""
    s = np.asarray(sorted_ids[:npp])
    pos = np.full(T * k, -1, dtype=np.int64)
    real = s < T * k
    pos[s[real]] = np.nonzero(real)[0]
    return pos


def covering_tokens(sorted_ids, npp, BM, T, k, prefer, n_min, seed=0):
    """Tokens such that every row block below the padded length holds at least
    one of their assignments (every block of an expert with assignments holds
    a real row, so every block can be covered), preferring tokens marked in
    `prefer`, topped up with random tokens to at least n_min.  Returns
    (tokens sorted ascending, number of blocks)."""
    s = np.asarray(sorted_ids)
    nblk = npp // BM
    rows = s[:nblk * BM].reshape(nblk, BM)
    blk = block_of_assignment(s, npp, T, k) // BM
    covered = np.zeros(nblk, dtype=bool)
    chosen = set()
    rng = np.random.default_rng(seed)
    for b in range(nblk):
        if covered[b]:
            continue
        cand = rows[b][rows[b] < T * k] // k
        good = cand[prefer[cand]]
        pool = good if good.size else cand
        t = int(pool[rng.integers(pool.size)])
        chosen.add(t)
        covered[blk[t * k:(t + 1) * k]] = True
    assert covered.all()
    rest = np.setdiff1d(np.arange(T), np.fromiter(chosen, dtype=np.int64))
    extra = max(0, min(n_min, T) - len(chosen))
    if extra:
        chosen.update(int(t) for t in rng.choice(rest, extra, replace=False))
    return np.array(sorted(chosen), dtype=np.int32), nblk


def blocks_covered(sorted_ids, npp, BM, T, k, tokens):
    """Row blocks below the padded length that hold an assignment of `tokens`."""
    blk = block_of_assignment(sorted_ids, npp, T, k) // BM
    a = (np.asarray(tokens, dtype=np.int64)[:, None] * k + np.arange(k)[None, :]).reshape(-1)
    b = blk[a]
    return np.unique(b[b >= 0]).size
