"""Pins of the oracle align (moe_align_block_size).

* Printed example: "Mixture of Experts", worked moe_align_block_size example.
* Worst-case sizing T*k + E*(BLOCK_M-1): "MoE Kernels, in depth" (Alignment)
  and the DeepSeek-V3 decode walk-through of "Mixture of Experts" (4,352 rows,
  272 blocks at T=64, k=8, E=256, BLOCK_M=16).
* Padded length = sum(ceil(count / BLOCK_M)) * BLOCK_M ("MoE Kernels, in
  depth", What to do next, item 2); counts of 0, 1 and exactly BLOCK_M per
  expert (Failure modes).
* Stable order: checked against Python's stable sort, a library routine.
"""
import json
import os

import numpy as np
import pytest

import oracle

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def test_printed_example():
    g = json.load(open(os.path.join(GOLD, "p2_align_example.json")))
    ids = np.array(g["topk_ids"], dtype=np.int32)
    T, k = ids.shape
    E, BM = g["num_experts"], g["block_size"]
    sorted_ids, block_expert, npp = oracle.align(ids, T, k, E, BM)
    assert npp == g["num_post_padded"]
    n_used = len(g["sorted_ids_used"])
    assert sorted_ids[:n_used].tolist() == g["sorted_ids_used"]
    assert (sorted_ids[n_used:] == T * k).all()
    assert len(sorted_ids) == T * k + E * (BM - 1)
    nb = len(g["block_expert_used"])
    assert block_expert[:nb].tolist() == g["block_expert_used"]
    assert (block_expert[nb:] == -1).all()


def test_v3_decode_capacity():
    g = json.load(open(os.path.join(GOLD, "p2_v3_decode_trace.json")))
    T, k, E, BM = g["T"], g["k"], g["E"], g["block_m"]
    rng = np.random.default_rng(0)
    ids = np.stack([rng.choice(E, k, replace=False) for _ in range(T)]).astype(np.int32)
    s, b, npp = oracle.align(ids, T, k, E, BM)
    assert len(s) == g["cap_rows"] and len(b) == g["max_blocks"]


def check_invariants(ids, T, k, E, BM, sorted_ids, block_expert, npp):
    n = T * k
    flat = ids.reshape(-1)
    counts = np.bincount(flat, minlength=E)
    assert npp == int(sum(-(-c // BM) * BM for c in counts))
    assert npp % BM == 0
    used = sorted_ids[:npp]
    real = used[used < n]
    # every assignment exactly once
    assert np.array_equal(np.sort(real), np.arange(n))
    assert (sorted_ids[npp:] == n).all() and (used[used >= n] == n).all()
    # blocks: one expert per block, non-decreasing, -1 only in the tail
    nb = npp // BM
    assert (block_expert[nb:] == -1).all() and (block_expert[:nb] >= 0).all()
    assert (np.diff(block_expert[:nb]) >= 0).all()
    for b in range(nb):
        rows = used[b * BM:(b + 1) * BM]
        rows = rows[rows < n]
        assert (flat[rows] == block_expert[b]).all()
    # within an expert: ascending assignment id == Python's stable sort by expert
    expect = [a for a in sorted(range(n), key=lambda a: flat[a])]
    assert real.tolist() == [a for a in used.tolist() if a < n]
    assert [a for a in used.tolist() if a < n] == expect


@pytest.mark.parametrize("T,k,E,BM", [(1, 1, 4, 4), (5, 2, 8, 16), (37, 8, 64, 16),
                                      (100, 6, 32, 64), (64, 8, 128, 128), (0, 8, 16, 16)])
def test_invariants_random(T, k, E, BM):
    rng = np.random.default_rng(T * 1000 + E)
    ids = np.stack([rng.choice(E, k, replace=False) for _ in range(T)]).astype(np.int32) \
        if T else np.zeros((0, k), np.int32)
    s, b, npp = oracle.align(ids, T, k, E, BM)
    check_invariants(ids, T, k, E, BM, s, b, npp)


def test_counts_zero_one_and_block_m():
    E, BM, k = 6, 4, 1
    # expert 0: 0 rows, 1: 1 row, 2: exactly BM rows, 3: BM+1 rows, 4/5: 0
    ids = np.array([1] + [2] * BM + [3] * (BM + 1), dtype=np.int32).reshape(-1, 1)
    rng = np.random.default_rng(2)
    ids = ids[rng.permutation(len(ids))]
    T = len(ids)
    s, b, npp = oracle.align(ids, T, k, E, BM)
    assert npp == BM + BM + 2 * BM
    check_invariants(ids, T, k, E, BM, s, b, npp)
    assert b[:4].tolist() == [1, 2, 3, 3]


def test_skewed_all_to_one_expert():
    T, k, E, BM = 50, 1, 8, 16
    ids = np.full((T, k), 5, dtype=np.int32)
    s, b, npp = oracle.align(ids, T, k, E, BM)
    assert npp == 64
    assert s[:50].tolist() == list(range(50)) and (s[50:] == 50).all()
    assert b[:4].tolist() == [5] * 4 and (b[4:] == -1).all()


def test_rejects_bad_ids_and_small_capacity():
    with pytest.raises(ValueError):
        oracle.align(np.array([[0, 9]], np.int32), 1, 2, 4, 4)
    with pytest.raises(ValueError):
        oracle.align(np.array([[0, 1]], np.int32), 1, 2, 4, 4, cap_rows=4)
