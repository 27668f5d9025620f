"""Pins of the oracle router.

* Printed values: "How an MoE Model Picks Its Experts During LLM Inference",
  Figure 1 (scores 0.881 / 0.870 -> weights 0.503 / 0.497), Figure 3 (rank keys
  8.900 / 8.899, rejected 8.881, gap 0.018, weights from the unbiased scores)
  and §2.1 (a bf16 bias flips the selection to experts 0 and 2).
* Closed form: softmax + renormalise over the selected experts equals a softmax
  over the selected logits only ("Mixture of Experts", fused_topk discussion).
* Brute force: group-limited top-k by exhaustive enumeration on tiny E.
* Ties: lowest expert id wins ("MoE Kernels, in depth", Router section).
* The square root of a softplus (§1.3, DeepSeek-V4's score): sqrt(ln 2) at a
  zero logit, the sqrt(l) and e^(l/2) asymptotes, and the same ranking as the
  sigmoid when there is no bias (both increase with the logit).
"""
import itertools
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def route_logits(logits, bias, k, scoring="sigmoid", n_group=1, topk_group=1, renorm=True,
                 scaling=1.0):
    """Feed given logits through the oracle: H = E, gate = identity (exact)."""
    logits = np.atleast_2d(np.asarray(logits, dtype=np.float32))
    T, E = logits.shape
    gate = np.eye(E, dtype=np.float32)
    return oracle.router(logits, "f32", gate, "f32", bias, T, E, E, k, scoring, n_group,
                         topk_group, renorm, scaling, want_logits=True)


def test_fig1_fig3_printed_values():
    g = json.load(open(os.path.join(GOLD, "p1_router_fig1_fig3.json")))
    tol = g["printed_tolerance"]
    logits, bias, k = g["logits"], g["bias"], g["k"]
    # Figure 1: no bias
    ids, w, gap, lg = route_logits(logits, None, k)
    f1 = g["fig1_softmaxless_sigmoid"]
    assert list(ids[0]) == f1["ids"]
    scores = [1 / (1 + math.exp(-float(np.float32(logits[i])))) for i in f1["ids"]]
    assert np.allclose(scores, f1["scores"], atol=tol)
    assert np.allclose(w[0], f1["weights"], atol=tol)
    # Figure 3: with the selection bias
    ids, w, gap, lg = route_logits(logits, np.array(bias, np.float32), k)
    f3 = g["fig3_biased"]
    assert list(ids[0]) == f3["ids"]
    keys = [1 / (1 + math.exp(-lg[0, i])) + float(np.float32(bias[i])) for i in f3["ids"]]
    assert np.allclose(keys, f3["keys"], atol=tol)
    rej = f3["first_rejected"]
    rkey = 1 / (1 + math.exp(-lg[0, rej["id"]])) + float(np.float32(bias[rej["id"]]))
    assert abs(rkey - rej["key"]) < tol
    assert abs(gap[0] - f3["gap"]) < 2 * tol
    # weights come from the unbiased scores 0.870 and 0.769, renormalised
    s = np.array(f3["weight_scores"])
    assert np.allclose(w[0], s / s.sum(), atol=2 * tol)


def test_bf16_bias_flips_selection():
    g = json.load(open(os.path.join(GOLD, "p1_router_fig1_fig3.json")))
    b16 = torch.tensor(g["bias"], dtype=torch.float32).to(torch.bfloat16).float().numpy()
    ids, w, gap, lg = route_logits(g["logits"], b16, g["k"])
    assert sorted(ids[0].tolist()) == g["bf16_bias"]["selected_set"]
    key5 = 1 / (1 + math.exp(-lg[0, 5])) + float(b16[5])
    assert abs(key5 - g["bf16_bias"]["key_expert5"]) < g["printed_tolerance"]


def test_softmax_renorm_equals_softmax_over_selected():
    rng = np.random.default_rng(7)
    for trial in range(50):
        E, k = int(rng.integers(4, 40)), 0
        k = int(rng.integers(1, min(E, 9) + 1))
        logits = rng.standard_normal((1, E)) * 3
        ids, w, gap, lg = route_logits(logits, None, k, scoring="softmax")
        sel = lg[0, ids[0]]
        closed = np.exp(sel - sel.max()) / np.exp(sel - sel.max()).sum()
        assert np.allclose(w[0], closed, rtol=1e-12, atol=1e-15)
        # the selected ones are the k largest logits, best first
        order = sorted(range(E), key=lambda e: (-lg[0, e], e))[:k]
        assert list(ids[0]) == order


def test_weights_sum_to_scaling_and_unbiased():
    rng = np.random.default_rng(8)
    E, k = 16, 4
    logits = rng.standard_normal((20, E))
    bias = rng.uniform(-0.1, 0.1, E).astype(np.float32)
    ids, w, gap, lg = route_logits(logits, bias, k, scaling=2.5)
    assert np.allclose(w.sum(1), 2.5, rtol=1e-12)
    ids2, w2, _, _ = route_logits(logits, bias, k, renorm=False, scaling=1.0)
    sig = 1 / (1 + np.exp(-lg))
    assert np.allclose(w2, np.take_along_axis(sig, ids2, 1), rtol=1e-12)


def test_top1_renormalised_weight_is_one():
    # "For top-1 normalized routing the selected weight becomes one."
    ids, w, gap, lg = route_logits([[0.3, -1.0, 2.0, 0.1]], None, 1)
    assert ids[0, 0] == 2 and w[0, 0] == pytest.approx(1.0, abs=1e-15)


def test_ties_go_to_lowest_id():
    ids, w, gap, lg = route_logits([[1.0, 2.0, 2.0, 2.0, 0.5, 2.0]], None, 3)
    assert list(ids[0]) == [1, 2, 3]
    assert gap[0] == 0.0
    ids, _, _, _ = route_logits([[0.0] * 8], None, 4, scoring="softmax")
    assert list(ids[0]) == [0, 1, 2, 3]


def brute_force_grouped(key, score, k, n_group, topk_group):
    """Literal definition by enumeration (independent of the oracle's rounds)."""
    E = len(key)
    gs = E // n_group
    gscore = [sum(sorted(key[g * gs:(g + 1) * gs])[-2:]) for g in range(n_group)]
    # the kept set is the unique subset S such that every member beats every
    # non-member under (score desc, id asc)
    kept = None
    for S in itertools.combinations(range(n_group), topk_group):
        out = [g for g in range(n_group) if g not in S]
        if all((gscore[a] > gscore[b]) or (gscore[a] == gscore[b] and a < b) for a in S for b in out):
            assert kept is None
            kept = S
    allowed = [e for e in range(E) if e // gs in kept]
    best = None
    for C in itertools.combinations(allowed, k):
        rest = [e for e in allowed if e not in C]
        if all((key[a] > key[b]) or (key[a] == key[b] and a < b) for a in C for b in rest):
            assert best is None
            best = C
    order = sorted(best, key=lambda e: (-key[e], e))
    return order


@pytest.mark.parametrize("E,n_group,topk_group,k", [
    (8, 2, 1, 2), (8, 4, 2, 3), (12, 3, 2, 4), (12, 4, 3, 5), (12, 2, 1, 6), (9, 3, 2, 2)])
def test_group_limited_topk_matches_brute_force(E, n_group, topk_group, k):
    rng = np.random.default_rng(E * 100 + n_group * 10 + k)
    for trial in range(30):
        logits = rng.standard_normal((1, E)) * 2
        bias = rng.uniform(-0.3, 0.3, E).astype(np.float32)
        ids, w, gap, lg = route_logits(logits, bias, k, n_group=n_group, topk_group=topk_group)
        score = 1 / (1 + np.exp(-lg[0]))
        key = list(score + bias.astype(np.float64))
        assert list(ids[0]) == brute_force_grouped(key, list(score), k, n_group, topk_group)
        ws = score[ids[0]]
        assert np.allclose(w[0], ws / ws.sum(), rtol=1e-12)


def test_n_group_one_is_plain_topk():
    rng = np.random.default_rng(11)
    logits = rng.standard_normal((5, 12))
    bias = rng.uniform(-0.1, 0.1, 12).astype(np.float32)
    a = route_logits(logits, bias, 3)
    b = route_logits(logits, bias, 3, n_group=1, topk_group=1)
    c = route_logits(logits, bias, 3, n_group=4, topk_group=4)  # all groups kept
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[0], c[0])


def test_logits_are_the_gate_product():
    # bf16 hidden x bf16 gate: compare with an exact rational computation
    rng = np.random.default_rng(5)
    T, H, E = 3, 40, 6
    x = torch.from_numpy(rng.standard_normal((T, H)).astype(np.float32)).to(torch.bfloat16)
    g = torch.from_numpy(rng.standard_normal((E, H)).astype(np.float32)).to(torch.bfloat16)
    xb = x.view(torch.int16).numpy().view(np.uint16)
    gb = g.view(torch.int16).numpy().view(np.uint16)
    ids, w, gap, lg = oracle.router(xb, "bf16", gb, "bf16", None, T, H, E, 2, "softmax",
                                    want_logits=True)
    from fractions import Fraction
    xd, gd = x.double().numpy(), g.double().numpy()
    for t in range(T):
        for e in range(E):
            exact = sum(Fraction(float(xd[t, h])) * Fraction(float(gd[e, h])) for h in range(H))
            assert abs(lg[t, e] - float(exact)) <= 1e-12 * max(1.0, abs(float(exact)))


def test_gap_definition():
    # 4 experts, k = 2: keys (sigmoid) ordered; the gap is key_2 - key_3
    logits = [[0.0, 3.0, 1.0, 2.0]]
    ids, w, gap, lg = route_logits(logits, None, 2)
    s = 1 / (1 + np.exp(-np.array(logits[0])))
    assert list(ids[0]) == [1, 3]
    assert gap[0] == pytest.approx(s[3] - s[2], abs=1e-15)
    # grouped: with one kept group of two experts there is no competitor at
    # the expert cut, so the gap is the group cut G_(1) - G_(2)
    logits = [[3.0, 2.9, 0.0, 0.0, 2.95, 2.95, 0.0, 0.0]]
    ids, w, gap, lg = route_logits(logits, None, 2, n_group=4, topk_group=1)
    s = 1 / (1 + np.exp(-lg[0]))
    gsc = [s[0] + s[1], s[2] + s[3], s[4] + s[5], s[6] + s[7]]
    assert list(ids[0]) == [4, 5]
    assert gap[0] == pytest.approx(gsc[2] - gsc[0], abs=1e-15)


def test_sqrt_softplus_scores_at_known_points():
    # unnormalised weights are the scores: sqrt(ln(1 + e^l))
    ids, w, gap, _ = route_logits([[0.0, 30.0, -30.0, 2.0]], None, 4, scoring="sqrt_softplus",
                                  renorm=False)
    s = dict(zip(ids[0].tolist(), w[0].tolist()))
    assert abs(s[0] - 0.8325546111576977) < 1e-12          # sqrt(ln 2)
    assert abs(s[1] - math.sqrt(30.0)) < 1e-10             # softplus(l) - l = ln(1 + e^-l)
    assert abs(s[2] / math.exp(-15.0) - 1.0) < 1e-6        # softplus(l) ~ e^l for l << 0
    assert list(ids[0]) == [1, 3, 0, 2]                    # increasing in the logit


def test_sqrt_softplus_ranks_like_sigmoid_without_bias():
    rng = np.random.default_rng(5)
    logits = rng.normal(size=(64, 24)).astype(np.float32)
    a = route_logits(logits, None, 6, scoring="sigmoid")
    b = route_logits(logits, None, 6, scoring="sqrt_softplus")
    assert np.array_equal(a[0], b[0])
    assert np.allclose(b[1].sum(axis=1), 1.0)
