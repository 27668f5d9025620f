"""Whole-layer pins of the oracle: router -> experts -> weighted combine on
cases small enough to derive by hand, so the composition is checked against
closed-form values rather than against the oracle's own parts.

Every logit is ln of a rational, so every score is a simple fraction:
sigmoid(ln a) = a / (1 + a) and softmax(ln a_e) = a_e / sum(a).  The experts
have F = 1 and act = silu(g) * u with g = +-ln 3, where silu(ln 3) = 0.75 ln 3
and silu(-ln 3) = -0.25 ln 3.  Experts that a wrong routing would pick see a
gate pre-activation of 50 and give outputs of about 2,500, far from any
expected value.

Sources: "How an MoE Model Picks Its Experts During LLM Inference" §1 (the
rank key is score + bias, the weight is the unbiased score) and §4
(renormalise, then scale); "Mixture of Experts" (grouped routing: group score
= sum of the two best keys, keep topk_group groups; routed scaling factor;
fused w13 = gate rows then up rows, w2 [E, H, F]); "MoE Kernels, in depth"
(SwiGLU silu(gate) * up; combine = sum over the k slots).
"""
import math

import numpy as np

import oracle

LN3 = math.log(3.0)
LN7 = math.log(7.0)


def f32(a):
    return np.ascontiguousarray(a, dtype=np.float32)


def experts():
    """E = 4, H = 2, F = 1: w13 [E, 2, 2] (gate row, up row), w2 [E, 2, 1]."""
    w13 = np.zeros((4, 2, 2))
    w2 = np.zeros((4, 2, 1))
    w13[0] = [[50.0, LN3], [50.0, 2.0]]     # x = [0, 1]: act = 0.75 ln3 * 2 = 1.5 ln3
    w2[0] = [[1.0], [3.0]]                  # -> [1.5 ln3, 4.5 ln3]
    w13[1] = [[50.0, -LN3], [50.0, 4.0]]    # x = [0, 1]: act = -0.25 ln3 * 4 = -ln3
    w2[1] = [[-2.0], [1.0]]                 # -> [2 ln3, -ln3]
    w13[2] = [[LN3, 50.0], [2.0, 50.0]]     # x = [1, 0]: act = 1.5 ln3
    w2[2] = [[1.0], [-1.0]]                 # -> [1.5 ln3, -1.5 ln3]
    w13[3] = [[-LN3, 50.0], [4.0, 50.0]]    # x = [1, 0]: act = -ln3
    w2[3] = [[0.5], [2.0]]                  # -> [-0.5 ln3, -2 ln3]
    return f32(w13), f32(w2)


def test_grouped_sigmoid_bias_renorm_scaling_layer():
    # token 0 sees logits ln 7, -ln 3, ln 3, 0 (scores 7/8, 1/4, 3/4, 1/2);
    # token 1 sees ln 3, ln 7, 0, -ln 3 (scores 3/4, 7/8, 1/2, 1/4)
    gate = f32([[LN7, LN3], [-LN3, LN7], [LN3, 0.0], [0.0, -LN3]])
    bias = f32([0.0, 0.0, 0.0, 0.3])
    x = f32([[1.0, 0.0], [0.0, 1.0]])
    w13, w2 = experts()
    y, ids, w, _ = oracle.moe_layer(x, "f32", gate, "f32", bias, w13, w2, "f32", 2, 2, 1, 4, 2,
                                    "sigmoid", n_group=2, topk_group=1, renormalize=True,
                                    scaling=2.5)
    # token 0: keys 7/8, 1/4, 3/4, 1/2 + 0.3; groups {0,1} = 1.125, {2,3} = 1.55:
    # keep {2,3}; by key e3 (0.8) then e2 (0.75) -- the plain top-2 would have
    # taken e0.  Weights from the unbiased scores 1/2 and 3/4: 2.5 * (0.4, 0.6).
    # token 1: keys 3/4, 7/8, 1/2, 1/4 + 0.3; groups 1.625 and 1.05: keep
    # {0,1}; e1 (7/8) then e0 (3/4): 2.5 * (7/13, 6/13).
    assert ids.tolist() == [[3, 2], [1, 0]]
    assert np.allclose(w, [[1.0, 1.5], [17.5 / 13, 15.0 / 13]], rtol=1e-6, atol=0)
    y0 = 1.0 * np.array([-0.5, -2.0]) + 1.5 * np.array([1.5, -1.5])
    y1 = (17.5 / 13) * np.array([2.0, -1.0]) + (15.0 / 13) * np.array([1.5, 4.5])
    assert np.allclose(y, LN3 * np.stack([y0, y1]), rtol=1e-6, atol=0)
    # = ln 3 * [[1.75, -4.25], [57.5/13, 50/13]]
    assert np.allclose(y, LN3 * np.array([[1.75, -4.25], [57.5 / 13, 50.0 / 13]]), rtol=1e-6)


def test_softmax_renormalised_layer():
    # one token x = [1, 0]; logits ln 1, ln 2, ln 8, ln 4 -> softmax 1/15,
    # 2/15, 8/15, 4/15; top-2 e2, e3; renormalised 2/3, 1/3 (a softmax over
    # the two selected logits); no scaling
    gate = f32([[0.0, 0.0], [math.log(2.0), 0.0], [math.log(8.0), 0.0], [math.log(4.0), 0.0]])
    x = f32([[1.0, 0.0]])
    w13, w2 = experts()
    y, ids, w, _ = oracle.moe_layer(x, "f32", gate, "f32", None, w13, w2, "f32", 1, 2, 1, 4, 2,
                                    "softmax")
    assert ids.tolist() == [[2, 3]]
    assert np.allclose(w, [[2.0 / 3.0, 1.0 / 3.0]], rtol=1e-6, atol=0)
    want = (2.0 / 3.0) * np.array([1.5, -1.5]) + (1.0 / 3.0) * np.array([-0.5, -2.0])
    assert np.allclose(y[0], LN3 * want, rtol=1e-6, atol=0)
    # without renormalisation the weights are the raw softmax scores 8/15, 4/15
    y, ids, w, _ = oracle.moe_layer(x, "f32", gate, "f32", None, w13, w2, "f32", 1, 2, 1, 4, 2,
                                    "softmax", renormalize=False)
    assert np.allclose(w, [[8.0 / 15.0, 4.0 / 15.0]], rtol=1e-6, atol=0)
    want = (8.0 / 15.0) * np.array([1.5, -1.5]) + (4.0 / 15.0) * np.array([-0.5, -2.0])
    assert np.allclose(y[0], LN3 * want, rtol=1e-6, atol=0)
