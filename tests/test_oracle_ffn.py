"""Pins of the oracle expert FFN and weighted combine.

* Hand-worked case: silu(ln 3) = ln 3 * sigmoid(ln 3) = 0.75 ln 3, with the
  gate rows first and the up rows second in w13 [E, 2F, H] and w2 [E, H, F]
  ("Mixture of Experts", fused w13 / w2 shapes; "MoE Kernels, in depth",
  SwiGLU silu(g) * u).  Non-square shapes catch a transposed operand.
* Grouped scatter equals the direct per-token sum, the check printed on
  "Mixture of Experts" (grouped vs direct), with SwiGLU experts.
* Top-1 renormalised routing: the weight is one and y is the expert output.
* Emulate modes round where the GPU path rounds (bf16 act / staged rows, or an
  e4m3 + UE8M0-per-32 re-quantisation, "How GPUs Fuse Communication and
  Computation During LLM Inference" §3.5): checked against torch casts.
"""
import math

import numpy as np
import pytest
import torch

import oracle


def f32(a):
    return np.ascontiguousarray(a, dtype=np.float32)


def test_hand_worked_single_expert():
    # H = 3, F = 2, E = 2; x = [1, 2, -1]
    H, F, E = 3, 2, 2
    x = f32([[1.0, 2.0, -1.0]])
    ln3 = math.log(3.0)
    w13 = np.zeros((E, 2 * F, H), np.float32)
    # expert 1: gate rows 0..F-1, up rows F..2F-1
    w13[1, 0] = [ln3, 0.0, 0.0]      # g0 = ln 3      -> silu = 0.75 ln 3
    w13[1, 1] = [0.0, 0.0, 0.0]      # g1 = 0         -> silu = 0
    w13[1, 2] = [0.0, 1.0, 0.0]      # u0 = 2
    w13[1, 3] = [5.0, 5.0, 5.0]      # u1 = 10 (multiplied by silu(0) = 0)
    w2 = np.zeros((E, H, F), np.float32)
    w2[1] = [[1.0, 7.0], [-2.0, 7.0], [0.5, 7.0]]
    w2[0] = 100.0                    # expert 0 must not contribute
    ids = np.array([[1]], np.int32)
    wts = np.array([[1.0]])
    y = oracle.moe_ffn(x, "f32", f32(w13), f32(w2), "f32", 1, H, F, E, 1, ids, wts)
    act0 = 1.5 * ln3                 # 0.75 ln3 * 2 (ln 3 is stored as f32: rtol 1e-7)
    assert np.allclose(y[0], [act0, -2 * act0, 0.5 * act0], rtol=1e-7, atol=0)
    # a routing weight of 0.25 scales the output linearly
    y = oracle.moe_ffn(x, "f32", f32(w13), f32(w2), "f32", 1, H, F, E, 1, ids, wts * 0.25)
    assert np.allclose(y[0], 0.25 * np.array([act0, -2 * act0, 0.5 * act0]), rtol=1e-7)


def test_silu_closed_forms():
    # one hidden unit: g = z, u = 1, w2 = 1 -> y = silu(z)
    H, F, E = 1, 1, 1
    for z, want in [(0.0, 0.0), (math.log(3.0), 0.75 * math.log(3.0)),
                    (-math.log(3.0), -0.25 * math.log(3.0)), (40.0, 40.0)]:
        w13 = f32([[[z], [1.0]]])
        w2 = f32([[[1.0]]])
        y = oracle.moe_ffn(f32([[1.0]]), "f32", w13, w2, "f32", 1, H, F, E, 1,
                           np.array([[0]], np.int32), np.array([[1.0]]))
        assert y[0, 0] == pytest.approx(want, rel=1e-7, abs=1e-15)


def test_grouped_scatter_equals_direct_sum():
    rng = np.random.default_rng(4)
    T, H, F, E, k = 7, 12, 5, 4, 2
    x = f32(rng.standard_normal((T, H)))
    w13 = f32(rng.standard_normal((E, 2 * F, H)) * 0.3)
    w2 = f32(rng.standard_normal((E, H, F)) * 0.3)
    ids = np.stack([rng.choice(E, k, replace=False) for _ in range(T)]).astype(np.int32)
    wts = rng.uniform(0.1, 1.0, (T, k))
    grouped = oracle.moe_ffn(x, "f32", w13, w2, "f32", T, H, F, E, k, ids, wts)
    direct = np.zeros((T, H))
    for t in range(T):
        for j in range(k):
            direct[t] += wts[t, j] * oracle.expert_ffn(x[t].astype(np.float64), w13, w2, "f32",
                                                       H, F, int(ids[t, j]))
    assert np.allclose(grouped, direct, rtol=1e-13, atol=1e-14)
    # a token list selects rows
    sub = oracle.moe_ffn(x, "f32", w13, w2, "f32", T, H, F, E, k, ids, wts, tokens=[5, 2])
    assert np.array_equal(sub, grouped[[5, 2]])


def test_top1_layer_is_the_expert_output():
    rng = np.random.default_rng(9)
    T, H, F, E = 4, 8, 6, 3
    x = f32(rng.standard_normal((T, H)))
    gate = f32(rng.standard_normal((E, H)))
    w13 = f32(rng.standard_normal((E, 2 * F, H)) * 0.5)
    w2 = f32(rng.standard_normal((E, H, F)) * 0.5)
    y, ids, w, gap = oracle.moe_layer(x, "f32", gate, "f32", None, w13, w2, "f32", T, H, F, E, 1,
                                      "softmax")
    assert np.allclose(w, 1.0)
    for t in range(T):
        want = oracle.expert_ffn(x[t].astype(np.float64), w13, w2, "f32", H, F, int(ids[t, 0]))
        assert np.allclose(y[t], want, rtol=1e-14, atol=1e-15)


def test_emulate_bf16_rounds_like_torch():
    rng = np.random.default_rng(10)
    T, H, F, E, k = 3, 16, 8, 2, 2
    x = f32(rng.standard_normal((T, H)))
    w13 = f32(rng.standard_normal((E, 2 * F, H)))
    w2 = f32(rng.standard_normal((E, H, F)))
    ids = np.array([[0, 1]] * T, np.int32)
    wts = np.full((T, k), 0.5)
    y1 = oracle.moe_ffn(x, "f32", w13, w2, "f32", T, H, F, E, k, ids, wts, emulate=1)
    # recompute with torch: act -> bf16, weighted expert output -> bf16, fp64 sum
    xt, a, b = (torch.from_numpy(v).double() for v in (x, w13, w2))
    want = torch.zeros(T, H, dtype=torch.float64)
    for j in range(k):
        e = j
        h = xt @ a[e].T
        act = (torch.nn.functional.silu(h[:, :F]) * h[:, F:]).to(torch.bfloat16).double()
        o = act @ b[e].T
        want += (0.5 * o).to(torch.bfloat16).double()
    assert np.allclose(y1, want.numpy(), rtol=0, atol=1e-12)


def test_emulate_fp8_requant_scale_rule():
    # act values of one 32-block: the scale is the smallest power of two with
    # amax / scale <= 448, so the largest magnitude lands in (224, 448]
    H, F, E = 1, 32, 1
    vals = np.linspace(-3.0, 1000.0, F)
    w13 = np.zeros((E, 2 * F, H), np.float32)
    w13[0, :F, 0] = 60.0             # gate: silu(60) = 60 (to fp64 precision)
    w13[0, F:, 0] = vals / 60.0      # up: act = vals
    w2 = np.zeros((E, H, F), np.float32)
    w2[0, 0, F - 1] = 1.0            # y = act[F-1] after re-quantisation
    y = oracle.moe_ffn(f32([[1.0]]), "f32", f32(w13), f32(w2), "f32", 1, H, F, E, 1,
                       np.array([[0]], np.int32), np.array([[1.0]]), emulate=2)
    act_last = 60.0 / (1 + math.exp(-60.0)) * float(np.float32(vals[-1] / 60.0))
    scale = 4.0  # 1000 / 448 = 2.23 -> next power of two
    q = torch.tensor(act_last / scale, dtype=torch.float64).to(torch.float8_e4m3fn).double().item()
    assert y[0, 0] == pytest.approx(torch.tensor(q * scale).to(torch.bfloat16).double().item())


def test_lowbit_ffn_equals_f32_ffn_on_decoded_values():
    # Low-bit experts ("How GPUs Fuse Communication and Computation During LLM
    # Inference" §1.1: FP8 activations, FP4 weights, one UE8M0 scale per 32
    # values along the contraction): the oracle's FP8 x FP4 FFN must equal its
    # f32 FFN on the same values decoded here, independently of the oracle --
    # e4m3 through torch's float8 cast, e2m1 from the OCP table, scales
    # 2^(s-127) applied per 32 values of x along H, of w13 along H and of w2
    # along F.  A scale read along the wrong axis or from the wrong block
    # changes the result.
    rng = np.random.default_rng(12)
    T, H, F, E, k = 3, 64, 64, 3, 2
    table = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])

    def fp4(shape):
        nib = rng.integers(0, 16, size=shape)
        vals = table[nib & 7] * np.where(nib & 8, -1.0, 1.0)
        packed = (nib[..., 0::2] | (nib[..., 1::2] << 4)).astype(np.uint8)
        return packed, vals

    def scales(shape):
        return rng.integers(127 - 4, 127 + 2, size=shape).astype(np.uint8)

    def apply(vals, sc):
        return vals * np.repeat(np.ldexp(1.0, sc.astype(np.int64) - 127), 32, axis=-1)

    x_codes = rng.integers(0, 0x7E, size=(T, H)).astype(np.uint8)   # finite, non-negative
    x_codes[1] |= 0x80                                               # negative row
    x_vals = torch.from_numpy(x_codes).view(torch.float8_e4m3fn).double().numpy()
    x_sc = scales((T, H // 32))
    w13_q, w13_v = fp4((E, 2 * F, H))
    w13_sc = scales((E, 2 * F, H // 32))
    w2_q, w2_v = fp4((E, H, F))
    w2_sc = scales((E, H, F // 32))
    ids = np.array([[0, 2], [1, 0], [2, 1]], np.int32)
    wts = np.array([[0.75, 0.25], [0.5, 0.5], [1.0, 0.125]])
    low = oracle.moe_ffn(x_codes, "e4m3", w13_q, w2_q, "e2m1", T, H, F, E, k, ids, wts,
                         x_scale=x_sc, w13_scale=w13_sc, w2_scale=w2_sc)
    ref = oracle.moe_ffn(f32(apply(x_vals, x_sc)), "f32", f32(apply(w13_v, w13_sc)),
                         f32(apply(w2_v, w2_sc)), "f32", T, H, F, E, k, ids, wts)
    assert np.allclose(low, ref, rtol=1e-12, atol=1e-12)
    assert np.abs(ref).max() > 1.0  # not vacuous
