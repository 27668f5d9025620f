"""Pins of the oracle's number-format decoders and roundings.

The decoders are checked against library casts (torch bf16 / float8_e4m3fn)
and against the OCP microscaling format tables (e2m1 values, UE8M0 = 2^(s-127)),
which the pages name but do not print ("How GPUs Fuse Communication and
Computation During LLM Inference", §1.1: FP4 weights, FP8 activations, one
scale per 32 values)."""
import math

import numpy as np
import pytest
import torch

import oracle


def test_bf16_decoder_matches_torch_all_codes():
    codes = np.arange(0, 1 << 16, dtype=np.uint32).astype(np.uint16)
    ref = torch.from_numpy(codes.view(np.int16)).view(torch.bfloat16).double().numpy()
    got = oracle.decode(codes, "bf16", 1, len(codes))[0]
    same = (got == ref) | (np.isnan(got) & np.isnan(ref))
    assert same.all()


def test_e4m3_decoder_matches_torch_all_codes():
    codes = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).double().numpy()
    got = np.array([oracle.e4m3_to_double(c) for c in codes])
    same = (got == ref) | (np.isnan(got) & np.isnan(ref))
    assert same.all()
    assert oracle.e4m3_to_double(0x7E) == 448.0  # largest finite
    assert math.isnan(oracle.e4m3_to_double(0x7F))


def test_e2m1_decoder_matches_format_table():
    # OCP MX FP4 E2M1 code table (sign bit 3): 0, .5, 1, 1.5, 2, 3, 4, 6
    table = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]
    for c in range(16):
        want = table[c & 7] * (-1.0 if c & 8 else 1.0)
        assert oracle.e2m1_to_double(c) == want


def test_ue8m0_decoder():
    for s in range(255):
        assert oracle.ue8m0_to_double(s) == math.ldexp(1.0, s - 127)
    assert math.isnan(oracle.ue8m0_to_double(255))


def test_packed_fp4_with_scales_decode():
    # one row of 64 values: low nibble first, one scale per 32 values
    rng = np.random.default_rng(3)
    nib = rng.integers(0, 16, size=64)
    packed = (nib[0::2] | (nib[1::2] << 4)).astype(np.uint8)
    scales = np.array([127 - 2, 127 + 1], dtype=np.uint8)
    got = oracle.decode(packed, "e2m1", 1, 64, scale=scales)[0]
    table = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]
    want = np.array([table[c & 7] * (-1 if c & 8 else 1) for c in nib], dtype=np.float64)
    want[:32] *= 0.25
    want[32:] *= 2.0
    assert np.array_equal(got, want)


def test_e4m3_with_scales_decode():
    codes = np.arange(64, dtype=np.uint8)
    scales = np.array([127, 127 - 4], dtype=np.uint8)
    got = oracle.decode(codes, "e4m3", 1, 64, scale=scales)[0]
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).double().numpy()
    ref[32:] /= 16.0
    assert np.array_equal(got, ref)


def test_round_bf16_matches_torch():
    rng = np.random.default_rng(0)
    vals = np.concatenate([rng.standard_normal(20000) * 10.0 ** rng.integers(-8, 8, 20000),
                           [1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, -(1.0 + 2 ** -8), 8.03, 8.13]])
    # torch casts float64 -> bf16 with a single rounding
    ref = torch.from_numpy(vals).to(torch.bfloat16).double().numpy()
    got = np.array([oracle.round_bf16(v) for v in vals])
    assert np.array_equal(got, ref)


def test_round_e4m3_matches_torch_in_range_and_saturates():
    rng = np.random.default_rng(1)
    vals = rng.uniform(-448, 448, 20000) * 10.0 ** rng.integers(-4, 1, 20000)
    ref = torch.from_numpy(vals).to(torch.float8_e4m3fn).double().numpy()
    got = np.array([oracle.round_e4m3(v) for v in vals])
    assert np.array_equal(got, ref)
    assert oracle.round_e4m3(1000.0) == 448.0
    assert oracle.round_e4m3(-460.0) == -448.0


# ---- FP8 cast of the layer input ("How GPUs Fuse ..." §1.1 cast kernel, §3.5
# scale rule: per 32 values the smallest 2^s with amax / 2^s <= 448) ----------

E4M3 = np.array([oracle.e4m3_to_double(c) for c in range(256)])
FINITE_POS = [c for c in range(1, 127)]  # 0x01 .. 0x7E (0x7F is NaN)


def _cast(rows):
    x = np.asarray(rows, dtype=np.float32)
    return oracle.quantize_e4m3(x, "f32", x.shape[0], x.shape[1])


def test_cast_worked_values():
    codes, scales = _cast([[1.0] * 32 + [0.0] * 32 + [-0.0] + [0.0] * 31])
    # 1.0 <= 448 * 2^s first at s = -8 (448/256 = 1.75; 448/512 = 0.875 < 1):
    # byte 127 - 8, and 1.0 / 2^-8 = 256 = 1.0 x 2^8 -> exponent field 15, code 0x78
    assert scales[0].tolist() == [119, 127, 127]
    assert (codes[0, :32] == 0x78).all() and (codes[0, 32:64] == 0).all()
    assert codes[0, 64] == 0x80  # -0 keeps its sign


def test_cast_round_trips_values_on_the_grid():
    rng = np.random.default_rng(3)
    for s in [-20, -8, 0, 5]:
        picks = rng.choice(FINITE_POS, size=(4, 32))
        signs = rng.choice([0, 0x80], size=(4, 32))
        picks[:, 0] = 0x7E  # 448: pins s for every row
        want = (picks | signs).astype(np.uint8)
        x = E4M3[want] * 2.0 ** s
        codes, scales = _cast(x)
        assert (scales == s + 127).all()
        assert np.array_equal(codes, want)


def test_cast_scale_is_the_smallest_and_error_within_half_a_step():
    rng = np.random.default_rng(4)
    x = (rng.standard_normal((16, 256)) * np.exp2(rng.integers(-12, 12, size=(16, 1)))).astype(np.float32)
    codes, scales = _cast(x)
    for t in range(16):
        for g in range(8):
            v = x[t, 32 * g:32 * g + 32].astype(np.float64)
            s = int(scales[t, g]) - 127
            amax = np.abs(v).max()
            assert amax <= 448 * 2.0 ** s and amax > 448 * 2.0 ** (s - 1)
            q = E4M3[codes[t, 32 * g:32 * g + 32]] * 2.0 ** s
            # spacing of e4m3 at |v|/2^s: 2^-9 below 2^-6, else 2^(floor(log2)-3)
            a = np.abs(v) / 2.0 ** s
            step = np.where(a < 2.0 ** -6, 2.0 ** -9, 2.0 ** (np.floor(np.log2(np.maximum(a, 1e-300))) - 3))
            assert (np.abs(q - v) <= 0.5 * step * 2.0 ** s + 1e-300).all()


def test_cast_ties_go_to_the_even_code():
    # halfway between 1.0 (0x38, even) and 1.125 (0x39), and between 1.125 and
    # 1.25 (0x3A, even); 448 in the row fixes s = 0
    codes, scales = _cast([[448.0, 1.0625, 1.1875, -1.0625] + [0.0] * 28])
    assert scales[0, 0] == 127
    assert codes[0, 1:4].tolist() == [0x38, 0x3A, 0xB8]
