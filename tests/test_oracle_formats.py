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
