"""Pins of the oracle's number formats against independent definitions.

The formats are named, not defined, on the pages (FP8 activations, MXFP4
weights, per-1x32 scaling: AITER #5609 "Add DeepSeek V4.1 Flash TP4 gfx950
MoE tuning", Configuration). Each check below uses a source other than the
oracle's own construction: literal value sets of the OCP formats, torch's
independent float8_e4m3fn / bfloat16 conversions, and closed forms.
"""
import math

import numpy as np
import pytest
import torch

from oracle import mx_formats as mx


def test_e2m1_table_is_the_ocp_value_set():
    pos = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]
    assert mx.E2M1_VALUES[:8].tolist() == pos
    assert mx.E2M1_VALUES[8:].tolist() == [-v for v in pos]
    assert math.copysign(1.0, mx.E2M1_VALUES[8]) == -1.0  # code 8 is -0


def test_e4m3_decode_matches_torch_for_all_256_codes():
    ref = torch.arange(256, dtype=torch.int32).to(torch.uint8).view(torch.float8_e4m3fn)
    ref = ref.to(torch.float64).numpy()
    ours = mx.E4M3_VALUES
    nan = np.isnan(ref)
    assert np.array_equal(nan, np.isnan(ours))
    assert nan.sum() == 2  # 0x7F and 0xFF
    assert np.array_equal(ref[~nan], ours[~nan])
    assert ours[0x7E] == 448.0 and ours[0x01] == 2.0 ** -9 and ours[0x38] == 1.0


def test_e4m3_encode_round_trips_every_finite_code():
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], dtype=np.uint8)
    vals = mx.E4M3_VALUES[codes]
    assert np.array_equal(mx.e4m3_encode(vals), codes)


def test_e4m3_encode_midpoints_round_to_even_and_saturate():
    pos = mx.E4M3_VALUES[:127]
    mids = (pos[:-1] + pos[1:]) / 2
    got = mx.e4m3_encode(mids)
    lo = np.arange(126)
    want = np.where(lo % 2 == 0, lo, lo + 1)
    assert np.array_equal(got, want.astype(np.uint8))
    assert mx.e4m3_encode(np.array([448.0, 463.9, 464.0, 1e9]))[:].tolist() == [0x7E] * 4
    assert mx.e4m3_encode(np.array([-1e9]))[0] == 0xFE
    # sign of zero is kept
    assert mx.e4m3_encode(np.array([-1e-30, 0.0]))[:].tolist() == [0x80, 0x00]


def test_e4m3_encode_matches_torch_on_in_range_values():
    g = torch.Generator().manual_seed(1)
    v = (torch.randn(200000, generator=g) * 40).clamp(-448, 448)
    v = torch.cat([v, torch.randn(20000, generator=g) * 1e-3])
    ref = v.to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    ours = mx.e4m3_encode(v.to(torch.float64).numpy())
    assert np.array_equal(ref, ours)


def test_bf16_round_matches_torch_on_float32_values():
    g = torch.Generator().manual_seed(2)
    v = torch.randn(200000, generator=g) * torch.exp(torch.randn(200000, generator=g) * 10)
    # exact ties: bf16 values plus half an ulp
    b = torch.randn(1000, generator=g).to(torch.bfloat16).to(torch.float32)
    ties = (b.view(torch.int32) + 0x8000).view(torch.float32)
    v = torch.cat([v, ties, b])
    ref = v.to(torch.bfloat16).to(torch.float64).numpy()
    ours = mx.bf16_round(v.to(torch.float64).numpy())
    assert np.array_equal(ref, ours)


def test_bf16_round_is_a_single_rounding_from_fp64():
    # 1 + 2^-8 + 2^-40 lies just above a bf16 tie: one rounding gives
    # 1 + 2^-7, rounding through float32 first would give 1.0.
    v = 1.0 + 2.0 ** -8 + 2.0 ** -40
    assert mx.bf16_round(np.array([v]))[0] == 1.0 + 2.0 ** -7
    assert mx.bf16_round(np.array([1.0 + 2.0 ** -8]))[0] == 1.0
    assert mx.bf16_round(np.array([3.4e38]))[0] == np.inf
    assert mx.bf16_round(np.array([3.39e38]))[0] == (2.0 - 2.0 ** -7) * 2.0 ** 127
    assert mx.bf16_round(np.array([2.0 ** -134]))[0] == 0.0
    assert mx.bf16_round(np.array([1.5 * 2.0 ** -133]))[0] == 2.0 ** -132


def test_unpack_e2m1_nibble_order():
    packed = np.array([[0x21, 0xF8]], dtype=np.uint8)
    assert mx.unpack_e2m1(packed).tolist() == [[1, 2, 8, 15]]


def test_dequant_mxfp4_applies_block_scale():
    packed = np.full((1, 32), 0x71, dtype=np.uint8)  # even k: code 1 (0.5), odd k: code 7 (6)
    scale = np.array([[127 - 3, 127 + 2]], dtype=np.uint8)
    d = mx.dequant_mxfp4(packed, scale)
    assert d[0, 0] == 0.5 / 8 and d[0, 1] == 6 / 8
    assert d[0, 32] == 0.5 * 4 and d[0, 63] == 6 * 4


def test_quant_scale_rule_hand_cases():
    x = np.zeros((4, 32))
    x[0, 3] = 448.0            # amax 448 -> e = 0 -> byte 127, code 0x7E exact
    x[1, :] = 1.0              # amax 1 -> e = -8 -> byte 119, x/2^e = 256
    x[2, 5] = -0.75            # amax 0.75 -> floor(log2) = -1 -> e = -9 -> byte 118
    codes, s = mx.quant_mxfp8(x)
    assert s[:, 0].tolist() == [127, 119, 118, 0]
    assert codes[0, 3] == 0x7E and codes[0, 0] == 0
    assert (codes[1] == mx.e4m3_encode(np.array([256.0]))[0]).all()
    assert mx.E4M3_VALUES[codes[1, 0]] == 256.0
    assert mx.E4M3_VALUES[codes[2, 5]] * 2.0 ** -9 == -0.75
    assert (codes[3] == 0).all()


def test_quant_error_bound_and_saturation():
    g = torch.Generator().manual_seed(3)
    x = (torch.randn(512, 256, generator=g, dtype=torch.float64)
         * torch.exp(torch.randn(512, 1, generator=g, dtype=torch.float64) * 3)).numpy()
    codes, s = mx.quant_mxfp8(x)
    dq = mx.dequant_mxfp8(codes, s)
    scale = np.repeat(mx.e8m0_value(s), 32, axis=-1)
    y = x / scale
    # E4M3 spacing at |y|: 2^(floor(log2|y|) - 3) for normals, 2^-9 below 2^-6
    ay = np.abs(y)
    with np.errstate(divide="ignore"):
        ex = np.floor(np.log2(np.where(ay > 0, ay, 1.0)))
    ulp = np.where(ay >= 2.0 ** -6, 2.0 ** (ex - 3), 2.0 ** -9)
    sat = ay > 448
    err = np.abs(dq - x) / scale
    assert (err[~sat] <= ulp[~sat] / 2 + 1e-300).all()
    assert np.all(np.abs(mx.E4M3_VALUES[codes[sat]]) == 448.0)
    # every block's max lies in [256, 512) before saturation
    blk = ay.reshape(512, 8, 32).max(-1)
    assert ((blk >= 256) & (blk < 512)).all()


def test_e8m0_value():
    assert mx.e8m0_value(127) == 1.0
    assert mx.e8m0_value(0) == 2.0 ** -127
    assert mx.e8m0_value(254) == 2.0 ** 127
    assert np.isnan(mx.e8m0_value(255))
