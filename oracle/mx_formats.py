"""Number formats of the block-scaled MoE layer, decoded and encoded in FP64.

TEST INFRASTRUCTURE ONLY. This file is part of the plain CPU oracle. Only
``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import it; the CUDA product path never does.

The pages name the formats without defining them: FP8 activations and MXFP4
weights with "per-1x32 scaling" (AITER #5609 "Add DeepSeek V4.1 Flash TP4
gfx950 MoE tuning", Configuration; AITER #5904 "Add tuned a8w4 fused-MoE
configs for DeepSeek V4.1-Flash (TP4 + EP, gfx950)", first paragraph:
"FP8 activations x MXFP4 weights, QuantType.per_1x32"). The plainest reading,
used here, is the OCP microscaling family those names come from:

* E2M1 (MXFP4 element): sign, 2 exponent bits with bias 1, 1 mantissa bit,
  no inf/NaN.
* E8M0 (MX block scale): an unsigned biased exponent, value 2^(b-127);
  b = 255 is NaN.
* E4M3 "fn" (FP8 activation): sign, 4 exponent bits with bias 7, 3 mantissa
  bits, no infinities, S.1111.111 is NaN, largest finite 448.

Every table is built from the bit-field definition, not typed in, so the
tests can check it against independently written values.
"""
from __future__ import annotations

import numpy as np


def _e2m1_from_bits(code: int) -> float:
    sign = -1.0 if (code >> 3) & 1 else 1.0
    exp = (code >> 1) & 3
    man = code & 1
    if exp == 0:  # subnormal: 0.man * 2^(1 - bias) with bias 1
        mag = man * 0.5
    else:
        mag = (1.0 + man / 2.0) * 2.0 ** (exp - 1)
    return sign * mag


def _e4m3_from_bits(code: int) -> float:
    sign = -1.0 if (code >> 7) & 1 else 1.0
    exp = (code >> 3) & 15
    man = code & 7
    if exp == 15 and man == 7:
        return float("nan")
    if exp == 0:  # subnormal: 0.man * 2^(1 - 7)
        mag = (man / 8.0) * 2.0 ** (1 - 7)
    else:
        mag = (1.0 + man / 8.0) * 2.0 ** (exp - 7)
    return sign * mag


E2M1_VALUES = np.array([_e2m1_from_bits(c) for c in range(16)], dtype=np.float64)
E4M3_VALUES = np.array([_e4m3_from_bits(c) for c in range(256)], dtype=np.float64)
E4M3_MAX = 448.0
E4M3_EMAX = 8  # floor(log2(448))

# Non-negative finite E4M3 magnitudes in code order 0x00..0x7E (ascending).
_E4M3_POS = E4M3_VALUES[:127]


def e8m0_value(b) -> np.ndarray:
    """E8M0 byte -> 2^(b-127) (NaN for 255)."""
    b = np.asarray(b).astype(np.int64)
    v = np.ldexp(1.0, b - 127)
    return np.where(b == 255, np.nan, v)


def e4m3_encode(v) -> np.ndarray:
    """Round float64 values to E4M3 codes: round to nearest, ties to the even
    code (even mantissa), saturating at +-448, keeping the sign of zero.
    The search is over the explicit table of finite magnitudes."""
    v = np.asarray(v, dtype=np.float64)
    a = np.minimum(np.abs(v), E4M3_MAX)
    # index of the first table magnitude >= a
    hi = np.searchsorted(_E4M3_POS, a, side="left")
    hi = np.minimum(hi, 126)
    lo = np.maximum(hi - 1, 0)
    d_hi = _E4M3_POS[hi] - a
    d_lo = a - _E4M3_POS[lo]
    pick_hi = (d_hi < d_lo) | ((d_hi == d_lo) & (hi % 2 == 0))
    mag = np.where(pick_hi, hi, lo).astype(np.uint8)
    sign = np.where(np.signbit(v), 0x80, 0).astype(np.uint8)
    return (mag | sign).astype(np.uint8)


def bf16_round(v) -> np.ndarray:
    """Round float64 values to the nearest bfloat16 value (ties to even),
    directly from float64 (one rounding, no float32 step). Returns float64."""
    v = np.asarray(v, dtype=np.float64)
    a = np.abs(v)
    _, e = np.frexp(a)  # a = m * 2^e, m in [0.5, 1)
    # bfloat16 keeps 8 significant bits; below 2^-126 the quantum is 2^-133
    q_exp = np.maximum(e - 8, -133)
    q = np.ldexp(np.round(np.ldexp(a, -q_exp)), q_exp)
    bf16_max = (2.0 - 2.0 ** -7) * 2.0 ** 127
    q = np.where(q > bf16_max, np.inf, q)
    return np.copysign(q, v)


def bf16_bits(v) -> np.ndarray:
    """bfloat16 bit patterns (uint16) of float64 values that are already
    bfloat16-representable (the output of ``bf16_round``)."""
    f32 = np.asarray(v, dtype=np.float64).astype(np.float32)
    return (f32.view(np.uint32) >> 16).astype(np.uint16)


def unpack_e2m1(packed: np.ndarray) -> np.ndarray:
    """uint8 [..., K/2] (element k in byte k/2, low nibble = even k) ->
    uint8 codes [..., K]."""
    p = np.asarray(packed, dtype=np.uint8)
    out = np.empty(p.shape[:-1] + (p.shape[-1] * 2,), dtype=np.uint8)
    out[..., 0::2] = p & 0x0F
    out[..., 1::2] = p >> 4
    return out


def dequant_mxfp4(packed: np.ndarray, scale: np.ndarray) -> np.ndarray:
    """MXFP4 weights -> float64: E2M1 value times the E8M0 scale of its
    32-element block along the last (K) axis."""
    codes = unpack_e2m1(packed)
    vals = E2M1_VALUES[codes]
    s = e8m0_value(scale)
    return vals * np.repeat(s, 32, axis=-1)


def dequant_mxfp8(codes: np.ndarray, scale: np.ndarray) -> np.ndarray:
    """E4M3 codes with one E8M0 scale per 32 along the last axis -> float64."""
    vals = E4M3_VALUES[np.asarray(codes, dtype=np.uint8)]
    s = e8m0_value(scale)
    return vals * np.repeat(s, 32, axis=-1)


def quant_mxfp8(x) -> tuple[np.ndarray, np.ndarray]:
    """Per-1x32 FP8 quantisation of the rows of ``x`` (float64 [..., K]).

    For each block of 32 consecutive values along K:
      amax = max |x|; if amax == 0 the scale byte is 0 and every code is 0;
      else e = floor(log2(amax)) - 8 (8 = the E4M3 maximum exponent),
      clamped to [-127, 127]; scale byte = e + 127; code = E4M3 round-to-
      nearest-even of x / 2^e, saturating at +-448.
    This is the OCP MX conversion, the reading taken for the pages'
    "per-1x32 scaling" (AITER #5609, Configuration).
    Returns (codes uint8 [..., K], scale bytes uint8 [..., K/32]).
    """
    x = np.asarray(x, dtype=np.float64)
    K = x.shape[-1]
    assert K % 32 == 0
    xb = x.reshape(x.shape[:-1] + (K // 32, 32))
    amax = np.abs(xb).max(axis=-1)
    _, ex = np.frexp(amax)          # amax = m * 2^ex, m in [0.5, 1)
    flog2 = ex - 1                  # floor(log2(amax)) for amax > 0
    e = np.clip(flog2 - E4M3_EMAX, -127, 127)
    zero = amax == 0
    e = np.where(zero, 0, e)
    scaled = np.ldexp(xb, -e[..., None])
    codes = e4m3_encode(scaled)
    codes = np.where(zero[..., None], np.uint8(0), codes)
    sbyte = np.where(zero, 0, e + 127).astype(np.uint8)
    return codes.reshape(x.shape).astype(np.uint8), sbyte
