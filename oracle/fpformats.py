"""Oracle: the two narrow floating-point formats of the layer, from their definitions.

TEST INFRASTRUCTURE ONLY. Nothing in the product path imports this package;
only the tests, the smoke check and the benchmark's CPU-baseline leg do.

Formats (OCP 8-bit floating point specification, E4M3 variant; OCP
microscaling / NVIDIA NVFP4 element type E2M1). The EpiLoRA page ("Fusing Many
LoRA Adapters into Low-Precision GEMMs for Serving and RL", Introduction and
§Design › The vLLM plugin › Implementation and correctness) only names FP8
and NVFP4; the bit layouts below are those public definitions:

E4M3 (byte: s eeee mmm, exponent bias 7)
  * exponent field 0: subnormal, value = m * 2^-9           (m = 0..7)
  * exponent field 1..15: normal, value = (1 + m/8) * 2^(e-7)
  * e = 15 and m = 7 is NaN; there is no infinity; the largest finite
    magnitude is (1 + 6/8) * 2^8 = 448.

E2M1 (nibble: s ee m, exponent bias 1)
  * exponent field 0: subnormal, value = m * 0.5            (m = 0..1)
  * exponent field 1..3: normal, value = (1 + m/2) * 2^(e-1)
  * magnitudes {0, 0.5, 1, 1.5, 2, 3, 4, 6}; no NaN, no infinity.

Rounding (the reading taken for conversions of a float32 value): round to
nearest, ties to the even code, and saturate magnitudes above the largest
finite value to it (the "satfinite" behaviour). Rounding is computed exactly
in float64: a float32 value divided by a power of two is exact, so
rint(v / quantum) * quantum is the correctly rounded result on that grid.
"""
from __future__ import annotations

import numpy as np

E4M3_MAX = 448.0
E4M3_MIN_NORMAL_EXP = -6      # smallest normal: 2^-6
E4M3_MANT_BITS = 3
E2M1_MAX = 6.0
E2M1_MIN_NORMAL_EXP = 0       # smallest normal: 1.0
E2M1_MANT_BITS = 1


def _floor_log2(a: np.ndarray) -> np.ndarray:
    """Exact floor(log2(a)) for a > 0 (frexp returns a = f * 2^e, f in [0.5, 1))."""
    _, e = np.frexp(a)
    return e.astype(np.int64) - 1


def _round_to_format(v, min_normal_exp: int, mant_bits: int, max_val: float) -> np.ndarray:
    """Round float values onto a sign-magnitude binary grid: RNE + satfinite."""
    v = np.asarray(v, dtype=np.float64)
    a = np.abs(v)
    safe = np.where(a > 0, a, 1.0)
    e = np.maximum(_floor_log2(safe), min_normal_exp)   # subnormals share the min-normal quantum
    quantum = np.ldexp(1.0, (e - mant_bits).astype(np.int64))
    r = np.rint(a / quantum) * quantum                   # np.rint rounds half to even
    r = np.minimum(r, max_val)                           # saturate to the largest finite value
    r = np.where(a > 0, r, 0.0)
    return np.copysign(r, v)


def e4m3_round(v) -> np.ndarray:
    """Nearest E4M3 value (as float64) of each element, ties to even, saturating."""
    return _round_to_format(v, E4M3_MIN_NORMAL_EXP, E4M3_MANT_BITS, E4M3_MAX)


def e2m1_round(v) -> np.ndarray:
    """Nearest E2M1 value (as float64) of each element, ties to even, saturating."""
    return _round_to_format(v, E2M1_MIN_NORMAL_EXP, E2M1_MANT_BITS, E2M1_MAX)


def _encode(r: np.ndarray, bias: int, mant_bits: int, exp_bits: int) -> np.ndarray:
    """Bit pattern of values already on the grid (finite, representable)."""
    r = np.asarray(r, dtype=np.float64)
    sign = np.signbit(r).astype(np.int64)
    a = np.abs(r)
    min_normal = 2.0 ** (1 - bias)
    safe = np.where(a > 0, a, 1.0)
    e = _floor_log2(safe)
    normal = a >= min_normal
    exp_field = np.where(normal, e + bias, 0)
    sub_quantum = 2.0 ** (1 - bias - mant_bits)
    mant_normal = np.rint((a / np.ldexp(1.0, e) - 1.0) * (1 << mant_bits))
    mant_sub = np.rint(a / sub_quantum)
    mant = np.where(normal, mant_normal, mant_sub).astype(np.int64)
    mant = np.where(a > 0, mant, 0)
    exp_field = np.where(a > 0, exp_field, 0)
    code = (sign << (exp_bits + mant_bits)) | (exp_field << mant_bits) | mant
    return code.astype(np.uint8)


def _decode(code, bias: int, mant_bits: int, exp_bits: int) -> np.ndarray:
    c = np.asarray(code).astype(np.int64)
    sign = (c >> (exp_bits + mant_bits)) & 1
    e = (c >> mant_bits) & ((1 << exp_bits) - 1)
    m = c & ((1 << mant_bits) - 1)
    sub = m * 2.0 ** (1 - bias - mant_bits)
    nor = (1.0 + m / float(1 << mant_bits)) * np.ldexp(1.0, (e - bias).astype(np.int64))
    v = np.where(e == 0, sub, nor)
    return np.where(sign == 1, -v, v)


def e4m3_encode(r) -> np.ndarray:
    """Byte code of E4M3-representable values."""
    return _encode(r, bias=7, mant_bits=3, exp_bits=4)


def e4m3_decode(code) -> np.ndarray:
    """float64 value of E4M3 byte codes (0x7F / 0xFF decode to NaN)."""
    c = np.asarray(code).astype(np.int64)
    v = _decode(c, bias=7, mant_bits=3, exp_bits=4)
    return np.where((c & 0x7F) == 0x7F, np.nan, v)


def e2m1_encode(r) -> np.ndarray:
    """4-bit code (in a uint8) of E2M1-representable values."""
    return _encode(r, bias=1, mant_bits=1, exp_bits=2)


def e2m1_decode(code) -> np.ndarray:
    return _decode(np.asarray(code).astype(np.int64) & 0xF, bias=1, mant_bits=1, exp_bits=2)


def fp32_to_e4m3_code(x) -> np.ndarray:
    """Conversion of float32 values to E4M3 codes (RNE, satfinite)."""
    return e4m3_encode(e4m3_round(np.asarray(x, dtype=np.float32)))


def fp32_to_e2m1_code(x) -> np.ndarray:
    """Conversion of float32 values to E2M1 codes (RNE, satfinite)."""
    return e2m1_encode(e2m1_round(np.asarray(x, dtype=np.float32)))


def pack_e2m1(codes: np.ndarray) -> np.ndarray:
    """Two E2M1 codes per byte along the last axis: element 2i in the low nibble."""
    c = np.asarray(codes, dtype=np.uint8)
    if c.shape[-1] % 2:
        raise ValueError("last axis must be even")
    return (c[..., 0::2] & 0xF) | ((c[..., 1::2] & 0xF) << 4)


def unpack_e2m1(packed: np.ndarray) -> np.ndarray:
    p = np.asarray(packed, dtype=np.uint8)
    out = np.empty(p.shape[:-1] + (p.shape[-1] * 2,), dtype=np.uint8)
    out[..., 0::2] = p & 0xF
    out[..., 1::2] = p >> 4
    return out
