"""Number formats used by the ResidualKV cache, written from their definitions.

TEST INFRASTRUCTURE.  This module belongs to the CPU oracle.  Only ``tests/``,
``__graft_entry__.smoke()`` and the ``cpu_baseline`` / ``--impl reference`` legs
of ``bench.py`` may import it; the CUDA product path never does.

Every routine takes and returns float64 arrays whose values are exactly
representable in the target format, so the oracle can keep doing its
arithmetic in float64 and round only where the method stores or feeds a value
in a narrower type.

Formats
-------
* OCP FP8 E4M3 ("e4m3fn"): 1 sign bit, 4 exponent bits (bias 7), 3 mantissa
  bits, no infinities, the all-ones pattern is NaN, largest finite 448.  The
  ResidualKV notes (section 2.4, last paragraph; section 3.3) say the reference
  vectors are kept in FP8 in deployment; E4M3 with round-to-nearest-even and
  saturation to +-448 is this library's reading.
* IEEE binary16 (FP16): p = 11 significant bits, emin = -14.  The group
  extremes are stored as two FP16 numbers per group (ResidualKV notes,
  section 3.3, the q_b formula).
* bfloat16: p = 8 significant bits, emin = -126 (fp32 exponent range).
  The tensor-core operands are bf16.
* binary32: numpy's float32 conversion (IEEE round-to-nearest-even).
"""
from __future__ import annotations

import numpy as np

__all__ = [
    "round_to_format",
    "bf16",
    "fp32",
    "fp16_rn",
    "fp16_rd",
    "fp16_ru",
    "FP16_MAX",
    "E4M3_MAX",
    "e4m3_encode",
    "e4m3_decode",
    "bf16_bits",
]

FP16_MAX = 65504.0
E4M3_MAX = 448.0


def round_to_format(x, p: int, emin: int, mode: str = "rn") -> np.ndarray:
    """Round float64 values to a binary format with ``p`` significant bits.

    ``emin`` is the exponent of the smallest normal number; below it the
    quantum stays 2**(emin - p + 1) (gradual underflow).  ``mode`` is "rn"
    (nearest, ties to even), "rd" (toward -inf) or "ru" (toward +inf).
    Overflow is not handled here: callers clamp to their format's maximum.
    The division by the quantum is a power-of-two scaling, hence exact.
    """
    x = np.asarray(x, dtype=np.float64)
    a = np.abs(x)
    _, ex = np.frexp(a)              # a = m * 2**ex with m in [0.5, 1)
    e = np.maximum(ex - 1, emin)     # a in [2**e, 2**(e+1)) for normals
    quantum = np.ldexp(1.0, (e - (p - 1)).astype(np.int64))
    y = a / quantum
    if mode == "rn":
        r = np.rint(y)               # numpy rint: round half to even
    elif mode == "rd":
        r = np.where(x >= 0, np.floor(y), np.ceil(y))
    elif mode == "ru":
        r = np.where(x >= 0, np.ceil(y), np.floor(y))
    else:
        raise ValueError(mode)
    out = np.copysign(r * quantum, x)
    return np.where(a == 0, x, out)


def bf16(x) -> np.ndarray:
    """Round to bfloat16, nearest-even (8 significant bits, fp32 exponent range)."""
    return round_to_format(x, 8, -126, "rn")


def bf16_bits(x) -> np.ndarray:
    """uint16 bit patterns of values already representable in bfloat16."""
    f = np.asarray(x, dtype=np.float32)
    return (f.view(np.uint32) >> 16).astype(np.uint16)


def fp32(x) -> np.ndarray:
    """Round to binary32 (nearest-even) and return the value as float64."""
    return np.asarray(np.asarray(x, dtype=np.float64).astype(np.float32), dtype=np.float64)


def fp16_rn(x) -> np.ndarray:
    """Round to binary16, nearest-even; magnitudes beyond 65504 saturate."""
    return np.clip(round_to_format(x, 11, -14, "rn"), -FP16_MAX, FP16_MAX)


def fp16_rd(x) -> np.ndarray:
    """Round to binary16 toward -inf (saturating at -65504 / +65504)."""
    return np.clip(round_to_format(x, 11, -14, "rd"), -FP16_MAX, FP16_MAX)


def fp16_ru(x) -> np.ndarray:
    """Round to binary16 toward +inf (saturating at -65504 / +65504)."""
    return np.clip(round_to_format(x, 11, -14, "ru"), -FP16_MAX, FP16_MAX)


def e4m3_decode(codes) -> np.ndarray:
    """Value of each E4M3 byte: (-1)^s * 2^(e-7) * (1 + m/8), subnormal m * 2^-9."""
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    s = (c >> 7) & 1
    e = (c >> 3) & 0xF
    m = c & 0x7
    mag = np.where(e == 0, m * 2.0 ** -9, (1.0 + m / 8.0) * np.ldexp(1.0, e - 7))
    mag = np.where((e == 15) & (m == 7), np.nan, mag)
    return np.where(s == 1, -mag, mag)


def e4m3_encode(x) -> np.ndarray:
    """E4M3 byte for each value: nearest-even, saturating to +-448 (no NaN out)."""
    x = np.asarray(x, dtype=np.float64)
    v = np.clip(round_to_format(x, 4, -6, "rn"), -E4M3_MAX, E4M3_MAX)
    a = np.abs(v)
    s = (np.signbit(v)).astype(np.int64)
    _, ex = np.frexp(a)
    e_unb = ex - 1
    normal = a >= 2.0 ** -6
    # normal: a = (1 + m/8) * 2^(E-7)
    E = np.where(normal, e_unb + 7, 0)
    mant = np.where(normal,
                    np.rint((a / np.ldexp(1.0, np.where(normal, e_unb, 0)) - 1.0) * 8.0),
                    np.rint(a / 2.0 ** -9))
    code = (s << 7) | (E.astype(np.int64) << 3) | mant.astype(np.int64)
    return code.astype(np.uint8)
