"""Pins of the oracle's number formats against library conversions and brute force."""
import os

import numpy as np
import pytest
import torch

from oracle import formats as F


def _fp8_lib_decode(codes):
    t = torch.tensor(np.asarray(codes, np.uint8)).view(torch.float8_e4m3fn)
    return t.to(torch.float64).numpy()


def test_e4m3_decode_all_codes_match_torch():
    codes = np.arange(256, dtype=np.uint8)
    ours = F.e4m3_decode(codes)
    lib = _fp8_lib_decode(codes)
    nan = np.isnan(lib)
    assert np.array_equal(np.isnan(ours), nan)
    assert nan.sum() == 2                       # 0x7f and 0xff
    assert np.array_equal(ours[~nan], lib[~nan])
    assert ours[0x7E] == 448.0 and ours[0x01] == 2.0 ** -9


def test_e4m3_encode_roundtrip_all_finite_codes():
    codes = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], dtype=np.uint8)
    vals = F.e4m3_decode(codes)
    back = F.e4m3_encode(vals)
    # +0 and -0 both decode to 0; keep sign via signbit in encode
    assert np.array_equal(back, codes)


def test_e4m3_encode_matches_torch_rne_random_and_midpoints():
    rng = np.random.default_rng(0)
    x = np.concatenate([rng.normal(0, 3, 20000), rng.uniform(-448, 448, 5000),
                        rng.normal(0, 0.01, 5000)]).astype(np.float32).astype(np.float64)
    pos = np.sort(np.unique(np.abs(F.e4m3_decode(np.arange(0, 0x7F, dtype=np.uint8)))))
    mids = (pos[1:] + pos[:-1]) / 2                 # exact ties
    x = np.concatenate([x, mids, -mids])
    ours = F.e4m3_decode(F.e4m3_encode(x))
    lib = torch.tensor(x, dtype=torch.float32).to(torch.float8_e4m3fn).to(torch.float64).numpy()
    assert np.array_equal(ours, lib)


def test_e4m3_saturates_to_448():
    x = np.array([449.0, 464.0, 1e6, -500.0])
    assert np.array_equal(F.e4m3_decode(F.e4m3_encode(x)), [448, 448, 448, -448])


def test_bf16_matches_torch():
    rng = np.random.default_rng(1)
    x = np.concatenate([rng.normal(0, 1, 50000), rng.normal(0, 1e-30, 1000),
                        rng.normal(0, 1e30, 1000)]).astype(np.float32)
    # exact ties: values with the 16 low bits equal to 0x8000
    ties = (rng.integers(0, 2 ** 31, 2000, dtype=np.uint32) & 0x7F7F0000) | 0x8000
    x = np.concatenate([x, ties.view(np.float32)]).astype(np.float64)
    x = x[np.isfinite(x)]
    lib = torch.tensor(x, dtype=torch.float32).to(torch.bfloat16).to(torch.float64).numpy()
    assert np.array_equal(F.bf16(x), lib)


def test_fp16_rn_matches_numpy():
    rng = np.random.default_rng(2)
    x = np.concatenate([rng.normal(0, 1, 50000), rng.normal(0, 1e-5, 5000),
                        rng.uniform(-6e4, 6e4, 5000)]).astype(np.float32).astype(np.float64)
    assert np.array_equal(F.fp16_rn(x), x.astype(np.float16).astype(np.float64))


def test_fp16_directed_brackets_by_brute_force():
    pos = np.arange(0, 0x7C00, dtype=np.uint16).view(np.float16).astype(np.float64)
    allv = np.concatenate([-pos[::-1], pos])
    allv = np.unique(allv)
    lo, hi = allv[:-1], allv[1:]
    # exactly representable values are fixed points
    assert np.array_equal(F.fp16_rd(allv), allv)
    assert np.array_equal(F.fp16_ru(allv), allv)
    # points strictly between two neighbours go to the neighbours
    rng = np.random.default_rng(3)
    t = rng.uniform(0.01, 0.99, lo.size)
    mid = lo + t * (hi - lo)
    ok = (mid > lo) & (mid < hi)
    assert np.array_equal(F.fp16_rd(mid[ok]), lo[ok])
    assert np.array_equal(F.fp16_ru(mid[ok]), hi[ok])


def test_fp32_is_ieee_single():
    x = np.array([1 + 2 ** -24, 1 + 3 * 2 ** -24, 0.1])
    assert F.fp32(x)[0] == 1.0
    assert F.fp32(x)[1] == 1 + 2 ** -22
    assert F.fp32(x)[2] == float(np.float32(0.1))


def test_parity_helper_bf16_rounding_matches_the_oracle():
    """The fast bf16 rounding the parity bounds use equals the oracle's general rounding
    on random values, exact ties and values next to ties."""
    import sys
    sys.path.insert(0, os.path.dirname(os.path.abspath(__file__)))
    from _common import bf16_near
    rng = np.random.default_rng(5)
    x = rng.normal(0, 1, 200000) * 10.0 ** rng.uniform(-8, 8, 200000)
    ties = (np.arange(1, 2000) * 2 + 1) * 2.0 ** -8 * 3.0       # between bf16 neighbours
    near = np.concatenate([ties * (1 + 2.0 ** -40), ties * (1 - 2.0 ** -40)])
    for v in (x, ties, near, -ties, np.array([0.0, -0.0, 1.0, 2.0 ** -120])):
        assert np.array_equal(bf16_near(v), F.bf16(v))
