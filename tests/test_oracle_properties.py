"""Property pins of the oracle over random inputs (hypothesis; skipped where it is not
installed).  Each property follows from the definitions in ResidualKV notes §2.4
(group quantisation, packing), §2.6 (reference schedule) and the E4M3 format, and is
checked against a brute-force or closed-form statement, not against the oracle itself."""
import numpy as np
import pytest

hypothesis = pytest.importorskip("hypothesis")
from hypothesis import given, settings  # noqa: E402
from hypothesis import strategies as st  # noqa: E402

from oracle import codec as C  # noqa: E402
from oracle import formats as F  # noqa: E402

ALL_E4M3 = F.e4m3_decode(np.arange(256, dtype=np.uint8))
FINITE_E4M3 = np.unique(ALL_E4M3[np.isfinite(ALL_E4M3)])


@settings(max_examples=300, deadline=None)
@given(st.floats(min_value=-600.0, max_value=600.0, allow_nan=False))
def test_e4m3_encode_is_nearest_and_saturates(x):
    v = float(F.e4m3_decode(F.e4m3_encode(np.array([x])))[0])
    if abs(x) >= 448.0:
        assert v == np.copysign(448.0, x)
        return
    best = np.min(np.abs(FINITE_E4M3 - x))
    assert abs(v - x) == best                     # a nearest E4M3 value (ties: any nearest)


@settings(max_examples=60, deadline=None)
@given(st.integers(min_value=0, max_value=2**31 - 1),
       st.sampled_from([2, 4]),
       st.floats(min_value=-3.0, max_value=3.0))
def test_group_quantisation_error_within_half_step(seed, bits, log_scale):
    """|z~ - z| <= Delta / 2 per element (plus the fp32 rounding of the two operand-mode
    operations), codes in [0, 2^b - 1]; Delta = (max16 - min16) / (2^b - 1)."""
    rng = np.random.default_rng(seed)
    z = rng.standard_normal((3, 64)) * 10.0 ** log_scale + rng.standard_normal() * 10.0 ** log_scale
    q, meta, overflow = C.quantize(z, bits, 32)
    assert not overflow.any()
    levels = 2 ** bits - 1
    assert q.min() >= 0 and q.max() <= levels
    zt = C.dequantize(q, meta, bits, 32)
    for gi, (a, b) in enumerate(((0, 32), (32, 64))):
        lo, hi = meta[:, gi, 0][:, None], meta[:, gi, 1][:, None]
        delta = (hi - lo) / levels
        # the stored range covers the group (extremes rounded outward)
        assert np.all(lo <= z[:, a:b]) and np.all(z[:, a:b] <= hi)
        slack = 4 * 2.0 ** -24 * (np.abs(z[:, a:b]) + np.abs(lo) + np.abs(hi))
        assert np.all(np.abs(zt[:, a:b] - z[:, a:b]) <= delta / 2 * (1 + 2.0 ** -20) + slack)


@settings(max_examples=40, deadline=None)
@given(st.integers(min_value=0, max_value=2**31 - 1), st.sampled_from([2, 4]))
def test_constant_groups_are_exact(seed, bits):
    rng = np.random.default_rng(seed)
    vals = F.fp16_rn(rng.standard_normal(2) * 100.0)      # FP16-representable constants
    z = np.concatenate([np.full(32, vals[0]), np.full(32, vals[1])])[None, :]
    q, meta, _ = C.quantize(z, bits, 32)
    assert np.all(q == 0)
    assert np.array_equal(C.dequantize(q, meta, bits, 32), z)


@settings(max_examples=60, deadline=None)
@given(st.integers(min_value=0, max_value=2**31 - 1), st.sampled_from([2, 4]),
       st.integers(min_value=1, max_value=4))
def test_pack_unpack_round_trip(seed, bits, n):
    rng = np.random.default_rng(seed)
    d_c = 64
    q = rng.integers(0, 2 ** bits, size=(n, d_c))
    packed = C.pack_codes(q, bits)
    assert packed.shape == (n, d_c * bits // 8)
    assert np.array_equal(C.unpack_codes(packed, bits, d_c), q)


@settings(max_examples=150, deadline=None)
@given(st.integers(min_value=1, max_value=6000), st.integers(min_value=1, max_value=40),
       st.floats(min_value=0.0, max_value=0.25), st.integers(min_value=0, max_value=8))
def test_schedule_invariants(T, s0, alpha, sink):
    """Strictly increasing positions below T; the sinks first; p_0 = n_sink; every gap
    after it at least s_0 and exactly s_0 + floor(alpha (p - n_sink))."""
    p = C.reference_positions(T, s0, alpha, sink)
    assert np.all(np.diff(p) > 0) and p.min() == 0 and p.max() < T
    k = min(sink, T)
    assert np.array_equal(p[:k], np.arange(k))
    if sink < T:
        assert p[k] == sink
        rest = p[k:]
        gaps = np.diff(rest)
        expect = s0 + np.floor(alpha * (rest[:-1] - sink)).astype(np.int64)
        assert np.array_equal(gaps, expect)
        # the last reference is the last schedule point below T
        nxt = rest[-1] + s0 + int(np.floor(alpha * (rest[-1] - sink)))
        assert nxt >= T
