"""Pins of the codec oracle against closed forms, printed values, brute force
and invariants the page states (ResidualKV notes, sections 2.2-2.8, 3.3)."""
import itertools
import math
import os

import numpy as np
import pytest
import torch

import oracle
from oracle import codec as C
from oracle import formats as F
from oracle import storage as S

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                rows.append(line.split())
    return rows


def _weights(rng, d_kv, d_ff, d_c, scale=1.0):
    def w(r, c):
        return F.bf16(scale * rng.normal(0, math.sqrt(2 / (r + c)), (r, c)))
    return {"Wc1": w(d_kv, d_ff), "Wc2": w(d_kv, d_ff), "Wc3": w(d_ff, d_c), "Wd": w(d_c, d_kv)}


# ---------------------------------------------------------------- schedule
def test_reference_count_is_ceil_T_over_s():
    assert len(C.reference_positions(256, 8)) == 32
    assert len(C.reference_positions(32768, 16)) == 2048
    assert len(C.reference_positions(1000, 16)) == 63
    assert C.reference_positions(40, 16).tolist() == [0, 16, 32]


def test_dynamic_schedule_with_alpha_zero_is_the_fixed_stride():
    """Section 2.6: alpha = 0 is the fixed stride, p_m = n_sink + m s_0."""
    for T, s in ((256, 8), (1000, 16), (4099, 10), (17, 32)):
        assert C.reference_positions(T, s, 0.0, 0).tolist() == list(range(0, T, s))
    # with sinks: 0 .. n_sink - 1, then n_sink, n_sink + s, ...
    assert C.reference_positions(40, 10, 0.0, 4).tolist() == [0, 1, 2, 3, 4, 14, 24, 34]


def test_dynamic_schedule_first_terms_by_hand():
    """p_{m+1} = p_m + s_0 + floor(alpha (p_m - n_sink)) with s_0 = 10,
    alpha = 0.1, n_sink = 4: 4, 4+10+0 = 14, 14+10+1 = 25, 25+10+2 = 37,
    37+10+3 = 50, 50+10+4 = 64, 64+10+6 = 80."""
    got = C.reference_positions(81, 10, 0.1, 4).tolist()
    assert got == [0, 1, 2, 3, 4, 14, 25, 37, 50, 64, 80]
    assert C.is_reference([3, 4, 5, 14, 24, 25], 10, 0.1, 4).tolist() == [
        True, True, False, True, False, True]


def test_dynamic_schedule_reproduces_table_vi_counts():
    """Table VI (section 4.6) counts at a 262K context with s_0 = 10.  The five
    counts are reproduced together, with no sink tokens, for an effective
    length T in [261881, 261890] (the page does not state the exact length);
    alpha = 0 there is ceil(T / 10)."""
    rows = [(float(a), int(n)) for a, n in _golden("table6_reference_counts.txt")]
    for T in (261881, 261885, 261890):
        for alpha, n in rows:
            assert len(C.reference_positions(T, 10, alpha, 0)) == n, (T, alpha)
    assert -(-261885 // 10) == 26189
    # just outside the window the alpha = 0 count moves
    assert len(C.reference_positions(261880, 10, 0.0, 0)) == 26188
    assert len(C.reference_positions(261891, 10, 0.0, 0)) == 26190


def test_dynamic_schedule_against_the_page_estimate():
    """Section 2.6's estimate log_{1+alpha}(1 + alpha (T - n_sink) / s_0) drops
    the floor.  The floor shortens each gap by less than one token, so the gaps
    lie between those of the real-valued recurrence with s_0 - 1 and with s_0,
    and the count between the two estimates (+1 for the last partial gap)."""
    for alpha in (0.001, 0.02, 0.05, 0.1):
        for T, sink in ((262144, 0), (98304, 0), (32768, 4)):
            n = len(C.reference_positions(T, 10, alpha, sink)) - sink
            lo = C.reference_count_estimate(T, 10, alpha, sink)
            hi = C.reference_count_estimate(T, 9, alpha, sink) + 1
            assert lo <= n <= hi, (alpha, T, n, lo, hi)


def test_dynamic_schedule_every_token_has_an_earlier_reference():
    """With the sinks kept as references, position 0 is always a reference, so
    no non-reference token has an empty pool; gaps never shrink."""
    for alpha, sink in ((0.02, 0), (0.05, 4), (0.1, 16)):
        rp = C.reference_positions(5000, 8, alpha, sink)
        assert rp[0] == 0 and np.all(np.diff(rp) >= 1)
        gaps = np.diff(rp[sink:])
        assert np.all(np.diff(gaps) >= 0) and gaps[0] == 8


def test_compress_with_dynamic_schedule_retrieves_only_earlier_references():
    """The write path over a dynamic schedule: every token's slots point at
    references strictly before it, k_i = min(k, references before it), and a
    reference's own row is [slot, -1, ...]."""
    rng = np.random.default_rng(7)
    sh = C.Shape(n_kv_heads=1, head_dim=16, d_c=16, d_ff=32, topk=4, group=16, bits=4,
                 stride=4, ref_alpha=0.25, ref_sink=2)
    T = 96
    kv = rng.normal(size=(T, sh.d_kv))
    st = C.compress_sequence(kv, _weights(rng, sh.d_kv, sh.d_ff, sh.d_c), sh, "fp64")
    rp = C.reference_positions(T, sh.stride, sh.ref_alpha, sh.ref_sink)
    assert st.pool.pos.tolist() == rp.tolist()
    for p in range(T):
        row = st.idx[p]
        if p in set(rp.tolist()):
            assert row[0] == rp.tolist().index(p) and np.all(row[1:] == -1)
            continue
        before = int(np.sum(rp < p))
        valid = row[row >= 0]
        assert len(valid) == min(sh.topk, before)
        assert np.all(st.pool.pos[valid] < p)


# ---------------------------------------------------------------- retrieval
def test_retrieval_equals_brute_force_over_subsets():
    rng = np.random.default_rng(10)
    for trial in range(60):
        R = int(rng.integers(1, 9))
        d = 6
        pool_vals = F.e4m3_decode(F.e4m3_encode(rng.normal(0, 1, (R, d))))
        pool_pos = np.arange(R) * 3
        q = rng.normal(0, 1, d)
        pos = int(rng.integers(1, 3 * R + 1))
        vis = [j for j in range(R) if pool_pos[j] < pos]
        if not vis:
            with pytest.raises(ValueError):
                C.retrieve(q, pool_vals, pool_pos, pos, 4)
            continue
        slots, dist = C.retrieve(q, pool_vals, pool_pos, pos, 4)
        k_i = min(4, len(vis))
        assert len(slots) == k_i
        # brute force: the k_i-subset of visible refs minimising rho^2
        best, best_set = None, None
        for sub in itertools.combinations(vis, k_i):
            rho2 = sum(float(np.sum((q - pool_vals[j]) ** 2)) for j in sub)
            if best is None or rho2 < best - 1e-12:
                best, best_set = rho2, set(sub)
        assert set(slots.tolist()) == best_set
        assert np.all(np.diff(dist) >= 0)
        assert all(pool_pos[j] < pos for j in slots)


def test_retrieval_warmup_k_i():
    s = 8
    rng = np.random.default_rng(11)
    T = 6 * s
    kv = rng.normal(0, 1, (T, 16))
    pool = C.build_pool(kv, T, s)
    for pos in range(1, T):
        if pos % s == 0:
            continue
        slots, _ = C.retrieve(kv[pos], pool.vals, pool.pos, pos, 4)
        n_vis = pos // s + 1
        assert len(slots) == min(4, n_vis)
    # warm-up, k_i = min(k, |T_ref,i|) (ResidualKV notes §2.1): tokens 1..s-1 see one
    # reference (position 0), token s+1 sees two
    assert len(C.retrieve(kv[1], pool.vals, pool.pos, 1, 4)[0]) == 1
    assert len(C.retrieve(kv[s + 1], pool.vals, pool.pos, s + 1, 4)[0]) == 2


def test_retrieval_tie_keeps_smaller_slot():
    pool_vals = np.array([[1.0, 0.0], [0.0, 1.0], [1.0, 0.0], [0.0, 1.0], [1.0, 0.0]])
    pool_pos = np.arange(5)
    slots, _ = C.retrieve(np.array([1.0, 0.0]), pool_vals, pool_pos, 10, 2)
    assert slots.tolist() == [0, 2]
    slots, _ = C.retrieve(np.array([0.5, 0.5]), pool_vals, pool_pos, 10, 4)
    assert slots.tolist() == [0, 1, 2, 3]


# ---------------------------------------------------------------- mean / Thm IV.1
def test_theorem_iv1_decomposition_with_oracle_mean():
    rng = np.random.default_rng(12)
    for _ in range(50):
        R, d = 12, 32
        pool = F.e4m3_decode(F.e4m3_encode(rng.normal(0, 1, (R, d))))
        q = rng.normal(0, 1, d)
        slots, dist = C.retrieve(q, pool, np.arange(R), R, 4)
        m = C.reference_mean(pool, slots, "fp64")
        rho2 = float(np.mean(dist))
        delta2 = float(np.sum((q - m) ** 2))
        V = float(np.mean(np.sum((pool[slots] - m) ** 2, axis=1)))
        assert abs(rho2 - (delta2 + V)) <= 1e-12 * rho2
        r2, d2, v2 = C.theorem_iv1_terms(q, pool, slots)
        assert abs(r2 - (d2 + v2)) <= 1e-12 * r2


def test_operand_mean_is_correctly_rounded_binary32():
    rng = np.random.default_rng(13)
    pool = F.e4m3_decode(F.e4m3_encode(rng.normal(0, 2, (40, 64))))
    for k in (1, 2, 3, 4):
        for _ in range(20):
            slots = rng.choice(40, k, replace=False)
            exact = C.reference_mean(pool, slots, "fp64")
            op = C.reference_mean(pool, slots, "operand")
            assert np.array_equal(op, F.fp32(op))
            ulp = np.spacing(np.abs(exact).astype(np.float32)).astype(np.float64)
            assert np.all(np.abs(op - exact) <= 0.5 * ulp)
            if k in (1, 2, 4):
                assert np.array_equal(op, exact)


# ---------------------------------------------------------------- f_c
def test_swish_closed_forms_and_library():
    assert C.swish(0.0) == 0.0
    assert abs(C.swish(1.0) - 0.7310585786300049) < 1e-15
    assert abs(C.swish(50.0) - 50.0) < 1e-12
    assert abs(C.swish(-50.0)) < 1e-18
    x = np.linspace(-20, 20, 1001)
    lib = torch.nn.functional.silu(torch.tensor(x)).numpy()
    assert np.max(np.abs(C.swish(x) - lib)) < 1e-14


def test_f_c_special_cases():
    rng = np.random.default_rng(14)
    d_kv, d_ff, d_c = 16, 24, 8
    W = _weights(rng, d_kv, d_ff, d_c)
    x = rng.normal(0, 1, (5, d_kv))
    zero = np.zeros_like(W["Wc2"])
    for mode in ("fp64", "operand"):
        assert np.all(C.f_c(x, W["Wc1"], zero, W["Wc3"], mode) == 0)
        assert np.all(C.f_c(x, zero, W["Wc2"], W["Wc3"], mode) == 0)   # Swish(0) = 0
    # one active path: x = e_0, W_c1 = a e_0 e_0^T, W_c2 = b e_0 e_0^T, W_c3 = e_0 e_0^T
    a, b = 1.5, -2.0
    e0 = np.zeros(d_kv); e0[0] = 1
    W1 = np.zeros((d_kv, d_ff)); W1[0, 0] = a
    W2 = np.zeros((d_kv, d_ff)); W2[0, 0] = b
    W3 = np.zeros((d_ff, d_c)); W3[0, 0] = 1
    out = C.f_c(e0[None], W1, W2, W3, "fp64")[0]
    assert abs(out[0] - a / (1 + math.exp(-a)) * b) < 1e-15
    assert np.all(out[1:] == 0)


def test_residual_maps_first_then_subtracts():
    rng = np.random.default_rng(15)
    d_kv, d_ff, d_c = 32, 48, 16
    W = _weights(rng, d_kv, d_ff, d_c, scale=3.0)
    kv = rng.normal(0, 1, (8, d_kv))
    m = kv + 0.3 * rng.normal(0, 1, kv.shape)
    for mode in ("fp64", "operand"):
        assert np.all(C.residual_code(kv, kv, W, mode) == 0)       # kv == mean -> z == 0
    z = C.residual_code(kv, m, W, "fp64")
    wrong = C.f_c(kv - m, W["Wc1"], W["Wc2"], W["Wc3"], "fp64")  # f_c of the difference
    assert np.linalg.norm(z - wrong) > 1e-2 * np.linalg.norm(z)
    # additivity of W_c3: f_c(kv) - f_c(m) = (h(kv) - h(m)) W_c3 exactly in fp64 math
    h = C.swiglu_hidden(kv, W["Wc1"], W["Wc2"], "fp64") - C.swiglu_hidden(m, W["Wc1"], W["Wc2"], "fp64")
    assert np.allclose(z, h @ W["Wc3"], rtol=0, atol=1e-12)


# ---------------------------------------------------------------- quantisation
def test_quant_ramp_gives_every_level():
    z = np.arange(16, dtype=np.float64)[None, :] / 15.0        # min 0, max 1 exact in FP16
    z = F.fp32(np.concatenate([z, z], axis=1))                  # two groups of 16 -> g=16
    q, meta, ovf = C.quantize(z, 4, 16)
    assert q[0, :16].tolist() == list(range(16))
    assert np.all(meta[0, :, 0] == 0) and np.all(meta[0, :, 1] == 1)
    z2 = F.fp32(np.array([[0, 1 / 3, 2 / 3, 1.0]]))
    q2, _, _ = C.quantize(z2, 2, 4)
    assert q2[0].tolist() == [0, 1, 2, 3]


def test_quant_round_half_even():
    # range [0, 15] -> Delta = 1 exactly; values at .5 go to the even level
    z = np.array([[0.0, 15.0, 2.5, 3.5, 4.5, 7.5, 0.5, 14.5]])
    q, _, _ = C.quantize(z, 4, 8)
    assert q[0].tolist() == [0, 15, 2, 4, 4, 8, 0, 14]


@pytest.mark.parametrize("bits", [4, 2])
@pytest.mark.parametrize("mode", ["operand", "fp64"])
def test_quant_error_within_half_step_and_page_bounds(bits, mode):
    rng = np.random.default_rng(16 + bits)
    z = F.fp32(rng.normal(0, 1, (200, 96)) * rng.uniform(0.01, 10, (200, 1)))
    q, meta, ovf = C.quantize(z, bits, 32, mode)
    assert not ovf.any()
    assert q.min() >= 0 and q.max() <= 2 ** bits - 1
    zt = C.dequantize(q, meta, bits, 32, mode)
    for gi, a in enumerate(range(0, 96, 32)):
        lo, hi = meta[:, gi, 0], meta[:, gi, 1]
        zg = z[:, a:a + 32]
        assert np.all(lo <= zg.min(axis=1)) and np.all(hi >= zg.max(axis=1))
        delta = (hi - lo) / (2 ** bits - 1)
        err = np.abs(zt[:, a:a + 32] - zg)
        assert np.all(err <= delta[:, None] * (0.5 + 1e-5))
    # the page's vector bound, with the stored (outward-rounded) range
    for i in range(200):
        e = np.linalg.norm(zt[i] - z[i])
        _, loose = C.quant_error_bounds(z[i], bits, 32)
        s = sum(32 * (meta[i, g, 1] - meta[i, g, 0]) ** 2 for g in range(3))
        tight = math.sqrt(s) / (2 * (2 ** bits - 1))
        assert e <= tight * (1 + 1e-5)
        assert e <= loose * (1 + 1e-3) + 1e-6


def test_quant_constant_groups_exact():
    z = np.zeros((3, 64))
    z[1, :32] = 0.375
    z[2, 32:] = -1.25
    q, meta, _ = C.quantize(z, 4, 32)
    assert np.all(q == 0)
    zt = C.dequantize(q, meta, 4, 32)
    assert np.array_equal(zt, z)


def test_pack_layout_and_roundtrip():
    assert C.pack_codes(np.array([[1, 2]]), 4).tolist() == [[0x21]]
    assert C.pack_codes(np.array([[1, 2, 3, 0]]), 2).tolist() == [[0x39]]
    rng = np.random.default_rng(17)
    for bits in (4, 2):
        q = rng.integers(0, 2 ** bits, (5, 64))
        p = C.pack_codes(q, bits)
        assert p.shape == (5, 64 * bits // 8)
        assert np.array_equal(C.unpack_codes(p, bits, 64), q)
    zb = F.bf16(rng.normal(0, 1, (4, 64)))
    assert np.array_equal(C.unpack_codes(C.pack_codes(zb, 16), 16, 64), zb)


def test_group_storage_matches_page():
    for bits, val in _golden("group_quant_storage.txt"):
        assert S.q_b(int(bits)) == float(val)
        # byte-level: one group of 32 = 32*b/8 payload bytes + 2 FP16 extremes (4 B)
        payload = 32 * int(bits) // 8 + 4
        assert payload / (32 * 2) == float(val)


def test_keep_ratio_worked_example():
    for full, total, rho, ratio, bits, pct, dec in _golden("kr_worked_example.txt"):
        kr = S.keep_ratio(int(full) / int(total), float(rho), int(bits), float(ratio))
        assert round(100 * kr, int(dec)) == float(pct)


# ---------------------------------------------------------------- decoder / RoPE
def _tiny_store(seed=20, T=48, bits=4):
    rng = np.random.default_rng(seed)
    sh = C.Shape(n_kv_heads=2, head_dim=8, d_c=32, d_ff=24, stride=8, bits=bits, rope_base=1e4)
    cent = rng.normal(0, 1, (4, sh.d_kv))
    kv = F.fp32(cent[rng.integers(0, 4, T)] + 0.3 * rng.normal(0, 1, (T, sh.d_kv)))
    W = _weights(rng, sh.d_kv, sh.d_ff, sh.d_c)
    return sh, kv, W


def test_zero_decoder_returns_reference_mean():
    sh, kv, W = _tiny_store()
    W0 = dict(W, Wd=np.zeros_like(W["Wd"]))
    st = C.compress_sequence(kv, W0, sh)
    pos = np.arange(1, 48)
    K, V, kvh = C.reconstruct(st, pos, W0)
    means = np.stack([C.reference_mean(st.pool.vals, st.idx[p][st.idx[p] >= 0]) for p in pos])
    assert np.array_equal(kvh, means)
    Km, Vm = C.split_kv(means, sh.n_kv_heads, sh.head_dim)
    assert np.array_equal(V, Vm)


def test_reference_tokens_read_back_their_fp8_value():
    sh, kv, W = _tiny_store()
    st = C.compress_sequence(kv, W, sh)
    refs = C.reference_positions(48, sh.stride)
    K, V, kvh = C.reconstruct(st, refs, W)
    fp8 = F.e4m3_decode(F.e4m3_encode(kv[refs]))
    assert np.array_equal(kvh, fp8)
    Kr, Vr = C.split_kv(fp8, sh.n_kv_heads, sh.head_dim)
    assert np.array_equal(V, Vr)
    assert np.array_equal(K[0], Kr[0])          # position 0: RoPE is the identity


def test_rope_closed_forms():
    for p, c, s in _golden("rope_unit_rotation.txt"):
        p, c, s = int(p), float(c), float(s)
        out = C.rope(np.array([[[0.6, -0.8]]]), np.array([p]), 1e4)[0, 0]
        assert abs(out[0] - (0.6 * c + 0.8 * s)) < 1e-15
        assert abs(out[1] - (-0.8 * c + 0.6 * s)) < 1e-15
    # rotate-half pairing for D=4: pairs (0,2) at theta_0=1 and (1,3) at theta_1=base^-1/2
    base = 100.0
    x = np.array([[[1.0, 0.0, 0.0, 0.0]]])
    out = C.rope(x, np.array([1]), base)[0, 0]
    assert np.allclose(out, [math.cos(1), 0, math.sin(1), 0], atol=1e-15)
    x = np.array([[[0.0, 1.0, 0.0, 0.0]]])
    out = C.rope(x, np.array([3]), base)[0, 0]
    a = 3 * base ** -0.5
    assert np.allclose(out, [0, math.cos(a), 0, math.sin(a)], atol=1e-15)


def test_rope_invariants():
    rng = np.random.default_rng(21)
    K = rng.normal(0, 1, (10, 4, 128))
    pos = rng.integers(0, 262144, 10)
    R = C.rope(K, pos, 5e5)
    pair = lambda A: A[..., :64] ** 2 + A[..., 64:] ** 2
    assert np.allclose(pair(R), pair(K), rtol=1e-12)
    assert np.array_equal(C.rope(K, np.zeros(10, int), 5e5), K)
    back = C.rope(R, -pos, 5e5)
    assert np.allclose(back, K, atol=1e-9)
    p1, p2 = rng.integers(0, 1000, 10), rng.integers(0, 1000, 10)
    assert np.allclose(C.rope(C.rope(K, p1, 5e5), p2, 5e5), C.rope(K, p1 + p2, 5e5), atol=1e-10)


def test_reconstruct_rotates_at_own_position():
    sh, kv, W = _tiny_store()
    st = C.compress_sequence(kv, W, sh)
    pos = np.array([13, 30, 47])
    K, V, kvh = C.reconstruct(st, pos, W)
    Kp, _ = C.split_kv(kvh, sh.n_kv_heads, sh.head_dim)
    assert np.allclose(C.rope(K, -pos, sh.rope_base), Kp, atol=1e-12)
    ref_pos = np.array([st.pool.pos[st.idx[p][0]] for p in pos])
    K_ref = C.rope(Kp, ref_pos, sh.rope_base)
    assert np.linalg.norm(K_ref - K) > 1e-3 * np.linalg.norm(K)


def test_whole_path_error_bound_holds():
    """Section 2.8: ||kv - KV_hat|| <= (eta + C_b) ||Delta|| with eta, gamma
    measured on the same tokens (a consistency check of encode + decode)."""
    sh, kv, W = _tiny_store(bits=4)
    st = C.compress_sequence(kv, W, sh, mode="fp64")
    nonref = np.array([p for p in range(48) if p % sh.stride])
    K, V, kvh = C.reconstruct(st, nonref, W, mode="fp64")
    means = np.stack([C.reference_mean(st.pool.vals, st.idx[p][st.idx[p] >= 0], "fp64") for p in nonref])
    Delta = kv[nonref] - means
    z = st.z[nonref]
    dn = np.linalg.norm(Delta, axis=1)
    eta = np.max(np.linalg.norm(Delta - z @ W["Wd"], axis=1) / dn)
    gamma = np.max(np.linalg.norm(z, axis=1) / dn)
    Cb = np.linalg.norm(W["Wd"], 2) * gamma * math.sqrt(sh.group / 2) / (2 ** sh.bits - 1)
    err = np.linalg.norm(kv[nonref] - kvh, axis=1)
    assert np.all(err <= (eta + Cb) * dn * (1 + 1e-9))


def test_operand_and_fp64_modes_agree_loosely():
    """bf16 operands perturb z by ~0.2 %; that flips ~1 % of the codes by one
    level, and every flip moves z-tilde by a whole step.  So the two modes
    share retrieval exactly, and differ in codes and K/V only by that much.
    (This is why the K/V parity tolerance is taken against operand mode.)"""
    sh, kv, W = _tiny_store(seed=22)
    a = C.compress_sequence(kv, W, sh, mode="operand")
    b = C.compress_sequence(kv, W, sh, mode="fp64")
    assert np.array_equal(a.idx, b.idx)
    nonref = np.array([p for p in range(48) if p % sh.stride])
    flips = np.abs(a.q[nonref] - b.q[nonref])
    assert flips.max() <= 1 and flips.mean() < 0.05
    pos = np.arange(48)
    Ka, Va, _ = C.reconstruct(a, pos, W, "operand")
    Kb, Vb, _ = C.reconstruct(b, pos, W, "fp64")
    rel = np.linalg.norm(np.concatenate([Ka - Kb, Va - Vb])) / np.linalg.norm(np.concatenate([Kb, Vb]))
    assert rel < 5e-2


def test_mean_hidden_from_reference_preactivations():
    """The weight-stationary form of the mean's hidden row (ResidualKV notes §2.3, f_c at
    the §2.2 mean): (1/k) sum_j r_j W taken per reference equals torch's
    silu(mean W_c1) * (mean W_c2) at the exact float64 mean; one reference gives the
    hidden row at that reference; repeating a reference or permuting the slots changes
    nothing."""
    import torch
    rng = np.random.default_rng(11)
    d_kv, d_ff = 64, 48
    pool = rng.normal(size=(9, d_kv))
    W1, W2 = rng.normal(size=(d_kv, d_ff)) / 8, rng.normal(size=(d_kv, d_ff)) / 8

    def torch_hidden(x):
        xt = torch.tensor(x)
        return (torch.nn.functional.silu(xt @ torch.tensor(W1)) * (xt @ torch.tensor(W2))).numpy()

    for slots in ([3], [0, 5], [1, 2, 7], [8, 4, 6, 0]):
        got = C.mean_hidden_from_refs(pool, slots, W1, W2)
        want = torch_hidden(pool[slots].mean(axis=0))
        assert np.allclose(got, want, rtol=1e-11, atol=1e-12), slots
    assert np.allclose(C.mean_hidden_from_refs(pool, [5], W1, W2), torch_hidden(pool[5]),
                       rtol=1e-12, atol=1e-13)
    assert np.allclose(C.mean_hidden_from_refs(pool, [5, 5], W1, W2),
                       C.mean_hidden_from_refs(pool, [5], W1, W2), rtol=1e-13, atol=1e-14)
    assert np.allclose(C.mean_hidden_from_refs(pool, [2, 7, 1], W1, W2),
                       C.mean_hidden_from_refs(pool, [1, 2, 7], W1, W2), rtol=1e-13, atol=1e-14)


def test_encoding_from_reference_preactivations():
    """encode_tokens with the mean's hidden row from the references: in fp64 the same z
    as mapping the mean row (linearity); in operand mode it differs only by the bf16
    rounding the mean row gets as a tensor-core operand (well under 1 % of z here), and
    the slots are the same."""
    import synth
    w = synth.workload("tiny")
    kv = synth.gen_kv(w, 21).double().numpy()
    W = {k: v.double().numpy() for k, v in synth.gen_weights(w, 22).items()}
    sh = C.Shape(w.n_kv_heads, w.head_dim, w.d_c, w.d_ff, w.topk, w.group, w.bits, w.stride,
                 w.rope_base)
    pool = C.build_pool(kv, w.T, w.stride)
    pos = np.array([9, 33, 100, 201, 255])
    a = C.encode_tokens(kv[pos], pos, pool, W, sh, "fp64", "row")
    b = C.encode_tokens(kv[pos], pos, pool, W, sh, "fp64", "refs")
    assert np.array_equal(a["idx"], b["idx"])
    assert np.allclose(a["z"], b["z"], rtol=1e-10, atol=1e-12)
    c = C.encode_tokens(kv[pos], pos, pool, W, sh, "operand", "row")
    e = C.encode_tokens(kv[pos], pos, pool, W, sh, "operand", "refs")
    assert np.array_equal(c["idx"], e["idx"])
    rel = np.linalg.norm(c["z"] - e["z"]) / np.linalg.norm(c["z"])
    assert 0 < rel < 1e-2
    with pytest.raises(ValueError):
        C.encode_tokens(kv[pos], pos, pool, W, sh, "fp64", "mean")
