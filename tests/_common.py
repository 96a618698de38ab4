"""Shared helpers of the GPU parity tests: run a workload through the CUDA library and
through the oracle on the same seeded inputs, and compare what is unique."""
from __future__ import annotations

import numpy as np
import torch

import synth
from oracle import codec as C
from oracle import formats as F


def oracle_shape(w: synth.Workload, alpha: float = 0.0, sink: int = 0) -> C.Shape:
    return C.Shape(w.n_kv_heads, w.head_dim, w.d_c, w.d_ff, w.topk, w.group, w.bits, w.stride,
                   w.rope_base, alpha, sink)


def np64(t: torch.Tensor) -> np.ndarray:
    return t.detach().to("cpu", torch.float64).numpy()


class _CAI:
    def __init__(self, ptr: int, nbytes: int):
        self.__cuda_array_interface__ = {"shape": (nbytes,), "typestr": "|u1",
                                         "data": (ptr, False), "version": 3}


def device_bytes(ptr: int, nbytes: int) -> torch.Tensor:
    """A uint8 CUDA tensor viewing library-owned device memory (copied out)."""
    return torch.as_tensor(_CAI(ptr, nbytes), device="cuda").clone()


def make_codec(w: synth.Workload, W: dict, T: int, batch: int = 1, max_rows: int = 0,
               out_dtype: str | None = None, bits: int | None = None, alpha: float = 0.0,
               sink: int = 0, mean_precompute: int = 0):
    from residual_kv_cache_gb300 import Codec, Config
    cfg = Config(n_kv_heads=w.n_kv_heads, head_dim=w.head_dim, d_c=w.d_c, d_ff=w.d_ff,
                 topk=w.topk, group=w.group, bits=w.bits if bits is None else bits,
                 ref_stride=w.stride, kv_dtype=w.kv_dtype,
                 out_dtype=out_dtype or w.out_dtype, rope_base=w.rope_base, batch=batch,
                 max_tokens=T, max_rows=max_rows, ref_alpha=alpha, ref_sink=sink,
                 mean_precompute=mean_precompute)
    Wd = {k: v.cuda().contiguous() for k, v in W.items()}
    return Codec(cfg, Wd)


def gpu_prefill(codec, kv_dev: torch.Tensor, stride: int, seq_id: int = 0, alpha: float = 0.0,
                sink: int = 0):
    """Write every position of one sequence: references (the schedule's positions) to
    the pool, the rest encoded."""
    T = kv_dev.shape[0]
    pos = np.arange(T, dtype=np.int32)
    isref = C.is_reference(pos, stride, alpha, sink)
    ref = pos[isref]
    non = pos[~isref]
    codec.pool_append(kv_dev, np.full(len(ref), seq_id, np.int32), ref, src_rows=ref)
    codec.compress(kv_dev, np.full(len(non), seq_id, np.int32), non, src_rows=non)
    return ref, non


def idx_parity(gpu_idx: np.ndarray, ora_idx: np.ndarray, kv: np.ndarray, pool_vals: np.ndarray,
               pool_pos: np.ndarray, positions: np.ndarray, rel_gap: float = 1e-4):
    """Compare retrieved slot lists.  Returns (n_exact, n_swapped, bad_rows): a row that
    differs is accepted only if every differing rank pairs two distances whose relative
    gap is below rel_gap (exact float64 distances), and every GPU slot is a visible,
    distinct reference."""
    exact = np.all(gpu_idx == ora_idx, axis=1)
    bad = []
    n_swap = 0
    for r in np.nonzero(~exact)[0]:
        g, o = gpu_idx[r], ora_idx[r]
        if np.sum(g >= 0) != np.sum(o >= 0):
            bad.append(r)
            continue
        k = int(np.sum(o >= 0))
        gs = g[:k]
        if (len(set(gs.tolist())) != k or np.any(gs < 0) or np.any(gs >= len(pool_pos))
                or np.any(pool_pos[np.clip(gs, 0, len(pool_pos) - 1)] >= positions[r])):
            bad.append(r)
            continue
        dg = np.sum((kv[r][None, :] - pool_vals[gs]) ** 2, axis=1)
        do = np.sum((kv[r][None, :] - pool_vals[o[:k]]) ** 2, axis=1)
        if np.all(np.abs(dg - do) <= rel_gap * do):
            n_swap += 1
        else:
            bad.append(r)
    return int(exact.sum()), n_swap, bad


def preround(z32: np.ndarray, meta: np.ndarray, bits: int, g: int = 32) -> np.ndarray:
    """The quantiser's pre-round value (z - min)/Delta in binary32, per coordinate."""
    n, d_c = z32.shape
    out = np.zeros((n, d_c))
    levels = np.float32(2 ** bits - 1)
    for gi, a in enumerate(range(0, d_c, g)):
        lo = meta[:, gi, 0].astype(np.float32)[:, None]
        hi = meta[:, gi, 1].astype(np.float32)[:, None]
        delta = (hi - lo) / levels
        with np.errstate(divide="ignore", invalid="ignore"):
            out[:, a:a + g] = ((z32[:, a:a + g].astype(np.float32) - lo) / delta).astype(np.float64)
    return out


def rel_fro(a: np.ndarray, b: np.ndarray) -> float:
    return float(np.linalg.norm((a - b).ravel()) / max(np.linalg.norm(b.ravel()), 1e-300))


# ---------------------------------------------------------------------------------
# Evaluation bounds.  The kernels multiply bf16 operands on the tensor cores and
# accumulate in fp32, 16 products per instruction, instructions issued in K order.
# GEMM-1/2 gives a1, a2 per hidden unit; the epilogue forms h = Swish(a1) a2 in fp32
# (fast exponential and division), d = h(kv) - h(mean) in fp32, and passes d to GEMM-3
# as two bf16 parts (hi, lo).  These helpers compute, from the oracle's own values only,
# a bound on how far any such evaluation can land from the exact value, and check the
# GPU's values against the interval it spans.
# Accumulation bound (first order): each addition into the running sum S_m is charged
# one unit in the last place of |S_m| (covering truncating as well as rounding adders),
# |err| <= u sum_m (|S_m| + sum_chunk |x w|), the second term for the adds inside one
# 16-product instruction.
# ---------------------------------------------------------------------------------
U32 = 2.0 ** -24


def fp32_chunked_bound(X: np.ndarray, W: np.ndarray, chunk: int = 16) -> np.ndarray:
    """Bound on |fl32(X W) - X W| for a K-ordered accumulation in 16-wide chunks.  The
    bound's own sums run in fp32 (torch, all host cores) and are widened by 2^-10 to
    cover their rounding."""
    Xt = torch.from_numpy(np.ascontiguousarray(X, dtype=np.float32))
    Wt = torch.from_numpy(np.ascontiguousarray(W, dtype=np.float32))
    Xa, Wa = Xt.abs(), Wt.abs()
    n, K = Xt.shape
    S = torch.zeros((n, Wt.shape[1]))
    acc = Xa @ Wa                                      # the in-chunk additions, all chunks
    for k0 in range(0, K, chunk):
        S.addmm_(Xt[:, k0:k0 + chunk], Wt[k0:k0 + chunk])
        acc.add_(S.abs())
    return (2.0 * U32 * (1.0 + 2.0 ** -10)) * acc.double().numpy()


def bf16_near(x: np.ndarray) -> np.ndarray:
    """Nearest bf16 value of each float64 (ties to even), by the bits of the binary64
    encoding: exact where the result is a normal bf16, which holds for the values these
    bounds round; anything else goes through the oracle's general rounding."""
    x = np.ascontiguousarray(x, dtype=np.float64)
    b = x.view(np.uint64)
    lsb = (b >> np.uint64(45)) & np.uint64(1)
    r = (b + np.uint64((1 << 44) - 1) + lsb) & ~np.uint64((1 << 45) - 1)
    out = r.view(np.float64)
    ax = np.abs(x)
    odd = ~np.isfinite(out) | ((ax < 2.0 ** -126) & (ax != 0)) | (np.abs(out) > 3.3895313892515355e38)
    if odd.any():
        out[odd] = F.bf16(x[odd])
    return out


def hidden_bounds(X: np.ndarray, Wc1: np.ndarray, Wc2: np.ndarray):
    """For operand rows X (bf16 values): exact h = Swish(X Wc1) * (X Wc2) and a bound dh
    on a fp32 evaluation's error (accumulation of a1 and a2, then Swish with a fast
    exponential and division, relative error <= |a1| 2^-22 + 2^-19, and the product)."""
    a1, a2 = X @ Wc1, X @ Wc2
    da1 = fp32_chunked_bound(X, Wc1)
    da2 = fp32_chunked_bound(X, Wc2)
    return swiglu_bounds(a1, a2, da1, da2)


def swiglu_bounds(a1, a2, da1, da2):
    """h = Swish(a1) * a2 for exact pre-activations, and the bound dh on a fp32
    evaluation from pre-activations within da1, da2 of them (Swish with a fast
    exponential and division, relative error <= |a1| 2^-22 + 2^-19, then the product)."""
    with np.errstate(over="ignore"):
        sig = 1.0 / (1.0 + np.exp(-a1))
    sw = a1 * sig
    dsw = np.abs(sig * (1.0 + a1 * (1.0 - sig)))       # |d Swish / d a1| <= 1.1
    h = sw * a2
    eps = np.abs(a1) * 2.0 ** -22 + 2.0 ** -19
    dh = dsw * da1 * (np.abs(a2) + da2) + np.abs(sw) * da2 + (eps + 2.0 ** -23) * np.abs(h) \
        + eps * np.abs(sw) * da2
    return h, dh


def z_bounds(d, dd, Wc3):
    """z = d W3 for the exact hidden difference d, and a half-width covering every d'
    within dd of it, its split into bf16 hi + lo (|d - hi - lo| <= 2^-18 |d|), and the
    fp32 accumulation of the 2 d_ff products (hi half first, then lo)."""
    aw = np.abs(Wc3)
    z = d @ Wc3
    ddt = dd + (2.0 ** -18 + 2.0 ** -23) * np.abs(d)
    ad = np.abs(d) + ddt
    w = ddt @ aw + fp32_chunked_bound(np.concatenate([ad, ad * 2.0 ** -8], axis=1),
                                      np.concatenate([aw, aw], axis=0))
    return z, w


def check_codes_interval(gq, gmeta, z, w, bits, g=32, window=1e-3):
    """Every GPU extreme must be the directed FP16 rounding of the extreme of some z' in
    [z - w, z + w]; every GPU code must be the rounding (in binary32, the kernel's
    precision) of (z' - min)/Delta under the GPU's own extremes for such a z', widened
    by `window` quantisation steps.  Returns a list of violations."""
    viol = []
    n, d_c = z.shape
    levels = 2 ** bits - 1
    for gi, a in enumerate(range(0, d_c, g)):
        zl, zh = z[:, a:a + g] - w[:, a:a + g], z[:, a:a + g] + w[:, a:a + g]
        lo_min, lo_max = F.fp16_rd(zl.min(1)), F.fp16_rd(zh.min(1))
        hi_min, hi_max = F.fp16_ru(zl.max(1)), F.fp16_ru(zh.max(1))
        glo, ghi = gmeta[:, gi, 0], gmeta[:, gi, 1]
        # a constant group stores the nearest FP16 of its value
        exact_const = (w[:, a:a + g].max(1) == 0) & (z[:, a:a + g].min(1) == z[:, a:a + g].max(1))
        okm = ((glo >= lo_min) & (glo <= lo_max) & (ghi >= hi_min) & (ghi <= hi_max)) | exact_const
        for r in np.nonzero(~okm)[0]:
            viol.append(("meta", int(r), gi, float(glo[r]), float(ghi[r]), float(lo_min[r]),
                         float(lo_max[r]), float(hi_min[r]), float(hi_max[r])))
        lo32 = glo.astype(np.float32)[:, None]
        delta = (ghi.astype(np.float32)[:, None] - lo32) / np.float32(levels)
        with np.errstate(divide="ignore", invalid="ignore"):
            ul = ((zl.astype(np.float32) - lo32) / delta).astype(np.float64) - window
            uh = ((zh.astype(np.float32) - lo32) / delta).astype(np.float64) + window
        qmin = np.clip(np.rint(ul), 0, levels)
        qmax = np.clip(np.rint(uh), 0, levels)
        zero = (delta[:, 0] == 0)
        qmin[zero] = 0
        qmax[zero] = 0
        q = gq[:, a:a + g]
        bad = (q < qmin) | (q > qmax)
        for r, c in zip(*np.nonzero(bad)):
            viol.append(("code", int(r), int(a + c), int(q[r, c]), float(ul[r, c]), float(uh[r, c])))
    return viol


def oracle_operand_rows(kv64_rows: np.ndarray, pool_vals: np.ndarray, idx_rows: np.ndarray):
    """bf16 kv rows and bf16 mean rows exactly as the oracle forms them."""
    means = np.stack([C.reference_mean(pool_vals, i[i >= 0]) for i in idx_rows])
    return F.bf16(kv64_rows), F.bf16(means)


def encoder_intervals(kv64_rows, pool_vals, idx_rows, W64):
    """The exact hidden difference d = h(kv) - h(mean) of the given tokens, its
    evaluation bound dd, and the code z with its half-width w."""
    xk, xm = oracle_operand_rows(kv64_rows, pool_vals, idx_rows)
    hk, dhk = hidden_bounds(xk, W64["Wc1"], W64["Wc2"])
    hm, dhm = hidden_bounds(xm, W64["Wc1"], W64["Wc2"])
    d = hk - hm
    dd = dhk + dhm + 2.0 ** -23 * np.abs(d)          # + the fp32 subtraction
    z, w = z_bounds(d, dd, W64["Wc3"])
    return dict(d=d, dd=dd, z=z, w=w)


def encoder_intervals_refs(kv64_rows, pool_vals, idx_rows, W64):
    """encoder_intervals for the mean's pre-activations taken from the references' own
    (mean_precompute): per slot P = fl32(r [W_c1 | W_c2]) within the chunked fp32 bound,
    the fp32 sum of the token's k <= 4 P rows (<= 3 additions, 2^-23 of the running sum
    each), the scaling by 1/k (exact for k = 1, 2, 4; one rounding for 3), then the same
    Swish, subtraction and GEMM-3 bounds."""
    xk = F.bf16(kv64_rows)
    hk, dhk = hidden_bounds(xk, W64["Wc1"], W64["Wc2"])
    P1, P2 = pool_vals @ W64["Wc1"], pool_vals @ W64["Wc2"]
    dP1, dP2 = fp32_chunked_bound(pool_vals, W64["Wc1"]), fp32_chunked_bound(pool_vals, W64["Wc2"])
    n = len(idx_rows)
    a1 = np.zeros((n, P1.shape[1]))
    a2, da1, da2 = np.zeros_like(a1), np.zeros_like(a1), np.zeros_like(a1)
    for r, i in enumerate(idx_rows):
        s = i[i >= 0]
        k = len(s)
        a1[r], a2[r] = P1[s].sum(0) / k, P2[s].sum(0) / k
        sum_err = 3 * 2.0 ** -23 * (np.abs(P1[s]).sum(0) + dP1[s].sum(0))
        da1[r] = (dP1[s].sum(0) + sum_err) / k + 2.0 ** -24 * np.abs(a1[r])
        sum_err = 3 * 2.0 ** -23 * (np.abs(P2[s]).sum(0) + dP2[s].sum(0))
        da2[r] = (dP2[s].sum(0) + sum_err) / k + 2.0 ** -24 * np.abs(a2[r])
    hm, dhm = swiglu_bounds(a1, a2, da1, da2)
    d = hk - hm
    dd = dhk + dhm + 2.0 ** -23 * np.abs(d)
    z, w = z_bounds(d, dd, W64["Wc3"])
    return dict(d=d, dd=dd, z=z, w=w)


def _requantize(z32, lo, hi, bits):
    """Codes of z under given FP16 extremes, as the quantiser takes them: binary32
    (z - min) / Delta with Delta = (max - min) / (2^b - 1), round half to even, clamped;
    also the pre-round values.  Rows of z: [n, g]; lo, hi: [n]."""
    levels = np.float32(2 ** bits - 1)
    lo32 = lo.astype(np.float32)[:, None]
    delta = (hi.astype(np.float32)[:, None] - lo32) / levels
    with np.errstate(divide="ignore", invalid="ignore"):
        u = ((z32.astype(np.float32) - lo32) / delta).astype(np.float64)
    q = np.clip(np.rint(u), 0, 2 ** bits - 1)
    q[np.broadcast_to(delta == 0, q.shape)] = 0
    return q, u


def code_parity_report(gq, gmeta, oq, ometa, oz, bits, g=32, window=1e-3, meta_rel=1e-6):
    """Counts for the method's code tolerance, over every code given: codes identical
    except +-1 where the oracle's binary32 pre-round value lies within `window` of a .5
    boundary; FP16 extremes identical except where the oracle's group extreme lies within
    `meta_rel` (relative) of an FP16 value.

    The extremes set Delta and min, so where a group's extremes differ its codes are
    compared with the oracle's z quantised under the GPU's extremes instead (the same
    window applies).  Keys:
      codes, identical (fraction over all codes), diff, not_pm1,
      beyond_window: differing codes outside the window (either kind of group),
      diff_other_extremes: differing codes in groups whose extremes differ,
      extremes_differ, extremes_within / extremes_beyond (meta_rel of an FP16 value)."""
    n, d_c = gq.shape
    G = d_c // g
    same = gq == oq
    diff = ~same
    step = np.abs(gq.astype(np.int64) - oq.astype(np.int64))
    meta_ne = gmeta != ometa                                     # [n, G, 2]
    gdiff = np.any(meta_ne, axis=2)
    gdiff_c = np.repeat(gdiff, g, axis=1)[:, :d_c]
    u = preround(oz, ometa, bits, g)
    with np.errstate(invalid="ignore"):
        in_win = np.abs(u - np.floor(u) - 0.5) < window
    beyond = int((diff & ~gdiff_c & ~in_win).sum())
    # groups whose extremes differ: the oracle's z under the GPU's extremes
    other = 0
    for r, gi in zip(*np.nonzero(gdiff)):
        a = gi * g
        q2, u2 = _requantize(oz[r:r + 1, a:a + g], gmeta[r:r + 1, gi, 0], gmeta[r:r + 1, gi, 1], bits)
        d2 = gq[r, a:a + g] != q2[0]
        if d2.any():
            fr = np.abs(u2[0] - np.floor(u2[0]) - 0.5)
            bad = d2 & ((np.abs(gq[r, a:a + g] - q2[0]) > 1) | (fr >= window))
            beyond += int(bad.sum())
    zg = oz[:, :G * g].reshape(n, G, g)
    ext = np.stack([zg.min(axis=2), zg.max(axis=2)], axis=2)     # [n, G, 2]
    near = F.fp16_rn(ext)
    close = np.abs(ext - near) <= meta_rel * np.maximum(np.abs(ext), 1e-30)
    other = int((diff & gdiff_c).sum())
    return {
        "codes": int(gq.size), "identical": float(same.mean()), "diff": int(diff.sum()),
        "not_pm1": int((step > 1).sum()), "beyond_window": beyond,
        "diff_other_extremes": other,
        "extremes_differ": int(meta_ne.sum()),
        "extremes_within": int((meta_ne & close).sum()),
        "extremes_beyond": int((meta_ne & ~close).sum()),
    }


def assert_code_parity(label, gq, gmeta, oq, ometa, oz, kv64_rows, pool_vals, idx_rows, W64,
                       bits, g=32):
    """The method's code tolerance, asserted over every code given, with the counts
    printed (pytest -rP or -s shows them).

    INT codes (bits 4, 2): at least 99.9 % identical over all codes, and a differing code
    only +-1 where the oracle's binary32 pre-round value lies within 1e-3 of a .5
    boundary.  Where a group's FP16 extremes differ, Delta and min differ and the group's
    codes move together; those codes are held to the same rule under the GPU's extremes.
    An extreme may differ where a correct evaluation of z puts the group's minimum or
    maximum on the other side of an FP16 value: every extreme and every code must lie in
    the interval derived from the arithmetic (check_codes_interval), and how many
    extremes differ by more than the oracle's distance of 1e-6 (relative) to an FP16 value
    is reported.

    Quantisation off (bits 16, z stored as bf16): every value inside its interval and at
    least 99 % identical (a correct evaluation moves z across a bf16 rounding boundary for
    a fraction of about E|dz| / ulp(z) of the values)."""
    iv = encoder_intervals(kv64_rows, pool_vals, idx_rows, W64)
    if bits == 16:
        lo, hi = F.bf16(iv["z"] - iv["w"]), F.bf16(iv["z"] + iv["w"])
        ident = float(np.mean(gq == oq))
        print(f"[codes {label}] bf16 z: {gq.size} values, identical {ident:.6f}")
        assert np.all((gq >= lo) & (gq <= hi))
        assert ident >= 0.99, f"only {ident:.5f} of bf16 z identical"
        return
    rep = code_parity_report(gq, gmeta, oq, ometa, oz, bits, g)
    print(f"[codes {label}] {rep}")
    assert rep["identical"] >= 0.999, f"only {rep['identical']:.5f} of codes identical"
    assert rep["not_pm1"] == 0, f"{rep['not_pm1']} codes differ by more than one level"
    assert rep["beyond_window"] == 0, f"{rep['beyond_window']} codes differ away from a .5 boundary"
    viol = check_codes_interval(gq, gmeta, iv["z"], iv["w"], bits, g)
    assert not viol, f"{len(viol)} codes or extremes outside their interval, first {viol[:3]}"
