"""CPU oracle of the ResidualKV cache codec: plain, slow, float64.

TEST INFRASTRUCTURE.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import this
module.  It shares no code with the CUDA library and imports nothing from it.

Source of every step: the page "ResidualKV:基于参考向量与残差的 KV Cache 压缩"
(study notes on arXiv 2602.08005v2), cited below as "ResidualKV notes" with
its section and equation.

Two arithmetic modes
--------------------
``mode="fp64"``    every product and sum in float64 on the values as given.
                   The storage formats the method itself prescribes are kept
                   (FP8 references, FP16 group extremes, b-bit codes).
``mode="operand"`` the same steps, but values are rounded where the GPU
                   library rounds them: bf16 for the tensor-core operands
                   kv, reference mean, weights and dequantised code; binary32
                   for the reference mean and for the code z before
                   quantisation.  The SwiGLU hidden rows stay exact: the
                   library forms h(kv) - h(mean) in binary32 and feeds it to
                   the last GEMM as two bf16 parts (about 16 significant
                   bits), which W_c3's linearity allows (section 2.3).
                   Accumulation stays float64.  The quantiser's decisions are
                   taken in binary32 (the kernel's precision) so that integer
                   codes can be compared exactly.

Readings of points the page leaves open (each one is also listed in the
design notes of the repository):
* the reference schedule starts at position 0 (fixed stride) or, for the
  dynamic schedule, at p_0 = n_sink with the n_sink sink tokens before it kept
  as references too; floor(alpha (p - n_sink)) is taken of one binary64 product;
* token i may retrieve references with position < i, ties broken by the
  smaller pool slot;
* "Swish" is x*sigmoid(x) (beta = 1), no biases;
* group extremes are stored as FP16, min rounded down and max rounded up;
  q = round-half-even((z - min)/Delta); a constant group stores its value;
* INT4 packs element 2t in the low nibble of byte t, INT2 element 4t+u in
  bits [2u, 2u+2);
* K is the first d_k columns of KV_hat laid out [head][dim], V the rest;
* RoPE is the rotate-half form with theta_j = base^(-2j/D) at the token's own
  0-based position.
"""
from __future__ import annotations

from dataclasses import dataclass

import math

import numpy as np

from . import formats as F

__all__ = [
    "Shape",
    "reference_positions",
    "is_reference",
    "reference_count_estimate",
    "store_references",
    "visible_slots",
    "retrieve",
    "reference_mean",
    "swish",
    "swiglu_hidden",
    "f_c",
    "residual_code",
    "quantize",
    "dequantize",
    "pack_codes",
    "unpack_codes",
    "decode",
    "split_kv",
    "rope_angles",
    "rope",
    "Pool",
    "build_pool",
    "encode_token",
    "encode_tokens",
    "Store",
    "compress_sequence",
    "reconstruct",
    "theorem_iv1_terms",
    "quant_error_bounds",
]


@dataclass(frozen=True)
class Shape:
    """Codec shape.  ``d_kv`` is 2*d_k = 2*N*D, the joint K/V width."""

    n_kv_heads: int
    head_dim: int
    d_c: int
    d_ff: int
    topk: int = 4
    group: int = 32
    bits: int = 4          # 4, 2, or 16 = quantisation off (z kept as bf16)
    stride: int = 16
    rope_base: float = 1e4
    ref_alpha: float = 0.0  # dynamic schedule growth (0: fixed stride)
    ref_sink: int = 0       # sink tokens, kept as references ahead of the schedule

    @property
    def d_k(self) -> int:
        return self.n_kv_heads * self.head_dim

    @property
    def d_kv(self) -> int:
        return 2 * self.d_k

    @property
    def n_groups(self) -> int:
        return -(-self.d_c // self.group)

    @property
    def code_bytes(self) -> int:
        """Bytes of one token's packed code."""
        if self.bits == 16:
            return 2 * self.d_c
        return -(-self.d_c * self.bits // 8)


# --------------------------------------------------------------------------
# Reference schedule (ResidualKV notes, section 2.6: fixed and dynamic stride)
# --------------------------------------------------------------------------
def reference_positions(T: int, stride: int, alpha: float = 0.0, sink: int = 0) -> np.ndarray:
    """Positions below T kept as references.

    Section 2.6: the gaps grow with the position, p_{m+1} = p_m + s_0 +
    floor(alpha (p_m - n_sink)), with s_0 = ``stride``; alpha = 0 is the fixed
    stride.  Readings: the schedule starts at p_0 = n_sink, and the n_sink sink
    tokens before it are references too (so every token has one before it);
    alpha (p_m - n_sink) is one binary64 product, then floored.
    """
    out = list(range(min(sink, T)))
    p = sink
    while p < T:
        out.append(p)
        p = p + stride + math.floor(alpha * (p - sink))
    return np.array(out, dtype=np.int64)


def is_reference(pos, stride: int, alpha: float = 0.0, sink: int = 0):
    pos = np.asarray(pos)
    if pos.size == 0:
        return np.zeros(pos.shape, dtype=bool)
    return np.isin(pos, reference_positions(int(pos.max()) + 1, stride, alpha, sink))


def reference_count_estimate(T: int, stride: int, alpha: float, sink: int = 0) -> float:
    """The page's closed-form estimate of the scheduled references (section 2.6),
    from the recurrence without the floor: log_{1+alpha}(1 + alpha (T - n_sink) / s_0);
    its alpha -> 0 limit is (T - n_sink) / s_0."""
    if alpha == 0.0:
        return (T - sink) / stride
    return math.log1p(alpha * (T - sink) / stride) / math.log1p(alpha)


# --------------------------------------------------------------------------
# Reference pool in FP8 (ResidualKV notes, section 2.4 last paragraph, 3.3)
# --------------------------------------------------------------------------
def store_references(kv_rows):
    """Store reference rows the way the pool keeps them.

    Returns (fp8 bytes, decoded values, squared norms).  The squared norm is
    the exact sum of the squared decoded values rounded once to binary32:
    every square of an E4M3 value has at most 8 significant bits between
    2**-18 and 448**2, so float64 sums of a few thousand of them are exact.
    """
    codes = F.e4m3_encode(kv_rows)
    vals = F.e4m3_decode(codes)
    norm2 = F.fp32(np.sum(vals * vals, axis=-1))
    return codes, vals, norm2


def visible_slots(pool_pos: np.ndarray, pos: int) -> np.ndarray:
    """Slots of the references token ``pos`` may use: the historical
    reference set T_ref,i, i.e. references strictly before it."""
    return np.nonzero(np.asarray(pool_pos) < pos)[0]


# --------------------------------------------------------------------------
# Retrieval (ResidualKV notes, section 2.2, the arg top-k_i equation)
# --------------------------------------------------------------------------
def retrieve(kv_i, pool_vals, pool_pos, pos: int, k: int):
    """Top-k_i nearest references by squared L2 distance.

    k_i = min(k, |T_ref,i|).  Distances are sum((kv_i - r_j)^2) in float64;
    equal distances keep the smaller slot first.  Returns (slots, distances),
    both ordered nearest first.
    """
    cand = visible_slots(pool_pos, pos)
    if cand.size == 0:
        raise ValueError("token has an empty reference pool")
    diff = np.asarray(kv_i, dtype=np.float64)[None, :] - pool_vals[cand]
    d = np.sum(diff * diff, axis=1)
    order = np.lexsort((cand, d))            # by distance, then by slot
    k_i = min(k, cand.size)
    sel = order[:k_i]
    return cand[sel], d[sel]


def reference_mean(pool_vals, slots, mode: str = "operand"):
    """Arithmetic mean of the retrieved references (section 2.2, mean eq.).

    The sum of at most four E4M3 values is exact in binary32 (their bits span
    2**-9 .. 2**11), so in operand mode the mean is that exact sum divided by
    k_i with one binary32 rounding (IEEE division, done by numpy in float32).
    """
    slots = np.asarray(slots)
    s = np.sum(pool_vals[slots], axis=0)
    if mode == "fp64":
        return s / len(slots)
    return np.asarray(s.astype(np.float32) / np.float32(len(slots)), dtype=np.float64)


# --------------------------------------------------------------------------
# SwiGLU compressor and latent residual (section 2.3)
# --------------------------------------------------------------------------
def swish(x):
    """Swish with beta = 1: x * sigmoid(x) = x / (1 + exp(-x))."""
    with np.errstate(over="ignore"):
        return x / (1.0 + np.exp(-x))


def swiglu_hidden(x, Wc1, Wc2, mode: str = "operand"):
    """Swish(x W_c1) (elementwise) x W_c2, the hidden row of f_c (section 2.3); exact
    in both modes (the operand mode rounds only x, see the module notes)."""
    return swish(x @ Wc1) * (x @ Wc2)


def mean_hidden_from_refs(pool_vals, slots, Wc1, Wc2):
    """The hidden row of f_c at the reference mean, with the mean's pre-activations
    taken from the references' own: mean_i W = (1/k_i) sum_j (kv_j W) for j in R_i,
    since x W is linear in x (section 2.3 maps the mean, which section 2.2 averages in
    KV space).  The references are the FP8-decoded pool rows, exact in bf16, so no
    operand is rounded; accumulation is float64.  This is the weight-stationary form of
    the mean half of the encoder: the products kv_j W_c1 / W_c2 are fixed per reference
    and can be kept beside the pool.
    """
    R = pool_vals[np.asarray(slots)]
    k = len(slots)
    a1 = (R @ Wc1).sum(axis=0) / k
    a2 = (R @ Wc2).sum(axis=0) / k
    return swish(a1) * a2


def f_c(x, Wc1, Wc2, Wc3, mode: str = "operand"):
    """f_c(x) = (Swish(x W_c1) * x W_c2) W_c3 (row-vector convention)."""
    if mode == "operand":
        x = F.bf16(x)
    return swiglu_hidden(x, Wc1, Wc2, mode) @ Wc3


def residual_code(kv, mean, W, mode: str = "operand"):
    """z = f_c(kv) - f_c(mean): map both, then subtract (boxed eq., 2.3).

    In operand mode the result is rounded to binary32, the precision in which
    the kernel holds z before quantising it.
    """
    Wc1, Wc2, Wc3 = W["Wc1"], W["Wc2"], W["Wc3"]
    z = f_c(kv, Wc1, Wc2, Wc3, mode) - f_c(mean, Wc1, Wc2, Wc3, mode)
    return F.fp32(z) if mode == "operand" else z


# --------------------------------------------------------------------------
# Per-token group quantisation (section 2.4, Delta / q / z-tilde equations)
# --------------------------------------------------------------------------
def _groups(d_c: int, g: int):
    return [(s, min(s + g, d_c)) for s in range(0, d_c, g)]


def quantize(z, bits: int, g: int = 32, mode: str = "operand"):
    """Asymmetric min-max quantisation of each token's code in groups of g.

    ``z`` is [n, d_c].  Returns (q, meta, overflow): q [n, d_c] integer codes
    (for bits == 16, the bf16 value of z instead), meta [n, G, 2] the FP16
    (min, max) of each group, overflow a bool [n] (an extreme saturated FP16).

    For a non-constant group the extremes are rounded outward to FP16 so the
    stored range covers the group; Delta = (max - min) / (2^b - 1) and
    q = round-half-even((z - min) / Delta), clamped to [0, 2^b - 1].
    A constant group (min == max) stores its value as both extremes, q = 0,
    and no division happens.  In operand mode the subtraction and the two
    divisions are binary32 operations, as in the kernel.
    """
    z = np.atleast_2d(np.asarray(z, dtype=np.float64))
    n, d_c = z.shape
    grp = _groups(d_c, g)
    meta = np.zeros((n, len(grp), 2), dtype=np.float64)
    overflow = np.zeros(n, dtype=bool)
    if bits == 16:
        return F.bf16(z), meta, overflow
    levels = 2 ** bits - 1
    q = np.zeros((n, d_c), dtype=np.int64)
    for gi, (a, b) in enumerate(grp):
        zg = z[:, a:b]
        zmin = zg.min(axis=1)
        zmax = zg.max(axis=1)
        const = zmin == zmax
        lo = np.where(const, F.fp16_rn(zmin), F.fp16_rd(zmin))
        hi = np.where(const, F.fp16_rn(zmax), F.fp16_ru(zmax))
        overflow |= (np.abs(zmin) > F.FP16_MAX) | (np.abs(zmax) > F.FP16_MAX)
        meta[:, gi, 0] = lo
        meta[:, gi, 1] = hi
        if mode == "operand":
            lo32 = lo.astype(np.float32)[:, None]
            hi32 = hi.astype(np.float32)[:, None]
            delta = (hi32 - lo32) / np.float32(levels)
            with np.errstate(divide="ignore", invalid="ignore"):
                u = (zg.astype(np.float32) - lo32) / delta
            u = u.astype(np.float64)
        else:
            delta = (hi - lo)[:, None] / levels
            with np.errstate(divide="ignore", invalid="ignore"):
                u = (zg - lo[:, None]) / delta
        with np.errstate(invalid="ignore"):
            qg = np.clip(np.rint(u), 0, levels)
        # constant group, or both extremes saturated to the same FP16 value
        qg = np.where(const[:, None] | (hi == lo)[:, None], 0, qg)
        q[:, a:b] = qg.astype(np.int64)
    return q, meta, overflow


def dequantize(q, meta, bits: int, g: int = 32, mode: str = "operand"):
    """z-tilde = q * Delta + min per group (binary32 products and sums in
    operand mode); for bits == 16 the stored bf16 values are returned."""
    q = np.atleast_2d(np.asarray(q))
    if bits == 16:
        return np.asarray(q, dtype=np.float64)
    n, d_c = q.shape
    levels = 2 ** bits - 1
    out = np.zeros((n, d_c), dtype=np.float64)
    for gi, (a, b) in enumerate(_groups(d_c, g)):
        lo = meta[:, gi, 0]
        hi = meta[:, gi, 1]
        if mode == "operand":
            lo32 = lo.astype(np.float32)[:, None]
            delta = (hi.astype(np.float32)[:, None] - lo32) / np.float32(levels)
            t = q[:, a:b].astype(np.float32) * delta
            out[:, a:b] = (t + lo32).astype(np.float64)
        else:
            delta = (hi - lo)[:, None] / levels
            out[:, a:b] = q[:, a:b] * delta + lo[:, None]
    return out


def pack_codes(q, bits: int) -> np.ndarray:
    """Byte layout of a token's code.

    INT4: element 2t in the low nibble of byte t, 2t+1 in the high nibble.
    INT2: element 4t+u in bits [2u, 2u+2) of byte t.
    bits == 16: the bf16 bit patterns, little-endian.
    """
    q = np.atleast_2d(np.asarray(q))
    n, d_c = q.shape
    if bits == 16:
        return F.bf16_bits(q).view(np.uint8).reshape(n, 2 * d_c)
    per = 8 // bits
    pad = (-d_c) % per
    qq = np.concatenate([q.astype(np.int64), np.zeros((n, pad), np.int64)], axis=1)
    qq = qq.reshape(n, -1, per)
    out = np.zeros(qq.shape[:2], dtype=np.int64)
    for u in range(per):
        out |= qq[:, :, u] << (bits * u)
    return out.astype(np.uint8)


def unpack_codes(packed, bits: int, d_c: int) -> np.ndarray:
    packed = np.atleast_2d(np.asarray(packed, dtype=np.uint8))
    n = packed.shape[0]
    if bits == 16:
        u16 = packed.reshape(n, -1).view(np.uint16).astype(np.uint32) << 16
        return u16.view(np.float32).astype(np.float64)
    per = 8 // bits
    mask = (1 << bits) - 1
    p = packed.astype(np.int64)
    parts = [(p >> (bits * u)) & mask for u in range(per)]
    return np.stack(parts, axis=2).reshape(n, -1)[:, :d_c]


# --------------------------------------------------------------------------
# Linear decoder, K/V split, RoPE (sections 2.1 and 2.5)
# --------------------------------------------------------------------------
def decode(z_tilde, Wd, mean, mode: str = "operand"):
    """KV_hat = z-tilde W_d + mean (boxed eq., 2.5).  No bias."""
    zt = F.bf16(z_tilde) if mode == "operand" else np.asarray(z_tilde, np.float64)
    return zt @ Wd + mean


def split_kv(kv_hat, n_kv_heads: int, head_dim: int):
    """K is the first N*D columns, V the rest, each laid out [head][dim]."""
    kv_hat = np.asarray(kv_hat)
    d_k = n_kv_heads * head_dim
    lead = kv_hat.shape[:-1]
    K = kv_hat[..., :d_k].reshape(*lead, n_kv_heads, head_dim)
    V = kv_hat[..., d_k:].reshape(*lead, n_kv_heads, head_dim)
    return K, V


def rope_angles(pos, head_dim: int, base: float):
    """pos * theta_j with theta_j = base^(-2j/D), j < D/2, in float64."""
    j = np.arange(head_dim // 2, dtype=np.float64)
    theta = np.power(float(base), -2.0 * j / head_dim)
    return np.asarray(pos, dtype=np.float64)[..., None] * theta


def rope(K, pos, base: float):
    """Rotate-half RoPE of K [..., N, D] at positions ``pos`` [...].

    Pairs (d, d + D/2): x' = x cos a - y sin a, y' = y cos a + x sin a.
    """
    K = np.asarray(K, dtype=np.float64)
    D = K.shape[-1]
    ang = rope_angles(pos, D, base)[..., None, :]      # [..., 1, D/2]
    c, s = np.cos(ang), np.sin(ang)
    x, y = K[..., : D // 2], K[..., D // 2:]
    return np.concatenate([x * c - y * s, y * c + x * s], axis=-1)


# --------------------------------------------------------------------------
# Whole-sequence helpers built from the steps above
# --------------------------------------------------------------------------
@dataclass
class Pool:
    codes: np.ndarray      # [R, d_kv] uint8 (E4M3)
    vals: np.ndarray       # [R, d_kv] decoded values
    norm2: np.ndarray      # [R] binary32 squared norms
    pos: np.ndarray        # [R] token positions


def build_pool(kv, T: int, stride: int, alpha: float = 0.0, sink: int = 0) -> Pool:
    rp = reference_positions(T, stride, alpha, sink)
    codes, vals, norm2 = store_references(np.asarray(kv, np.float64)[rp])
    return Pool(codes, vals, norm2, rp)


def encode_token(kv_i, pos: int, pool: Pool, W, shape: Shape, mode: str = "operand"):
    """Write path of one non-reference token.

    Returns a dict with the retrieved slots (padded with -1 to k), their
    distances, the mean, z, the integer codes and the FP16 extremes.
    """
    slots, dist = retrieve(kv_i, pool.vals, pool.pos, pos, shape.topk)
    m = reference_mean(pool.vals, slots, mode)
    z = residual_code(np.asarray(kv_i, np.float64)[None, :], m[None, :], W, mode)
    q, meta, ovf = quantize(z, shape.bits, shape.group, mode)
    idx = np.full(shape.topk, -1, dtype=np.int64)
    idx[: len(slots)] = slots
    return {"idx": idx, "dist": dist, "mean": m, "z": z[0], "q": q[0],
            "meta": meta[0], "overflow": bool(ovf[0])}


def encode_tokens(kv, positions, pool: Pool, W, shape: Shape, mode: str = "operand",
                  mean_from: str = "row"):
    """encode_token over many tokens, batching the f_c products.

    mean_from="row" maps the mean row itself (f_c(mean), as written in section 2.3);
    "refs" takes the mean's hidden row from the references' pre-activations
    (``mean_hidden_from_refs``), the same value in exact arithmetic, rounded
    differently: the mean is then never rounded to a tensor-core operand.
    """
    if mean_from not in ("row", "refs"):
        raise ValueError("mean_from must be 'row' or 'refs'")
    kv = np.asarray(kv, np.float64)
    positions = np.asarray(positions, dtype=np.int64)
    n = len(positions)
    idx = np.full((n, shape.topk), -1, dtype=np.int64)
    dist = np.full((n, shape.topk), np.nan)
    means = np.zeros((n, shape.d_kv))
    h_mean = np.zeros((n, shape.d_ff)) if mean_from == "refs" else None
    for r, p in enumerate(positions):
        slots, d = retrieve(kv[r], pool.vals, pool.pos, int(p), shape.topk)
        idx[r, : len(slots)] = slots
        dist[r, : len(slots)] = d
        means[r] = reference_mean(pool.vals, slots, mode)
        if h_mean is not None:
            h_mean[r] = mean_hidden_from_refs(pool.vals, slots, W["Wc1"], W["Wc2"])
    if not n:
        z = np.zeros((0, shape.d_c))
    elif h_mean is None:
        z = residual_code(kv, means, W, mode)
    else:
        x = F.bf16(kv) if mode == "operand" else kv
        z = (swiglu_hidden(x, W["Wc1"], W["Wc2"], mode) - h_mean) @ W["Wc3"]
        z = F.fp32(z) if mode == "operand" else z
    q, meta, ovf = quantize(z, shape.bits, shape.group, mode)
    return {"idx": idx, "dist": dist, "mean": means, "z": z, "q": q,
            "meta": meta, "overflow": ovf}


@dataclass
class Store:
    """Everything the cache keeps for one sequence."""

    shape: Shape
    pool: Pool
    idx: np.ndarray        # [T, k] slots, -1 padded; a reference has [slot,-1,..]
    q: np.ndarray          # [T, d_c] integer codes (bf16 values if bits == 16)
    meta: np.ndarray       # [T, G, 2] FP16 extremes
    z: np.ndarray          # [T, d_c] code before quantisation (0 for references)
    dist: np.ndarray       # [T, k] retrieval distances (nan for references)

    @property
    def packed(self) -> np.ndarray:
        return pack_codes(self.q, self.shape.bits)


def compress_sequence(kv, W, shape: Shape, mode: str = "operand",
                      mean_from: str = "row") -> Store:
    """Write all T tokens: references go to the pool, the rest are encoded.

    A reference's own row gets idx [slot, -1, ...] and an all-zero code with
    zero extremes, so that reading it back yields the stored reference.
    """
    kv = np.asarray(kv, np.float64)
    T = kv.shape[0]
    pool = build_pool(kv, T, shape.stride, shape.ref_alpha, shape.ref_sink)
    idx = np.full((T, shape.topk), -1, dtype=np.int64)
    q = np.zeros((T, shape.d_c))
    meta = np.zeros((T, shape.n_groups, 2))
    z = np.zeros((T, shape.d_c))
    dist = np.full((T, shape.topk), np.nan)
    idx[pool.pos, 0] = np.arange(len(pool.pos))
    nonref = np.nonzero(~is_reference(np.arange(T), shape.stride, shape.ref_alpha,
                                      shape.ref_sink))[0]
    enc = encode_tokens(kv[nonref], nonref, pool, W, shape, mode, mean_from)
    idx[nonref] = enc["idx"]
    q[nonref] = enc["q"]
    meta[nonref] = enc["meta"]
    z[nonref] = enc["z"]
    dist[nonref] = enc["dist"]
    return Store(shape, pool, idx, q, meta, z, dist)


def reconstruct(store: Store, positions, W, mode: str = "operand"):
    """Read path for the selected positions: returns K, V [n, N, D] and the
    pre-RoPE KV_hat [n, d_kv]."""
    sh = store.shape
    positions = np.asarray(positions, dtype=np.int64)
    zt = dequantize(store.q[positions], store.meta[positions], sh.bits, sh.group, mode)
    means = np.stack([
        reference_mean(store.pool.vals, store.idx[p][store.idx[p] >= 0], mode)
        for p in positions
    ]) if len(positions) else np.zeros((0, sh.d_kv))
    kv_hat = decode(zt, W["Wd"], means, mode)
    K, V = split_kv(kv_hat, sh.n_kv_heads, sh.head_dim)
    K = rope(K, positions, sh.rope_base)
    return K, V, kv_hat


# --------------------------------------------------------------------------
# Section 2.8: Theorem IV.1 and the quantisation error bound
# --------------------------------------------------------------------------
def theorem_iv1_terms(kv_i, pool_vals, slots):
    """(rho^2, ||Delta||^2, V) of Theorem IV.1 for one token, in float64."""
    R = pool_vals[np.asarray(slots)]
    m = R.mean(axis=0)
    rho2 = np.mean(np.sum((kv_i[None, :] - R) ** 2, axis=1))
    delta2 = np.sum((kv_i - m) ** 2)
    V = np.mean(np.sum((R - m[None, :]) ** 2, axis=1))
    return rho2, delta2, V


def quant_error_bounds(z, bits: int, g: int = 32):
    """The two right-hand sides of the quantisation error bound (2.8):
    sqrt(sum_G |G| range_G^2) / (2(2^b-1)) and sqrt(g/2)/(2^b-1) * ||z||."""
    z = np.asarray(z, np.float64)
    s = 0.0
    for a, b in _groups(len(z), g):
        s += (b - a) * (z[a:b].max() - z[a:b].min()) ** 2
    levels = 2 ** bits - 1
    return np.sqrt(s) / (2 * levels), np.sqrt(g / 2) / levels * np.linalg.norm(z)
