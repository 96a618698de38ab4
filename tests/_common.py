"""Shared helpers of the GPU parity tests: run a workload through the CUDA library and
through the oracle on the same seeded inputs, and compare what is unique."""
from __future__ import annotations

import numpy as np
import torch

import synth
from oracle import codec as C
from oracle import formats as F


def oracle_shape(w: synth.Workload) -> C.Shape:
    return C.Shape(w.n_kv_heads, w.head_dim, w.d_c, w.d_ff, w.topk, w.group, w.bits, w.stride,
                   w.rope_base)


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
               out_dtype: str | None = None, bits: int | None = None):
    from residual_kv_cache_gb300 import Codec, Config
    cfg = Config(n_kv_heads=w.n_kv_heads, head_dim=w.head_dim, d_c=w.d_c, d_ff=w.d_ff,
                 topk=w.topk, group=w.group, bits=w.bits if bits is None else bits,
                 ref_stride=w.stride, kv_dtype=w.kv_dtype,
                 out_dtype=out_dtype or w.out_dtype, rope_base=w.rope_base, batch=batch,
                 max_tokens=T, max_rows=max_rows)
    Wd = {k: v.cuda().contiguous() for k, v in W.items()}
    return Codec(cfg, Wd)


def gpu_prefill(codec, kv_dev: torch.Tensor, stride: int, seq_id: int = 0):
    """Write every position of one sequence: references to the pool, the rest encoded."""
    T = kv_dev.shape[0]
    pos = np.arange(T, dtype=np.int32)
    ref = pos[pos % stride == 0]
    non = pos[pos % stride != 0]
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


def code_parity(gq: np.ndarray, gmeta: np.ndarray, oq: np.ndarray, ometa: np.ndarray,
                oz: np.ndarray, bits: int, g: int = 32):
    """Returns (identical fraction, list of violations).  A differing code is allowed
    only as +-1 where the oracle's pre-round value is within 1e-3 of a .5 boundary;
    groups whose FP16 extremes differ are allowed only where the oracle's extreme lies
    within 1e-6 (relative) of an FP16 value boundary."""
    same = gq == oq
    frac = float(same.mean())
    viol = []
    meta_diff = np.any(gmeta != ometa, axis=2)             # [n, G]
    for r, gi in zip(*np.nonzero(meta_diff)):
        zg = oz[r, gi * g:(gi + 1) * g]
        for e, val in ((0, zg.min()), (1, zg.max())):
            if gmeta[r, gi, e] == ometa[r, gi, e]:
                continue
            near = F.fp16_rn(val)
            if abs(val - near) > 1e-6 * max(abs(val), 1e-30):
                viol.append(("meta", int(r), int(gi), e))
    u = preround(oz, ometa, bits, g)
    diff = np.nonzero(~same)
    for r, c in zip(*diff):
        if meta_diff[r, c // g]:
            continue
        d = abs(int(gq[r, c]) - int(oq[r, c]))
        fr = u[r, c] - np.floor(u[r, c])
        if d != 1 or abs(fr - 0.5) >= 1e-3:
            viol.append(("code", int(r), int(c), int(gq[r, c]), int(oq[r, c]), float(u[r, c])))
    return frac, viol


def rel_fro(a: np.ndarray, b: np.ndarray) -> float:
    return float(np.linalg.norm((a - b).ravel()) / max(np.linalg.norm(b.ravel()), 1e-300))
