"""Storage accounting of the ResidualKV cache (ResidualKV notes, section 3.3).

TEST INFRASTRUCTURE: imported only by tests, the smoke check and the bench's
CPU baseline.

The page defines the keep ratio KR as the GPU KV storage relative to a full
FP16 KV cache, with q_b = b/16 + 2/32 the relative size of b-bit codes stored
with two FP16 extremes per 32 values, and
    KR = beta*q_4 + (1 - beta) * (rho_ref/2 + q_b * d_c / (2 d_k)),
where beta is the fraction of full-attention layers and rho_ref the
reference density (references kept in FP8, i.e. half an FP16 entry).
"""
from __future__ import annotations

__all__ = ["q_b", "keep_ratio", "compute_ratio", "layer_bytes"]


def q_b(bits: int, group: int = 32) -> float:
    """Relative size of b-bit group codes with two FP16 extremes per group."""
    if bits == 16:
        return 1.0
    return bits / 16.0 + 2.0 / group


def keep_ratio(beta: float, rho_ref: float, bits: int, dc_over_2dk: float,
               full_layer_bits: int = 4, group: int = 32) -> float:
    """KR of the page (section 3.3, KR formula)."""
    return beta * q_b(full_layer_bits, group) + (1.0 - beta) * (
        0.5 * rho_ref + q_b(bits, group) * dc_over_2dk)


def compute_ratio(beta: float, r: float) -> float:
    """CR = beta + (1 - beta) r (section 3.3)."""
    return beta + (1.0 - beta) * r


def layer_bytes(T: int, stride: int, d_kv: int, d_c: int, bits: int,
                group: int = 32, topk: int = 4, with_index: bool = True) -> dict:
    """Bytes one codec layer keeps for T tokens, against FP16 K/V.

    References: d_kv FP8 bytes each.  Every token (reference or not) has a
    code row and its extremes, which matches the page's formula charging q_b
    on all tokens of a sparse layer.  ``with_index`` adds the k int32 slots
    per token that the page's formula does not count.
    """
    n_ref = -(-T // stride)
    ref = n_ref * d_kv
    code_row = 2 * d_c if bits == 16 else -(-d_c * bits // 8)
    meta_row = 0 if bits == 16 else 4 * (-(-d_c // group))
    codes = T * (code_row + meta_row)
    idx = T * 4 * topk if with_index else 0
    fp16 = T * d_kv * 2
    total = ref + codes + idx
    return {"refs": ref, "codes": codes, "index": idx, "total": total,
            "fp16": fp16, "fraction": total / fp16}
