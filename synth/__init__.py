"""Seeded synthetic inputs shared by the CPU oracle and the CUDA library tests.

This module holds none of the codec's arithmetic: it only draws random
numbers (torch CPU generator, so every machine gets the same values) and
names the workloads.  The oracle and the GPU path both consume what it
returns; neither imports the other.

Workloads (the synthetic stand-ins for the page's model KV caches):

* ``tiny``      one fp32 layer: T=256, N=2, D=64 (2d_k=256), d_c=64, d_ff=128,
                stride 8, INT4, 16 centroids, noise 0.3, RoPE base 1e4.
* ``llama8b``   one Llama-3.1-8B-shaped layer: N=8, D=128 (2d_k=2048),
                d_c=512, d_ff=1536, T=32768, stride 16, INT4, bf16 kv from a
                64-centroid mixture with noise 0.25 scaled to unit RMS,
                RoPE base 5e5; 64 decode steps reading 30 % each.
* ``qwen7b``    Qwen2.5-7B-shaped stack: 28 layers, N=4, D=128 (2d_k=1024),
                d_c=256, d_ff=768, T=131072, stride 16, INT4, 256 centroids,
                selection in contiguous 64-token blocks, RoPE base 1e6.
* ``batched``   Llama layer shape, B=16 sequences x T=16384, one new token per
                sequence per step, 30 % of each history read per step.
* ``long_int2`` Llama layer shape, T=262144, INT2; ``long_bf16z`` the same
                distribution at T=65536 with quantisation off (bf16 z).
* ``t1_*``      the codec shapes of Table I (section 3.1): Qwen2.5-7B (2d_k=1024,
                d_c=384, d_ff=3072), Qwen3-VL-8B (2048, 384, 3072), Qwen2.5-32B
                (2048, 512, 4096); llama8b's input distribution, T=8192.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, replace

import torch

__all__ = ["Workload", "WORKLOADS", "workload", "gen_kv", "gen_weights",
           "gen_selection", "gen_block_selection"]


@dataclass(frozen=True)
class Workload:
    name: str
    n_kv_heads: int
    head_dim: int
    d_c: int
    d_ff: int
    T: int
    stride: int
    bits: int
    kv_dtype: str            # "fp32" | "bf16"
    out_dtype: str           # "fp32" | "bf16"
    n_centroids: int
    noise: float
    unit_rms: bool
    rope_base: float
    topk: int = 4
    group: int = 32
    batch: int = 1
    layers: int = 1
    steps: int = 64
    sel_frac: float = 0.3
    sel_block: int = 1       # 1 = random positions, 64 = contiguous blocks

    @property
    def d_kv(self) -> int:
        return 2 * self.n_kv_heads * self.head_dim

    @property
    def n_sel(self) -> int:
        return int(round(self.sel_frac * self.T))


WORKLOADS = {
    "tiny": Workload("tiny", 2, 64, 64, 128, 256, 8, 4, "fp32", "fp32", 16, 0.3,
                     False, 1e4),
    "llama8b": Workload("llama8b", 8, 128, 512, 1536, 32768, 16, 4, "bf16", "bf16",
                        64, 0.25, True, 5e5),
    "qwen7b": Workload("qwen7b", 4, 128, 256, 768, 131072, 16, 4, "bf16", "bf16",
                       256, 0.25, True, 1e6, layers=28, sel_block=64),
    "batched": Workload("batched", 8, 128, 512, 1536, 16384, 16, 4, "bf16", "bf16",
                        64, 0.25, True, 5e5, batch=16),
    "long_int2": Workload("long_int2", 8, 128, 512, 1536, 262144, 16, 2, "bf16",
                          "bf16", 64, 0.25, True, 5e5, steps=16),
    "long_bf16z": Workload("long_bf16z", 8, 128, 512, 1536, 65536, 16, 16, "bf16",
                           "bf16", 64, 0.25, True, 5e5, steps=16),
    # the codec shapes of the page's Table I (2d_k, d_c, d_ff), with the llama8b
    # input distribution
    "t1_qwen25_7b": Workload("t1_qwen25_7b", 4, 128, 384, 3072, 8192, 16, 4, "bf16", "bf16",
                             64, 0.25, True, 1e6),
    "t1_qwen3vl_8b": Workload("t1_qwen3vl_8b", 8, 128, 384, 3072, 8192, 16, 4, "bf16", "bf16",
                              64, 0.25, True, 5e6),
    "t1_qwen25_32b": Workload("t1_qwen25_32b", 8, 128, 512, 4096, 8192, 16, 4, "bf16", "bf16",
                              64, 0.25, True, 1e6),
}


def workload(name: str, **overrides) -> Workload:
    return replace(WORKLOADS[name], **overrides)


def _gen(seed: int) -> torch.Generator:
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    return g


def gen_kv(w: Workload, seed: int, T: int | None = None, device: str = "cpu") -> torch.Tensor:
    """[T, 2d_k] pre-RoPE joint K/V rows: centroid[c_i] + noise * N(0, 1).

    Centroids ~ N(0, 1), c_i uniform.  For the Llama/Qwen-shaped workloads the
    whole tensor is then scaled to unit RMS.  Returned in the workload's kv dtype.
    On the CPU (the default) every machine draws the same values; with a CUDA
    `device` the draws come from that device's generator, seeded the same way: the
    same distribution, other values (for timing runs of full-size stacks, where
    drawing gigabytes on the host would take minutes).
    """
    T = w.T if T is None else T
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    cent = torch.randn(w.n_centroids, w.d_kv, generator=g, dtype=torch.float32, device=device)
    c = torch.randint(0, w.n_centroids, (T,), generator=g, device=device)
    kv = cent[c] + w.noise * torch.randn(T, w.d_kv, generator=g, dtype=torch.float32, device=device)
    if w.unit_rms:
        kv = kv / kv.pow(2).mean().sqrt()
    return kv.to(torch.float32 if w.kv_dtype == "fp32" else torch.bfloat16)


def _xavier(rows: int, cols: int, g: torch.Generator) -> torch.Tensor:
    std = math.sqrt(2.0 / (rows + cols))
    return (std * torch.randn(rows, cols, generator=g, dtype=torch.float32)).to(torch.bfloat16)


def gen_weights(w: Workload, seed: int) -> dict:
    """Codec weights, Xavier-normal, stored in bf16, in the page's shapes:
    W_c1, W_c2 [2d_k, d_ff]; W_c3 [d_ff, d_c]; W_d [d_c, 2d_k]."""
    g = _gen(seed)
    return {
        "Wc1": _xavier(w.d_kv, w.d_ff, g),
        "Wc2": _xavier(w.d_kv, w.d_ff, g),
        "Wc3": _xavier(w.d_ff, w.d_c, g),
        "Wd": _xavier(w.d_c, w.d_kv, g),
    }


def gen_selection(T: int, n: int, seed: int) -> torch.Tensor:
    """n distinct positions of [0, T), sorted (int32)."""
    g = _gen(seed)
    return torch.randperm(T, generator=g)[:n].sort().values.to(torch.int32)


def gen_block_selection(T: int, block: int, frac: float, seed: int) -> torch.Tensor:
    """Positions of round(frac * T/block) random contiguous blocks, sorted."""
    g = _gen(seed)
    nb = T // block
    pick = torch.randperm(nb, generator=g)[: int(round(frac * nb))].sort().values
    pos = (pick[:, None] * block + torch.arange(block)[None, :]).reshape(-1)
    return pos.to(torch.int32)
