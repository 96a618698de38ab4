"""The restore's two set-up paths agree bit for bit.  A selection restored in one call
has CTAs that cross token tiles: their later tiles are set up from records, extremes and
codes that the loader warps staged in shared memory, with z~ in alternating TMEM buffers
when d_c <= 256.  The same rows restored in calls of at most 128 tokens have every CTA
on a single tile, set up from global memory.  Every row is computed with the same
arithmetic either way (ResidualKV notes §2.4 dequantisation, §2.5 decode and mean, §2.1
RoPE at the token's position), so the outputs must be identical; covered for INT4, INT2
and bf16 z, bf16 and fp32 outputs, staged codes (rows of at most 128 bytes) and codes
read from global memory."""
import numpy as np
import pytest
import torch

import synth

from _common import gpu_prefill, make_codec

pytestmark = pytest.mark.gpu
cuda = pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA GPU")


@cuda
@pytest.mark.parametrize("name,T,bits,out", [
    ("tiny", 32768, 4, "bf16"),      # d_c = 64: 32-byte code rows, staged
    ("tiny", 32768, 2, "fp32"),      # 16-byte code rows, staged
    ("tiny", 32768, 16, "bf16"),     # bf16 z, 128-byte rows, staged
    ("llama8b", 16384, 4, "bf16"),   # 256-byte rows, read from global memory; one z~ buffer
    ("llama8b", 16384, 16, "fp32"),  # bf16 z, 1 KB rows
])
def test_restore_staged_tiles_equal_single_tile_calls(name, T, bits, out):
    w = synth.workload(name)
    kv = synth.gen_kv(w, 901, T=T).cuda()
    c = make_codec(w, synth.gen_weights(w, 902), T=T, bits=bits, out_dtype=out)
    gpu_prefill(c, kv, w.stride)
    torch.cuda.synchronize()
    assert c.get_status() == 0
    n = T - 1000                                    # a ragged last tile
    sel = synth.gen_selection(T, n, 903).cuda()
    zero = torch.zeros(n, dtype=torch.int32, device="cuda")
    K1, V1 = c.reconstruct(zero, sel)
    K2, V2 = torch.full_like(K1, float("nan")), torch.full_like(V1, float("nan"))
    for i in range(0, n, 128):
        j = min(n, i + 128)
        c.reconstruct(zero[i:j], sel[i:j], K2[i:j], V2[i:j])
    torch.cuda.synchronize()
    assert c.get_status() == 0
    units = ((n + 127) // 128) * (w.d_kv // 128)
    assert units > 2 * torch.cuda.get_device_properties(0).multi_processor_count
    assert torch.equal(K1, K2) and torch.equal(V1, V2)
    assert torch.isfinite(K1.float()).all() and torch.isfinite(V1.float()).all()
