"""One launch restoring several contexts' selections (rkv_reconstruct_multi): the same
computation as one rkv_reconstruct per context (ResidualKV notes §2.5 decode and mean,
§2.1 RoPE at the token's own position, §2.7 only the selected tokens), so the outputs
must be identical bit for bit.  The token tiles of all problems are numbered one after
the other and dealt to the CTAs in a stride (CTA b takes tiles b, b + G, ...), so a CTA
works on several problems (it switches storage, pool and W_d between two tiles, and
prefetches the next tile's W_d while the current one runs); covered with INT4 code rows read from global
memory (Llama shape, one z~ buffer) and staged (Qwen shape, two z~ buffers), fp32
outputs (the tiny shape), empty and one-token problems, two sequences per context."""
import numpy as np
import pytest
import torch

import residual_kv_cache_gb300 as rkv
import synth

from _common import gpu_prefill, make_codec

pytestmark = pytest.mark.gpu
cuda = pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA GPU")


def _layers(name, L, T, seed, batch=1):
    """L contexts of one shape, each with its own weights and kv rows, prefilled."""
    w = synth.workload(name)
    cs = []
    for l in range(L):
        c = make_codec(w, synth.gen_weights(w, seed + 10 * l), T=T, batch=batch)
        for s in range(batch):
            gpu_prefill(c, synth.gen_kv(w, seed + 10 * l + 1 + s, T=T).cuda(), w.stride, seq_id=s)
        cs.append(c)
    torch.cuda.synchronize()
    assert all(c.get_status() == 0 for c in cs)
    return w, cs


def _check_equal(cs, seqs, poss):
    K1, V1 = rkv.reconstruct_multi(cs, seqs, poss)
    singles = [c.reconstruct(s, p) for c, s, p in zip(cs, seqs, poss)]
    torch.cuda.synchronize()
    for c in cs:
        assert c.get_status() == 0
    for (k1, v1), (k2, v2) in zip(zip(K1, V1), singles):
        assert torch.equal(k1, k2) and torch.equal(v1, v2)


@cuda
@pytest.mark.parametrize("name,T,sizes", [
    ("llama8b", 4096, [3000, 0, 1, 2900, 128, 1000]),
    ("qwen7b", 4096, [4000, 257, 3333]),
    ("tiny", 256, [200, 77, 256, 1]),
])
def test_multi_equals_single_restores(name, T, sizes):
    w, cs = _layers(name, len(sizes), T, 1500)
    g = torch.Generator().manual_seed(1501)
    poss = [torch.randint(0, T, (n,), generator=g, dtype=torch.int32).cuda() for n in sizes]
    seqs = [torch.zeros_like(p) for p in poss]
    tiles = sum((n + 127) // 128 for n in sizes) * (w.d_kv // 128)
    assert tiles > torch.cuda.get_device_properties(0).multi_processor_count or name == "tiny"
    _check_equal(cs, seqs, poss)


@cuda
def test_multi_two_sequences_per_context():
    w, cs = _layers("llama8b", 3, 1024, 1510, batch=2)
    g = torch.Generator().manual_seed(1511)
    seqs = [torch.randint(0, 2, (700,), generator=g, dtype=torch.int32).cuda() for _ in cs]
    poss = [torch.randint(0, 1024, (700,), generator=g, dtype=torch.int32).cuda() for _ in cs]
    _check_equal(cs, seqs, poss)


@cuda
def test_multi_flags_the_context_of_a_bad_selection():
    w, cs = _layers("llama8b", 3, 1024, 1520)
    poss = [torch.arange(300, dtype=torch.int32).cuda() for _ in cs]
    poss[1][17] = 5000                                # past max_tokens in problem 1 only
    seqs = [torch.zeros_like(p) for p in poss]
    K, V = rkv.reconstruct_multi(cs, seqs, poss)
    torch.cuda.synchronize()
    flags = [c.get_status() for c in cs]
    assert flags[0] == 0 and flags[2] == 0 and flags[1] & rkv.FLAG_BAD_INDEX
    assert torch.count_nonzero(K[1][17]) == 0 and torch.count_nonzero(V[1][17]) == 0


@cuda
def test_multi_rejects_mismatched_contexts():
    w, cs = _layers("llama8b", 2, 1024, 1530)
    t = make_codec(w, synth.gen_weights(w, 1533), T=2048)        # another max_tokens
    p = torch.arange(10, dtype=torch.int32).cuda()
    z = torch.zeros_like(p)
    with pytest.raises(rkv.RkvError):
        rkv.reconstruct_multi([cs[0], t], [z, z], [p, p])
    with pytest.raises(ValueError):
        rkv.reconstruct_multi([], [], [])
    with pytest.raises(rkv.RkvError):
        rkv.reconstruct_multi([cs[0]] * 33, [z] * 33, [p] * 33)
