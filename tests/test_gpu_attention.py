"""GPU parity of the sparse-layer attention (ResidualKV notes section 2.7) against the
oracle.

Tolerances:
* on the same K/V rows (the library's own restore outputs, or seeded random rows):
  relative Frobenius error <= 1e-5.  The kernel works in fp32: a score is a
  128-term dot product (relative error ~1e-6), exp and the chunk merge add a few
  ulps, and the output is a convex combination of V rows;
* end to end against the oracle's own restore: <= 1e-2, the restore's tolerance,
  since attention is a smooth function of K and V.
"""
import numpy as np
import pytest
import torch

import synth
from oracle import attention as A
from oracle import codec as C

from _common import gpu_prefill, make_codec, np64, oracle_shape, rel_fro

pytestmark = pytest.mark.gpu
cuda = pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA GPU")


def _weights64(W):
    return {k: np64(v) for k, v in W.items()}


@pytest.fixture(scope="module")
def llama_small():
    w = synth.workload("llama8b")
    T = 2048
    kv = synth.gen_kv(w, 61, T=T)
    W = synth.gen_weights(w, 62)
    c = make_codec(w, W, T=T)
    gpu_prefill(c, kv.cuda(), w.stride)
    torch.cuda.synchronize()
    assert c.get_status() == 0
    st = C.compress_sequence(np64(kv), _weights64(W), oracle_shape(w), "operand")
    return dict(w=w, T=T, codec=c, store=st, W64=_weights64(W))


def _q(Hq, D, seed):
    g = torch.Generator().manual_seed(seed)
    return torch.randn(Hq, D, generator=g, dtype=torch.float32)


@cuda
@pytest.mark.parametrize("Hq", [8, 32, 64])
def test_attention_on_restored_rows(llama_small, Hq):
    """Query groups of 1, 4 and 8 heads over one restore's K/V (bf16 outputs)."""
    r = llama_small
    c, T = r["codec"], r["T"]
    sel = synth.gen_selection(T, int(round(0.3 * T)), 71)
    K, V = c.reconstruct(torch.zeros_like(sel).cuda(), sel.cuda())
    q = _q(Hq, r["w"].head_dim, 72 + Hq)
    out = c.sparse_attention(q.cuda(), K, V)
    torch.cuda.synchronize()
    ref = A.sparse_attention(q.double().numpy(), np64(K), np64(V))
    assert rel_fro(np64(out), ref) <= 1e-5


@cuda
def test_attention_end_to_end_against_the_oracle_restore(llama_small):
    r = llama_small
    c, st, T = r["codec"], r["store"], r["T"]
    sel = synth.gen_selection(T, int(round(0.3 * T)), 73).numpy()
    # tokens whose retrieval is a validated near-tie swap have no unique oracle answer
    same = np.all(c.ref_idx[0].cpu().numpy()[sel] == st.idx[sel], axis=1)
    sel = sel[same]
    K, V = c.reconstruct(torch.zeros(len(sel), dtype=torch.int32).cuda(),
                         torch.from_numpy(sel.astype(np.int32)).cuda())
    q = _q(32, 128, 74)
    out = c.sparse_attention(q.cuda(), K, V)
    Ko, Vo, _ = C.reconstruct(st, sel.astype(np.int64), r["W64"], "operand")
    ref = A.sparse_attention(q.double().numpy(), Ko, Vo)
    assert rel_fro(np64(out), ref) <= 1e-2


@cuda
@pytest.mark.parametrize("n", [1, 127, 128, 129, 1000, 20000, 33000, 100000])
def test_attention_token_counts(llama_small, n):
    """Seeded random K/V rows: one token (o = v exactly), chunk edges, many chunks."""
    c = llama_small["codec"]
    g = torch.Generator().manual_seed(80 + n)
    K = torch.randn(n, 8, 128, generator=g).to(torch.bfloat16)
    V = torch.randn(n, 8, 128, generator=g).to(torch.bfloat16)
    q = _q(32, 128, 81 + n)
    out = c.sparse_attention(q.cuda(), K.cuda(), V.cuda())
    torch.cuda.synchronize()
    if n == 1:
        vv = np64(V)[0]                                   # [N, D]
        assert np.array_equal(np64(out), np.repeat(vv, 4, axis=0))
        return
    ref = A.sparse_attention(q.double().numpy(), np64(K), np64(V))
    assert rel_fro(np64(out), ref) <= 1e-5


@cuda
def test_attention_fp32_rows_and_small_heads():
    """fp32 restore outputs, D = 64, N = 2 (the tiny shape), 2 query heads per group."""
    w = synth.workload("tiny")
    T = w.T
    kv = synth.gen_kv(w, 91)
    W = synth.gen_weights(w, 92)
    c = make_codec(w, W, T=T)
    gpu_prefill(c, kv.cuda(), w.stride)
    sel = synth.gen_selection(T, 200, 93)
    K, V = c.reconstruct(torch.zeros_like(sel).cuda(), sel.cuda())
    assert K.dtype == torch.float32
    q = _q(4, 64, 94)
    out = c.sparse_attention(q.cuda(), K, V)
    torch.cuda.synchronize()
    assert c.get_status() == 0
    ref = A.sparse_attention(q.double().numpy(), np64(K), np64(V))
    assert rel_fro(np64(out), ref) <= 1e-5


@cuda
def test_attention_rejects_bad_arguments(llama_small):
    import residual_kv_cache_gb300 as rkv
    c = llama_small["codec"]
    K = torch.zeros(10, 8, 128, dtype=torch.bfloat16, device="cuda")
    for Hq in (4, 12, 72):                                # not a multiple of N, or > 8 N
        with pytest.raises(rkv.RkvError) as e:
            c.sparse_attention(torch.zeros(Hq, 128, device="cuda"), K, K)
        assert e.value.status == -1
    with pytest.raises(rkv.RkvError):
        c.sparse_attention(torch.zeros(8, 128, device="cuda"), K[:0], K[:0])
    with pytest.raises(ValueError):
        c.sparse_attention(torch.zeros(8, 128, device="cuda"), K.float(), K)
