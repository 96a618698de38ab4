"""GPU parity of the restore fused into the sparse layer's attention (ResidualKV notes
section 2.7, Fig. 7 and the output equation o = softmax(q K_hat^T / sqrt(D)) V_hat over the
selected tokens) against the oracle.

The fused read hands the restored rows to the attention in bf16 (where a bf16 restore
stores them), so its oracle is ``attention.attend_restored``: the oracle's own restore,
rounded to bf16, then the float64 attention.  Tolerances (relative Frobenius error):
* storage written by the oracle: <= 2e-4.  The kernel's fp32 rows agree with the oracle's
  to ~1e-6 relative before rounding (the fp32 restore test bounds them by 1e-5), so their
  bf16 roundings differ only for the few elements that lie that close to a rounding
  boundary, by one bf16 unit (2^-8 relative); the attention carries such a flip into o
  scaled by the token's weight.  Everything else the kernel does stays near fp32: the
  query and the weights reach the tensor core as bf16 high + low parts (relative error
  below 2^-16), the products are exact, the sums fp32;
* the plain restore's own bf16 rows (the rows the fused kernel builds, bit for bit): <= 2e-5
  against the float64 attention over them, the unfused kernel's bound with room for the
  two splits and the tensor core's fp32 accumulation order;
* storage written by the library, end to end against the oracle's restore: <= 1e-2, the
  restore's tolerance (attention is a smooth function of K and V).
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

TOL_ORACLE = 2e-4
TOL_SAME_ROWS = 2e-5


def _weights64(W):
    return {k: np64(v) for k, v in W.items()}


def _q(Hq, D, seed, scale=1.0):
    g = torch.Generator().manual_seed(seed)
    return torch.randn(Hq, D, generator=g, dtype=torch.float32) * scale


def _oracle_store(name, T, seed):
    w = synth.workload(name)
    kv64 = np64(synth.gen_kv(w, seed, T=T))
    W = synth.gen_weights(w, seed + 1)
    W64 = _weights64(W)
    st = C.compress_sequence(kv64, W64, oracle_shape(w), "operand")
    c = make_codec(w, W, T=T, out_dtype="bf16")
    R = len(st.pool.pos)
    c.pool_fp8[0, :R] = torch.from_numpy(st.pool.codes).cuda()
    c.ref_idx[0] = torch.from_numpy(st.idx.astype(np.int32)).cuda()
    c.codes[0] = torch.from_numpy(st.packed).cuda()
    c.meta[0] = torch.from_numpy(st.meta.astype(np.float16)).cuda()
    return dict(w=w, T=T, W64=W64, st=st, codec=c)


@pytest.fixture(scope="module")
def llama_store():
    """Oracle-written storage of a 2048-token llama8b-shaped sequence (N = 8, d_c = 512:
    256-byte code rows read from global memory, one z~ buffer)."""
    return _oracle_store("llama8b", 2048, 1301)


@pytest.fixture(scope="module")
def qwen_store():
    """Oracle-written storage of a 2048-token qwen7b-shaped sequence (N = 4, d_c = 256:
    staged 128-byte code rows, two z~ buffers)."""
    return _oracle_store("qwen7b", 2048, 1311)


def _fused_vs_oracle(r, sel, Hq, seed, scale=1.0):
    c = r["codec"]
    sel_d = torch.from_numpy(sel.astype(np.int32)).cuda()
    zero = torch.zeros_like(sel_d)
    q = _q(Hq, 128, seed, scale)
    out = c.restore_attend(zero, sel_d, q.cuda())
    torch.cuda.synchronize()
    assert c.get_status() == 0
    Ko, Vo, _ = C.reconstruct(r["st"], sel.astype(np.int64), r["W64"], "operand")
    ref = A.attend_restored(q.double().numpy(), Ko, Vo)
    return np64(out), ref


@cuda
@pytest.mark.parametrize("n", [129, 700, 2048])
@pytest.mark.parametrize("Hq", [8, 32, 64])
def test_fused_llama_shape_against_the_oracle(llama_store, Hq, n):
    """Query groups of 1, 4 and 8 heads; a ragged tile, several tiles, every token."""
    r = llama_store
    sel = synth.gen_selection(r["T"], n, 1320 + n).numpy()
    got, ref = _fused_vs_oracle(r, sel, Hq, 1330 + Hq)
    err = rel_fro(got, ref)
    print(f"llama Hq={Hq} n={n}: rel err {err:.3e}")
    assert err <= TOL_ORACLE


@cuda
@pytest.mark.parametrize("n,scale", [(130, 1.0), (1500, 1.0), (2048, 4.0)])
def test_fused_qwen_shape_against_the_oracle(qwen_store, n, scale):
    """Seven query heads per key/value head (28 over 4), as in Qwen2.5-7B; a query scaled
    by 4 sharpens the softmax."""
    r = qwen_store
    sel = synth.gen_selection(r["T"], n, 1340 + n).numpy()
    got, ref = _fused_vs_oracle(r, sel, 28, 1350 + n, scale)
    err = rel_fro(got, ref)
    print(f"qwen n={n} scale={scale}: rel err {err:.3e}")
    assert err <= TOL_ORACLE


@cuda
def test_fused_one_token_returns_its_value_row(llama_store):
    """One selected token: every weight is exp(0) = 1, so o is the token's bf16 V_hat row
    (the plain restore's output) exactly, for every query head of its group."""
    r = llama_store
    c = r["codec"]
    for p in (0, 1, 17, 2047):
        pos = torch.tensor([p], dtype=torch.int32, device="cuda")
        zero = torch.zeros_like(pos)
        _, V = c.reconstruct(zero, pos)
        out = c.restore_attend(zero, pos, _q(32, 128, 1360 + p).cuda())
        torch.cuda.synchronize()
        assert torch.equal(out, V[0].float().repeat_interleave(4, dim=0)), p


@cuda
@pytest.mark.parametrize("name", ["llama8b", "qwen7b"])
def test_fused_on_the_plain_restore_rows(name):
    """Library-written storage of 32768 tokens, a selection of 30000: the fused output
    against the float64 attention over the plain restore's bf16 rows, and against the
    unfused kernel on those rows; many tiles per query head."""
    w = synth.workload(name)
    T = 32768
    kv = synth.gen_kv(w, 1370, T=T).cuda()
    c = make_codec(w, synth.gen_weights(w, 1371), T=T, out_dtype="bf16")
    gpu_prefill(c, kv, w.stride)
    torch.cuda.synchronize()
    assert c.get_status() == 0
    n = 30000
    sel = synth.gen_selection(T, n, 1372).cuda()
    zero = torch.zeros_like(sel)
    Hq = 7 * w.n_kv_heads if name == "qwen7b" else 4 * w.n_kv_heads
    q = _q(Hq, 128, 1373).cuda()
    out = c.restore_attend(zero, sel, q)
    K, V = c.reconstruct(zero, sel)
    unfused = c.sparse_attention(q, K, V)
    torch.cuda.synchronize()
    assert c.get_status() == 0
    ref = A.sparse_attention(q.double().cpu().numpy(), np64(K), np64(V))
    err = rel_fro(np64(out), ref)
    print(f"{name} same rows: rel err {err:.3e}, unfused {rel_fro(np64(unfused), ref):.3e}")
    assert err <= TOL_SAME_ROWS
    assert rel_fro(np64(out), np64(unfused)) <= 2 * TOL_SAME_ROWS


@cuda
def test_fused_end_to_end_against_the_oracle_restore():
    """Storage written by the library (retrieval, encoder, quantiser on the GPU) against
    the oracle's own write and restore: the restore's end-to-end tolerance."""
    w = synth.workload("llama8b")
    T = 2048
    kv = synth.gen_kv(w, 1380, T=T)
    W = synth.gen_weights(w, 1381)
    c = make_codec(w, W, T=T, out_dtype="bf16")
    gpu_prefill(c, kv.cuda(), w.stride)
    torch.cuda.synchronize()
    st = C.compress_sequence(np64(kv), _weights64(W), oracle_shape(w), "operand")
    sel = synth.gen_selection(T, 600, 1382).numpy()
    # tokens whose retrieval is a validated near-tie swap have no unique oracle answer
    same = np.all(c.ref_idx[0].cpu().numpy()[sel] == st.idx[sel], axis=1)
    sel = sel[same]
    q = _q(32, 128, 1383)
    out = c.restore_attend(torch.zeros(len(sel), dtype=torch.int32, device="cuda"),
                           torch.from_numpy(sel.astype(np.int32)).cuda(), q.cuda())
    torch.cuda.synchronize()
    assert c.get_status() == 0
    Ko, Vo, _ = C.reconstruct(st, sel.astype(np.int64), _weights64(W), "operand")
    assert rel_fro(np64(out), A.attend_restored(q.double().numpy(), Ko, Vo)) <= 1e-2


@cuda
def test_fused_back_to_back_calls(llama_store):
    """Calls queued back to back (each launch may start while the previous merge runs)
    give exactly what each gives alone."""
    r = llama_store
    c = r["codec"]
    sels = [synth.gen_selection(r["T"], n, 1390 + n).cuda() for n in (300, 1000, 77)]
    qs = [_q(32, 128, 1395 + i).cuda() for i in range(3)]
    alone = []
    for s, q in zip(sels, qs):
        alone.append(c.restore_attend(torch.zeros_like(s), s, q).clone())
        torch.cuda.synchronize()
    outs = [c.restore_attend(torch.zeros_like(s), s, q) for s, q in zip(sels, qs)]
    torch.cuda.synchronize()
    for a, b in zip(alone, outs):
        assert torch.equal(a, b)


@cuda
def test_fused_bad_selection_counts_as_zero_rows(llama_store):
    """An out-of-range position raises RKV_FLAG_BAD_INDEX and enters the softmax as a
    zero K_hat / V_hat row, as in the unfused read."""
    import residual_kv_cache_gb300 as rkv
    r = llama_store
    c = r["codec"]
    sel = synth.gen_selection(r["T"], 200, 1400).numpy()
    sel_bad = sel.copy()
    sel_bad[57] = r["T"] + 5
    q = _q(32, 128, 1401)
    out = c.restore_attend(torch.zeros(200, dtype=torch.int32, device="cuda"),
                           torch.from_numpy(sel_bad.astype(np.int32)).cuda(), q.cuda())
    torch.cuda.synchronize()
    flags = c.get_status()
    assert flags & rkv.FLAG_BAD_INDEX
    Ko, Vo, _ = C.reconstruct(r["st"], sel.astype(np.int64), r["W64"], "operand")
    Ko[57] = 0.0
    Vo[57] = 0.0
    assert rel_fro(np64(out), A.attend_restored(q.double().numpy(), Ko, Vo)) <= TOL_ORACLE


@cuda
def test_fused_rejects_unsupported_shapes(llama_store):
    import residual_kv_cache_gb300 as rkv
    c = llama_store["codec"]
    sel = torch.arange(10, dtype=torch.int32, device="cuda")
    zero = torch.zeros_like(sel)
    for Hq in (4, 12, 72):                          # not a multiple of N, or more than 8 N
        with pytest.raises(rkv.RkvError) as e:
            c.restore_attend(zero, sel, torch.zeros(Hq, 128, device="cuda"))
        assert e.value.status == -1
    with pytest.raises(rkv.RkvError):
        c.restore_attend(zero[:0], sel[:0], torch.zeros(8, 128, device="cuda"))
    # head_dim 64 (the tiny shape) and fp32 outputs are not supported
    w = synth.workload("tiny")
    t = make_codec(w, synth.gen_weights(w, 1410), T=256)
    with pytest.raises(rkv.RkvError):
        t.restore_attend(zero, sel, torch.zeros(4, 64, device="cuda"))
    wl = synth.workload("llama8b")
    f = make_codec(wl, synth.gen_weights(wl, 1411), T=256, out_dtype="fp32")
    with pytest.raises(rkv.RkvError):
        f.restore_attend(zero, sel, torch.zeros(8, 128, device="cuda"))


@cuda
def test_fused_selection_over_two_sequences():
    """A selection drawn from two sequences of one context: one softmax over all its rows,
    the same as restoring them and attending over the restored rows."""
    w = synth.workload("llama8b")
    T = 1024
    kvs = [synth.gen_kv(w, 1420 + s, T=T) for s in range(2)]
    c = make_codec(w, synth.gen_weights(w, 1422), T=T, batch=2, out_dtype="bf16")
    for s in range(2):
        gpu_prefill(c, kvs[s].cuda(), w.stride, seq_id=s)
    torch.cuda.synchronize()
    assert c.get_status() == 0
    g = torch.Generator().manual_seed(1423)
    seq = torch.randint(0, 2, (900,), generator=g, dtype=torch.int32).cuda()
    pos = torch.randint(0, T, (900,), generator=g, dtype=torch.int32).cuda()
    q = _q(32, 128, 1424).cuda()
    out = c.restore_attend(seq, pos, q)
    K, V = c.reconstruct(seq, pos)
    torch.cuda.synchronize()
    assert c.get_status() == 0
    ref = A.sparse_attention(q.double().cpu().numpy(), np64(K), np64(V))
    assert rel_fro(np64(out), ref) <= TOL_SAME_ROWS
