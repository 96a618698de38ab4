"""GPU parity of the encoder with the mean's pre-activations taken from the references'
own (mean_precompute = 1): mean_i W = (1/k_i) sum_j r_j W for W = W_c1, W_c2 (ResidualKV
notes §2.3 maps the §2.2 mean; x W is linear in x), kept per pool slot and summed per
token, so GEMM-1/2 runs on kv rows only.

The oracle is ``codec.encode_tokens(..., mean_from="refs")``: the same steps in float64
with the references exact (FP8 values are bf16 values) and the kv row rounded to bf16 as
the tensor core reads it.  Checks:
* the per-slot table P = r [W_c1 | W_c2] against float64 products: within the a-priori
  bound of an fp32 sum of 2d_k products (2d_k 2^-23 sum |r_d w_d|) everywhere, and
  within 1e-6 relative (Frobenius) overall;
* codes by the method's rule over every token whose retrieval matched: >= 99.9 %
  identical, a differing code only +-1 and only within 1e-3 of a .5 boundary (the GPU
  sums the slots' fp32 P rows, the oracle exact float64 products); then every code and
  FP16 extreme inside the interval of z that the fp32 arithmetic allows
  (``encoder_intervals_refs``);
* the restore end to end against the oracle's (<= 1e-2, the restore's tolerance);
* several sequences in one pass, appends in any order of sequences, and decode-style
  appends one reference at a time.
"""
import numpy as np
import pytest
import torch

import synth
from oracle import codec as C

from _common import check_codes_interval, code_parity_report, device_bytes, \
    encoder_intervals_refs, gpu_prefill, make_codec, np64, oracle_shape, rel_fro

pytestmark = pytest.mark.gpu
cuda = pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA GPU")


def _weights64(W):
    return {k: np64(v) for k, v in W.items()}


def _run(name, T, seed_kv=41, seed_w=42):
    w = synth.workload(name)
    kv = synth.gen_kv(w, seed_kv, T=T)
    W = synth.gen_weights(w, seed_w)
    codec = make_codec(w, W, T=T, mean_precompute=1)
    ref, non = gpu_prefill(codec, kv.cuda(), w.stride)
    torch.cuda.synchronize()
    assert codec.get_status() == 0
    sh = oracle_shape(w)
    W64 = _weights64(W)
    store = C.compress_sequence(np64(kv), W64, sh, "operand", mean_from="refs")
    return dict(w=w, kv=kv, kv64=np64(kv), W=W, W64=W64, codec=codec, store=store, sh=sh,
                ref=ref, non=non, T=T)


@pytest.fixture(scope="module")
def tiny():
    return _run("tiny", 256)


@pytest.fixture(scope="module")
def llama():
    return _run("llama8b", 4096)


@pytest.fixture(scope="module")
def qwen():
    return _run("qwen7b", 4096)


def _codes_rule(codec, store, sh, rows, label, kv64, W64, seq=0):
    """The method's code rule, then every code and FP16 extreme inside the interval the
    arithmetic allows (an extreme differs where a correct fp32 evaluation of z puts the
    group's minimum or maximum across an FP16 value)."""
    gq = C.unpack_codes(codec.codes[seq].cpu().numpy()[rows], sh.bits, sh.d_c)
    gmeta = codec.meta[seq].cpu().numpy().astype(np.float64)[rows]
    rep = code_parity_report(gq, gmeta, store.q[rows], store.meta[rows], store.z[rows], sh.bits,
                             sh.group)
    print(f"[codes {label}] {rep}")
    assert rep["identical"] >= 0.999, f"only {rep['identical']:.5f} of codes identical"
    assert rep["not_pm1"] == 0
    assert rep["beyond_window"] == 0
    iv = encoder_intervals_refs(kv64[rows], store.pool.vals, store.idx[rows], W64)
    viol = check_codes_interval(gq, gmeta, iv["z"], iv["w"], sh.bits, sh.group)
    assert not viol, f"{len(viol)} codes or extremes outside their interval, first {viol[:3]}"
    return rep


def _same_idx_rows(codec, store, non, seq=0):
    gidx = codec.ref_idx[seq].cpu().numpy().astype(np.int64)
    return non[np.all(gidx[non] == store.idx[non], axis=1)]


@cuda
@pytest.mark.parametrize("name", ["tiny", "llama", "qwen"])
def test_reference_preactivation_table(name, request):
    r = request.getfixturevalue(name)
    c, st, w = r["codec"], r["store"], r["w"]
    R = len(st.pool.pos)
    ptr, nbytes = c.debug_scratch(3)
    P = device_bytes(ptr, nbytes).view(torch.float32).cpu().numpy().reshape(-1, 2 * w.d_ff)[:R]
    W1, W2 = r["W64"]["Wc1"], r["W64"]["Wc2"]
    nt = w.d_ff // 128
    cols = np.concatenate([np.concatenate([W1[:, 128 * n:128 * n + 128], W2[:, 128 * n:128 * n + 128]],
                                          axis=1) for n in range(nt)], axis=1)
    exact = st.pool.vals @ cols
    # a-priori bound of an fp32 sum of 2d_k exact products (one unit of 2^-23 per
    # addition, whatever the order), and the typical error far below it
    bound = np.abs(st.pool.vals) @ np.abs(cols) * (w.d_kv * 2.0 ** -23)
    assert np.all(np.abs(P - exact) <= bound)
    assert rel_fro(P, exact) <= 1e-6


@cuda
@pytest.mark.parametrize("name", ["tiny", "llama", "qwen"])
def test_codes_by_the_method_rule(name, request):
    r = request.getfixturevalue(name)
    rows = _same_idx_rows(r["codec"], r["store"], r["non"])
    assert len(rows) >= 0.99 * len(r["non"])
    _codes_rule(r["codec"], r["store"], r["sh"], rows, name, r["kv64"], r["W64"])


@cuda
@pytest.mark.parametrize("name", ["llama", "qwen"])
def test_restore_end_to_end(name, request):
    r = request.getfixturevalue(name)
    c, st, T = r["codec"], r["store"], r["T"]
    sel = synth.gen_selection(T, int(round(0.3 * T)), 43)
    K, V = c.reconstruct(torch.zeros_like(sel).cuda(), sel.cuda())
    torch.cuda.synchronize()
    assert c.get_status() == 0
    Ko, Vo, _ = C.reconstruct(st, sel.numpy().astype(np.int64), r["W64"], "operand")
    same = np.all(c.ref_idx[0].cpu().numpy()[sel.numpy()] == st.idx[sel.numpy()], axis=1)
    assert same.mean() > 0.9
    assert rel_fro(np64(K)[same], Ko[same]) <= 1e-2
    assert rel_fro(np64(V)[same], Vo[same]) <= 1e-2


@cuda
def test_two_sequences_interleaved_and_one_pass():
    """Two sequences: references appended in calls that interleave the sequences (rows
    of sequence 1 first, so the pool tiles of one call are not in increasing order), the
    other tokens of both encoded in one pass (rows grouped by sequence)."""
    w = synth.workload("llama8b")
    T = 1024
    kvs = [synth.gen_kv(w, 50 + s, T=T) for s in range(2)]
    W = synth.gen_weights(w, 52)
    c = make_codec(w, W, T=T, batch=2, mean_precompute=1)
    kv_all = torch.cat(kvs).cuda()
    pos = np.arange(T, dtype=np.int32)
    ref = pos[pos % w.stride == 0]
    non = pos[pos % w.stride != 0]
    for lo, hi in ((0, 20), (20, len(ref))):
        seqs = np.concatenate([np.ones(hi - lo, np.int32), np.zeros(hi - lo, np.int32)])
        ps = np.concatenate([ref[lo:hi], ref[lo:hi]]).astype(np.int32)
        src = (seqs * T + ps).astype(np.int32)
        c.pool_append(kv_all, seqs, ps, src_rows=src)
    seqs = np.concatenate([np.zeros(len(non), np.int32), np.ones(len(non), np.int32)])
    ps = np.concatenate([non, non]).astype(np.int32)
    c.compress(kv_all, seqs, ps, src_rows=(seqs * T + ps).astype(np.int32))
    torch.cuda.synchronize()
    assert c.get_status() == 0
    sh = oracle_shape(w)
    for s in range(2):
        st = C.compress_sequence(np64(kvs[s]), _weights64(W), sh, "operand", mean_from="refs")
        rows = _same_idx_rows(c, st, non, seq=s)
        assert len(rows) >= 0.99 * len(non)
        _codes_rule(c, st, sh, rows, f"seq {s}", np64(kvs[s]), _weights64(W), seq=s)


@cuda
def test_decode_style_appends():
    """A prefill of the first half, then one token per call: each reference appended alone
    (its pool tile's P recomputed) before the tokens that follow it are encoded."""
    w = synth.workload("qwen7b")
    T = 512
    kv = synth.gen_kv(w, 60, T=T)
    W = synth.gen_weights(w, 61)
    c = make_codec(w, W, T=T, mean_precompute=1)
    kvd = kv.cuda()
    half = 256
    pos = np.arange(half, dtype=np.int32)
    ref, non = pos[pos % w.stride == 0], pos[pos % w.stride != 0]
    c.pool_append(kvd, np.zeros_like(ref), ref, src_rows=ref)
    c.compress(kvd, np.zeros_like(non), non, src_rows=non)
    for p in range(half, T):
        one = np.array([p], np.int32)
        if p % w.stride == 0:
            c.pool_append(kvd, np.zeros(1, np.int32), one, src_rows=one)
        else:
            c.compress(kvd, np.zeros(1, np.int32), one, src_rows=one)
    torch.cuda.synchronize()
    assert c.get_status() == 0
    sh = oracle_shape(w)
    st = C.compress_sequence(np64(kv), _weights64(W), sh, "operand", mean_from="refs")
    allnon = np.arange(T)[np.arange(T) % w.stride != 0]
    rows = _same_idx_rows(c, st, allnon)
    assert len(rows) >= 0.99 * len(allnon)
    _codes_rule(c, st, sh, rows, "decode", np64(kv), _weights64(W))


@cuda
def test_mode_is_validated():
    import residual_kv_cache_gb300 as rkv
    w = synth.workload("tiny")
    with pytest.raises(rkv.RkvError):
        make_codec(w, synth.gen_weights(w, 70), T=256, mean_precompute=2)
    c = make_codec(w, synth.gen_weights(w, 71), T=256)
    with pytest.raises(rkv.RkvError):
        c.debug_scratch(3)                       # no table without the mode


@cuda
def test_dynamic_schedule_and_int2():
    """The dynamic-stride schedule (alpha = 0.1, two sink tokens) with INT2 codes: the pool
    tiles a call touches follow the schedule's slots."""
    w = synth.workload("llama8b")
    T = 1024
    kv = synth.gen_kv(w, 80, T=T)
    W = synth.gen_weights(w, 81)
    c = make_codec(w, W, T=T, bits=2, alpha=0.1, sink=2, mean_precompute=1)
    ref, non = gpu_prefill(c, kv.cuda(), w.stride, alpha=0.1, sink=2)
    torch.cuda.synchronize()
    assert c.get_status() == 0
    sh = C.Shape(**{**oracle_shape(w, 0.1, 2).__dict__, "bits": 2})
    st = C.compress_sequence(np64(kv), _weights64(W), sh, "operand", mean_from="refs")
    rows = _same_idx_rows(c, st, non)
    assert len(rows) >= 0.99 * len(non)
    _codes_rule(c, st, sh, rows, "dyn int2", np64(kv), _weights64(W))
