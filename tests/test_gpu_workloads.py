"""Full-size workloads on the GPU, checked on sampled outputs the oracle computes one by
one (the oracle cannot encode a quarter-million tokens in seconds):

* llama8b    T=32768 prefill in the bench's launch configuration, 64 sampled tokens
             plus a sampled decode-step restore;
* long_int2  T=262144, INT2 codes, tokens sampled across the whole sequence (pools up
             to 16384 references);
* long_bf16z T=65536 with quantisation off;
* qwen7b     one layer of the Qwen2.5-7B-shaped stack (T=131072) read in contiguous
             64-token blocks;
* batched    16 sequences x 16384 with single-token decode writes interleaved with
             reads of each sequence's history.
"""
import numpy as np
import pytest
import torch

import synth
from oracle import codec as C

from _common import (assert_code_parity, gpu_prefill, idx_parity, make_codec, np64, oracle_shape,
                     rel_fro)

pytestmark = pytest.mark.gpu
cuda = pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA GPU")


def _sample_positions(T, stride, n, seed):
    rng = np.random.default_rng(seed)
    non = np.nonzero(np.arange(T) % stride)[0]
    # always include the first and last non-reference tokens (warm-up and full pool)
    pick = rng.choice(non, n - 2, replace=False)
    return np.unique(np.concatenate([pick, non[:1], non[-1:]]))


def _check_sampled(c, w, kv64, W64, pos, seq=0, bits=None):
    sh = oracle_shape(w)
    if bits is not None:
        sh = C.Shape(**{**sh.__dict__, "bits": bits})
    pool = C.build_pool(kv64, kv64.shape[0], w.stride)
    enc = C.encode_tokens(kv64[pos], pos, pool, W64, sh, "operand")
    gidx = c.ref_idx[seq].cpu().numpy().astype(np.int64)[pos]
    _, _, bad = idx_parity(gidx, enc["idx"], kv64[pos], pool.vals, pool.pos, pos)
    assert not bad, f"retrieval differs beyond near-ties at positions {pos[bad][:5]}"
    same = np.all(gidx == enc["idx"], axis=1)
    rows = pos[same]
    gq = C.unpack_codes(c.codes[seq].cpu().numpy()[rows], sh.bits, sh.d_c)
    gm = c.meta[seq].cpu().numpy().astype(np.float64)[rows]
    assert_code_parity(f"{w.name} T={kv64.shape[0]} sampled", gq, gm, enc["q"][same],
                       enc["meta"][same], enc["z"][same], kv64[rows], pool.vals,
                       enc["idx"][same], W64, sh.bits, sh.group)
    return pool, sh


def _check_restore(c, w, kv64, W64, pool, sh, sel, seq=0):
    """Restore `sel` on the GPU and compare with the oracle restoring the same tokens
    from its own encoding of them.  Tokens whose GPU retrieval is a (validated)
    near-tie swap have no unique oracle answer and are left out of the comparison."""
    sel = np.asarray(sel, dtype=np.int64)
    K, V = c.reconstruct(torch.full((len(sel),), seq, dtype=torch.int32).cuda(),
                         torch.from_numpy(sel.astype(np.int32)).cuda())
    torch.cuda.synchronize()
    assert c.get_status() == 0
    isref = sel % w.stride == 0
    idx = np.full((len(sel), sh.topk), -1)
    q = np.zeros((len(sel), sh.d_c))
    meta = np.zeros((len(sel), sh.n_groups, 2))
    idx[isref, 0] = sel[isref] // w.stride
    nr = ~isref
    if nr.any():
        enc = C.encode_tokens(kv64[sel[nr]], sel[nr], pool, W64, sh, "operand")
        idx[nr], q[nr], meta[nr] = enc["idx"], enc["q"], enc["meta"]
    gidx = c.ref_idx[seq].cpu().numpy().astype(np.int64)[sel]
    _, _, bad = idx_parity(gidx[nr], idx[nr], kv64[sel[nr]], pool.vals, pool.pos, sel[nr])
    assert not bad
    same = np.all(gidx == idx, axis=1)
    assert same.mean() > 0.9
    zt = C.dequantize(q, meta, sh.bits, sh.group)
    means = np.stack([C.reference_mean(pool.vals, i[i >= 0]) for i in idx])
    kvh = C.decode(zt, W64["Wd"], means)
    Ko, Vo = C.split_kv(kvh, sh.n_kv_heads, sh.head_dim)
    Ko = C.rope(Ko, sel, sh.rope_base)
    assert rel_fro(np64(K)[same], Ko[same]) <= 1e-2
    assert rel_fro(np64(V)[same], Vo[same]) <= 1e-2


def _prefill(name, seed, T=None, bits=None, **kw):
    w = synth.workload(name) if T is None else synth.workload(name, T=T)
    kv = synth.gen_kv(w, seed)
    W = synth.gen_weights(w, seed + 1)
    c = make_codec(w, W, T=w.T, bits=bits, **kw)
    gpu_prefill(c, kv.cuda(), w.stride)
    torch.cuda.synchronize()
    assert c.get_status() == 0
    return w, c, np64(kv), {k: np64(v) for k, v in W.items()}


@cuda
def test_llama8b_full_size_sampled():
    w, c, kv64, W64 = _prefill("llama8b", 201)
    pos = _sample_positions(w.T, w.stride, 64, 202)
    pool, sh = _check_sampled(c, w, kv64, W64, pos)
    sel = synth.gen_selection(w.T, w.n_sel, 203).numpy()[::40]   # 246 of one step's 9830
    _check_restore(c, w, kv64, W64, pool, sh, sel)


@cuda
def test_long_context_int2_sampled():
    w, c, kv64, W64 = _prefill("long_int2", 211)
    pos = _sample_positions(w.T, w.stride, 24, 212)
    pool, sh = _check_sampled(c, w, kv64, W64, pos)
    sel = synth.gen_selection(w.T, w.n_sel, 213).numpy()[::2048]
    _check_restore(c, w, kv64, W64, pool, sh, sel)


@cuda
def test_long_context_quant_off_sampled():
    w, c, kv64, W64 = _prefill("long_bf16z", 221)
    pos = _sample_positions(w.T, w.stride, 32, 222)
    pool, sh = _check_sampled(c, w, kv64, W64, pos)
    sel = synth.gen_selection(w.T, w.n_sel, 223).numpy()[::256]
    _check_restore(c, w, kv64, W64, pool, sh, sel)


@cuda
def test_qwen7b_layer_block_selection():
    w, c, kv64, W64 = _prefill("qwen7b", 231)
    pos = _sample_positions(w.T, w.stride, 48, 232)
    pool, sh = _check_sampled(c, w, kv64, W64, pos)
    blocks = synth.gen_block_selection(w.T, w.sel_block, w.sel_frac, 233).numpy()
    # all restored on the GPU; a strided sample of them checked against the oracle
    n = len(blocks)
    K, V = c.reconstruct(torch.zeros(n, dtype=torch.int32).cuda(),
                         torch.from_numpy(blocks).cuda())
    torch.cuda.synchronize()
    assert c.get_status() == 0
    _check_restore(c, w, kv64, W64, pool, sh, blocks[::301])


@cuda
def test_batched_decode_steps():
    """16 sequences prefilled, then decode steps that append one token per sequence
    (a reference every 16th position, otherwise a single-token compress) and restore
    30 % of each sequence's history."""
    w = synth.workload("batched")
    B, T0, steps = w.batch, w.T, 3
    Tcap = T0 + 32
    W = synth.gen_weights(w, 241)
    W64 = {k: np64(v) for k, v in W.items()}
    c = make_codec(w, W, T=Tcap, batch=B)
    kvs = [synth.gen_kv(w, 250 + b, T=T0 + steps) for b in range(B)]
    for b in range(B):
        gpu_prefill_part(c, kvs[b][:T0].cuda(), w.stride, b)
    sh = oracle_shape(w)
    dev_rows = torch.stack([kv[T0:T0 + steps] for kv in kvs], dim=1).cuda()   # [steps, B, d_kv]
    for s in range(steps):
        p = T0 + s
        seq = np.arange(B, dtype=np.int32)
        pos = np.full(B, p, dtype=np.int32)
        if p % w.stride == 0:
            c.pool_append(dev_rows[s].contiguous(), seq, pos)
        else:
            c.compress(dev_rows[s].contiguous(), seq, pos)
        # read 30 % of every sequence's history in one call
        sels = [synth.gen_selection(p + 1, int(round(0.3 * (p + 1))), 260 + 17 * s + b) for b in range(B)]
        sq = torch.cat([torch.full((len(x),), b, dtype=torch.int32) for b, x in enumerate(sels)])
        K, V = c.reconstruct(sq.cuda(), torch.cat(sels).cuda())
        torch.cuda.synchronize()
        assert c.get_status() == 0
    # oracle: the new tokens of two sequences and a sample of their last reads
    for b in (0, B - 1):
        kv64 = np64(kvs[b])
        pool = C.build_pool(kv64, T0 + steps, w.stride)
        newp = np.array([T0 + s for s in range(steps) if (T0 + s) % w.stride])
        enc = C.encode_tokens(kv64[newp], newp, pool, W64, sh, "operand")
        gidx = c.ref_idx[b].cpu().numpy().astype(np.int64)[newp]
        _, _, bad = idx_parity(gidx, enc["idx"], kv64[newp], pool.vals, pool.pos, newp)
        assert not bad
        _check_restore(c, w, kv64, W64, pool, sh, np.concatenate([newp, np.arange(0, T0, 997)]), b)


def gpu_prefill_part(codec, kv_dev, stride, seq_id):
    T = kv_dev.shape[0]
    pos = np.arange(T, dtype=np.int32)
    ref = pos[pos % stride == 0]
    non = pos[pos % stride != 0]
    codec.pool_append(kv_dev, np.full(len(ref), seq_id, np.int32), ref, src_rows=ref)
    codec.compress(kv_dev, np.full(len(non), seq_id, np.int32), non, src_rows=non)
