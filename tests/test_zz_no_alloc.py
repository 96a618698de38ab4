"""The allocation-free retrieval entry point, called through the C ABI, returns the
same slots as the retrieval inside rkv_compress (the existing entry point) on the same
pool, on two calls in a row that share its fixed scratch array.

Callers that use it cannot allocate device memory while they run (a runtime that owns
all device memory through its own arena, or a step that must not pay cudaMalloc's
implicit synchronisation); this file runs last so that a failure here leaves every
other test already run."""
import ctypes

import numpy as np
import pytest
import torch

import synth

from _common import gpu_prefill, make_codec

pytestmark = pytest.mark.gpu
cuda = pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA GPU")


def _noalloc(queries, qpos, pool, norm2, ppos, topk, out, flags):
    import residual_kv_cache_gb300 as rkv
    n, d = queries.shape
    R = pool.shape[0]
    return rkv.lib().rkv_retrieve_noalloc(
        queries.data_ptr(), qpos.data_ptr(), n, pool.data_ptr(), norm2.data_ptr(),
        ppos.data_ptr(), R, d, topk, out.data_ptr(),
        flags.data_ptr() if flags is not None else None,
        torch.cuda.current_stream().cuda_stream)


@cuda
def test_noalloc_retrieval_equals_compress_retrieval_on_two_calls():
    w = synth.workload("llama8b")
    T = 4096
    kv = synth.gen_kv(w, 301, T=T).cuda()
    c = make_codec(w, synth.gen_weights(w, 302), T=T)
    ref, non = gpu_prefill(c, kv, w.stride)
    torch.cuda.synchronize()
    assert c.get_status() == 0
    R = len(ref)
    pool = c.pool_bf16[0, :R]
    norm2 = c.pool_norm2[0, :R]
    ppos = c.pool_pos[0, :R]
    expected = c.ref_idx[0].long()
    flags = torch.zeros(1, dtype=torch.int32, device="cuda")

    # call 1: every non-reference token, in order
    q1 = torch.from_numpy(non.astype(np.int64)).cuda()
    out1 = torch.full((len(non), w.topk), -7, dtype=torch.int32, device="cuda")
    assert _noalloc(kv[q1].contiguous(), q1.int(), pool, norm2, ppos, w.topk, out1, flags) == 0
    torch.cuda.synchronize()
    assert int(flags.item()) == 0
    assert torch.equal(out1.long(), expected[q1])

    # call 2, right after: another set of rows in another order (the scratch now holds
    # the first call's lists)
    q2 = q1.flip(0)[::3].contiguous()
    out2 = torch.full((len(q2), w.topk), -7, dtype=torch.int32, device="cuda")
    assert _noalloc(kv[q2].contiguous(), q2.int(), pool, norm2, ppos, w.topk, out2, flags) == 0
    torch.cuda.synchronize()
    assert int(flags.item()) == 0
    assert torch.equal(out2.long(), expected[q2])


@cuda
def test_noalloc_retrieval_rejects_sizes_beyond_its_scratch():
    import residual_kv_cache_gb300 as rkv
    d, R, n = 256, 256 * 16, 128 * 65          # 65 x 16 tiles > 1024
    q = torch.zeros((n, d), dtype=torch.bfloat16, device="cuda")
    qpos = torch.ones(n, dtype=torch.int32, device="cuda")
    pool = torch.zeros((R, d), dtype=torch.bfloat16, device="cuda")
    norm2 = torch.zeros(R, dtype=torch.float32, device="cuda")
    ppos = torch.zeros(R, dtype=torch.int32, device="cuda")
    out = torch.empty((n, 4), dtype=torch.int32, device="cuda")
    flags = torch.zeros(1, dtype=torch.int32, device="cuda")
    assert _noalloc(q, qpos, pool, norm2, ppos, 4, out, flags) == -3     # RKV_ECAPACITY
    assert b"1024" in rkv.lib().rkv_last_error()


@cuda
def test_noalloc_retrieval_across_pool_tiles_topk_and_null_flags():
    """A pool of 1024 references (four 256-slot tiles, so the merge combines partial
    lists across tile boundaries) and 2048 queries spread over the sequence, its last
    tokens included: the same slots as rkv_compress stores; with topk = 2 the first two
    of them; and with no caller flags, the same result on two calls in a row."""
    w = synth.workload("llama8b")
    T = 16384
    kv = synth.gen_kv(w, 311, T=T).cuda()
    c = make_codec(w, synth.gen_weights(w, 312), T=T)
    ref, non = gpu_prefill(c, kv, w.stride)
    torch.cuda.synchronize()
    assert c.get_status() == 0
    R = len(ref)
    assert R == 1024
    pool = c.pool_bf16[0, :R]
    norm2 = c.pool_norm2[0, :R]
    ppos = c.pool_pos[0, :R]
    expected = c.ref_idx[0].long()
    rng = np.random.default_rng(313)
    pick = np.sort(np.concatenate([rng.choice(non[:-64], 2048 - 64, replace=False), non[-64:]]))
    q = torch.from_numpy(pick.astype(np.int64)).cuda()
    rows = kv[q].contiguous()
    flags = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = torch.full((len(pick), 4), -7, dtype=torch.int32, device="cuda")
    assert _noalloc(rows, q.int(), pool, norm2, ppos, 4, out, flags) == 0
    torch.cuda.synchronize()
    assert int(flags.item()) == 0
    assert torch.equal(out.long(), expected[q])
    # the nearest two, nearest first, are the first two of the nearest four
    out2 = torch.full((len(pick), 2), -7, dtype=torch.int32, device="cuda")
    assert _noalloc(rows, q.int(), pool, norm2, ppos, 2, out2, flags) == 0
    torch.cuda.synchronize()
    assert int(flags.item()) == 0
    assert torch.equal(out2.long(), expected[q][:, :2])
    # no caller flags: the library's own status word, cleared by each call
    for _ in range(2):
        out3 = torch.full((len(pick), 4), -7, dtype=torch.int32, device="cuda")
        assert _noalloc(rows, q.int(), pool, norm2, ppos, 4, out3, None) == 0
        torch.cuda.synchronize()
        assert torch.equal(out3.long(), expected[q])
