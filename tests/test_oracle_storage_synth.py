"""Storage accounting against the page's KR formula, and the seeded inputs."""
import numpy as np
import torch

import synth
from oracle import storage as S


def test_layer_bytes_equals_page_formula_with_beta_zero():
    for bits in (4, 2, 16):
        for d_kv, d_c in ((2048, 512), (1024, 256), (256, 64)):
            b = S.layer_bytes(T=16 * 1024, stride=16, d_kv=d_kv, d_c=d_c, bits=bits,
                              with_index=False)
            kr = S.keep_ratio(0.0, 1 / 16, bits, d_c / d_kv)
            assert abs(b["fraction"] - kr) < 1e-15


def test_storage_fractions_of_the_long_context_workloads():
    # Llama layer shape, stride 16: INT4 10.94 %, INT2 7.81 %, bf16 z 28.13 %
    want = {4: 10.94, 2: 7.81, 16: 28.13}
    for bits, pct in want.items():
        b = S.layer_bytes(262144, 16, 2048, 512, bits, with_index=False)
        assert abs(100 * b["fraction"] - pct) <= 0.005


def test_synthetic_inputs_are_deterministic_and_shaped():
    w = synth.workload("tiny")
    a, b = synth.gen_kv(w, 5), synth.gen_kv(w, 5)
    assert a.dtype == torch.float32 and a.shape == (256, 256)
    assert torch.equal(a, b)
    w2 = synth.workload("llama8b")
    kv = synth.gen_kv(w2, 1, T=2048)
    assert kv.dtype == torch.bfloat16 and kv.shape == (2048, 2048)
    rms = kv.float().pow(2).mean().sqrt().item()
    assert abs(rms - 1.0) < 1e-2
    W = synth.gen_weights(w2, 2)
    assert W["Wc1"].shape == (2048, 1536) and W["Wd"].shape == (512, 2048)
    sel = synth.gen_selection(32768, w2.n_sel, 3)
    assert len(sel) == 9830 and len(torch.unique(sel)) == 9830
    assert torch.all(sel[1:] > sel[:-1])
    blk = synth.gen_block_selection(131072, 64, 0.3, 4)
    assert len(blk) == 614 * 64
    assert torch.all(blk.view(-1, 64)[:, 1:] - blk.view(-1, 64)[:, :-1] == 1)
