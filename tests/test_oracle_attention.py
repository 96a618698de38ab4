"""Pins of oracle/attention.py (ResidualKV notes section 2.7, the sparse-layer
attention over restored K/V) against closed forms and a library routine."""
import math

import numpy as np
import pytest
import torch

from oracle import attention as A


def _rand(rng, *shape):
    return rng.normal(size=shape)


def test_matches_torch_sdpa_in_float64():
    """With one key/value head per query head, o is torch's scaled dot-product
    attention (default scale 1/sqrt(D)) of the same float64 tensors."""
    rng = np.random.default_rng(1)
    for n, N, D in ((1, 1, 8), (37, 4, 16), (300, 2, 128)):
        q, K, V = _rand(rng, N, D), _rand(rng, n, N, D), _rand(rng, n, N, D)
        got = A.sparse_attention(q, K, V)
        ref = torch.nn.functional.scaled_dot_product_attention(
            torch.tensor(q)[:, None, :], torch.tensor(K).permute(1, 0, 2),
            torch.tensor(V).permute(1, 0, 2))[:, 0, :].numpy()
        assert np.allclose(got, ref, rtol=1e-12, atol=1e-12)


def test_grouped_query_heads_read_their_group():
    """H_q = 8 query heads over N = 2 key/value heads: heads 0-3 read kv head 0,
    heads 4-7 kv head 1; a query that matches no key averages V uniformly."""
    rng = np.random.default_rng(2)
    n, D = 5, 4
    K = np.zeros((n, 2, D))
    V = _rand(rng, n, 2, D)
    q = np.zeros((8, D))
    out = A.sparse_attention(q, K, V)
    assert np.allclose(out[:4], V[:, 0].mean(0)) and np.allclose(out[4:], V[:, 1].mean(0))
    # head 5 with a huge score on token 3 of kv head 1 returns that token's value
    K[3, 1, 0] = 1.0
    q[5, 0] = 1e3
    out = A.sparse_attention(q, K, V)
    assert np.allclose(out[5], V[3, 1], atol=1e-12)
    assert np.allclose(out[1], V[:, 0].mean(0))


def test_closed_forms():
    """One token returns its value; two tokens with score gap g weight them
    1/(1+e^-g) and 1/(1+e^g); a shift of every score leaves o unchanged."""
    rng = np.random.default_rng(3)
    D = 16
    V = _rand(rng, 1, 1, D)
    assert np.allclose(A.sparse_attention(_rand(rng, 1, D), _rand(rng, 1, 1, D), V)[0], V[0, 0])
    q = np.zeros((1, D)); q[0, 0] = 1.0
    K = np.zeros((2, 1, D)); K[0, 0, 0] = 2.0 * math.sqrt(D)   # scores 2 and 0
    V = _rand(rng, 2, 1, D)
    w0 = 1 / (1 + math.exp(-2.0))
    assert np.allclose(A.sparse_attention(q, K, V)[0], w0 * V[0, 0] + (1 - w0) * V[1, 0],
                       rtol=1e-14)
    K2 = K.copy(); K2[:, 0, 1] = 5.0; q2 = q.copy(); q2[0, 1] = 0.3   # both scores + 1.5/sqrt(D)
    assert np.allclose(A.sparse_attention(q2, K2, V), A.sparse_attention(q, K, V), rtol=1e-12)


def test_rejects_empty_selection_and_bad_groups():
    with pytest.raises(ValueError):
        A.sparse_attention(np.zeros((2, 4)), np.zeros((0, 1, 4)), np.zeros((0, 1, 4)))
    with pytest.raises(ValueError):
        A.sparse_attention(np.zeros((3, 4)), np.zeros((2, 2, 4)), np.zeros((2, 2, 4)))


def test_attend_restored_rounds_rows_as_torch_bf16():
    """The one-pass read (ResidualKV notes section 2.7, Fig. 7) attends over the restored
    rows rounded to bf16: the same as torch's scaled dot-product attention over the rows
    converted by torch to bfloat16 (nearest-even) and back; one token returns its value
    rounded to bf16; with rows="f64" nothing is rounded."""
    rng = np.random.default_rng(4)
    n, N, D = 200, 2, 128
    q, K, V = _rand(rng, N, D), _rand(rng, n, N, D) * 3.0, _rand(rng, n, N, D)
    Kb = torch.tensor(K).to(torch.bfloat16).double()
    Vb = torch.tensor(V).to(torch.bfloat16).double()
    ref = torch.nn.functional.scaled_dot_product_attention(
        torch.tensor(q)[:, None, :], Kb.permute(1, 0, 2), Vb.permute(1, 0, 2))[:, 0, :].numpy()
    got = A.attend_restored(q, K, V)
    assert np.allclose(got, ref, rtol=1e-12, atol=1e-12)
    assert not np.allclose(got, A.sparse_attention(q, K, V), rtol=1e-6, atol=0)
    assert np.array_equal(A.attend_restored(q, K, V, rows="f64"), A.sparse_attention(q, K, V))
    one = A.attend_restored(q[:1], K[:1, :1], V[:1, :1])
    assert np.array_equal(one[0], torch.tensor(V[0, 0]).to(torch.bfloat16).double().numpy())
    with pytest.raises(ValueError):
        A.attend_restored(q, K, V, rows="fp8")
