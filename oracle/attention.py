"""Sparse attention over restored K/V, written out in float64.

Test infrastructure, like the rest of ``oracle/``: only ``tests/``,
``__graft_entry__.smoke()`` and the CPU legs of ``bench.py`` may import it.  It
shares no code with the CUDA library.

ResidualKV notes, section 2.7 (the OmniKV combination): a sparse layer restores
only the selected tokens I_t and computes

    o = softmax(q K_hat[I_t]^T / sqrt(D)) V_hat[I_t]

for the current query q.  Readings of what the section leaves open:
* grouped-query attention as in the Llama / Qwen models the page uses: with H_q
  query heads and N key/value heads, query head h reads key/value head
  h // (H_q / N);
* q arrives already rotated at the decode position (the restored K_hat is rotated
  at each token's own position);
* the softmax runs over exactly the selected tokens, with no mask or sink beyond
  them.
"""
from __future__ import annotations

import numpy as np

from . import formats as F

__all__ = ["sparse_attention", "attend_restored"]


def sparse_attention(q, K, V):
    """q [H_q, D]; K, V [n, N, D] (the restored rows of the selected tokens).

    Returns o [H_q, D] in float64.  An empty selection (n = 0) has no softmax and
    is rejected.
    """
    q = np.asarray(q, np.float64)
    K = np.asarray(K, np.float64)
    V = np.asarray(V, np.float64)
    n, N, D = K.shape
    Hq = q.shape[0]
    if n == 0:
        raise ValueError("softmax over an empty selection")
    if q.shape[1] != D or Hq % N != 0:
        raise ValueError("q must be [H_q, D] with H_q a multiple of N")
    group = Hq // N
    out = np.empty((Hq, D))
    for h in range(Hq):
        g = h // group
        s = K[:, g, :] @ q[h] / np.sqrt(D)           # [n] scores
        w = np.exp(s - s.max())
        out[h] = (w / w.sum()) @ V[:, g, :]
    return out


def attend_restored(q, K_hat, V_hat, rows: str = "bf16"):
    """The sparse layer's read as one pass (ResidualKV notes section 2.7, Fig. 7: the
    selected tokens are restored and attended without a stored K/V copy): the output
    equation over the restored rows as the read consumes them.

    K_hat, V_hat [n, N, D] are the restored rows in float64 (``codec.reconstruct``);
    ``rows`` names the format they are handed to the attention in: "bf16" rounds them
    (nearest-even) as a bf16 restore output is rounded, "f64" keeps them.  Reading of
    the page: it fixes no format for the restored rows, and a fused read rounds them
    where an unfused one would store them.
    """
    if rows == "bf16":
        K_hat, V_hat = F.bf16(K_hat), F.bf16(V_hat)
    elif rows != "f64":
        raise ValueError("rows must be 'bf16' or 'f64'")
    return sparse_attention(q, K_hat, V_hat)
