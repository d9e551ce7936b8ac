"""Verify-step attention, written out plainly in fp64.

Test infrastructure only (see the package docstring).

"推测解码" (world.lapla.si/zh/specdec), section 几段话一起写: besides the
shared weights, every sequence has its own KV cache that must be read on
every step (Llama 3.1 8B: about 131 KB per token over its layers), and at
batch 64 with 4,096 cached tokens that read dominates the step. The verify
pass runs the gamma + 1 new positions of each sequence at once; each of them
attends to the cached tokens and to the new positions up to itself.

Layout (the reading shared with the CUDA library), for one layer:
  q        [B, n_new, Hq, D]     the new positions' queries
  k, v     [B, Lmax, Hkv, D]     the cache; rows < seq_lens[b] are valid and
                                 the last n_new of them are the new positions
  seq_lens [B]                   cached length including the new positions
Query head h reads KV head h // (Hq / Hkv) (grouped-query attention). New
position i of sequence b sits at P = seq_lens[b] - n_new + i and attends to
cache rows 0..P. Output o[b, i, h] = sum_j softmax_j(q . k_j * scale) v_j with
scale = 1 / sqrt(D).
"""
from __future__ import annotations

import numpy as np


def verify_attention(q, k, v, seq_lens, scale=None) -> np.ndarray:
    """fp64 attention of the new positions over their causal window."""
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    B, n_new, Hq, D = q.shape
    Hkv = k.shape[2]
    assert Hq % Hkv == 0
    G = Hq // Hkv
    scale = 1.0 / np.sqrt(D) if scale is None else scale
    out = np.zeros((B, n_new, Hq, D))
    for b in range(B):
        L = int(seq_lens[b])
        assert n_new <= L <= k.shape[1]
        for h in range(Hq):
            kh = k[b, :L, h // G]                      # [L, D]
            vh = v[b, :L, h // G]
            s = (q[b, :, h] @ kh.T) * scale            # [n_new, L]
            for i in range(n_new):
                P = L - n_new + i                      # visible rows 0..P
                row = s[i, :P + 1]
                e = np.exp(row - row.max())
                out[b, i, h] = (e / e.sum()) @ vh[:P + 1]
    return out
