"""The clustered LM head of a small drafter, written out plainly in fp64.

Test infrastructure only (see the package docstring).

"多詞元預測視覺化指南" (the Gemma 4 MTP visual guide), section 高效嵌入器:
the drafter's output head would multiply its hidden state by the whole
vocabulary table; instead the token embeddings are grouped into clusters of
similar tokens, each cluster gets one embedding, the hidden state is scored
against those (cluster logits), the most likely cluster is chosen, and only
that cluster's tokens get token logits.

Readings where the page is silent (each is also the CUDA library's):
* The clusters partition the vocabulary. Rows of W_sorted are the token
  embeddings grouped by cluster: cluster c owns rows starts[c] ..
  starts[c+1] - 1, and row r is token token_of_row[r].
* top_k >= 1 clusters are kept: the largest cluster logits, ties to the
  lower cluster index (top_k = 1 is the page's single cluster).
* The draft distribution is softmax(z / T) over the kept clusters' tokens
  (every other token has probability 0). Greedy takes its argmax (lowest
  token ID on ties); sampling inverts its prefix sum in token-ID order at
  u * S with u the Philox uniform of (row, position, purpose 2) -- the
  draft purpose of the verify step's random numbers -- exactly as the verify
  step draws its replacements.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

from . import philox
from .verify import GREEDY, SAMPLE, greedy_argmax, invert_cdf

DRAFT = 2


def draft_uniform(seed: int, b, i) -> np.ndarray:
    """u = k / 2^24 in [0, 1) from Philox counter (b, i, 2, 0)."""
    return philox.uniform24(seed, b, i, DRAFT).astype(np.float64) * philox.TWO_M24


def top_clusters(y_row, k: int) -> np.ndarray:
    """Indices of the k largest entries, ties to the lower index."""
    y_row = np.asarray(y_row, dtype=np.float64)
    order = np.lexsort((np.arange(y_row.shape[0]), -y_row))
    return order[:k]


@dataclass
class ClusterHeadResult:
    clusters: np.ndarray              # [M, top_k] kept clusters, best first
    tokens: np.ndarray                # [M] drafted token
    member_ids: list                  # per row: token IDs of the kept tokens (token-ID order)
    member_logits: list               # per row: their logits z (fp64), same order
    cluster_gaps: list = field(default_factory=list)   # k-th minus (k+1)-th cluster logit
    margins: list = field(default_factory=list)        # draw margin, or greedy top-2 gap


def cluster_head(h, E, W_sorted, starts, token_of_row, top_k: int, temperature: float,
                 seed: int, mode: int, position: int = 0, rows=None) -> ClusterHeadResult:
    """h [M, d], E [n_c, d], W_sorted [V, d], starts [n_c + 1], token_of_row [V]."""
    h = np.asarray(h, dtype=np.float64)
    E = np.asarray(E, dtype=np.float64)
    W = np.asarray(W_sorted, dtype=np.float64)
    starts = np.asarray(starts, dtype=np.int64)
    tor = np.asarray(token_of_row, dtype=np.int64)
    M = h.shape[0]
    rows = np.arange(M) if rows is None else np.asarray(rows)
    y = h @ E.T                                       # cluster logits
    res = ClusterHeadResult(np.zeros((M, top_k), dtype=np.int64), np.zeros(M, dtype=np.int64),
                            [], [])
    for m in range(M):
        sel = top_clusters(y[m], top_k)
        res.clusters[m] = sel
        ys = np.sort(y[m])[::-1]
        res.cluster_gaps.append(float(ys[top_k - 1] - ys[top_k]) if top_k < y.shape[1]
                                else float("inf"))
        r = np.concatenate([np.arange(starts[c], starts[c + 1]) for c in sel])
        ids = tor[r]
        z = W[r] @ h[m]
        order = np.argsort(ids, kind="stable")
        ids, z = ids[order], z[order]
        res.member_ids.append(ids)
        res.member_logits.append(z)
        if mode == GREEDY:
            a, gap = greedy_argmax(z)
            res.tokens[m] = ids[a]
            res.margins.append(gap)
        else:
            x = z / temperature
            w = np.exp(x - x.max())
            v, margin = invert_cdf(w, draft_uniform(seed, int(rows[m]), position))
            res.tokens[m] = ids[int(v)]
            res.margins.append(float(margin))
    return res
