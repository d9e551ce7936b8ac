"""Pins for the clustered-LM-head oracle (oracle/cluster_head.py), on CPU.

* keeping every cluster reduces it to the full head: the member logits are
  h W^T and greedy is the plain argmax ("多詞元預測視覺化指南", sections
  高效嵌入器 and 什麼是多詞元預測);
* the kept clusters are the top-k by a brute-force scan;
* the law of the drawn token over all 2^24 uniforms is the softmax
  restricted to the kept clusters (exact enumeration), and a planted draw
  from the full softmax breaks it;
* the drawn token only depends on the kept tokens' logits.
"""
import numpy as np
import pytest

from oracle import cluster_head as oc
from oracle import philox
from oracle import verify as ov

N24 = 1 << 24


def _case(seed, M=4, d=16, V=60, n_c=7):
    rng = np.random.default_rng(seed)
    h = rng.normal(size=(M, d))
    W = rng.normal(size=(V, d)) * 0.7
    cut = np.sort(rng.choice(np.arange(1, V), size=n_c - 1, replace=False))
    starts = np.concatenate([[0], cut, [V]])
    perm = rng.permutation(V)                     # token IDs of the grouped rows
    E = np.stack([W[starts[c]:starts[c + 1]].mean(axis=0) for c in range(n_c)])
    return h, E, W, starts, perm


def test_all_clusters_is_the_full_head():
    h, E, W, starts, tor = _case(0)
    n_c = len(starts) - 1
    res = oc.cluster_head(h, E, W, starts, tor, n_c, 1.0, 0, ov.GREEDY)
    full = np.zeros((h.shape[0], W.shape[0]))
    full[:, tor] = h @ W.T                        # logits by token ID
    for m in range(h.shape[0]):
        np.testing.assert_array_equal(res.member_ids[m], np.arange(W.shape[0]))
        np.testing.assert_allclose(res.member_logits[m], full[m], rtol=1e-12, atol=1e-12)
        assert res.tokens[m] == int(np.argmax(full[m]))


@pytest.mark.parametrize("k", [1, 2, 3])
def test_kept_clusters_are_the_top_k(k):
    h, E, W, starts, tor = _case(1)
    res = oc.cluster_head(h, E, W, starts, tor, k, 1.0, 0, ov.GREEDY)
    y = h @ E.T
    for m in range(h.shape[0]):
        best = []
        for _ in range(k):
            cand = [c for c in range(y.shape[1]) if c not in best]
            best.append(max(cand, key=lambda c: (y[m, c], -c)))
        assert list(res.clusters[m]) == best
        members = np.sort(np.concatenate([tor[starts[c]:starts[c + 1]] for c in best]))
        np.testing.assert_array_equal(res.member_ids[m], members)
        # greedy: argmax over the kept tokens only
        z_full = np.zeros(W.shape[0])
        z_full[tor] = W @ h[m]
        assert res.tokens[m] == members[np.argmax(z_full[members])]


def _draw_law(ids, z, T):
    """Law of the oracle's draw over every u = j / 2^24."""
    x = z / T
    w = np.exp(x - x.max())
    u = np.arange(N24, dtype=np.float64) * philox.TWO_M24
    v, _ = ov.invert_cdf(w, u)
    law = np.zeros(int(ids.max()) + 1)
    np.add.at(law, ids[v], 1.0 / N24)
    return law


@pytest.mark.slow
def test_draw_law_is_the_restricted_softmax():
    h, E, W, starts, tor = _case(2, M=1)
    res = oc.cluster_head(h, E, W, starts, tor, 2, 0.8, 0, ov.SAMPLE)
    ids, z = res.member_ids[0], res.member_logits[0]
    law = _draw_law(ids, z, 0.8)
    p = np.exp(z / 0.8 - (z / 0.8).max())
    p /= p.sum()
    want = np.zeros_like(law)
    want[ids] = p
    np.testing.assert_allclose(law, want, rtol=0, atol=len(ids) * 2.0 ** -24)
    # a planted draw from the full softmax puts mass outside the kept clusters
    z_full = np.zeros(W.shape[0])
    z_full[tor] = W @ h[0]
    bad = _draw_law(np.arange(W.shape[0]), z_full, 0.8)
    assert bad[np.setdiff1d(np.arange(W.shape[0]), ids)].sum() > 1e-3


def test_draw_uses_the_draft_counter_and_only_kept_logits():
    h, E, W, starts, tor = _case(3)
    a = oc.cluster_head(h, E, W, starts, tor, 2, 1.0, 42, ov.SAMPLE, position=3)
    # changing a row of a cluster that is not kept changes nothing
    keep = set(int(c) for c in a.clusters[0])
    other = next(c for c in range(len(starts) - 1) if c not in keep)
    W2 = W.copy()
    W2[starts[other]] += 5.0
    E2 = E.copy()                                 # keep the selection itself unchanged
    b = oc.cluster_head(h[:1], E2, W2, starts, tor, 2, 1.0, 42, ov.SAMPLE, position=3)
    assert b.tokens[0] == a.tokens[0]
    # the uniform is Philox (row, position, purpose 2)
    u = oc.draft_uniform(42, 0, 3)
    assert u == float(philox.uniform24(42, 0, 3, 2)) * 2.0 ** -24
