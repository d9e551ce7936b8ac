"""Tree verification: the verify rule applied at every fork of a token tree.

Test infrastructure only (see the package docstring).

"推测解码" (world.lapla.si/zh/specdec), section 不要第二个模型: Medusa-style
heads arrange several guesses into a tree that the large model checks in one
pass, and EAGLE applies the same acceptance rule at every fork of the guess
tree, which keeps the output distribution unchanged.

Layout (the reading shared with the CUDA library). A tree of N nodes, the
same for every sequence of the batch: node 0 is the root (the position after
the committed text); every other node n holds one guessed token tok[n] and
has a parent parent[n] < n. hidden[b, n] is the target state after the path
root -> n, so p_n = softmax(W hidden[b, n] / T) is the large model's
distribution for the children of n; draft_logits[b, n] gives q_n, the
distribution the children of n were drawn from.

Readings where the pages are silent (each is also the CUDA library's):

* Siblings are tried in increasing node index. Each is kept iff
  r * q_u(x) <= f(x), with f = p_u for the first child; after a sibling is
  rejected, f becomes max(0, f - q_u) / S, S its sum, for the next sibling.
  For siblings drawn independently from q_u this keeps the law of the
  emitted token equal to p_u (the rule of "推测解码", section 通过的规则,
  applied once per sibling).
* A kept child becomes the new node; a node whose children are all
  rejected (or that has none) emits one token drawn from the current f by
  the chain rule's inversion: weights max(0, f - q_u) of the last rejection
  (unnormalised), or p_u if nothing was rejected, at t = u * S.
* If a residual sums to 0 (possible only through rounding), testing stops
  and the token is drawn from p_u (the chain rule's fallback).
* Random draws: the acceptance uniform of node c is the chain's r at
  position c - 1; the draw at depth j (j tokens kept) is the chain's u at
  position j. A chain-shaped tree (parent[n] = n - 1) therefore reproduces
  the chain verify step exactly.
* Greedy: at node u take a = argmax p_u (lowest ID on ties); move to the
  first child whose token is a, else emit a and stop.
* Outputs: tokens kept along the path then the drawn token, -1 padded to N;
  the kept nodes, -1 padded; n_accepted = number of kept nodes.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

from . import philox
from .verify import (GREEDY, SAMPLE, accept_test, greedy_argmax, invert_cdf, lm_head_logits,
                     residual_weights, softmax_t)


def children_of(parent) -> list:
    """Children of every node, in increasing node index; checks the shape.

    parent[0] must be -1 and 0 <= parent[n] < n for n >= 1 (so node indices
    are a topological order and the tree is connected).
    """
    parent = [int(x) for x in parent]
    if len(parent) < 1 or parent[0] != -1:
        raise ValueError("parent[0] must be -1 (the root)")
    kids = [[] for _ in parent]
    for n in range(1, len(parent)):
        if not 0 <= parent[n] < n:
            raise ValueError(f"parent[{n}] = {parent[n]} is not an earlier node")
        kids[parent[n]].append(n)
    return kids


@dataclass
class TreeSequenceResult:
    tokens: np.ndarray            # [N] int64, -1 padded
    nodes: np.ndarray             # [N] int64 kept node indices, -1 padded
    n_accepted: int
    accept_margins: list = field(default_factory=list)   # |r - f(x)/q(x)| per tested child
    sample_margin: float = float("inf")
    greedy_gaps: list = field(default_factory=list)


def verify_tree_sequence_sampling(p_rows, q_rows, tok, parent, r_at, u_at) -> TreeSequenceResult:
    """Sampling-mode tree verify of one sequence, from its probabilities.

    p_rows [N, V], q_rows [N, V], tok [N] (tok[0] unused), parent [N];
    r_at(c) the acceptance uniform of child c, u_at(j) the draw uniform at
    depth j.
    """
    kids = children_of(parent)
    N = len(kids)
    tokens = np.full(N, -1, dtype=np.int64)
    nodes = np.full(N, -1, dtype=np.int64)
    res = TreeSequenceResult(tokens=tokens, nodes=nodes, n_accepted=0)
    u, depth = 0, 0
    while True:
        f = p_rows[u]
        w_last = None
        kept = None
        for c in kids[u]:
            x = int(tok[c])
            f_x, q_x = f[x], q_rows[u, x]
            r = r_at(c)
            res.accept_margins.append(abs(r - f_x / q_x) if q_x > 0 else float("inf"))
            if accept_test(f_x, q_x, r):
                kept = c
                break
            w = residual_weights(f, q_rows[u])
            S = np.cumsum(w)[-1]
            if not S > 0.0:
                w_last = None          # rounding left nothing: draw from p_u
                break
            w_last = w
            f = w / S
        if kept is not None:
            tokens[depth] = tok[kept]
            nodes[depth] = kept
            depth += 1
            u = kept
            continue
        w = w_last if w_last is not None else p_rows[u]
        v, margin = invert_cdf(w, u_at(depth))
        tokens[depth] = int(v)
        res.n_accepted = depth
        res.sample_margin = float(margin)
        return res


def verify_tree_sequence_greedy(z_rows, tok, parent) -> TreeSequenceResult:
    """Greedy tree verify: follow the child whose token is the target argmax."""
    kids = children_of(parent)
    N = len(kids)
    tokens = np.full(N, -1, dtype=np.int64)
    nodes = np.full(N, -1, dtype=np.int64)
    res = TreeSequenceResult(tokens=tokens, nodes=nodes, n_accepted=0)
    u, depth = 0, 0
    while True:
        a, gap = greedy_argmax(z_rows[u])
        res.greedy_gaps.append(gap)
        match = next((c for c in kids[u] if int(tok[c]) == a), None)
        tokens[depth] = a
        if match is None:
            res.n_accepted = depth
            return res
        nodes[depth] = match
        depth += 1
        u = match


@dataclass
class TreeResult:
    out_tokens: np.ndarray        # [B, N] int64
    nodes: np.ndarray             # [B, N] int64
    n_accepted: np.ndarray        # [B] int64
    z: np.ndarray                 # [B, N, V]
    sequences: list

    def decision_margin(self, b: int, mode: int) -> float:
        s = self.sequences[b]
        if mode == GREEDY:
            return min(s.greedy_gaps)
        return min([s.sample_margin] + list(s.accept_margins))


def verify_tree_from_logits(z, zq, parent, node_tokens, temperature: float, seed: int, mode: int,
                            seq_ids=None) -> TreeResult:
    """Tree verify given target logits z [B, N, V] and draft logits zq."""
    z = np.asarray(z, dtype=np.float64)
    tok = np.asarray(node_tokens, dtype=np.int64)
    B, N, V = z.shape
    seq_ids = np.arange(B) if seq_ids is None else np.asarray(seq_ids)
    out = np.full((B, N), -1, dtype=np.int64)
    nodes = np.full((B, N), -1, dtype=np.int64)
    n_acc = np.zeros(B, dtype=np.int64)
    seqs = []
    if mode == GREEDY:
        for bi in range(B):
            s = verify_tree_sequence_greedy(z[bi], tok[bi], parent)
            out[bi], nodes[bi], n_acc[bi] = s.tokens, s.nodes, s.n_accepted
            seqs.append(s)
        return TreeResult(out, nodes, n_acc, z, seqs)
    p, _ = softmax_t(z, temperature)
    q, _ = softmax_t(np.asarray(zq, dtype=np.float64), temperature)
    for bi in range(B):
        b = int(seq_ids[bi])
        s = verify_tree_sequence_sampling(
            p[bi], q[bi], tok[bi], parent,
            lambda c, b=b: float(philox.accept_uniform(seed, b, c - 1)),
            lambda j, b=b: philox.sample_uniform(seed, b, j))
        out[bi], nodes[bi], n_acc[bi] = s.tokens, s.nodes, s.n_accepted
        seqs.append(s)
    return TreeResult(out, nodes, n_acc, z, seqs)


def verify_tree(hidden, W, parent, node_tokens, draft_logits, temperature: float, seed: int,
                mode: int, seq_ids=None) -> TreeResult:
    """The whole tree verify step: LM-head logits in fp64, then the walk.

    hidden [B, N, d], W [V, d], parent [N], node_tokens [B, N],
    draft_logits [B, N, V] (unused in greedy mode).
    """
    z = lm_head_logits(hidden, W)
    return verify_tree_from_logits(z, draft_logits, parent, node_tokens, temperature, seed, mode,
                                   seq_ids=seq_ids)
