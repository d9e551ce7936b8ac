"""The speculative-decoding verify step, written out plainly in fp64.

Test infrastructure only (see the package docstring).

Notation follows "推测解码" (world.lapla.si/zh/specdec): the small model
guesses gamma tokens x_0..x_{gamma-1}; the large model reads its weights once
and scores gamma + 1 positions (section 先让小模型猜). p is the large model's
probability for a token, q the small model's (section 通过的规则).

Row layout (the reading shared with the CUDA library): hidden[b, i] is the
target state whose next-token distribution p_{b,i} scores draft x_{b,i} for
i < gamma; hidden[b, gamma] is the extra position: the pass that checks
the guesses also scores the position after the last one. draft_logits[b, i]
gives q_{b,i}.

Readings where the pages are silent (each is also the CUDA library's):

* p and q are both softmax at the same temperature T; greedy mode ignores T
  and the draft logits.
* r is in (0, 1] and equality keeps the draft (the page: keep iff r <= p/q).
  The test is evaluated as r*q <= p, which keeps a draft whose q underflowed
  to 0 (the limit of min(1, p/q)).
* The replacement is drawn by inverting the prefix sum of
  w = max(0, p - q) in token-ID order at t = u * S, S being that prefix
  sum's last entry: the token is the smallest v with C_v > t. Strict ">"
  means a token with w = 0 is never drawn (the page: over-guessed tokens do
  not come back). If S == 0 (possible only through rounding) the draw falls
  back to p.
* The bonus token (all gamma drafts kept) is drawn from p at position gamma
  by the same inversion with w = p.
* Greedy argmax takes the lowest token ID among equal maxima.
* out_tokens positions after n_accepted hold -1.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

from . import philox

SAMPLE = 0
GREEDY = 1


# ---------------------------------------------------------------- inputs --

def bf16_bits_to_f64(bits) -> np.ndarray:
    """Exact value of bf16 bit patterns (uint16 array) as float64.

    bf16 is the top half of an IEEE binary32, so placing the 16 bits in the
    high half of a binary32 and widening is exact.
    """
    bits = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return bits.view(np.float32).astype(np.float64)


# ------------------------------------------------------- LM head and p/q --

def lm_head_logits(hidden, W) -> np.ndarray:
    """z[..., v] = sum_k hidden[..., k] * W[v, k], in fp64.

    The LM head multiplies the decoder's hidden state by the vocabulary
    weight matrix ("多詞元預測視覺化指南", section 高效嵌入器).
    """
    hidden = np.asarray(hidden, dtype=np.float64)
    W = np.asarray(W, dtype=np.float64)
    return hidden @ W.T


def softmax_t(logits, T: float):
    """p = softmax(logits / T) over the last axis, and its log-normaliser.

    Returns (p, lse) with lse = log sum_v exp(logits_v / T), computed with
    the maximum subtracted first.
    """
    y = np.asarray(logits, dtype=np.float64) / T
    m = y.max(axis=-1, keepdims=True)
    e = np.exp(y - m)
    s = e.sum(axis=-1, keepdims=True)
    return e / s, (m + np.log(s))[..., 0]


# --------------------------------------------------- the decision rules --

def accept_test(p_x, q_x, r):
    """Keep draft x iff r <= p(x)/q(x), evaluated as r*q(x) <= p(x).

    "推测解码", section 通过的规则: q <= p keeps the draft outright (every
    r <= 1 passes); q > p keeps it with probability p/q.
    """
    return np.asarray(r) * np.asarray(q_x) <= np.asarray(p_x)


def accept_margin(p_x: float, q_x: float, r: float) -> float:
    """Distance of the acceptance uniform r from the threshold p(x)/q(x).

    The keep/reject decision of "推测解码", section 通过的规则, flips only if
    r moves across p/q, so |r - p/q| is how far that decision is from being
    taken the other way. A draft whose q underflowed to 0 is kept for every
    r (the limit of min(1, p/q)), so its margin is infinite.
    """
    if not q_x > 0:
        return float("inf")
    return abs(r - p_x / q_x)


def residual_weights(p_row, q_row) -> np.ndarray:
    """w = max(0, p - q), the part of p that q under-covers.

    "推测解码", section 通过的规则: after a rejection the replacement comes
    from max(0, p - q), renormalised.
    """
    return np.maximum(0.0, np.asarray(p_row) - np.asarray(q_row))


def invert_cdf(w, u):
    """Smallest token v with C_v > u * S, C the prefix sum of w by token ID.

    S is C's last entry. u may be an array; the result then has its shape.
    Returns (token, margin): margin is the distance, in units of u, from u
    to the nearest boundary of the chosen token's interval [C_{v-1}, C_v)/S.
    """
    C = np.cumsum(np.asarray(w, dtype=np.float64))
    S = C[-1]
    u = np.asarray(u, dtype=np.float64)
    t = u * S
    v = np.searchsorted(C, t, side="right")
    v = np.minimum(v, C.shape[0] - 1)
    lo = np.where(v > 0, C[np.maximum(v - 1, 0)], 0.0)
    margin = np.minimum(t - lo, C[v] - t) / S
    return v, margin


def greedy_argmax(z_row):
    """argmax over token IDs with ties to the lowest ID, and the top-2 gap."""
    z_row = np.asarray(z_row, dtype=np.float64)
    v = int(np.argmax(z_row))          # numpy returns the first maximum
    if z_row.shape[0] > 1:
        top2 = np.partition(z_row, -2)[-2:]
        gap = float(top2[1] - top2[0])
    else:
        gap = float("inf")
    return v, gap


# ------------------------------------------------------- one sequence --

@dataclass
class SequenceResult:
    tokens: np.ndarray            # [gamma + 1] int64, -1 padded
    n_accepted: int               # j: drafts kept, 0..gamma
    accept_margins: list = field(default_factory=list)   # |r - p/q| per tested i
    sample_margin: float = float("inf")                  # distance of u to a CDF boundary
    greedy_gaps: list = field(default_factory=list)      # top-1 minus top-2 logit per tested row


def verify_sequence_sampling(p_rows, q_rows, x, r, u_at) -> SequenceResult:
    """Sampling-mode verify of one sequence, from its probabilities.

    p_rows [gamma+1, V], q_rows [gamma, V], x [gamma] draft tokens,
    r [gamma] acceptance uniforms, u_at(j) the sampling uniform for
    position j. Steps in the order of "推测解码", section
    留下对的，换掉错的: check the guesses from the first; keep each that
    passes; at the first that fails, stop, replace it with a token the large
    model draws, and drop every later guess; if all pass, the pass also
    yields the token at position gamma.
    """
    gamma = len(x)
    tokens = np.full(gamma + 1, -1, dtype=np.int64)
    res = SequenceResult(tokens=tokens, n_accepted=gamma)
    j = gamma
    for i in range(gamma):
        p_x = p_rows[i, x[i]]
        q_x = q_rows[i, x[i]]
        res.accept_margins.append(accept_margin(p_x, q_x, r[i]))
        if accept_test(p_x, q_x, r[i]):
            tokens[i] = x[i]
        else:
            j = i
            break
    if j < gamma:
        w = residual_weights(p_rows[j], q_rows[j])
        if not np.cumsum(w)[-1] > 0.0:
            w = p_rows[j]
    else:
        w = p_rows[gamma]
    v, margin = invert_cdf(w, u_at(j))
    tokens[j] = int(v)
    res.n_accepted = j
    res.sample_margin = float(margin)
    return res


def verify_sequence_greedy(z_rows, x) -> SequenceResult:
    """Greedy-mode verify: keep drafts while each equals the target argmax.

    maxstudionews.com article 1664 (the verify paragraph): a candidate that
    matches the large model's prediction is kept, otherwise decoding rolls
    back to the first divergence, where the large model's own token stands.
    If every draft matches, the argmax at position gamma is the extra token.
    """
    gamma = len(x)
    tokens = np.full(gamma + 1, -1, dtype=np.int64)
    res = SequenceResult(tokens=tokens, n_accepted=gamma)
    for i in range(gamma + 1):
        a, gap = greedy_argmax(z_rows[i])
        res.greedy_gaps.append(gap)
        if i == gamma or x[i] != a:
            tokens[i] = a
            res.n_accepted = i
            break
        tokens[i] = x[i]
    return res


# ----------------------------------------------------------- the step --

@dataclass
class VerifyResult:
    out_tokens: np.ndarray        # [B, gamma+1] int64
    n_accepted: np.ndarray        # [B] int64
    z: np.ndarray | None          # [B, gamma+1, V] target logits (fp64)
    lse_p: np.ndarray | None      # [B, gamma+1]   log-normaliser of z/T
    lse_q: np.ndarray | None      # [B, gamma]     log-normaliser of zq/T
    p_x: np.ndarray | None        # [B, gamma]     p_i(x_i)
    q_x: np.ndarray | None        # [B, gamma]     q_i(x_i)
    sequences: list               # SequenceResult per sequence (margins)

    def decision_margin(self, b: int, mode: int) -> float:
        """Smallest margin among the decisions sequence b actually took."""
        s = self.sequences[b]
        if mode == GREEDY:
            return min(s.greedy_gaps)
        return min([s.sample_margin] + list(s.accept_margins))


def verify_from_logits(z, zq, draft_tokens, temperature: float, seed: int, mode: int,
                       seq_ids=None) -> VerifyResult:
    """Verify step given target logits z [B, gamma+1, V] and draft logits zq.

    seq_ids gives the sequence index b used for the Philox counters of each
    row of z (default 0..B-1); it lets a caller verify a subset of a larger
    batch with the same random draws the full batch would use.
    """
    z = np.asarray(z, dtype=np.float64)
    x = np.asarray(draft_tokens, dtype=np.int64)
    B, g1, V = z.shape
    gamma = g1 - 1
    seq_ids = np.arange(B) if seq_ids is None else np.asarray(seq_ids)
    out = np.full((B, g1), -1, dtype=np.int64)
    n_acc = np.zeros(B, dtype=np.int64)
    seqs = []
    if mode == GREEDY:
        for bi in range(B):
            s = verify_sequence_greedy(z[bi], x[bi])
            out[bi], n_acc[bi] = s.tokens, s.n_accepted
            seqs.append(s)
        return VerifyResult(out, n_acc, z, None, None, None, None, seqs)

    zq = np.asarray(zq, dtype=np.float64)
    p, lse_p = softmax_t(z, temperature)
    q, lse_q = softmax_t(zq, temperature)
    rows = np.arange(gamma)
    p_x = np.stack([p[bi, rows, x[bi]] for bi in range(B)]) if gamma else np.zeros((B, 0))
    q_x = np.stack([q[bi, rows, x[bi]] for bi in range(B)]) if gamma else np.zeros((B, 0))
    for bi in range(B):
        b = int(seq_ids[bi])
        r = philox.accept_uniform(seed, b, np.arange(gamma))
        s = verify_sequence_sampling(p[bi], q[bi], x[bi], r,
                                     lambda j, b=b: philox.sample_uniform(seed, b, j))
        out[bi], n_acc[bi] = s.tokens, s.n_accepted
        seqs.append(s)
    return VerifyResult(out, n_acc, z, lse_p, lse_q, p_x, q_x, seqs)


def verify(hidden, W, draft_tokens, draft_logits, temperature: float, seed: int,
           mode: int, seq_ids=None) -> VerifyResult:
    """The whole verify step: LM-head logits in fp64, then the rule.

    hidden [B, gamma+1, d], W [V, d], draft_tokens [B, gamma],
    draft_logits [B, gamma, V] (unused in greedy mode), all as exact fp64
    values of the inputs the library receives.
    """
    z = lm_head_logits(hidden, W)
    return verify_from_logits(z, draft_logits, draft_tokens, temperature, seed, mode,
                              seq_ids=seq_ids)
