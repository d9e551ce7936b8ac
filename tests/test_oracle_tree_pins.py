"""Pins for the tree-verification oracle (oracle/tree.py), on CPU.

Each ties the oracle to something other than itself:
* a chain-shaped tree reproduces the (separately pinned) chain verify step
  token for token, random draws included;
* exact enumeration with rational arithmetic shows that the rule the
  oracle follows -- siblings tried in order, f -> max(0, f - q)/S after each
  rejection, the draw from the last residual -- makes the first H tokens of
  "this step, then the target model" follow the target's own law
  ("推测解码", sections 不要第二个模型 and 和大模型写的一样);
* the oracle's walk, run on many random draws, matches that exact law
  (chi-square), and fails it when a mistake is planted in it;
* greedy trees follow the target's argmax path.
"""
import itertools
from fractions import Fraction as F

import numpy as np
import pytest

from oracle import tree as ot
from oracle import verify as ov

# ------------------------------------------------ synthetic path models --
# Target P(. | path) and draft Q(. | path) over V = 3 tokens, rational and
# different at every path, so a mistake in which node's distribution is used
# shows in the law.

_PD = [(F(1, 2), F(1, 3), F(1, 6)), (F(1, 5), F(3, 5), F(1, 5)), (F(1, 10), F(3, 10), F(3, 5)),
       (F(2, 7), F(2, 7), F(3, 7)), (F(5, 8), F(1, 8), F(1, 4))]
_QD = [(F(1, 3), F(1, 3), F(1, 3)), (F(3, 5), F(1, 5), F(1, 5)), (F(1, 4), F(1, 2), F(1, 4)),
       (F(1, 8), F(1, 8), F(3, 4)), (F(2, 5), F(1, 10), F(1, 2))]
V3 = 3


def _h(path):
    return sum((i + 3) * (t + 1) for i, t in enumerate(path)) + 7 * len(path)


def P(path):
    return _PD[_h(path) % len(_PD)]


def Q(path):
    return _QD[(_h(path) + 2) % len(_QD)]


# -------------------------------------------------- exact law of the rule --

def _rule_law(kids, tok, u, path):
    """Exact law of the tokens emitted from node u on (tuples -> Fraction)."""
    f = list(P(path))
    q = Q(path)
    law = {}
    stay = F(1)
    for c in kids[u]:
        x = tok[c]
        a = min(F(1), f[x] / q[x])
        for seq, pr in _rule_law(kids, tok, c, path + (x,)).items():
            law[(x,) + seq] = law.get((x,) + seq, F(0)) + stay * a * pr
        stay *= 1 - a
        w = [max(F(0), f[v] - q[v]) for v in range(V3)]
        S = sum(w)
        if S == 0:
            break
        f = [wv / S for wv in w]
    for v in range(V3):
        if f[v]:
            law[(v,)] = law.get((v,), F(0)) + stay * f[v]
    return law


def _paths(parent):
    """Node -> tuple of node indices from the root's first child down to it."""
    out = {0: ()}
    for n in range(1, len(parent)):
        out[n] = out[parent[n]] + (n,)
    return out


def _step_then_target(parent, H):
    """Exact law of the first H tokens: one tree step, then the target.

    Draft tokens are drawn independently: node n's token from Q at the path
    of its parent.
    """
    kids = ot.children_of(parent)
    npath = _paths(parent)
    N = len(parent)
    total = {}
    for assign in itertools.product(range(V3), repeat=N - 1):
        tok = (0,) + assign
        pw = F(1)
        for n in range(1, N):
            pw *= Q(tuple(tok[m] for m in npath[parent[n]]))[tok[n]]
        for seq, pr in _rule_law(kids, tok, 0, ()).items():
            ext = {seq: pr}
            while len(next(iter(ext))) < H:
                nxt = {}
                for s, ps in ext.items():
                    for v in range(V3):
                        nxt[s + (v,)] = nxt.get(s + (v,), F(0)) + ps * P(s)[v]
                ext = nxt
            for s, ps in ext.items():
                s = s[:H]
                total[s] = total.get(s, F(0)) + pw * ps
    return total


def _target_law(H):
    law = {}
    for s in itertools.product(range(V3), repeat=H):
        pr = F(1)
        for k in range(H):
            pr *= P(s[:k])[s[k]]
        law[s] = pr
    return law


TREES = {
    "two siblings": [-1, 0, 0],
    "siblings, first with a child": [-1, 0, 0, 1],
    "three siblings, first with two": [-1, 0, 0, 0, 1, 1],
    "chain of three": [-1, 0, 1, 2],
}


@pytest.mark.parametrize("name", sorted(TREES))
def test_rule_keeps_the_target_law_exactly(name):
    parent = TREES[name]
    depth = max(len(p) for p in _paths(parent).values())
    H = depth + 1
    got = _step_then_target(parent, H)
    want = _target_law(H)
    assert sum(got.values()) == 1
    assert got == want


def test_rule_without_renormalising_breaks_the_law():
    """The exact check has teeth: keep f = max(0, f - q) unnormalised after a
    rejection and the law of the first token is no longer P."""
    parent = TREES["three siblings, first with two"]
    kids = ot.children_of(parent)
    law1 = {v: F(0) for v in range(V3)}
    for assign in itertools.product(range(V3), repeat=len(parent) - 1):
        tok = (0,) + assign
        pw = F(1)
        for n in range(1, len(parent)):
            pw *= Q(())[tok[n]] if parent[n] == 0 else Q((tok[parent[n]],))[tok[n]]
        f = list(P(()))
        q = Q(())
        stay = F(1)
        for c in kids[0]:
            x = tok[c]
            a = min(F(1), f[x] / q[x])
            law1[x] += pw * stay * a
            stay *= 1 - a
            f = [max(F(0), f[v] - q[v]) for v in range(V3)]       # planted: no 1/S
        S = sum(f)
        for v in range(V3):
            if S:
                law1[v] += pw * stay * f[v] / S
    assert any(law1[v] != P(())[v] for v in range(V3))


# ---------------------------------------- the oracle's walk, by sampling --

def _rows_for(parent, tok, Vp):
    """p_rows / q_rows of one draft assignment, from the path models."""
    npath = _paths(parent)
    N = len(parent)
    p = np.zeros((N, Vp))
    q = np.zeros((N, Vp))
    for n in range(N):
        path = tuple(tok[m] for m in npath[n])
        p[n, :V3] = [float(x) for x in P(path)]
        q[n, :V3] = [float(x) for x in Q(path)]
    return p, q


def _sample_first_two(parent, trials, seed):
    """Histogram of the first two tokens of (oracle step, then target)."""
    rng = np.random.default_rng(seed)
    npath = _paths(parent)
    N = len(parent)
    hist = np.zeros((V3, V3))
    for _ in range(trials):
        tok = [0] * N
        for n in range(1, N):
            qq = np.array([float(x) for x in Q(tuple(tok[m] for m in npath[parent[n]]))])
            tok[n] = int(rng.choice(V3, p=qq))
        p_rows, q_rows = _rows_for(parent, tok, V3)
        r = rng.random(N) * (1 - 2 ** -53) + 2 ** -53        # (0, 1]
        uu = rng.random(N)
        s = ot.verify_tree_sequence_sampling(p_rows, q_rows, np.array(tok), parent,
                                             lambda c: r[c], lambda j: uu[j])
        t0 = int(s.tokens[0])
        if s.n_accepted >= 1:
            t1 = int(s.tokens[1])
        else:
            t1 = int(rng.choice(V3, p=[float(x) for x in P((t0,))]))
        hist[t0, t1] += 1
    return hist


def _chi2_ok(hist, law, trials):
    exp = np.array([[float(law[(a, b)]) for b in range(V3)] for a in range(V3)]) * trials
    chi2 = float(((hist - exp) ** 2 / exp).sum())
    # 8 degrees of freedom: P(chi2 > 30) < 2e-4
    return chi2, chi2 < 30.0


@pytest.mark.parametrize("name", ["two siblings", "three siblings, first with two"])
def test_oracle_walk_matches_the_exact_law(name):
    parent = TREES[name]
    trials = 12000
    hist = _sample_first_two(parent, trials, 5)
    chi2, ok = _chi2_ok(hist, _target_law(2), trials)
    assert ok, chi2


def test_walk_with_a_planted_residual_from_p_fails(monkeypatch):
    """Drawing from p instead of the residual after rejections breaks the
    sampled law (the same planted mistake as the chain pins)."""
    parent = TREES["three siblings, first with two"]
    monkeypatch.setattr(ot, "residual_weights", lambda f, q: np.asarray(f))
    trials = 12000
    hist = _sample_first_two(parent, trials, 5)
    chi2, ok = _chi2_ok(hist, _target_law(2), trials)
    assert not ok, chi2


# ------------------------------------------------------ chain equivalence --

def _chain_case(seed, B=24, gamma=4, V=40):
    rng = np.random.default_rng(seed)
    z = rng.normal(size=(B, gamma + 1, V)) * 2.0
    zq = z[:, :gamma] + rng.normal(size=(B, gamma, V)) * 0.7
    x = np.zeros((B, gamma), dtype=np.int64)
    for b in range(B):
        for i in range(gamma):
            e = np.exp(zq[b, i] - zq[b, i].max())
            x[b, i] = rng.choice(V, p=e / e.sum())
    return z, zq, x


@pytest.mark.parametrize("seed", [0, 1, 2])
@pytest.mark.parametrize("mode", [ov.SAMPLE, ov.GREEDY])
def test_chain_shaped_tree_reproduces_the_chain_step(seed, mode):
    z, zq, x = _chain_case(seed)
    B, g1, V = z.shape
    gamma = g1 - 1
    chain = ov.verify_from_logits(z, zq, x, 0.8, 77 + seed, mode)
    parent = [-1] + list(range(gamma))
    tok = np.concatenate([np.zeros((B, 1), dtype=np.int64), x], axis=1)
    zq_t = np.concatenate([zq, np.zeros((B, 1, V))], axis=1)
    tr = ot.verify_tree_from_logits(z, zq_t, parent, tok, 0.8, 77 + seed, mode)
    np.testing.assert_array_equal(tr.out_tokens, chain.out_tokens)
    np.testing.assert_array_equal(tr.n_accepted, chain.n_accepted)
    for b in range(B):
        n = tr.n_accepted[b]
        np.testing.assert_array_equal(tr.nodes[b, :n], np.arange(1, n + 1))
        assert (tr.nodes[b, n:] == -1).all()


# ---------------------------------------------------------------- greedy --

def test_greedy_tree_follows_the_argmax_path():
    """Greedy verify on a tree that holds the target's argmax path among
    decoys emits that path: argmax decoding of the target ("推测解码",
    section 先让小模型猜; maxstudionews.com article 1664)."""
    rng = np.random.default_rng(3)
    V = 30
    # root with children 1 (decoy), 2 (argmax); node 2 with children 3
    # (argmax), 4 (argmax again: the first one counts); node 3 with child 5 (decoy)
    parent = [-1, 0, 0, 2, 2, 3]
    z = rng.normal(size=(1, 6, V))
    a = [int(np.argmax(z[0, n])) for n in range(6)]
    tok = np.zeros((1, 6), dtype=np.int64)
    tok[0, 1] = (a[0] + 1) % V
    tok[0, 2] = a[0]
    tok[0, 3] = a[2]
    tok[0, 4] = a[2]
    tok[0, 5] = (a[3] + 5) % V
    r = ot.verify_tree_from_logits(z, None, parent, tok, 1.0, 0, ov.GREEDY)
    assert r.n_accepted[0] == 2
    assert list(r.nodes[0]) == [2, 3, -1, -1, -1, -1]
    assert list(r.out_tokens[0]) == [a[0], a[2], a[3], -1, -1, -1]


def test_children_of_checks_the_shape():
    assert ot.children_of([-1, 0, 0, 1]) == [[1, 2], [3], [], []]
    for bad in ([0, 0], [-1, 1], [-1, 0, 3, 0], []):
        with pytest.raises(ValueError):
            ot.children_of(bad)
