"""Pins of the fp64 oracle to things other than itself (CPU only).

Each test ties one oracle function to a library routine, a brute-force
computation, an exact enumeration over every 24-bit uniform value, a
statistical bound, or a number printed on "推测解码"
(world.lapla.si/zh/specdec). The mutation tests at the end plant plausible
mistakes in the oracle and check that the pins catch them.
"""
import json
import math
import os
import subprocess
import sys

import numpy as np
import pytest

from oracle import formulas, philox
from oracle import verify as ov

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
N24 = 1 << 24


def _load(name):
    with open(os.path.join(GOLDEN, name), encoding="utf-8") as f:
        return json.load(f)


# ------------------------------------------------------------ Philox --

def test_philox_matches_triton_interpreter():
    """The oracle's Philox4x32-10 equals triton's, word for word."""
    pytest.importorskip("triton")
    rng = np.random.default_rng(123)
    rows = [[0, 0, 0, 0, 0, 0], [0xFFFFFFFF] * 6, [1, 2, 3, 4, 5, 6],
            [0, 0, 0, 0, 0xFFFFFFFF, 0], [0, 0, 1, 0, 42, 0], [7, 3, 0, 0, 1, 1]]
    rows += rng.integers(0, 1 << 32, size=(250, 6), dtype=np.uint64).tolist()
    env = dict(os.environ, TRITON_INTERPRET="1")
    helper = os.path.join(os.path.dirname(__file__), "philox_triton_ref.py")
    proc = subprocess.run([sys.executable, helper], input=json.dumps(rows), env=env,
                          capture_output=True, text=True, timeout=300)
    assert proc.returncode == 0, proc.stderr[-2000:]
    ref = np.array(json.loads(proc.stdout), dtype=np.uint64)
    arr = np.array(rows, dtype=np.uint64)
    got = np.stack(philox.philox4x32_10(*[arr[:, i] for i in range(6)]), axis=1)
    np.testing.assert_array_equal(got, ref)


def test_uniform_maps_ranges_and_lattice():
    seed = 0x1234_5678_9ABC_DEF0
    b = np.repeat(np.arange(200), 50)
    i = np.tile(np.arange(50), 200)
    r = philox.accept_uniform(seed, b, i)
    u = philox.sample_uniform(seed, b, i)
    assert np.all(r > 0) and np.all(r <= 1)
    assert np.all(u >= 0) and np.all(u < 1)
    # both are exact multiples of 2^-24, so they are exact in fp32
    assert np.all(np.float32(r).astype(np.float64) == r)
    assert np.all(np.float32(u).astype(np.float64) == u)
    assert np.all((r * N24) == np.round(r * N24))
    # r and u come from different counters (purpose word) and differ
    assert np.mean(r - u == 2.0 ** -24) < 0.01


def test_uniforms_are_uniform():
    scipy_stats = pytest.importorskip("scipy.stats")
    seed = 987654321
    b = np.arange(100_000)
    u = philox.sample_uniform(seed, b, 0)
    r = philox.accept_uniform(seed, b, 3)
    assert scipy_stats.kstest(u, "uniform").pvalue > 1e-4
    assert scipy_stats.kstest(r, "uniform").pvalue > 1e-4
    # the seed's high word matters (key word 1)
    u2 = philox.sample_uniform(seed + (1 << 32), b[:1000], 0)
    assert np.mean(u2 == u[:1000]) < 0.01


# ---------------------------------------------------------- bf16 / GEMM --

def test_bf16_decoding_known_patterns():
    bits = np.array([0x3F80, 0xBF80, 0x4049, 0x0000, 0x8000, 0x7F7F, 0x0001, 0x7F80, 0x3C00],
                    dtype=np.uint16)
    want = [1.0, -1.0, 3.140625, 0.0, -0.0, 3.3895313892515355e38, 2.0 ** -133,
            math.inf, 2.0 ** -7]
    got = ov.bf16_bits_to_f64(bits)
    for g, w in zip(got, want):
        assert g == w


def test_lm_head_logits_brute_force():
    rng = np.random.default_rng(5)
    h = rng.standard_normal((2, 3, 7))
    W = rng.standard_normal((11, 7))
    z = ov.lm_head_logits(h, W)
    for b in range(2):
        for i in range(3):
            for v in range(11):
                acc = 0.0
                for k in range(7):
                    acc += h[b, i, k] * W[v, k]
                assert abs(z[b, i, v] - acc) < 1e-12


# ------------------------------------------------------------- softmax --

def test_softmax_closed_forms():
    p, lse = ov.softmax_t(np.full((3, 10), 4.25), 0.7)
    np.testing.assert_allclose(p, 0.1, rtol=0, atol=1e-15)
    np.testing.assert_allclose(lse, 4.25 / 0.7 + math.log(10), rtol=1e-15)
    # softmax([0, ln 3]) = (1/4, 3/4)
    p, lse = ov.softmax_t(np.array([0.0, math.log(3.0)]), 1.0)
    np.testing.assert_allclose(p, [0.25, 0.75], rtol=1e-15)
    assert abs(lse - math.log(4.0)) < 1e-15
    # temperature: softmax(T*z / T) == softmax(z / 1)
    rng = np.random.default_rng(1)
    z = rng.standard_normal(50) * 3
    a, _ = ov.softmax_t(z * 0.37, 0.37)
    b_, _ = ov.softmax_t(z, 1.0)
    np.testing.assert_allclose(a, b_, rtol=1e-13)
    # huge logits do not overflow
    p, _ = ov.softmax_t(np.array([1000.0, 1000.0 - math.log(3.0)]), 1.0)
    np.testing.assert_allclose(p, [0.75, 0.25], rtol=1e-13)


# ---------------------------------------------------- exact enumeration --

_LATTICE = {}


def _lattice(kind):
    """Every value the acceptance ("r") or sampling ("u") uniform can take."""
    if kind not in _LATTICE:
        k = np.arange(N24, dtype=np.float64)
        _LATTICE[kind] = (k + 1.0) * 2.0 ** -24 if kind == "r" else k * 2.0 ** -24
    return _LATTICE[kind]


def _accept_law(p_x, q_x):
    """P(keep) over every acceptance uniform r = (k+1)/2^24, k < 2^24."""
    return np.count_nonzero(ov.accept_test(p_x, q_x, _lattice("r"))) / N24


def _draw_law(w, V):
    """Law of invert_cdf(w, u) over every sampling uniform u = k/2^24."""
    v, _ = ov.invert_cdf(w, _lattice("u"))
    return np.bincount(v, minlength=V) / N24


def _position_law(p, q):
    """Law of the token written at one position, given it is reached.

    The draft x is drawn from q; it is kept with the oracle's acceptance law,
    else the oracle's residual draw replaces it. Returns (law, P(keep)).
    """
    V = p.shape[0]
    res = _draw_law(ov.residual_weights(p, q), V)
    law = np.zeros(V)
    keep = 0.0
    for x in range(V):
        if q[x] == 0:
            continue
        a = _accept_law(p[x], q[x])
        keep += q[x] * a
        law[x] += q[x] * a
        law += q[x] * (1.0 - a) * res
    return law, keep


@pytest.mark.slow
def test_enumeration_committed_law_equals_p():
    """V=8, gamma=2: the token written at each position has law p exactly,
    up to the 2^-24 lattice of the uniforms ("推测解码", section
    和大模型写的一样)."""
    rng = np.random.default_rng(2024)
    V = 8
    p = rng.dirichlet(np.ones(V), size=3)
    q = rng.dirichlet(np.ones(V) * 0.7, size=2)
    tol = 4.0 / N24
    law0, keep0 = _position_law(p[0], q[0])
    np.testing.assert_allclose(law0, p[0], rtol=0, atol=tol)
    law1, keep1 = _position_law(p[1], q[1])
    np.testing.assert_allclose(law1, p[1], rtol=0, atol=tol)
    # reaching position 1 happens with probability sum_v min(p0, q0)
    assert abs(keep0 - np.minimum(p[0], q[0]).sum()) < tol
    # the bonus at position 2 is drawn from p2
    bonus = _draw_law(p[2], V)
    np.testing.assert_allclose(bonus, p[2], rtol=0, atol=2.0 / N24)
    # so P(n_accepted = 2, bonus = v) = keep0 * keep1 * p2(v)
    joint = keep0 * keep1 * bonus
    np.testing.assert_allclose(joint, np.minimum(p[0], q[0]).sum()
                               * np.minimum(p[1], q[1]).sum() * p[2], atol=3 * tol)


def test_worked_fragment():
    """The page's 地 / 慢 example: 慢 is kept with probability 0.09/0.33 and
    never comes back as a replacement; 地 takes 0.19/0.24 of the residual."""
    fx = _load("slow_ground_fragment.json")
    p = np.array(fx["p"])
    q = np.array(fx["q"])
    for x in range(3):
        assert abs(_accept_law(p[x], q[x]) - fx["expect"]["accept_prob"][x]) <= 1.0 / N24
    res = _draw_law(ov.residual_weights(p, q), 3)
    assert res[1] == 0.0
    np.testing.assert_allclose(res, fx["expect"]["residual"], atol=2.0 / N24)
    assert abs(formulas.acceptance_rate(p, q) - fx["expect"]["acceptance_rate"]) < 1e-15
    law, _ = _position_law(p, q)
    np.testing.assert_allclose(law, p, atol=4.0 / N24)


def test_invert_cdf_boundaries():
    w = np.array([0.0, 0.25, 0.0, 0.5, 0.25])
    cases = {0.0: 1, 0.2499: 1, 0.25: 3, 0.7499: 3, 0.75: 4, 0.999999: 4}
    for u, want in cases.items():
        v, m = ov.invert_cdf(w, u)
        assert int(v) == want, (u, v)
    _, m = ov.invert_cdf(w, 0.3)
    assert abs(m - 0.05) < 1e-15


# ------------------------------------------------ decision margins --
# The parity rule forgives a token mismatch only where the oracle's decision
# was close: |r - p/q| < 1e-4 for an acceptance test, u within 1e-4 of a CDF
# boundary for a draw, a top-2 logit gap below 1e-3 in greedy mode. A wrong
# margin would silently widen what the rule forgives, so each is pinned to
# values worked out by hand below.

def check_accept_margins():
    """The page's worked fragment ("推测解码", section 和大模型写的一样):
    p = (0.32, 0.09, 0.59), q = (0.13, 0.33, 0.54) over (地, 慢, third).
    Drafts x = (慢, 地) with r = (0.2, 0.5): p/q(慢) = 0.09/0.33 = 3/11, so
    r = 0.2 keeps it with margin 3/11 - 1/5 = 4/55; p/q(地) = 0.32/0.13 =
    32/13 (> 1), so r = 0.5 keeps it with margin 32/13 - 1/2 = 51/26. With
    r = (0.5, .) the first test fails with margin 1/2 - 3/11 = 5/22 and no
    second test is taken. A draft with q(x) = 0 is kept at any r: margin inf."""
    p = np.array([0.32, 0.09, 0.59])
    q = np.array([0.13, 0.33, 0.54])
    rows_p = np.stack([p, p, p])
    rows_q = np.stack([q, q])
    u_at = lambda j: 0.5
    s = ov.verify_sequence_sampling(rows_p, rows_q, np.array([1, 0]), np.array([0.2, 0.5]), u_at)
    assert s.n_accepted == 2
    assert len(s.accept_margins) == 2
    assert abs(s.accept_margins[0] - 4.0 / 55.0) < 1e-15, s.accept_margins
    assert abs(s.accept_margins[1] - 51.0 / 26.0) < 1e-14, s.accept_margins
    s = ov.verify_sequence_sampling(rows_p, rows_q, np.array([1, 0]), np.array([0.5, 0.5]), u_at)
    assert s.n_accepted == 0 and len(s.accept_margins) == 1
    assert abs(s.accept_margins[0] - 5.0 / 22.0) < 1e-15, s.accept_margins
    pz = np.array([[0.5, 0.5, 0.0], [0.5, 0.5, 0.0]])
    qz = np.array([[0.0, 1.0, 0.0]])
    s = ov.verify_sequence_sampling(pz, qz, np.array([0]), np.array([1.0]), u_at)
    assert s.n_accepted == 1 and s.accept_margins == [math.inf]


def check_greedy_gaps():
    """Top-1 minus top-2 logit, by hand: (0.1, 0.7, 0.4, -1) -> token 1,
    gap 0.7 - 0.4 = 0.3; an exact tie (1, 3, 2.5, 3) -> the lower ID 1 and
    gap 0; three equal maxima -> token 0, gap 0; one token -> gap inf. In a
    sequence, the gaps of every row the walk tested are kept in order."""
    v, gap = ov.greedy_argmax([0.1, 0.7, 0.4, -1.0])
    assert v == 1 and abs(gap - 0.3) < 1e-15
    assert ov.greedy_argmax([1.0, 3.0, 2.5, 3.0]) == (1, 0.0)
    assert ov.greedy_argmax([2.0, 2.0, 2.0]) == (0, 0.0)
    assert ov.greedy_argmax([5.0]) == (0, math.inf)
    z = np.array([[0.0, 2.0, 1.5], [4.0, 1.0, 3.0], [0.0, 0.0, 9.0]])
    s = ov.verify_sequence_greedy(z, np.array([1, 2]))
    assert s.n_accepted == 1 and list(s.tokens) == [1, 0, -1]
    np.testing.assert_allclose(s.greedy_gaps, [0.5, 1.0], rtol=0, atol=1e-15)


def check_draw_margins():
    """w = (1, 2, 1): C = (1, 3, 4), S = 4, token 1 owns [1/4, 3/4) of u.
    u = 0.3 sits 0.05 above its lower edge and u = 0.7 0.05 below its upper
    edge (margin 0.05 both times); u = 0.74 is 0.01 from the upper edge;
    u = 0.25 and u = 0.75 sit exactly on a boundary (margin 0, tokens 1 and
    2 under the strict C_v > u S); u = 0.9 is token 2, 0.1 from its upper
    edge; u = 0 is token 0 on its lower edge."""
    w = np.array([1.0, 2.0, 1.0])
    cases = [(0.3, 1, 0.05), (0.7, 1, 0.05), (0.74, 1, 0.01), (0.25, 1, 0.0), (0.75, 2, 0.0),
             (0.9, 2, 0.1), (0.0, 0, 0.0)]
    for u, tok, margin in cases:
        v, m = ov.invert_cdf(w, u)
        assert int(v) == tok, (u, v)
        assert abs(float(m) - margin) < 1e-15, (u, m, margin)


def test_accept_margin_pin():
    check_accept_margins()


def test_greedy_gap_pin():
    check_greedy_gaps()


def test_draw_margin_pin():
    check_draw_margins()


# ------------------------------------------------------------- statistics --

def _run_oracle_rows(p, q, x, seed, gamma):
    """verify_from_logits on B sequences built from per-position p and q."""
    B = x.shape[0]
    with np.errstate(divide="ignore"):
        z = np.broadcast_to(np.log(p), (B,) + p.shape)
        zq = np.broadcast_to(np.log(q), (B,) + q.shape)
    return ov.verify_from_logits(z, zq, x, 1.0, seed, ov.SAMPLE)


def _chi_square_chunk(args):
    """One worker's share: the oracle on `x` under its own seed; returns the
    first-token counts, the kept count and the bonus-token counts."""
    p, q, x, seed = args
    res = _run_oracle_rows(p, q, x, seed=seed, gamma=1)
    V = p.shape[1]
    first = np.bincount(res.out_tokens[:, 0], minlength=V)
    kept = int(np.sum(res.n_accepted == 1))
    bonus = np.bincount(res.out_tokens[res.n_accepted == 1, 1], minlength=V)
    return first, kept, bonus


@pytest.mark.slow
def test_chi_square_and_acceptance_rate():
    """10^6 sequences at V=64, gamma=1 through the whole oracle (Philox draws
    included): the first written token follows p0 (chi-square), the kept
    fraction matches sum_v min(p0, q0) within 4 binomial sigmas, and bonus
    tokens after a kept draft follow p1 ("推测解码", sections 和大模型写的一样
    and 接受率 α). The sequences run as 16 chunks, each under its own seed
    (independent Philox streams), on a pool of spawned worker processes."""
    scipy_stats = pytest.importorskip("scipy.stats")
    import concurrent.futures as cf
    import multiprocessing as mp
    rng = np.random.default_rng(77)
    V, B, chunks = 64, 1_000_000, 16
    p = rng.dirichlet(np.ones(V), size=2)
    q = rng.dirichlet(np.ones(V) * 0.5, size=1)
    x = rng.choice(V, size=(B, 1), p=q[0])
    parts = [(p, q, x[c * (B // chunks):(c + 1) * (B // chunks)], 31337 + c) for c in range(chunks)]
    workers = max(1, min(chunks, len(os.sched_getaffinity(0))))
    env = {k: os.environ.get(k) for k in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS")}
    for k in env:
        os.environ[k] = "1"   # one BLAS thread per worker (inherited by the spawned processes)
    try:
        with cf.ProcessPoolExecutor(max_workers=workers, mp_context=mp.get_context("spawn")) as ex:
            outs = list(ex.map(_chi_square_chunk, parts))
    finally:
        for k, v in env.items():
            if v is None:
                os.environ.pop(k, None)
            else:
                os.environ[k] = v
    counts = sum(o[0] for o in outs)
    kept = sum(o[1] for o in outs)
    c1 = sum(o[2] for o in outs)
    assert counts.sum() == B
    stat = scipy_stats.chisquare(counts, p[0] * B)
    assert stat.pvalue > 1e-4, stat
    alpha = np.minimum(p[0], q[0]).sum()
    assert abs(kept / B - alpha) < 4 * math.sqrt(alpha * (1 - alpha) / B)
    assert scipy_stats.chisquare(c1, p[1] * c1.sum()).pvalue > 1e-4


@pytest.mark.slow
def test_tokens_per_step_matches_printed_value():
    """i.i.d. positions with sum min(p, q) = 0.642 and gamma = 4: the mean
    number of tokens per step is (1 - a^5)/(1 - a) = 2.4887, which the page
    prints as 2.49 (section 接受率 α)."""
    pv = _load("printed_values.json")["tokens_per_read"]
    a, gamma = pv["alpha"], pv["gamma"]
    rng = np.random.default_rng(9)
    V = 16
    base = np.zeros(V)
    base[:8] = rng.dirichlet(np.ones(8))
    other = np.zeros(V)
    other[8:] = rng.dirichlet(np.ones(8))
    q_row = a * base + (1 - a) * other        # overlaps base in mass a exactly
    assert abs(np.minimum(base, q_row).sum() - a) < 1e-12
    p = np.tile(base, (gamma + 1, 1))
    q = np.tile(q_row, (gamma, 1))
    B = 40_000
    x = np.stack([rng.choice(V, size=B, p=q_row) for _ in range(gamma)], axis=1)
    res = _run_oracle_rows(p, q, x, seed=4242, gamma=gamma)
    tokens = res.n_accepted + 1
    want = formulas.expected_tokens_per_step(a, gamma)
    assert round(want, pv["decimals"]) == pv["printed"]
    assert abs(want - (1 - a ** (gamma + 1)) / (1 - a)) < 1e-12
    assert abs(tokens.mean() - want) < 4 * tokens.std() / math.sqrt(B)
    assert tokens.min() >= 1 and tokens.max() <= gamma + 1


def test_speedup_and_arithmetic_printed_values():
    pv = _load("printed_values.json")
    s = pv["speedup"]
    sp = {g: formulas.speedup(s["alpha"], g, s["c"]) for g in range(1, 21)}
    assert max(sp, key=sp.get) == s["best_gamma"]
    assert round(sp[s["best_gamma"]], s["decimals"]) == s["printed"]
    ar = pv["arithmetic_and_speed"]
    extra_arith = formulas.arithmetic_factor(ar["alpha"], ar["gamma"]) - 1
    extra_speed = formulas.speedup(ar["alpha"], ar["gamma"], 0.0) - 1
    assert round(100 * extra_arith) == ar["extra_arithmetic_percent"]
    assert round(100 * extra_speed) == ar["extra_speed_percent"]
    # with alpha = 1 every guess is kept: gamma + 1 tokens per read
    assert formulas.expected_tokens_per_step(1.0, 4) == pv["positions_per_read"]["positions"]


# ---------------------------------------------------------------- greedy --

def _brute_argmax(row):
    best = 0
    for v in range(1, len(row)):
        if row[v] > row[best]:
            best = v
    return best


def test_greedy_equals_argmax_decoding():
    """Greedy verify writes exactly what argmax decoding would: the drafts up
    to the first mismatch, then the target argmax there."""
    rng = np.random.default_rng(3)
    V, gamma = 20, 5
    for trial in range(200):
        z = rng.integers(-3, 4, size=(gamma + 1, V)).astype(np.float64)   # many ties
        amax = [_brute_argmax(z[i]) for i in range(gamma + 1)]
        k = rng.integers(0, gamma + 1)
        x = np.array(amax[:gamma])
        if k < gamma:
            x[k] = (amax[k] + 1 + rng.integers(0, V - 1)) % V
        s = ov.verify_sequence_greedy(z, x)
        assert s.n_accepted == k
        assert list(s.tokens[:k + 1]) == amax[:k + 1]
        assert np.all(s.tokens[k + 1:] == -1)


def test_sampling_invariants():
    """1 <= tokens <= gamma+1; kept prefix equals the drafts; -1 padding; a
    replacement never lands on a token with p <= q ("推测解码", sections
    留下对的，换掉错的 and 通过的规则)."""
    rng = np.random.default_rng(11)
    B, gamma, V = 400, 4, 12
    z = rng.standard_normal((B, gamma + 1, V)) * 2
    zq = z[:, :gamma] + rng.standard_normal((B, gamma, V)) * 1.5
    x = rng.integers(0, V, size=(B, gamma))
    res = ov.verify_from_logits(z, zq, x, 0.8, 99, ov.SAMPLE)
    p, _ = ov.softmax_t(z, 0.8)
    q, _ = ov.softmax_t(zq, 0.8)
    for b in range(B):
        j = res.n_accepted[b]
        assert 0 <= j <= gamma
        assert np.all(res.out_tokens[b, :j] == x[b, :j])
        assert np.all(res.out_tokens[b, j + 1:] == -1)
        t = res.out_tokens[b, j]
        assert 0 <= t < V
        if j < gamma:
            assert p[b, j, t] > q[b, j, t]
            # the rejected draft really failed its test
            r = philox.accept_uniform(99, b, j)
            assert r * q[b, j, x[b, j]] > p[b, j, x[b, j]]


def test_subset_verification_uses_the_same_draws():
    rng = np.random.default_rng(12)
    B, gamma, V = 30, 3, 9
    z = rng.standard_normal((B, gamma + 1, V))
    zq = z[:, :gamma] + rng.standard_normal((B, gamma, V))
    x = rng.integers(0, V, size=(B, gamma))
    full = ov.verify_from_logits(z, zq, x, 1.0, 5, ov.SAMPLE)
    idx = np.array([3, 17, 29])
    sub = ov.verify_from_logits(z[idx], zq[idx], x[idx], 1.0, 5, ov.SAMPLE, seq_ids=idx)
    np.testing.assert_array_equal(sub.out_tokens, full.out_tokens[idx])


# ------------------------------------------------------ planted mistakes --

def test_pins_catch_a_residual_drawn_from_p(monkeypatch):
    """Drawing the replacement from p instead of max(0, p - q) breaks the
    enumeration pin."""
    rng = np.random.default_rng(2024)
    p = rng.dirichlet(np.ones(8))
    q = rng.dirichlet(np.ones(8) * 0.7)
    monkeypatch.setattr(ov, "residual_weights", lambda pr, qr: np.asarray(pr))
    law, _ = _position_law(p, q)
    assert np.abs(law - p).max() > 1e-3


def test_pins_catch_an_inverted_ratio(monkeypatch):
    """Testing r <= q/p instead of r <= p/q breaks the enumeration pin."""
    fx = _load("slow_ground_fragment.json")
    p, q = np.array(fx["p"]), np.array(fx["q"])
    monkeypatch.setattr(ov, "accept_test", lambda px, qx, r: np.asarray(r) * px <= qx)
    law, _ = _position_law(p, q)
    assert np.abs(law - p).max() > 1e-3


def test_pins_catch_a_weak_inequality_in_the_draw(monkeypatch):
    """Choosing the first v with C_v >= t lets a zero-weight token be drawn
    at u = 0 (the page: over-guessed tokens do not come back)."""
    def bad_invert(w, u):
        C = np.cumsum(w)
        v = np.searchsorted(C, np.asarray(u) * C[-1], side="left")
        return v, np.zeros_like(np.asarray(u, dtype=float))
    monkeypatch.setattr(ov, "invert_cdf", bad_invert)
    res = _draw_law(np.array([0.0, 0.5, 0.5]), 3)
    assert res[0] > 0


def test_pins_catch_an_inverted_accept_margin(monkeypatch):
    """A margin measured against q/p instead of p/q fails its pin."""
    monkeypatch.setattr(ov, "accept_margin",
                        lambda px, qx, r: abs(r - qx / px) if px > 0 else math.inf)
    with pytest.raises(AssertionError):
        check_accept_margins()


def test_pins_catch_a_margin_from_one(monkeypatch):
    """A margin taken as the distance of p/q from 1 (ignoring r) fails."""
    monkeypatch.setattr(ov, "accept_margin",
                        lambda px, qx, r: abs(1.0 - px / qx) if qx > 0 else math.inf)
    with pytest.raises(AssertionError):
        check_accept_margins()


def test_pins_catch_a_top1_minus_top3_gap(monkeypatch):
    """A gap to the third-largest logit instead of the second fails."""
    def bad(z_row):
        z_row = np.asarray(z_row, dtype=np.float64)
        v = int(np.argmax(z_row))
        if z_row.shape[0] < 3:
            return v, math.inf
        top3 = np.sort(z_row)[-3:]
        return v, float(top3[2] - top3[0])
    monkeypatch.setattr(ov, "greedy_argmax", bad)
    with pytest.raises(AssertionError):
        check_greedy_gaps()


def test_pins_catch_a_gap_that_skips_ties(monkeypatch):
    """A gap to the next distinct value (so an exact tie reads as a wide
    margin) fails."""
    def bad(z_row):
        z_row = np.asarray(z_row, dtype=np.float64)
        v = int(np.argmax(z_row))
        vals = np.unique(z_row)
        return v, float(vals[-1] - vals[-2]) if vals.shape[0] > 1 else math.inf
    monkeypatch.setattr(ov, "greedy_argmax", bad)
    with pytest.raises(AssertionError):
        check_greedy_gaps()


def test_pins_catch_a_lower_edge_only_draw_margin(monkeypatch):
    """A draw margin measured to the lower edge only fails at u = 0.7."""
    good = ov.invert_cdf

    def bad(w, u):
        C = np.cumsum(np.asarray(w, dtype=np.float64))
        v, _ = good(w, u)
        lo = C[v - 1] if v > 0 else 0.0
        return v, (np.asarray(u) * C[-1] - lo) / C[-1]
    monkeypatch.setattr(ov, "invert_cdf", bad)
    with pytest.raises(AssertionError):
        check_draw_margins()


def test_pins_catch_an_unnormalised_draw_margin(monkeypatch):
    """A draw margin left in units of w (not divided by S) fails."""
    good = ov.invert_cdf

    def bad(w, u):
        v, m = good(w, u)
        return v, m * np.cumsum(np.asarray(w, dtype=np.float64))[-1]
    monkeypatch.setattr(ov, "invert_cdf", bad)
    with pytest.raises(AssertionError):
        check_draw_margins()
