"""The vocabulary-parallel verify step (specdec_shard_*) on one GPU.

Each test splits W_lm and the draft logits into G vocabulary slices and
runs every slice's three calls on cuda:0 in turn, standing in for the G
GPUs of a tensor-parallel LM head: the all-gathers are concatenations in
rank order and the final max-reduce an elementwise max, which is what the
collectives of verify_vocab_parallel() compute. No slice's kernels wait on
another's (the exchange happens between calls), so running them one after
another on one GPU is the same computation.

Results are checked against the fp64 oracle on the whole vocabulary under
the parity rule of the single-GPU step (tests/parity.py), and against the
single-GPU step itself: tokens and counts must agree except where the
oracle's margin is below the rule's threshold (the draw's position is
split across slices in a different order of additions).
"""
import numpy as np
import pytest
import torch

from oracle import verify as ov
from target_model_verify_gb300 import workloads as wl

from . import parity

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from target_model_verify_gb300 import build
    build.build()
    import target_model_verify_gb300  # noqa: F401  (fails loudly if the library is missing)
    torch.cuda.init()


def _run_sharded(inp, bounds, T, seed, mode):
    """All slices' calls, the exchanges emulated in rank order."""
    import target_model_verify_gb300 as tv
    W, dl = inp["W_lm"], inp["draft_logits"]
    B, g1, _ = inp["hidden"].shape
    V = W.shape[0]
    G = len(bounds) - 1
    shards, dls = [], []
    for g in range(G):
        v0, v1 = bounds[g], bounds[g + 1]
        shards.append(tv.VocabShard(W[v0:v1].contiguous(), v0, V, B, g1 - 1, mode, T))
        dls.append(dl[:, :, v0:v1].contiguous() if mode == ov.SAMPLE else None)
    recs = [sh.score(inp["hidden"], inp["draft_tokens"], dls[g]).clone()
            for g, sh in enumerate(shards)]
    all_rec = torch.cat(recs)
    outs, naccs, sums = [], [], []
    for g, sh in enumerate(shards):
        out = torch.full((B, g1), -7, dtype=torch.int32, device=DEV)
        nacc = torch.full((B,), -7, dtype=torch.int32, device=DEV)
        s = sh.accept(all_rec, G, inp["draft_tokens"], dls[g], seed, out, nacc)
        outs.append(out)
        naccs.append(nacc)
        sums.append(s.clone())
    if mode == ov.SAMPLE:
        all_sums = torch.cat([s.reshape(-1) for s in sums])
        for g, sh in enumerate(shards):
            sh.draw(all_sums, G, g, dls[g], seed, outs[g])
    torch.cuda.synchronize()
    for sh in shards:
        assert tv.read_status(sh.workspace) == 0
    # every slice decided alike: same kept prefix and counts everywhere
    for g in range(1, G):
        assert torch.equal(naccs[g], naccs[0])
    out = torch.stack(outs).amax(dim=0)
    if mode == ov.SAMPLE:
        # exactly one slice drew each sequence's token
        nacc = naccs[0].long()
        drawn = torch.stack([o.gather(1, nacc[:, None])[:, 0] for o in outs])
        assert torch.all((drawn >= 0).sum(dim=0) == 1)
    return out.cpu().numpy(), naccs[0].cpu().numpy()


@pytest.mark.parametrize("mode", [ov.SAMPLE, ov.GREEDY])
@pytest.mark.parametrize("B,gamma,d,V,bounds", [
    (4, 4, 256, 3001, (0, 1000, 2100, 3001)),          # three uneven slices, ragged tails
    (2, 1, 64, 128, (0, 128)),                         # one slice: the single-GPU step
    (30, 4, 128, 2049, (0, 640, 1281, 1900, 2049)),    # four slices, pairs with stream-K
    # (up to B * chunks = 128 the accept call decides and sums in one kernel)
    (64, 3, 128, 3000, (0, 1501, 3000)),               # row-owner tiles on each slice
    (48, 3, 64, 20000, (0, 9000, 20000)),              # B * chunks > 128: accept, then sums
    (4, 3, 64, 3000, tuple(3000 * g // 40 for g in range(41))),   # 40 slices: two lanes' worth
])
def test_sharded_step_matches_the_oracle(B, gamma, d, V, bounds, mode):
    w = wl.get("llama3_8b_head", B=B, gamma=gamma, d=d, V=V, temperature=0.9, sigma=0.5)
    inp = wl.generate(w, 17 + B, device=DEV)
    out, nacc = _run_sharded(inp, bounds, w.temperature, 5, mode)
    res = parity.run_oracle(inp, w.temperature, 5, mode)
    parity.assert_tokens(out, nacc, res, mode)
    parity.check_structure(out, nacc, inp["draft_tokens"].cpu().numpy(), V)
    ref_out, ref_nacc, _ = parity.run_library(inp, w.temperature, 5, mode, debug=False)
    diff = np.nonzero((out != ref_out).any(axis=1) | (nacc != ref_nacc))[0]
    for b in diff:   # only where the oracle itself sat on a boundary
        m = parity.first_difference_margin(res, int(b), out[b], int(nacc[b]), mode)
        assert m < (parity.GREEDY_GAP if mode == ov.GREEDY else parity.SAMPLE_MARGIN), (b, m)


@pytest.mark.parametrize("mode", [ov.SAMPLE, ov.GREEDY])
def test_sharded_llama_head_four_slices(mode):
    """The Llama-3-8B-shaped head split over four GPUs' worth of slices,
    eight sequences, every sequence against the fp64 oracle."""
    w = wl.get("llama3_8b_head", B=8)
    inp = wl.generate(w, 9, device=DEV)
    V = w.V
    bounds = tuple(V * g // 4 for g in range(5))
    out, nacc = _run_sharded(inp, bounds, w.temperature, 3, mode)
    res = parity.run_oracle(inp, w.temperature, 3, mode)
    parity.assert_tokens(out, nacc, res, mode)
    parity.check_structure(out, nacc, inp["draft_tokens"].cpu().numpy(), V)


def test_sharded_token_out_of_range_sets_status():
    import target_model_verify_gb300 as tv
    w = wl.get("llama3_8b_head", B=3, gamma=4, d=128, V=1000, sigma=0.5)
    inp = wl.generate(w, 4, device=DEV)
    bad = dict(inp, draft_tokens=inp["draft_tokens"].clone())
    bad["draft_tokens"][1, 0] = w.V + 5
    bounds = (0, 500, 1000)
    shards = [tv.VocabShard(inp["W_lm"][a:b].contiguous(), a, w.V, w.B, w.gamma, ov.SAMPLE, 1.0)
              for a, b in zip(bounds[:-1], bounds[1:])]
    dls = [inp["draft_logits"][:, :, a:b].contiguous() for a, b in zip(bounds[:-1], bounds[1:])]
    all_rec = torch.cat([sh.score(bad["hidden"], bad["draft_tokens"], dls[g]).clone()
                         for g, sh in enumerate(shards)])
    out = torch.empty(w.B, w.gamma + 1, dtype=torch.int32, device=DEV)
    nacc = torch.empty(w.B, dtype=torch.int32, device=DEV)
    shards[0].accept(all_rec, 2, bad["draft_tokens"], dls[0], 1, out, nacc)
    assert tv.read_status(shards[0].workspace) == tv._b.SPECDEC_ERR_TOKEN_RANGE
    assert int(nacc[1]) == -1 and bool((out[1] == -1).all())
    assert int(nacc[0]) >= 0 and int(nacc[2]) >= 0


def test_sharded_committed_token_law():
    """Distribution preservation through the vocabulary-parallel step: with
    the vocabulary split in four uneven slices, 2 * 10^5 draws (10^4
    identical rows x 20 calls, each its own seed) of the first written token
    follow p0 (chi-square), and the kept fraction is sum min(p0, q0) ("推测解码",
    sections 和大模型写的一样 and 接受率 α). The acceptance test and the draw
    both cross slices: the guesses land in every slice, and the replacement
    is drawn from the slices' running sums."""
    import math
    stats = pytest.importorskip("scipy.stats")
    import target_model_verify_gb300 as tv
    V, d, B, calls = 64, 64, 10000, 20
    bounds = (0, 9, 30, 47, 64)
    w = wl.get("llama3_8b_head", B=1, gamma=1, d=d, V=V, sigma=0.8, w_std=0.3)
    base = wl.generate(w, 123, device=DEV)
    hidden = base["hidden"].expand(B, -1, -1).contiguous()
    dl = base["draft_logits"].expand(B, -1, -1).contiguous()
    res1 = parity.run_oracle(base, 1.0, 0, ov.SAMPLE)
    p0, _ = ov.softmax_t(res1.z[0, 0], 1.0)
    q0, _ = ov.softmax_t(parity.to_f64(base["draft_logits"])[0, 0], 1.0)
    rng = np.random.default_rng(6)
    G = len(bounds) - 1
    shards = [tv.VocabShard(base["W_lm"][a:b].contiguous(), a, V, B, 1, ov.SAMPLE, 1.0)
              for a, b in zip(bounds[:-1], bounds[1:])]
    dls = [dl[:, :, a:b].contiguous() for a, b in zip(bounds[:-1], bounds[1:])]
    counts = np.zeros(V)
    kept = 0
    for c in range(calls):
        x = torch.as_tensor(rng.choice(V, size=(B, 1), p=q0), dtype=torch.int32, device=DEV)
        recs = torch.cat([sh.score(hidden, x, dls[g]).clone() for g, sh in enumerate(shards)])
        outs, sums, nacc = [], [], None
        for g, sh in enumerate(shards):
            o = torch.empty(B, 2, dtype=torch.int32, device=DEV)
            n = torch.empty(B, dtype=torch.int32, device=DEV)
            sums.append(sh.accept(recs, G, x, dls[g], 1000 + c, o, n).clone().reshape(-1))
            outs.append(o)
            nacc = n
        all_sums = torch.cat(sums)
        for g, sh in enumerate(shards):
            sh.draw(all_sums, G, g, dls[g], 1000 + c, outs[g])
        out = torch.stack(outs).amax(dim=0)
        counts += np.bincount(out[:, 0].cpu().numpy(), minlength=V)
        kept += int((nacc == 1).sum())
    n = B * calls
    assert stats.chisquare(counts, p0 * n).pvalue > 1e-4
    alpha = np.minimum(p0, q0).sum()
    assert abs(kept / n - alpha) < 4 * math.sqrt(alpha * (1 - alpha) / n)
