"""The drafter's clustered LM head on the GPU (specdec_cluster_head) against
the fp64 oracle (oracle/cluster_head.py).

Rule: kept clusters exact except where the k-th and (k+1)-th cluster logits
are within 1e-3; tokens exact except at a draw margin below 1e-4 (greedy:
a top-2 logit gap below 1e-3); such rows counted, at most max(1, 0.1 %).
Kept tokens' logits within 5e-3 (the LM head's logit tolerance).
"""
import numpy as np
import pytest
import torch

from oracle import cluster_head as oc
from oracle import verify as ov

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _head(seed, M, d, V, n_c, ragged=True):
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    if ragged:
        cut = torch.sort(torch.randperm(V - 1, generator=g)[:n_c - 1] + 1).values
        starts = torch.cat([torch.tensor([0]), cut, torch.tensor([V])]).int()
    else:
        starts = torch.arange(0, V + 1, V // n_c).int()
    tor = torch.randperm(V, generator=g).int()
    W = (torch.randn(V, d, generator=g) * 0.02).to(torch.bfloat16)
    E = torch.stack([W[starts[c]:starts[c + 1]].float().mean(0) for c in range(n_c)]).to(torch.bfloat16)
    h = torch.randn(M, d, generator=g)
    h = (h / h.pow(2).mean(-1, keepdim=True).sqrt() * 3.0).to(torch.bfloat16)
    return {k: v.to(DEV) for k, v in dict(h=h, E=E, W=W, starts=starts, tor=tor).items()}


def _compare(x, top_k, T, seed, mode, position=0):
    import target_model_verify_gb300 as tv
    M, V = x["h"].shape[0], x["W"].shape[0]
    logits = torch.full((M, V), float("-inf"), device=DEV)
    tok, cl = tv.cluster_head(x["h"], x["E"], x["W"], x["starts"], x["tor"], top_k=top_k,
                              temperature=T, seed=seed, position=position, mode=mode,
                              logits_out=logits)
    torch.cuda.synchronize()
    f = lambda t: t.float().cpu().double().numpy()
    res = oc.cluster_head(f(x["h"]), f(x["E"]), f(x["W"]), x["starts"].cpu().numpy(),
                          x["tor"].cpu().numpy(), top_k, T, seed, mode, position)
    tok, cl, lg = tok.cpu().numpy(), cl.cpu().numpy(), logits.cpu().numpy()
    excused = 0
    thr = 1e-3 if mode == ov.GREEDY else 1e-4
    for m in range(M):
        if not np.array_equal(cl[m], res.clusters[m]):
            assert res.cluster_gaps[m] < 1e-3, (m, cl[m], res.clusters[m])
            excused += 1
            continue
        ids = res.member_ids[m]
        np.testing.assert_allclose(lg[m, ids], res.member_logits[m], rtol=0, atol=5e-3)
        assert np.isinf(np.delete(lg[m], ids)).all()
        if tok[m] != res.tokens[m]:
            assert res.margins[m] < thr, (m, tok[m], res.tokens[m], res.margins[m])
            excused += 1
    assert excused <= max(1, int(0.001 * M)), excused
    return tok


@pytest.mark.parametrize("mode", [ov.SAMPLE, ov.GREEDY])
@pytest.mark.parametrize("M,d,V,n_c,top_k,T", [
    (3, 64, 1000, 16, 1, 1.0),     # ragged clusters, one kept
    (8, 128, 3001, 40, 3, 0.8),    # several kept, odd vocabulary
    (64, 64, 2048, 64, 8, 1.2),    # the most rows and the most kept clusters
    (1, 4096, 500, 5, 5, 1.0),     # every cluster kept: the full head, the widest rows
])
def test_cluster_head_matches_oracle(mode, M, d, V, n_c, top_k, T):
    x = _head(M + V, M, d, V, n_c)
    _compare(x, top_k, T, 7, mode, position=2)


@pytest.mark.parametrize("top_k", [1, 4])
def test_cluster_head_gemma_shape(top_k):
    """Gemma-E2B-shaped head: V = 262,144, d = 1536, 2,048 clusters of 128."""
    x = _head(5, 8, 1536, 262144, 2048, ragged=False)
    _compare(x, top_k, 1.0, 3, ov.SAMPLE)


@pytest.mark.parametrize("mode", [ov.SAMPLE, ov.GREEDY])
def test_cluster_head_more_than_1024_kept_tokens(mode):
    """2,000 kept tokens per row: the draw orders them with the bitonic sort
    (up to 256 it counts ranks)."""
    x = _head(12, 4, 64, 6000, 12, ragged=False)
    _compare(x, 4, 1.0, 9, mode, position=1)


def test_cluster_head_draws_follow_the_uniforms():
    """Different positions and seeds give the oracle's different draws."""
    x = _head(9, 16, 64, 1000, 8)
    a = _compare(x, 2, 1.0, 1, ov.SAMPLE, position=0)
    b = _compare(x, 2, 1.0, 1, ov.SAMPLE, position=1)
    assert (a != b).any()


def test_cluster_head_bad_starts_set_status():
    import target_model_verify_gb300 as tv
    x = _head(10, 2, 64, 1000, 8)
    starts = x["starts"].clone()
    starts[-1] = 5000                 # the last cluster runs past the table
    ws = torch.empty(tv._b.specdec_cluster_head_workspace_size(2, 8, 8, 512), dtype=torch.uint8,
                     device=DEV)
    tv.cluster_head(x["h"], x["E"], x["W"], starts, x["tor"], top_k=8, max_cluster=512,
                    mode=ov.GREEDY, workspace=ws)
    assert tv.read_status(ws) == tv._b.SPECDEC_ERR_INVALID_ARG
    # the next good call on the same workspace clears the status word
    tv.cluster_head(x["h"], x["E"], x["W"], x["starts"], x["tor"], top_k=8, max_cluster=512,
                    mode=ov.GREEDY, workspace=ws)
    assert tv.read_status(ws) == 0


def test_prepared_cluster_head_rereads_hidden():
    """ClusterHeadStep gives cluster_head()'s tokens, and sees hidden refilled in place."""
    import target_model_verify_gb300 as tv
    x = _head(11, 16, 256, 4000, 32)
    step = tv.ClusterHeadStep(x["h"], x["E"], x["W"], x["starts"], x["tor"], top_k=2,
                              temperature=0.9)
    for seed, pos in ((1, 0), (1, 3), (2, 3)):
        tok, cl = tv.cluster_head(x["h"], x["E"], x["W"], x["starts"], x["tor"], top_k=2,
                                  temperature=0.9, seed=seed, position=pos)
        got_tok, got_cl = step(seed, pos)
        assert torch.equal(tok, got_tok) and torch.equal(cl, got_cl)
    x["h"].copy_(x["h"].flip(0))
    want = _compare(x, 2, 0.9, 2, ov.SAMPLE, position=3)
    got, _ = step(2, 3)
    torch.cuda.synchronize()
    assert np.array_equal(got.cpu().numpy(), want)


def test_cluster_head_bad_starts_set_status_one_kept_cluster():
    """The same report on the path where the member kernel selects the one
    kept cluster itself (M <= 8, top_k = 1): the last cluster is made the
    best one for both rows, and its end runs past the table."""
    import target_model_verify_gb300 as tv
    x = _head(13, 2, 64, 1000, 8)
    E = x["E"].clone()
    E[-1] = (x["h"].float().sum(0) * 4.0).to(torch.bfloat16)
    starts = x["starts"].clone()
    starts[-1] = 5000
    ws = torch.empty(tv._b.specdec_cluster_head_workspace_size(2, 8, 1, 4096), dtype=torch.uint8,
                     device=DEV)
    _, cl = tv.cluster_head(x["h"], E, x["W"], starts, x["tor"], top_k=1, max_cluster=4096,
                            mode=ov.GREEDY, workspace=ws)
    assert tv.read_status(ws) == tv._b.SPECDEC_ERR_INVALID_ARG
    assert (cl[:, 0] == 7).all()
    tv.cluster_head(x["h"], x["E"], x["W"], x["starts"], x["tor"], top_k=1, max_cluster=512,
                    mode=ov.GREEDY, workspace=ws)
    assert tv.read_status(ws) == 0
