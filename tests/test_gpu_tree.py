"""Tree verification on the GPU (specdec_verify_tree) against the fp64 tree
oracle, on the same seeded inputs.

Rule: out_tokens, out_nodes and n_accepted bit-exact, except for sequences
whose walk took a decision with a margin below 1e-4 (sampling: |r - f/q| or
the draw's distance to a CDF boundary; greedy: a top-2 logit gap below
1e-3), which are counted and must stay under max(1, 0.1 %).
"""
import numpy as np
import pytest
import torch

from oracle import tree as ot
from oracle import verify as ov
from target_model_verify_gb300 import workloads as wl

from .parity import GREEDY_GAP, SAMPLE_MARGIN, to_f64

pytestmark = pytest.mark.gpu
DEV = "cuda"

TREES = {
    "root_only": (-1,),
    "star4": (-1, 0, 0, 0, 0),
    "binary7": (-1, 0, 0, 1, 1, 2, 2),
    "chain5": (-1, 0, 1, 2, 3),
    "wide_root": tuple([-1] + [0] * 12 + [1, 1, 2]),
    "tree26": wl.TREE26,
}


def _run(inp, T, seed, mode):
    import target_model_verify_gb300 as tv
    dl = inp["draft_logits"] if mode == ov.SAMPLE else None
    out, nodes, nacc = tv.verify_tree(inp["hidden"], inp["W_lm"], inp["parent"], inp["node_tokens"],
                                      dl, T, seed, mode)
    torch.cuda.synchronize()
    return out.cpu().numpy(), nodes.cpu().numpy(), nacc.cpu().numpy()


def _oracle(inp, T, seed, mode, rows=None):
    idx = None if rows is None else torch.as_tensor(np.asarray(rows), device=inp["hidden"].device)
    sel = (lambda t: t) if idx is None else (lambda t: t.index_select(0, idx))
    h = to_f64(sel(inp["hidden"]))
    W = to_f64(inp["W_lm"])
    tok = sel(inp["node_tokens"]).cpu().numpy().astype(np.int64)
    dl = to_f64(sel(inp["draft_logits"])) if mode == ov.SAMPLE else None
    return ot.verify_tree(h, W, inp["parent"], tok, dl, T, seed, mode, seq_ids=rows)


def _compare(lib, res, mode, rows=None):
    out, nodes, nacc = lib
    rows = list(range(len(res.sequences))) if rows is None else list(rows)
    thr = GREEDY_GAP if mode == ov.GREEDY else SAMPLE_MARGIN
    exact = excused = 0
    fails = []
    for k, r in enumerate(rows):
        same = (nacc[r] == res.n_accepted[k] and np.array_equal(out[r], res.out_tokens[k])
                and np.array_equal(nodes[r], res.nodes[k]))
        if same:
            exact += 1
        elif res.decision_margin(k, mode) < thr:
            excused += 1
        else:
            fails.append((r, out[r].tolist(), nodes[r].tolist(), int(nacc[r]),
                          res.out_tokens[k].tolist(), res.nodes[k].tolist(), int(res.n_accepted[k])))
    assert not fails, f"tree mismatches beyond the margin rule: {fails[:3]}"
    assert excused <= max(1, int(0.001 * len(rows))), (exact, excused)
    return exact, excused


def _structure(lib, inp):
    """Invariants of any result: a root-down path of kept nodes, their
    tokens, then one in-range token, then -1."""
    out, nodes, nacc = lib
    parent = inp["parent"]
    tok = inp["node_tokens"].cpu().numpy()
    V = inp["W_lm"].shape[0]
    N = len(parent)
    for b in range(out.shape[0]):
        j = int(nacc[b])
        assert 0 <= j <= N - 1
        prev = 0
        for i in range(j):
            n = int(nodes[b, i])
            assert parent[n] == prev
            assert out[b, i] == tok[b, n]
            prev = n
        assert 0 <= out[b, j] < V
        assert (out[b, j + 1:] == -1).all() and (nodes[b, j:] == -1).all()


@pytest.mark.parametrize("mode", [ov.SAMPLE, ov.GREEDY])
@pytest.mark.parametrize("tree", sorted(TREES))
@pytest.mark.parametrize("B,d,V,T", [
    (3, 64, 1000, 1.0),       # ragged vocabulary (1000 = 7*128 + 104), vector loads
    (5, 200, 2049, 0.8),      # V % 4 != 0 (scalar loads in the walk), d % 64 != 0
])
def test_tree_small_shapes(mode, tree, B, d, V, T):
    w = wl.get("llama3_8b_head_tree26", B=B, d=d, V=V, temperature=T, sigma=0.6, tree=TREES[tree])
    inp = wl.generate_tree(w, 100 + B + len(TREES[tree]), device=DEV)
    lib = _run(inp, T, 9, mode)
    _structure(lib, inp)
    _compare(lib, _oracle(inp, T, 9, mode), mode)


@pytest.mark.parametrize("mode", [ov.SAMPLE, ov.GREEDY])
def test_tree_many_sequences_and_seeds(mode):
    """B = 48 on the 26-node tree: several token tiles (M = 1248 rows), many
    walks, three seeds."""
    w = wl.get("llama3_8b_head_tree26_b8", B=48, d=128, V=3001)
    inp = wl.generate_tree(w, 4, device=DEV)
    for seed in (0, 1, 2):
        lib = _run(inp, w.temperature, seed, mode)
        _structure(lib, inp)
        _compare(lib, _oracle(inp, w.temperature, seed, mode), mode)


@pytest.mark.parametrize("mode", [ov.SAMPLE, ov.GREEDY])
def test_tree_llama_head(mode):
    """The Llama-3-8B-shaped head with the 26-node tree, B = 4; sequences 0
    and 3 checked against the oracle, all against the structure."""
    w = wl.get("llama3_8b_head_tree26_b8", B=4)
    inp = wl.generate_tree(w, 7, device=DEV)
    lib = _run(inp, w.temperature, 3, mode)
    _structure(lib, inp)
    rows = [0, 3]
    _compare(lib, _oracle(inp, w.temperature, 3, mode, rows=rows), mode, rows)


def test_chain_shaped_tree_matches_the_chain_entry_point():
    """A chain-shaped tree through specdec_verify_tree gives the chain step's
    tokens (both paths share the random draws)."""
    import target_model_verify_gb300 as tv
    w = wl.get("llama3_8b_head", B=64, d=128, V=2000)
    inp = wl.generate(w, 5, device=DEV)
    gamma = w.gamma
    hid = inp["hidden"]
    tok = torch.cat([torch.zeros(w.B, 1, dtype=torch.int32, device=DEV), inp["draft_tokens"]], 1)
    dl = torch.cat([inp["draft_logits"], torch.zeros_like(inp["draft_logits"][:, :1])], 1)
    parent = tuple([-1] + list(range(gamma)))
    for mode in (ov.SAMPLE, ov.GREEDY):
        out_c, nacc_c = tv.verify(hid, inp["W_lm"], inp["draft_tokens"],
                                  inp["draft_logits"] if mode == ov.SAMPLE else None, 1.0, 11, mode)
        out_t, nodes_t, nacc_t = tv.verify_tree(hid, inp["W_lm"], parent, tok.contiguous(),
                                                dl.contiguous() if mode == ov.SAMPLE else None,
                                                1.0, 11, mode)
        torch.cuda.synchronize()
        same = (out_c == out_t).all(dim=1) & (nacc_c == nacc_t)
        # decisions computed by different kernels may differ only at rounding-level margins
        assert int(same.sum()) >= w.B - 1, (out_c[~same], out_t[~same])


def test_tree_token_out_of_range_sets_status():
    import target_model_verify_gb300 as tv
    w = wl.get("llama3_8b_head_tree26", B=2, d=64, V=1000)
    inp = wl.generate_tree(w, 1, device=DEV)
    inp["node_tokens"][1, 5] = 1000
    ws = tv.alloc_tree_workspace(2, len(w.tree), 64, 1000, device=DEV)
    out, nodes, nacc = tv.verify_tree(inp["hidden"], inp["W_lm"], inp["parent"],
                                      inp["node_tokens"], inp["draft_logits"], 1.0, 0, ov.SAMPLE,
                                      workspace=ws)
    assert tv.read_status(ws) == tv._b.SPECDEC_ERR_TOKEN_RANGE
    nacc, out, nodes = nacc.cpu(), out.cpu(), nodes.cpu()
    assert nacc[1] == -1 and (out[1] == -1).all() and (nodes[1] == -1).all()
    assert nacc[0] >= 0 and out[0, 0] >= 0
    # the next good call on the same workspace clears the status
    inp["node_tokens"][1, 5] = 3
    tv.verify_tree(inp["hidden"], inp["W_lm"], inp["parent"], inp["node_tokens"],
                   inp["draft_logits"], 1.0, 0, ov.SAMPLE, workspace=ws)
    assert tv.read_status(ws) == 0


def test_tree_first_token_law_on_the_gpu():
    """A star of 4 siblings, 20000 identical sequences: the emitted first
    token follows p_root (chi-square), whatever the draws."""
    import target_model_verify_gb300 as tv
    V, d, B = 64, 64, 20000
    w = wl.get("llama3_8b_head_tree26", B=1, d=d, V=V, sigma=1.0, tree=(-1, 0, 0, 0, 0))
    one = wl.generate_tree(w, 3, device=DEV)
    rep = lambda t: t.expand(B, *t.shape[1:]).contiguous()
    g = torch.Generator(device=DEV)
    g.manual_seed(5)
    # independent sibling draws per sequence, from q_root
    q = torch.softmax(one["draft_logits"][0, 0].double(), -1)
    tok = torch.zeros(B, 5, dtype=torch.int32, device=DEV)
    tok[:, 1:] = torch.multinomial(q.float(), B * 4, replacement=True, generator=g).view(B, 4).int()
    out, nodes, nacc = tv.verify_tree(rep(one["hidden"]), one["W_lm"], w.tree, tok,
                                      rep(one["draft_logits"]), 1.0, 12345, ov.SAMPLE)
    first = out[:, 0].long().cpu().numpy()
    p = ov.softmax_t(ov.lm_head_logits(to_f64(one["hidden"][0, 0]), to_f64(one["W_lm"])), 1.0)[0]
    counts = np.bincount(first, minlength=V)
    exp = p * B
    keep = exp >= 5
    chi2 = float((((counts[keep] - exp[keep]) ** 2) / exp[keep]).sum())
    dof = int(keep.sum()) - 1
    assert chi2 < dof + 6 * np.sqrt(2 * dof), (chi2, dof)


def test_tree_step_replays_in_a_cuda_graph():
    """The 26-node tree step on the Llama-3-8B head, captured once in a CUDA
    graph: every replay writes the direct call's tokens, nodes and counts
    (split LM-head tiles get a fresh fix-up tag each replay)."""
    import target_model_verify_gb300 as tv
    w = wl.get("llama3_8b_head_tree26_b8")
    inp = wl.generate_tree(w, 4, device=DEV)
    B, N = w.B, w.N
    ws = tv.alloc_tree_workspace(B, N, w.d, w.V, torch.bfloat16, ov.SAMPLE, device=DEV)

    def bufs():
        return tuple(torch.empty(*s, dtype=torch.int32, device=DEV) for s in ((B, N), (B, N), (B,)))

    def step(o, n, a):
        tv.verify_tree(inp["hidden"], inp["W_lm"], inp["parent"], inp["node_tokens"],
                       inp["draft_logits"], w.temperature, 17, ov.SAMPLE, out_tokens=o,
                       out_nodes=n, n_accepted=a, workspace=ws)

    ref = bufs()
    step(*ref)
    torch.cuda.synchronize()
    got = bufs()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        step(*got)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step(*got)
    for _ in range(3):
        for t in got:
            t.fill_(-7)
        graph.replay()
        torch.cuda.synchronize()
        assert tv.read_status(ws) == 0
        for a, b in zip(got, ref):
            assert torch.equal(a, b)
