"""Guard bands around every buffer the library writes.

Each entry point gets its workspace and its output buffers carved out of a
larger allocation whose 4 KB margins before and after are filled with a
byte pattern. After the call, every margin byte must still hold the
pattern: a kernel that strays past the end (or before the start) of its
workspace segment or of an output buffer would overwrite it. The shapes
cover the schedules whose writes are the easiest to get wrong: stream-K
fix-up slots (one token tile split between clusters), the row-owner
epilogue's bulk tensor stores of 32 x 32 logit tiles (clipped at a ragged
vocabulary edge), two token tiles, and vocabulary sizes that are not a
multiple of the 128- or 256-row tiles.
"""
import numpy as np
import pytest
import torch

from oracle import verify as ov
from target_model_verify_gb300 import workloads as wl

from . import parity

pytestmark = pytest.mark.gpu

DEV = "cuda:0"
GUARD = 4096
PATTERN = 0xA5


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from target_model_verify_gb300 import build
    build.build()
    import target_model_verify_gb300  # noqa: F401  (fails loudly if the library is missing)
    torch.cuda.init()


class Guarded:
    """`nbytes` of usable memory with GUARD pattern bytes on either side.

    The usable part starts GUARD bytes into the allocation, so it keeps the
    allocation's alignment (at least 256 bytes)."""

    def __init__(self, nbytes, device=DEV, pinned=False):
        self.n = int(nbytes)
        total = GUARD + self.n + GUARD
        if device == "cpu":
            self.whole = torch.full((total,), PATTERN, dtype=torch.uint8, pin_memory=pinned)
        else:
            self.whole = torch.full((total,), PATTERN, dtype=torch.uint8, device=device)
        self.body = self.whole[GUARD:GUARD + self.n]

    def typed(self, dtype, shape):
        return self.body.view(dtype).view(*shape)

    def check(self, what):
        torch.cuda.synchronize()
        w = self.whole.cpu().numpy()
        before = np.nonzero(w[:GUARD] != PATTERN)[0]
        after = np.nonzero(w[GUARD + self.n:] != PATTERN)[0]
        assert before.size == 0, f"{what}: {before.size} bytes written before the buffer"
        assert after.size == 0, f"{what}: {after.size} bytes written past the end (first at +{after[0]})"


def _out_buffers(B, cols, device=DEV, pinned=False):
    o = Guarded(B * cols * 4, device, pinned)
    n = Guarded(B * 4, device, pinned)
    return o, n


# (B, gamma, d, V): full-size heads and small ragged ones
CHAIN_SHAPES = [
    pytest.param(1, 4, 4096, 128256, id="llama_b1_streamk"),
    pytest.param(64, 4, 4096, 128256, id="llama_b64_two_tiles"),
    pytest.param(256, 4, 4096, 128256, id="llama_b256_row_owner"),
    pytest.param(1, 4, 256, 3001, id="b1_ragged_vocab"),
    pytest.param(30, 4, 128, 2049, id="pairs_streamk_ragged"),
    pytest.param(16, 4, 128, 2049, id="single_ctas_80_rows_ragged"),
    pytest.param(60, 4, 128, 700, id="two_tiles_ragged"),
    pytest.param(40, 4, 64, 3000, id="pairs_208_rows_ragged"),
    pytest.param(22, 4, 128, 2049, id="single_ctas_112_rows_ragged"),
    pytest.param(64, 3, 128, 3000, id="row_owner_streamk_ragged"),
    pytest.param(100, 4, 64, 3000, id="row_owner_two_tiles_ragged"),
]


@pytest.mark.parametrize("mode", [ov.SAMPLE, ov.GREEDY])
@pytest.mark.parametrize("B,gamma,d,V", CHAIN_SHAPES)
def test_verify_stays_inside_its_buffers(B, gamma, d, V, mode):
    import target_model_verify_gb300 as tv
    w = wl.get("llama3_8b_head", B=B, gamma=gamma, d=d, V=V, sigma=0.5)
    inp = wl.generate(w, 3, device=DEV)
    ws = Guarded(tv.workspace_bytes(B, gamma, d, V, torch.bfloat16, mode))
    o, n = _out_buffers(B, gamma + 1)
    dl = inp["draft_logits"] if mode == ov.SAMPLE else None
    out, nacc = tv.verify(inp["hidden"], inp["W_lm"], inp["draft_tokens"], dl, 1.0, 7, mode,
                          out_tokens=o.typed(torch.int32, (B, gamma + 1)),
                          n_accepted=n.typed(torch.int32, (B,)), workspace=ws.body)
    torch.cuda.synchronize()
    assert tv.read_status(ws.body) == 0
    ws.check("workspace")
    o.check("out_tokens")
    n.check("n_accepted")
    parity.check_structure(out.cpu().numpy(), nacc.cpu().numpy(),
                           inp["draft_tokens"].cpu().numpy(), V)


@pytest.mark.parametrize("mode", [ov.SAMPLE, ov.GREEDY])
@pytest.mark.parametrize("B,gamma,d,V", [
    pytest.param(64, 3, 128, 3000, id="row_owner_bulk_stores_ragged"),
    pytest.param(100, 4, 64, 3000, id="row_owner_two_tiles_ragged"),
    pytest.param(30, 4, 128, 2049, id="pairs_streamk_ragged"),
    pytest.param(3, 4, 256, 1000, id="single_ctas_ragged"),
    pytest.param(40, 4, 64, 3000, id="pairs_208_rows_ragged"),
    pytest.param(22, 4, 128, 3000, id="single_ctas_112_rows_ragged"),
])
def test_debug_outputs_stay_inside_their_buffers(B, gamma, d, V, mode):
    """The debug call writes the logits into the caller's buffer (through the
    bulk tensor stores on the row-owner path), plus the log-normalisers,
    p(x), q(x) and argmax: each buffer guarded on both sides."""
    import target_model_verify_gb300 as tv
    w = wl.get("llama3_8b_head", B=B, gamma=gamma, d=d, V=V, sigma=0.5)
    inp = wl.generate(w, 4, device=DEV)
    M = B * (gamma + 1)
    ws = Guarded(tv.workspace_bytes(B, gamma, d, V, torch.bfloat16, mode))
    o, n = _out_buffers(B, gamma + 1)
    bufs = {"logits": Guarded(M * V * 4), "lse_p": Guarded(M * 4), "lse_q": Guarded(B * gamma * 4),
            "p_x": Guarded(B * gamma * 4), "q_x": Guarded(B * gamma * 4),
            "argmax": Guarded(M * 4)}
    shapes = {"logits": (M, V), "lse_p": (M,), "lse_q": (B * gamma,), "p_x": (B * gamma,),
              "q_x": (B * gamma,), "argmax": (M,)}
    dbg = {k: g.typed(torch.int32 if k == "argmax" else torch.float32, shapes[k])
           for k, g in bufs.items()}
    dl = inp["draft_logits"] if mode == ov.SAMPLE else None
    tv.verify(inp["hidden"], inp["W_lm"], inp["draft_tokens"], dl, 1.0, 7, mode,
              out_tokens=o.typed(torch.int32, (B, gamma + 1)),
              n_accepted=n.typed(torch.int32, (B,)), workspace=ws.body, debug=dbg)
    torch.cuda.synchronize()
    assert tv.read_status(ws.body) == 0
    ws.check("workspace")
    o.check("out_tokens")
    n.check("n_accepted")
    for k, g in bufs.items():
        g.check(k)
    # the guarded logits are the real ones
    z = (inp["hidden"].float().reshape(M, d) @ inp["W_lm"].float().T)
    assert (dbg["logits"] - z).abs().max().item() < 5e-3


@pytest.mark.parametrize("mode", [ov.SAMPLE, ov.GREEDY])
@pytest.mark.parametrize("name,over", [
    pytest.param("llama3_8b_head_tree26_b8", {}, id="tree26_b8_full"),
    pytest.param("llama3_8b_head_tree26", {"d": 128, "V": 3001}, id="tree26_ragged"),
    pytest.param("llama3_8b_head_tree26_b8", {"d": 128, "V": 3000}, id="tree26_b8_vector_loads"),
])
def test_tree_stays_inside_its_buffers(name, over, mode):
    import target_model_verify_gb300 as tv
    w = wl.get(name, **over)
    inp = wl.generate_tree(w, 5, device=DEV)
    B, N = w.B, w.N
    ws = Guarded(tv.tree_workspace_bytes(B, N, w.d, w.V, torch.bfloat16, mode))
    o, n = _out_buffers(B, N)
    nodes = Guarded(B * N * 4)
    dl = inp["draft_logits"] if mode == ov.SAMPLE else None
    tv.verify_tree(inp["hidden"], inp["W_lm"], inp["parent"], inp["node_tokens"], dl, 1.0, 3, mode,
                   out_tokens=o.typed(torch.int32, (B, N)),
                   out_nodes=nodes.typed(torch.int32, (B, N)),
                   n_accepted=n.typed(torch.int32, (B,)), workspace=ws.body)
    torch.cuda.synchronize()
    assert tv.read_status(ws.body) == 0
    ws.check("workspace")
    o.check("out_tokens")
    nodes.check("out_nodes")
    n.check("n_accepted")


@pytest.mark.parametrize("B,L,n_new,lens", [
    pytest.param(3, 1100, 5, (1000, 37, 1100), id="splits_ragged_lengths"),
    pytest.param(64, 4096, 5, None, id="llama_b64_l4096"),
])
def test_attention_stays_inside_its_buffers(B, L, n_new, lens):
    import target_model_verify_gb300 as tv
    Hq, Hkv, D = 32, 8, 128
    g = torch.Generator(device=DEV)
    g.manual_seed(9)
    q = torch.randn(B, n_new, Hq, D, generator=g, device=DEV).to(torch.bfloat16)
    k = torch.randn(B, L, Hkv, D, generator=g, device=DEV).to(torch.bfloat16)
    v = torch.randn(B, L, Hkv, D, generator=g, device=DEV).to(torch.bfloat16)
    seq = torch.tensor(lens if lens is not None else [L] * B, dtype=torch.int32, device=DEV)
    ws = Guarded(tv.attention_workspace_bytes(B, n_new, Hq, Hkv, D, L))
    out = Guarded(B * n_new * Hq * D * 4)
    tv.verify_attention(q, k, v, seq, out=out.typed(torch.float32, (B, n_new, Hq, D)),
                        workspace=ws.body)
    torch.cuda.synchronize()
    assert tv.read_status(ws.body) == 0
    ws.check("workspace")
    out.check("out")


@pytest.mark.parametrize("mode", [ov.SAMPLE, ov.GREEDY])
@pytest.mark.parametrize("M,top_k", [(1, 1), (8, 4), (64, 2)])
def test_cluster_head_stays_inside_its_buffers(M, top_k, mode):
    import target_model_verify_gb300 as tv
    from target_model_verify_gb300 import _binding as b
    d, V, n_c = 256, 5003, 40
    g = torch.Generator(device="cpu")
    g.manual_seed(M)
    cut = torch.sort(torch.randperm(V - 1, generator=g)[:n_c - 1] + 1).values
    starts = torch.cat([torch.tensor([0]), cut, torch.tensor([V])]).int()
    tor = torch.randperm(V, generator=g).int()
    W = (torch.randn(V, d, generator=g) * 0.02).to(torch.bfloat16)
    E = torch.stack([W[starts[c]:starts[c + 1]].float().mean(0) for c in range(n_c)]).to(torch.bfloat16)
    h = (torch.randn(M, d, generator=g) * 3.0).to(torch.bfloat16)
    h, E, W, starts, tor = (t.to(DEV) for t in (h, E, W, starts, tor))
    max_cluster = int((starts[1:] - starts[:-1]).max())
    ws = Guarded(b.specdec_cluster_head_workspace_size(M, n_c, top_k, max_cluster))
    tokens = Guarded(M * 4)
    clusters = Guarded(M * top_k * 4)
    logits = Guarded(M * V * 4)
    rc = b.specdec_cluster_head(h.data_ptr(), E.data_ptr(), W.data_ptr(), starts.data_ptr(),
                                tor.data_ptr(), M, d, V, n_c, top_k, max_cluster, 1.0, 11, 2, mode,
                                tokens.body.data_ptr(), clusters.body.data_ptr(),
                                logits.body.data_ptr(), ws.body.data_ptr(), ws.n,
                                torch.cuda.current_stream().cuda_stream)
    assert rc == 0, tv.status_string(rc)
    torch.cuda.synchronize()
    assert tv.read_status(ws.body) == 0
    for what, gb in (("workspace", ws), ("tokens", tokens), ("clusters", clusters),
                     ("logits", logits)):
        gb.check(what)


@pytest.mark.parametrize("pinned", [True, False])
@pytest.mark.parametrize("mode", [ov.SAMPLE, ov.GREEDY])
def test_host_entry_point_stays_inside_its_buffers(mode, pinned):
    """specdec_verify_host: the device workspace (with its staging segments)
    and the host output buffers, pinned (written by the GPU through the
    mapping) or pageable (written by copies)."""
    import target_model_verify_gb300 as tv
    w = wl.get("llama3_8b_head", B=3, gamma=4, d=256, V=3001, sigma=0.5)
    inp = wl.generate(w, 6, device=DEV)
    B, g1 = w.B, w.gamma + 1
    host = {k: (inp[k].cpu().pin_memory() if pinned else inp[k].cpu().clone())
            for k in ("hidden", "draft_tokens", "draft_logits")}
    ws = Guarded(tv.workspace_bytes(B, w.gamma, w.d, w.V, torch.bfloat16, mode, host=True))
    o, n = _out_buffers(B, g1, device="cpu", pinned=pinned)
    out, nacc = tv.verify_host(host["hidden"], inp["W_lm"], host["draft_tokens"],
                               host["draft_logits"] if mode == ov.SAMPLE else None, 1.0, 5, mode,
                               out_tokens=o.typed(torch.int32, (B, g1)),
                               n_accepted=n.typed(torch.int32, (B,)), workspace=ws.body)
    ws.check("workspace")
    o.check("out_tokens (host)")
    n.check("n_accepted (host)")
    dev_out, dev_nacc, _ = parity.run_library(inp, 1.0, 5, mode, debug=False)
    np.testing.assert_array_equal(out.numpy(), dev_out)
    np.testing.assert_array_equal(nacc.numpy(), dev_nacc)


@pytest.mark.parametrize("mode", [ov.SAMPLE, ov.GREEDY])
@pytest.mark.parametrize("B,gamma,d,V,bounds", [
    pytest.param(4, 4, 256, 3001, (0, 1000, 3001), id="two_slices_ragged"),
    pytest.param(64, 3, 128, 3000, (0, 1499, 3000), id="row_owner_slices_ragged"),
    pytest.param(8, 4, 4096, 128256, (0, 32064, 64128, 96192, 128256), id="llama_four_slices"),
    pytest.param(48, 3, 64, 20000, (0, 9000, 20000), id="accept_then_sums_kernels"),
])
def test_vocab_parallel_calls_stay_inside_their_buffers(B, gamma, d, V, bounds, mode):
    """specdec_shard_score / _accept / _draw: every slice's workspace,
    records, sums and outputs guarded, the exchanges done in between."""
    import target_model_verify_gb300 as tv
    from target_model_verify_gb300 import _binding as b
    w = wl.get("llama3_8b_head", B=B, gamma=gamma, d=d, V=V, sigma=0.5)
    inp = wl.generate(w, 8, device=DEV)
    G = len(bounds) - 1
    shards, guards, dls = [], [], []
    for g in range(G):
        v0, v1 = bounds[g], bounds[g + 1]
        sh = tv.VocabShard(inp["W_lm"][v0:v1].contiguous(), v0, V, B, gamma, mode, 1.0)
        gw = Guarded(sh.workspace.numel())
        gr = Guarded(b.specdec_shard_record_bytes(B, gamma))
        gs = Guarded(B * 8)
        sh.workspace, sh.records, sh.sums = gw.body, gr.body, gs.typed(torch.float32, (B, 2))
        shards.append(sh)
        guards.append((gw, gr, gs))
        dls.append(inp["draft_logits"][:, :, v0:v1].contiguous() if mode == ov.SAMPLE else None)
    recs = torch.cat([sh.score(inp["hidden"], inp["draft_tokens"], dls[g]).clone()
                      for g, sh in enumerate(shards)])
    outs = [_out_buffers(B, gamma + 1) for _ in range(G)]
    sums = []
    for g, sh in enumerate(shards):
        o, n = outs[g]
        s = sh.accept(recs, G, inp["draft_tokens"], dls[g], 5,
                      o.typed(torch.int32, (B, gamma + 1)), n.typed(torch.int32, (B,)))
        sums.append(s.clone().reshape(-1))
    if mode == ov.SAMPLE:
        all_sums = torch.cat(sums)
        for g, sh in enumerate(shards):
            sh.draw(all_sums, G, g, dls[g], 5, outs[g][0].typed(torch.int32, (B, gamma + 1)))
    torch.cuda.synchronize()
    for g, (gw, gr, gs) in enumerate(guards):
        assert tv.read_status(gw.body) == 0
        gw.check(f"workspace of slice {g}")
        gr.check(f"records of slice {g}")
        gs.check(f"sums of slice {g}")
        outs[g][0].check(f"out_tokens of slice {g}")
        outs[g][1].check(f"n_accepted of slice {g}")
    out = torch.stack([o.typed(torch.int32, (B, gamma + 1)) for o, _ in outs]).amax(dim=0)
    nacc = outs[0][1].typed(torch.int32, (B,))
    parity.check_structure(out.cpu().numpy(), nacc.cpu().numpy(),
                           inp["draft_tokens"].cpu().numpy(), V)
