"""GPU parity: the C-ABI library against the fp64 oracle on seeded inputs.

Every test calls the library through its C ABI (ctypes) on cuda:0 and
compares with the oracle on byte-identical inputs, under the rule stated in
tests/parity.py. Small cases cover several vocabulary tiles, a ragged
vocabulary tail, several token tiles and the degenerate cases; the
full-size workloads are checked on every sequence the oracle can afford and
on structural invariants for the rest.
"""
import math

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


def _gen(name, seed, **over):
    w = wl.get(name, **over)
    return w, wl.generate(w, seed, device=DEV)


def _full_check(w, inp, seed, mode, rows=None):
    T = w.temperature
    out, nacc, dbg = parity.run_library(inp, T, seed, mode)
    res = parity.run_oracle(inp, T, seed, mode, seq_ids=rows)
    rep = parity.assert_tokens(out, nacc, res, mode, rows)
    parity.assert_intermediates(dbg, res, mode, w.B, w.gamma, rows)
    parity.check_structure(out, nacc, inp["draft_tokens"].cpu().numpy(), w.V)
    return out, nacc, rep


# ------------------------------------------------------------ Philox --

def test_philox_uniforms_match_oracle():
    import target_model_verify_gb300 as tv
    from oracle import philox
    seed = 0xDEADBEEF12345678
    for purpose, fn in ((0, philox.accept_uniform), (1, philox.sample_uniform)):
        got = tv.philox_uniforms(seed, 300, 33, purpose, device=DEV).cpu().double().numpy()
        b = np.repeat(np.arange(300), 33).reshape(300, 33)
        i = np.tile(np.arange(33), 300).reshape(300, 33)
        np.testing.assert_array_equal(got, fn(seed, b, i))


# ------------------------------------------------- small, several tiles --

@pytest.mark.parametrize("seed", [0, 1, 2])
def test_tiny_fp32_sampling(seed):
    w, inp = _gen("tiny_fp32", seed)
    _full_check(w, inp, seed, ov.SAMPLE)


@pytest.mark.parametrize("mode", [ov.SAMPLE, ov.GREEDY])
@pytest.mark.parametrize("B,gamma,d,V,T", [
    (3, 4, 256, 1000, 0.8),     # ragged vocabulary tail (1000 = 7*128 + 104)
    (2, 1, 64, 128, 1.0),       # one tile, gamma = 1
    (60, 4, 128, 700, 1.3),     # M = 300: two token tiles of 160
    (1, 32, 192, 2049, 0.5),    # gamma at its maximum, ragged tail
    (7, 3, 8, 300, 1.0),        # d = 8: one zero-padded k-slice
    (30, 4, 200, 2049, 0.9),    # M = 150: cluster pairs with 2-D boxes (d % 64 != 0), odd tile count
    (30, 4, 128, 1920, 1.1),    # M = 150: cluster pairs with 3-D boxes, 15 tiles (one past the end)
    (16, 4, 128, 2049, 1.0),    # M = 80: single CTAs (pairs start at 128-row tiles), 2 slices a stage
    (22, 4, 128, 2049, 0.9),    # M = 110: single CTAs with 112-row tiles, 1 slice a stage
    (40, 4, 64, 3000, 1.0),     # M = 200: one token tile of 208, clusters, q streamed whole
    (64, 3, 128, 2049, 0.9),    # M = 256: tokens on the MMA's M side, stream-K, V % 4 != 0
    (64, 3, 200, 1000, 1.0),    # M = 256, tokens on M with 2-D boxes and a ragged k-slice
    (100, 4, 64, 3001, 1.0),    # M = 500: two token tiles of 256 on M, the last one partial
    (128, 3, 192, 1024, 1.2),   # M = 512: two full token tiles on M, vector logit stores
    (1024, 4, 64, 1000, 1.0),   # M = 5120: twenty token tiles, 1,024 sampler sequences
    (8, 4, 128, 1500, 0.05),    # cold: logits / T spread over hundreds, p nearly one-hot
    (8, 4, 128, 1500, 20.0),    # hot: p and q nearly uniform
])
def test_bf16_small_shapes(mode, B, gamma, d, V, T):
    w = wl.get("llama3_8b_head", B=B, gamma=gamma, d=d, V=V, temperature=T, sigma=0.4)
    inp = wl.generate(w, 11 + B, device=DEV)
    _full_check(w, inp, 5, mode)


@pytest.mark.parametrize("mode", [ov.SAMPLE, ov.GREEDY])
def test_largest_vocabulary(mode):
    """V one below the largest vocabulary the library takes (2^22 - 1:
    1,024 sampler chunks, the last one ragged; 32,768 vocabulary tiles)."""
    w, inp = _gen("llama3_8b_head", 3, B=1, gamma=2, d=64, V=(1 << 22) - 1, w_std=0.3)
    _full_check(w, inp, 5, mode)


def test_fp32_small_shapes_greedy():
    w = wl.get("tiny_fp32", B=5, gamma=3, d=40, V=777)
    inp = wl.generate(w, 3, device=DEV)
    _full_check(w, inp, 9, ov.GREEDY)
    _full_check(w, inp, 9, ov.SAMPLE)


# ------------------------------------------------------ full-size heads --

@pytest.mark.parametrize("seed", [0, 1, 2])
@pytest.mark.parametrize("mode", [ov.SAMPLE, ov.GREEDY])
def test_llama3_8b_head(seed, mode):
    w, inp = _gen("llama3_8b_head", seed)
    _full_check(w, inp, seed, mode)


@pytest.mark.parametrize("gamma", [1, 2, 3, 4, 6, 8])
def test_gemma_e2b_head_gamma_sweep(gamma):
    w, inp = _gen(f"gemma_e2b_head_g{gamma}", 0)
    _full_check(w, inp, 0, ov.SAMPLE)


@pytest.mark.parametrize("name,bound", [
    ("llama3_8b_head", 1.0e-6),       # 16 accumulators (16-row token tile)
    ("llama3_8b_head_b4", 2.0e-6),    # 8 (32-row tile)
    ("gemma_e2b_head_g8", 1.0e-6),    # 16, d = 1536
])
def test_logit_error_with_dealt_accumulators(name, bound):
    """Narrow token tiles deal each tile's k-slices across up to 16 tensor-
    memory accumulators that the epilogue adds in fp32 (lmhead_tc.cu,
    issue_stage). The tensor core's fp32 additions truncate, so one
    accumulator's error grows with the count and size of its additions: a CPU
    model of exact 16-term blocks added with truncation gives 6.5e-6 rms at
    d = 4096 (5.4e-6 measured with one accumulator), 3.4e-7 with 16. The rms
    logit error against fp64 must sit well under the one-accumulator figure."""
    w, inp = _gen(name, 2)
    _, _, dbg = parity.run_library(inp, w.temperature, 2, ov.SAMPLE)
    z = ov.lm_head_logits(parity.to_f64(inp["hidden"]), parity.to_f64(inp["W_lm"]))
    dz = dbg["logits"].view(w.B, w.gamma + 1, w.V).double().cpu().numpy() - z
    rms = float(np.sqrt(np.mean(dz ** 2)))
    print(f"{name}: logit error rms {rms:.2e}, max {np.abs(dz).max():.2e}")
    assert rms < bound, rms


@pytest.mark.parametrize("B", [4, 16, 64, 256])
@pytest.mark.parametrize("mode", [ov.SAMPLE, ov.GREEDY])
def test_llama3_8b_head_batch_sweep(B, mode):
    w, inp = _gen(f"llama3_8b_head_b{B}", 1)
    rows = sorted(set([0, B // 3, B // 2, B - 1]))
    _full_check(w, inp, 3, mode, rows=rows)


@pytest.mark.parametrize("mode", [ov.SAMPLE, ov.GREEDY])
def test_head_70b(mode):
    """70B-shaped head with 5 % near-duplicate hidden rows. Near-duplicate
    rows give near-identical logit rows, not ties inside a row, so the
    argmax near-ties (top-2 gap < 1e-3) that actually arise among the
    checked rows are counted and reported (-s prints them); decisions at
    such ties are the only ones the parity rule lets differ."""
    w, inp = _gen("head_70b_b32_g7", 2)
    rows = [0, 7, 19, 31]
    T = w.temperature
    out, nacc, dbg = parity.run_library(inp, T, 4, mode)
    res = parity.run_oracle(inp, T, 4, mode, seq_ids=rows)
    rep = parity.assert_tokens(out, nacc, res, mode, rows)
    parity.assert_intermediates(dbg, res, mode, w.B, w.gamma, rows)
    parity.check_structure(out, nacc, inp["draft_tokens"].cpu().numpy(), w.V)
    gaps = [ov.greedy_argmax(res.z[k, i])[1] for k in range(len(rows)) for i in range(w.gamma + 1)]
    ties = sum(g < parity.GREEDY_GAP for g in gaps)
    print(f"70B head, {len(gaps)} checked rows: {ties} argmax near-ties (gap < {parity.GREEDY_GAP}), "
          f"smallest gap {min(gaps):.3g}; decisions excused by the margin rule: {rep.excused}")


# ------------------------------------------------------------ behaviour --

def test_deterministic_and_seed_sensitive():
    w, inp = _gen("llama3_8b_head", 0, V=5000, d=512)
    a = parity.run_library(inp, 1.0, 77, ov.SAMPLE)
    b = parity.run_library(inp, 1.0, 77, ov.SAMPLE)
    np.testing.assert_array_equal(a[0], b[0])
    assert torch.equal(a[2]["logits"], b[2]["logits"])
    assert torch.equal(a[2]["lse_p"], b[2]["lse_p"])


def test_all_accepted_and_all_rejected():
    """q == p keeps every draft (bonus written at position gamma); a draft
    with p = 0 is always rejected and never comes back as the replacement."""
    w = wl.get("llama3_8b_head", B=4, gamma=4, d=128, V=600, sigma=0.3)
    inp = wl.generate(w, 21, device=DEV)
    # draft logits equal to the target's own logits: q == p up to bf16 rounding
    z = (inp["hidden"].float() @ inp["W_lm"].float().T)[:, :4]
    inp_eq = dict(inp, draft_logits=z.to(torch.bfloat16).contiguous())
    out, nacc, _ = parity.run_library(inp_eq, 1.0, 3, ov.SAMPLE)
    res = parity.run_oracle(inp_eq, 1.0, 3, ov.SAMPLE)
    parity.assert_tokens(out, nacc, res, ov.SAMPLE)
    # strongly wrong drafts: q concentrated on a token the target gives ~0
    zq = torch.full_like(inp["draft_logits"], -30.0)
    x = torch.argmin(z, dim=-1).int()
    zq.scatter_(2, x.long().unsqueeze(-1), 30.0)
    inp_bad = dict(inp, draft_logits=zq.contiguous(), draft_tokens=x.contiguous())
    out, nacc, _ = parity.run_library(inp_bad, 1.0, 3, ov.SAMPLE)
    assert np.all(nacc == 0)
    assert np.all(out[:, 0] != x[:, 0].cpu().numpy())
    res = parity.run_oracle(inp_bad, 1.0, 3, ov.SAMPLE)
    parity.assert_tokens(out, nacc, res, ov.SAMPLE)


def test_greedy_ignores_temperature_and_draft_logits():
    w, inp = _gen("llama3_8b_head", 4, V=3000, d=256)
    a = parity.run_library(inp, 1.0, 1, ov.GREEDY, debug=False)
    b = parity.run_library(dict(inp, draft_logits=None), 0.3, 99, ov.GREEDY, debug=False)
    np.testing.assert_array_equal(a[0], b[0])


def test_draft_token_out_of_range_sets_status():
    import target_model_verify_gb300 as tv
    w, inp = _gen("llama3_8b_head", 5, B=3, V=1000, d=128)
    bad = inp["draft_tokens"].clone()
    bad[1, 2] = w.V            # out of [0, V)
    ws = tv.alloc_workspace(w.B, w.gamma, w.d, w.V, torch.bfloat16, ov.SAMPLE, device=DEV)
    out, nacc = tv.verify(inp["hidden"], inp["W_lm"], bad, inp["draft_logits"], 1.0, 0,
                          ov.SAMPLE, workspace=ws)
    assert tv.read_status(ws) == tv._b.SPECDEC_ERR_TOKEN_RANGE
    nacc = nacc.cpu().numpy()
    assert nacc[1] == -1 and np.all(out[1].cpu().numpy() == -1)
    assert nacc[0] >= 0 and nacc[2] >= 0
    # the next good call on the same workspace clears the status
    tv.verify(inp["hidden"], inp["W_lm"], inp["draft_tokens"], inp["draft_logits"], 1.0, 0,
              ov.SAMPLE, workspace=ws)
    assert tv.read_status(ws) == 0


def test_empty_batch_is_a_noop():
    import target_model_verify_gb300 as tv
    w = wl.get("llama3_8b_head", B=1, V=256, d=64)
    inp = wl.generate(w, 0, device=DEV)
    h = inp["hidden"][:0]
    out, nacc = tv.verify(h, inp["W_lm"], inp["draft_tokens"][:0], inp["draft_logits"][:0],
                          1.0, 0, ov.SAMPLE,
                          workspace=torch.empty(256, dtype=torch.uint8, device=DEV))
    assert out.shape == (0, 5) and nacc.shape == (0,)


def test_host_entry_point_matches_device_entry_point():
    import target_model_verify_gb300 as tv
    w, inp = _gen("llama3_8b_head", 6, B=2, V=4000, d=256)
    dev_out, dev_nacc, _ = parity.run_library(inp, 1.0, 8, ov.SAMPLE, debug=False)
    host = {k: v.cpu().pin_memory() for k, v in inp.items() if k != "W_lm"}
    out, nacc = tv.verify_host(host["hidden"], inp["W_lm"], host["draft_tokens"],
                               host["draft_logits"], 1.0, 8, ov.SAMPLE)
    np.testing.assert_array_equal(out.numpy(), dev_out)
    np.testing.assert_array_equal(nacc.numpy(), dev_nacc)


@pytest.mark.parametrize("pinned", [True, False])
@pytest.mark.parametrize("mode", [ov.SAMPLE, ov.GREEDY])
def test_host_entry_point_pinned_and_pageable(pinned, mode):
    """Pinned buffers take the mapped path (the GPU reads and writes host
    memory), pageable ones the copy engines; both give the device entry
    point's results, including shapes whose sizes are not multiples of 16
    bytes (B * gamma * 4 = 12 bytes of draft tokens)."""
    import target_model_verify_gb300 as tv
    w, inp = _gen("llama3_8b_head", 11, B=3, gamma=1, V=3001, d=64)
    dev_out, dev_nacc, _ = parity.run_library(inp, 1.0, 5, mode, debug=False)
    host = {k: (v.cpu().pin_memory() if pinned else v.cpu().clone())
            for k, v in inp.items() if k not in ("W_lm", "sigma")}
    out_t = torch.full((w.B, w.gamma + 1), -7, dtype=torch.int32)
    nacc_t = torch.full((w.B,), -7, dtype=torch.int32)
    if pinned:
        out_t, nacc_t = out_t.pin_memory(), nacc_t.pin_memory()
    out, nacc = tv.verify_host(host["hidden"], inp["W_lm"], host["draft_tokens"],
                               host["draft_logits"] if mode == ov.SAMPLE else None, 1.0, 5, mode,
                               out_tokens=out_t, n_accepted=nacc_t)
    np.testing.assert_array_equal(out.numpy(), dev_out)
    np.testing.assert_array_equal(nacc.numpy(), dev_nacc)


def test_prepared_host_step_rereads_its_buffers_each_call():
    """HostStep: bound once; each call re-reads the pinned inputs the caller
    refilled and matches the device entry point for that input and seed."""
    import target_model_verify_gb300 as tv
    w, inp0 = _gen("llama3_8b_head", 6, B=3, V=4000, d=256)
    _, inp1 = _gen("llama3_8b_head", 7, B=3, V=4000, d=256)
    inp1["W_lm"] = inp0["W_lm"]
    host = {k: v.cpu().pin_memory() for k, v in inp0.items() if k not in ("W_lm", "sigma")}
    step = tv.HostStep(host["hidden"], inp0["W_lm"], host["draft_tokens"], host["draft_logits"],
                       1.0, ov.SAMPLE)
    for seed, inp in ((8, inp0), (9, inp1), (8, inp0)):
        for k in host:
            host[k].copy_(inp[k].cpu())
        out, nacc = step(seed)
        dev_out, dev_nacc, _ = parity.run_library(inp, 1.0, seed, ov.SAMPLE, debug=False)
        np.testing.assert_array_equal(out.numpy(), dev_out)
        np.testing.assert_array_equal(nacc.numpy(), dev_nacc)


def test_tokens_per_step_match_the_closed_form():
    """Independent positions with one p and one q everywhere: the number of
    drafts kept follows P(j = k) = alpha^k (1 - alpha) (k < gamma), alpha^gamma
    (k = gamma), so the tokens written per step average (1 - alpha^(gamma+1))
    / (1 - alpha) ("推测解码", section 接受率 α), alpha = sum_v min(p, q)."""
    import target_model_verify_gb300 as tv
    V, d, B, gamma = 64, 64, 20000, 4
    w = wl.get("llama3_8b_head", B=1, gamma=gamma, d=d, V=V, sigma=0.8, w_std=0.3)
    base = wl.generate(w, 5, device=DEV)
    hidden = base["hidden"][:, :1].expand(B, gamma + 1, d).contiguous()
    dl = base["draft_logits"][:, :1].expand(B, gamma, V).contiguous()
    one = {"hidden": base["hidden"][:, :2].contiguous(), "W_lm": base["W_lm"],
           "draft_tokens": base["draft_tokens"][:, :1].contiguous(),
           "draft_logits": base["draft_logits"][:, :1].contiguous()}
    res = parity.run_oracle(one, 1.0, 0, ov.SAMPLE)
    p = ov.softmax_t(res.z[0, 0], 1.0)[0]
    q = ov.softmax_t(parity.to_f64(base["draft_logits"][0, 0]), 1.0)[0]
    alpha = float(np.minimum(p, q).sum())
    g = torch.Generator(device=DEV)
    g.manual_seed(3)
    x = torch.multinomial(torch.as_tensor(q, device=DEV).float(), B * gamma, replacement=True,
                          generator=g).view(B, gamma).int()
    _, nacc = tv.verify(hidden, base["W_lm"], x, dl, 1.0, 77, ov.SAMPLE)
    n = (nacc.double() + 1).cpu().numpy()
    pk = np.array([alpha ** k * (1 - alpha) for k in range(gamma)] + [alpha ** gamma])
    vals = np.arange(1, gamma + 2)
    mean, var = float((pk * vals).sum()), float((pk * vals ** 2).sum() - (pk * vals).sum() ** 2)
    assert abs(mean - (1 - alpha ** (gamma + 1)) / (1 - alpha)) < 1e-12
    assert abs(n.mean() - mean) < 5 * np.sqrt(var / B), (n.mean(), mean, alpha)
    counts = np.bincount(n.astype(int) - 1, minlength=gamma + 1)
    assert np.all(np.abs(counts / B - pk) < 5 * np.sqrt(pk * (1 - pk) / B) + 1e-12)


def test_chi_square_committed_token_law():
    """Distribution preservation on the GPU: over 10^6 draws (10^4 identical
    rows x 100 calls, each call its own seed) the first written token follows
    p0 and the kept fraction is sum min(p0, q0) ("推测解码", sections
    和大模型写的一样 and 接受率 α)."""
    stats = pytest.importorskip("scipy.stats")
    import target_model_verify_gb300 as tv
    V, d, B, calls = 64, 64, 10000, 100
    w = wl.get("llama3_8b_head", B=1, gamma=1, d=d, V=V, sigma=0.8, w_std=0.3)
    base = wl.generate(w, 123, device=DEV)
    hidden = base["hidden"].expand(B, -1, -1).contiguous()
    dl = base["draft_logits"].expand(B, -1, -1).contiguous()
    res1 = parity.run_oracle(base, 1.0, 0, ov.SAMPLE)
    p0, _ = ov.softmax_t(res1.z[0, 0], 1.0)
    q0, _ = ov.softmax_t(parity.to_f64(base["draft_logits"])[0, 0], 1.0)
    rng = np.random.default_rng(5)
    ws = tv.alloc_workspace(B, 1, d, V, torch.bfloat16, ov.SAMPLE, device=DEV)
    counts = np.zeros(V)
    kept = 0
    for c in range(calls):
        x = torch.as_tensor(rng.choice(V, size=(B, 1), p=q0), dtype=torch.int32, device=DEV)
        out, nacc = tv.verify(hidden, base["W_lm"], x, dl, 1.0, 1000 + c, ov.SAMPLE,
                              workspace=ws)
        counts += np.bincount(out[:, 0].cpu().numpy(), minlength=V)
        kept += int((nacc == 1).sum())
    n = B * calls
    assert stats.chisquare(counts, p0 * n).pvalue > 1e-4
    alpha = np.minimum(p0, q0).sum()
    assert abs(kept / n - alpha) < 4 * math.sqrt(alpha * (1 - alpha) / n)


def test_bounded_wait_reports_timeout_and_context_survives():
    """Failure detection without a fault: a wait on a barrier nothing arms
    runs out after its bound, the kernel reports SPECDEC_ERR_TIMEOUT through
    the status word, and the next verify call on the same context is exact."""
    import time

    import target_model_verify_gb300 as tv
    b = tv._b
    n = b.specdec_verify_workspace_size(1, 4, 64, 256, b.SPECDEC_BF16, b.SPECDEC_GREEDY)
    ws = torch.empty(n, dtype=torch.uint8, device=DEV)
    t0 = time.time()
    st = b.specdec_selftest_wait_timeout(ws.data_ptr(), n, torch.cuda.current_stream().cuda_stream)
    dt = time.time() - t0
    assert st == b.SPECDEC_ERR_TIMEOUT
    assert 0.5 < dt < 30
    w, inp = _gen("llama3_8b_head", 8, B=2, V=1500, d=256)
    _full_check(w, inp, 2, ov.SAMPLE)


_GEMMA_PQ = {}


def _gemma_pq():
    """p and q of one Gemma-E2B-shaped position (fp64 oracle), cached."""
    if not _GEMMA_PQ:
        w = wl.get("gemma_e2b_head_g1")
        base = wl.generate(w, 21, device=DEV)
        one = {"hidden": base["hidden"].contiguous(), "W_lm": base["W_lm"],
               "draft_tokens": base["draft_tokens"].contiguous(),
               "draft_logits": base["draft_logits"].contiguous()}
        res = parity.run_oracle(one, 1.0, 0, ov.SAMPLE)
        p = ov.softmax_t(res.z[0, 0], 1.0)[0]
        q = ov.softmax_t(parity.to_f64(base["draft_logits"][0, 0]), 1.0)[0]
        _GEMMA_PQ.update(base=base, p=p, q=q)
    return _GEMMA_PQ


@pytest.mark.parametrize("gamma", [1, 2, 3, 4, 6, 8])
def test_gemma_tokens_per_step_follow_the_closed_form(gamma):
    """Gemma-E2B-shaped head (d = 1536, V = 262,144), gamma swept over
    {1, 2, 3, 4, 6, 8}: with one p and one q at every position and fresh
    draft tokens from q, the mean number of tokens per step is
    (1 - alpha^(gamma+1)) / (1 - alpha), alpha = sum_v min(p, q) ("推测解码",
    section 接受率 α); 4,000 sequences, within 5 standard errors."""
    import target_model_verify_gb300 as tv
    pq = _gemma_pq()
    base, p, q = pq["base"], pq["p"], pq["q"]
    alpha = float(np.minimum(p, q).sum())
    d, V = base["hidden"].shape[-1], base["W_lm"].shape[0]
    B, calls = 500, 8
    hidden = base["hidden"][:, :1].expand(B, gamma + 1, d).contiguous()
    dl = base["draft_logits"][:, :1].expand(B, gamma, V).contiguous()
    ws = tv.alloc_workspace(B, gamma, d, V, torch.bfloat16, ov.SAMPLE, device=DEV)
    g = torch.Generator(device=DEV)
    g.manual_seed(40 + gamma)
    qt = torch.as_tensor(q, device=DEV).float()
    n = []
    for c in range(calls):
        x = torch.multinomial(qt, B * gamma, replacement=True, generator=g).view(B, gamma).int()
        _, nacc = tv.verify(hidden, base["W_lm"], x, dl, 1.0, 500 + c, ov.SAMPLE, workspace=ws)
        n.append((nacc.double() + 1).cpu().numpy())
    n = np.concatenate(n)
    pk = np.array([alpha ** k * (1 - alpha) for k in range(gamma)] + [alpha ** gamma])
    vals = np.arange(1, gamma + 2)
    mean = (1 - alpha ** (gamma + 1)) / (1 - alpha)
    var = float((pk * vals ** 2).sum() - mean ** 2)
    assert 0.5 < alpha < 0.8, alpha
    assert abs(n.mean() - mean) < 5 * np.sqrt(var / n.size), (n.mean(), mean, alpha)


def test_verify_step_replays_in_a_cuda_graph():
    """The step captured once in a CUDA graph gives, on every replay, exactly
    what the same call gives when launched directly -- logits, records and
    tokens. The Llama-3-8B head splits vocabulary tiles between CTAs
    (stream-K), and every replay repeats the same launch parameters, so this
    also checks that a split tile is never finished from the previous
    replay's partial (the workspace's call count keeps the fix-up tags
    distinct)."""
    import target_model_verify_gb300 as tv
    w, inp = _gen("llama3_8b_head", 13)
    B, g1, V = w.B, w.gamma + 1, w.V
    ws = tv.alloc_workspace(B, w.gamma, w.d, V, torch.bfloat16, ov.SAMPLE, device=DEV)

    def buffers():
        return (torch.empty(B, g1, dtype=torch.int32, device=DEV),
                torch.empty(B, dtype=torch.int32, device=DEV),
                {"logits": torch.empty(B * g1, V, device=DEV),
                 "lse_p": torch.empty(B * g1, device=DEV),
                 "lse_q": torch.empty(B * w.gamma, device=DEV),
                 "p_x": torch.empty(B * w.gamma, device=DEV),
                 "q_x": torch.empty(B * w.gamma, device=DEV)})

    def step(out, nacc, dbg):
        tv.verify(inp["hidden"], inp["W_lm"], inp["draft_tokens"], inp["draft_logits"], 1.0, 21,
                  ov.SAMPLE, out_tokens=out, n_accepted=nacc, workspace=ws, debug=dbg)

    ref = buffers()
    step(*ref)
    torch.cuda.synchronize()
    got = buffers()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        step(*got)                      # warm-up on the capture's stream kind
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step(*got)
    for _ in range(3):
        for t in (got[0], got[1], *got[2].values()):
            t.fill_(-7)
        graph.replay()
        torch.cuda.synchronize()
        assert tv.read_status(ws) == 0
        assert torch.equal(got[0], ref[0]) and torch.equal(got[1], ref[1])
        for k in ref[2]:
            assert torch.equal(got[2][k], ref[2][k]), k
