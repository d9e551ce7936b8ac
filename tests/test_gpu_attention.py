"""Verify-step attention on the GPU (specdec_verify_attention) against the
fp64 oracle (oracle/attention.py) on the same seeded bf16 inputs.

Tolerance, from the arithmetic: q.k is exact products summed in fp32; the
probabilities enter the value contraction rounded to bf16 (relative error
at most 2^-9 each), so the output, a convex combination of values, moves by
at most 2^-9 * max|v| from that rounding; the bound used is twice that plus
1e-5.
"""
import numpy as np
import pytest
import torch

from oracle import attention as oa

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _inputs(seed, B, n_new, Hq, Hkv, Lmax, lens=None):
    g = torch.Generator(device=DEV)
    g.manual_seed(seed)
    q = torch.randn(B, n_new, Hq, 128, generator=g, device=DEV).to(torch.bfloat16)
    k = torch.randn(B, Lmax, Hkv, 128, generator=g, device=DEV).to(torch.bfloat16)
    v = torch.randn(B, Lmax, Hkv, 128, generator=g, device=DEV).to(torch.bfloat16)
    if lens is None:
        lens = torch.randint(n_new, Lmax + 1, (B,), generator=g, device=DEV)
    lens = torch.as_tensor(lens, device=DEV).to(torch.int32)
    return q, k, v, lens


def _check(q, k, v, lens, out, rows=None):
    f = lambda t: t.detach().float().cpu().double().numpy()
    qs, ks, vs, ls = f(q), f(k), f(v), lens.cpu().numpy()
    rows = list(range(q.shape[0])) if rows is None else rows
    want = oa.verify_attention(qs[rows], ks[rows], vs[rows], ls[rows])
    got = out.detach().cpu().double().numpy()[rows]
    tol = 2 * 2.0 ** -9 * np.abs(vs).max() + 1e-5
    err = np.abs(got - want).max()
    assert err <= tol, (err, tol)
    return err


@pytest.mark.parametrize("B,n_new,Hq,Hkv,Lmax", [
    (1, 5, 32, 8, 300),      # Llama grouping, one sequence: many splits
    (3, 1, 8, 2, 40),        # one new position
    (2, 5, 4, 4, 1000),      # no grouping, ragged last block
    (5, 8, 16, 2, 777),      # 64 query rows per KV head (the limit)
    (64, 5, 32, 8, 256),     # enough KV heads for one split per sequence
    (1, 5, 4, 1, 16400),     # one KV head: 64 splits, merged 32 per lane pass
    (2, 8, 64, 8, 700),      # 64 query rows per KV head: four row tiles, two stages
])
def test_attention_matches_oracle(B, n_new, Hq, Hkv, Lmax):
    import target_model_verify_gb300 as tv
    q, k, v, lens = _inputs(B + Lmax, B, n_new, Hq, Hkv, Lmax)
    out = tv.verify_attention(q, k, v, lens)
    torch.cuda.synchronize()
    _check(q, k, v, lens, out)


def test_attention_edge_lengths():
    """seq_len = n_new (only the new positions) and seq_len = Lmax."""
    import target_model_verify_gb300 as tv
    q, k, v, lens = _inputs(9, 4, 5, 8, 2, 500, lens=[5, 500, 64, 65])
    out = tv.verify_attention(q, k, v, lens)
    torch.cuda.synchronize()
    _check(q, k, v, lens, out)


def test_attention_llama_layer_sampled():
    """Llama-3-8B-shaped layer, B = 4 x 4,096 cached tokens, gamma + 1 = 5."""
    import target_model_verify_gb300 as tv
    q, k, v, lens = _inputs(11, 4, 5, 32, 8, 4096, lens=[4096, 3000, 4096, 17])
    out = tv.verify_attention(q, k, v, lens)
    torch.cuda.synchronize()
    _check(q, k, v, lens, out, rows=[0, 3])


def test_attention_bad_length_sets_status():
    import target_model_verify_gb300 as tv
    q, k, v, lens = _inputs(12, 3, 5, 8, 2, 100, lens=[50, 200, 4])
    ws = torch.empty(tv.attention_workspace_bytes(3, 5, 8, 2, 128, 100), dtype=torch.uint8,
                     device=DEV)
    out = tv.verify_attention(q, k, v, lens, workspace=ws)
    assert tv.read_status(ws) == tv._b.SPECDEC_ERR_INVALID_ARG
    assert float(out[1].abs().max()) == 0.0 and float(out[2].abs().max()) == 0.0
    _check(q, k, v, lens, out, rows=[0])
    lens[1], lens[2] = 100, 5
    tv.verify_attention(q, k, v, lens, workspace=ws)
    assert tv.read_status(ws) == 0
