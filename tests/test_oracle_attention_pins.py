"""Pins for the verify-step attention oracle (oracle/attention.py), on CPU.

* a library routine: torch's scaled_dot_product_attention in fp64 with an
  explicit mask and the KV heads repeated for the query groups;
* closed forms: identical keys average the visible values; one visible key
  returns its value;
* the causal window: a change after position P leaves the query at P alone,
  a change at or before P moves it (and a planted maskless oracle fails);
* the grouped-query map: query head h reads KV head h // G.
"""
import numpy as np
import pytest
import torch

from oracle import attention as oa


def _case(seed, B=3, n_new=5, Hq=8, Hkv=2, D=16, Lmax=40):
    rng = np.random.default_rng(seed)
    q = rng.normal(size=(B, n_new, Hq, D))
    k = rng.normal(size=(B, Lmax, Hkv, D))
    v = rng.normal(size=(B, Lmax, Hkv, D))
    lens = rng.integers(n_new, Lmax + 1, size=B)
    return q, k, v, lens


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_matches_torch_sdpa_in_fp64(seed):
    q, k, v, lens = _case(seed)
    got = oa.verify_attention(q, k, v, lens)
    B, n_new, Hq, D = q.shape
    G = Hq // k.shape[2]
    for b in range(B):
        L = int(lens[b])
        qb = torch.tensor(q[b]).permute(1, 0, 2)                          # [Hq, n_new, D]
        kb = torch.tensor(k[b, :L]).permute(1, 0, 2).repeat_interleave(G, 0)
        vb = torch.tensor(v[b, :L]).permute(1, 0, 2).repeat_interleave(G, 0)
        pos = torch.arange(L - n_new, L)[:, None]
        mask = torch.arange(L)[None, :] <= pos                            # [n_new, L]
        ref = torch.nn.functional.scaled_dot_product_attention(qb, kb, vb, attn_mask=mask)
        np.testing.assert_allclose(got[b], ref.permute(1, 0, 2).numpy(), rtol=1e-12, atol=1e-12)


def test_identical_keys_average_the_visible_values():
    q, k, v, lens = _case(3)
    k[:] = k[:, :1]                                   # every key equal: uniform weights
    got = oa.verify_attention(q, k, v, lens)
    B, n_new, Hq, D = q.shape
    G = Hq // k.shape[2]
    for b in range(B):
        L = int(lens[b])
        for i in range(n_new):
            P = L - n_new + i
            for h in range(Hq):
                np.testing.assert_allclose(got[b, i, h], v[b, :P + 1, h // G].mean(axis=0),
                                           rtol=1e-12, atol=1e-12)


def test_one_visible_key_returns_its_value():
    q, k, v, _ = _case(4, n_new=1)
    lens = np.ones(q.shape[0], dtype=np.int64)
    got = oa.verify_attention(q, k, v, lens)
    G = q.shape[2] // k.shape[2]
    for h in range(q.shape[2]):
        np.testing.assert_allclose(got[:, 0, h], v[:, 0, h // G], rtol=1e-13)


def test_causal_window():
    q, k, v, lens = _case(5)
    base = oa.verify_attention(q, k, v, lens)
    B, n_new = q.shape[:2]
    b = 1
    L = int(lens[b])
    i = 2
    P = L - n_new + i
    for pos, moves in ((P + 1, False), (L - 1, False), (P, True), (0, True)):
        if pos >= L or (pos > P) == moves:
            continue
        k2 = k.copy()
        k2[b, pos] += 3.0
        v2 = v.copy()
        v2[b, pos] -= 2.0
        got = oa.verify_attention(q, k2, v2, lens)
        changed = not np.allclose(got[b, i], base[b, i])
        assert changed == moves, (pos, P, moves)
        # the other sequences never move
        np.testing.assert_array_equal(got[0], base[0])


def test_a_maskless_attention_fails_the_causal_pin(monkeypatch):
    """Planted mistake: every new position sees all L rows."""
    q, k, v, lens = _case(6)

    def no_mask(q, k, v, seq_lens, scale=None):
        B, n_new, Hq, D = q.shape
        G = Hq // k.shape[2]
        out = np.zeros(q.shape)
        for b in range(B):
            L = int(seq_lens[b])
            for h in range(Hq):
                s = q[b, :, h] @ k[b, :L, h // G].T / np.sqrt(D)
                e = np.exp(s - s.max(axis=1, keepdims=True))
                out[b, :, h] = (e / e.sum(axis=1, keepdims=True)) @ v[b, :L, h // G]
        return out

    monkeypatch.setattr(oa, "verify_attention", no_mask)
    base = oa.verify_attention(q, k, v, lens)
    k2, v2 = k.copy(), v.copy()
    L = int(lens[1])
    k2[1, L - 1] += 3.0
    v2[1, L - 1] -= 2.0
    got = oa.verify_attention(q, k2, v2, lens)
    assert not np.allclose(got[1, 0], base[1, 0])     # the first new position saw the last row


def test_grouped_query_map():
    q, k, v, lens = _case(7, Hq=6, Hkv=3)
    for hk in range(3):
        v[:, :, hk] = hk + 1.0                        # constant value per KV head
    got = oa.verify_attention(q, k, v, lens)
    for h in range(6):
        np.testing.assert_allclose(got[:, :, h], h // 2 + 1.0, rtol=1e-13)
