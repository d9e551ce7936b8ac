"""Seeded synthetic inputs for the verify step.

This module makes inputs only. It holds none of the verify step's own
arithmetic (no target softmax, no acceptance test, no residual draw), so the
CUDA library and the CPU oracle can both be fed from it without sharing
code. It does play the small model: draft logits are W (h + sigma * eps)
rounded to the input dtype, and the draft tokens are drawn from
softmax(draft_logits / T) with this module's own seeded torch generator.

The shapes follow the LM heads the pages name: a Llama-3-8B-shaped head
(d = 4096, V = 128256; "推测解码", section 一次一个词元), a Gemma-E2B-shaped
head (d = 1536, V = 262144; "多詞元預測視覺化指南", sections Gemma 4 的 MTP
and 高效嵌入器), and a 70B-shaped head (d = 8192) for the Chinchilla-70B
pairing (section 快多少). No trained weights exist here: W ~ N(0, w_std^2)
and the hidden rows are Gaussian with unit RMS.
"""
from __future__ import annotations

from dataclasses import dataclass, replace

import torch

SAMPLE = 0
GREEDY = 1


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    gamma: int
    d: int
    V: int
    dtype: str = "bf16"              # "bf16" or "fp32" for hidden, W and draft logits
    temperature: float = 1.0
    w_std: float = 0.02
    unit_rms: bool = True            # hidden rows scaled to RMS 1 (else N(0, 1))
    sigma: float = 0.7               # draft noise, or the low end of U[lo, hi] per sequence
    sigma_hi: float | None = None    # set: sigma_b ~ U[sigma, sigma_hi] per sequence
    near_dup_frac: float = 0.0       # share of hidden rows replaced by a near copy of another
    tree: tuple | None = None        # token tree (parent of every node) instead of a chain

    @property
    def N(self) -> int:
        """Rows per sequence: gamma + 1 positions, or the tree's nodes."""
        return len(self.tree) if self.tree is not None else self.gamma + 1

    @property
    def n_draft(self) -> int:
        """Draft-logit rows per sequence (every tree node has one)."""
        return len(self.tree) if self.tree is not None else self.gamma

    @property
    def M(self) -> int:
        return self.B * self.N

    @property
    def elem_bytes(self) -> int:
        return 2 if self.dtype == "bf16" else 4

    def algorithmic_bytes(self, mode: int = SAMPLE) -> int:
        """W + hidden + draft tokens (+ draft logits in sampling mode)."""
        e = self.elem_bytes
        n_tok = self.B * (self.N - 1 if self.tree is not None else self.gamma)
        n = self.V * self.d * e + self.M * self.d * e + n_tok * 4
        if mode == SAMPLE:
            n += self.B * self.n_draft * self.V * e
        return n

    def flops(self) -> int:
        return 2 * self.M * self.V * self.d


# Draft-noise sigmas give sum_v min(p, q) near 0.65 (Llama head) and 0.64
# (Gemma head) for these weight and hidden scales (set by bisection on the
# mean overlap of the two softmaxes on sample rows).
_LLAMA_SIGMA = 0.71
_GEMMA_SIGMA = 1.19

WORKLOADS: dict[str, Workload] = {}


def _add(w: Workload) -> None:
    WORKLOADS[w.name] = w


_add(Workload("tiny_fp32", B=1, gamma=4, d=64, V=512, dtype="fp32", w_std=0.125,
              unit_rms=False, sigma=0.5))
_add(Workload("llama3_8b_head", B=1, gamma=4, d=4096, V=128256, sigma=_LLAMA_SIGMA))
for _g in (1, 2, 3, 4, 6, 8):
    _add(Workload(f"gemma_e2b_head_g{_g}", B=1, gamma=_g, d=1536, V=262144, sigma=_GEMMA_SIGMA))
for _b in (1, 4, 16, 64, 256):
    _add(Workload(f"llama3_8b_head_b{_b}", B=_b, gamma=4, d=4096, V=128256,
                  sigma=0.2, sigma_hi=1.5))
_add(Workload("head_70b_b32_g7", B=32, gamma=7, d=8192, V=128256, temperature=0.7,
              w_std=0.015, sigma=0.3, sigma_hi=1.0, near_dup_frac=0.05))

# A static token tree of 26 nodes, depth 5 (4, 7, 7, 5, 2 nodes per level):
# widest near the root, where the guesses are least certain, in the manner of
# the Medusa / EAGLE trees ("推测解码", section 不要第二个模型).
TREE26 = (-1, 0, 0, 0, 0, 1, 1, 1, 2, 2, 3, 4, 5, 5, 6, 7, 8, 10, 11, 12, 12, 13, 14, 16, 19, 21)
_add(Workload("llama3_8b_head_tree26", B=1, gamma=1, d=4096, V=128256, sigma=_LLAMA_SIGMA,
              tree=TREE26))
_add(Workload("llama3_8b_head_tree26_b8", B=8, gamma=1, d=4096, V=128256, sigma=0.2,
              sigma_hi=1.5, tree=TREE26))


def get(name: str, **overrides) -> Workload:
    """A named workload, optionally with fields replaced (e.g. smaller V)."""
    return replace(WORKLOADS[name], **overrides)


def _torch_dtype(w: Workload):
    return torch.bfloat16 if w.dtype == "bf16" else torch.float32


@torch.no_grad()
def generate(w: Workload, seed: int, device="cpu") -> dict:
    """Inputs of one verify step, as contiguous tensors on `device`.

    Returns hidden [B, gamma+1, d], W_lm [V, d], draft_logits [B, gamma, V]
    (all in the workload's dtype), draft_tokens [B, gamma] int32 and the
    per-sequence draft noise sigma [B] (float32).
    """
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    dt = _torch_dtype(w)
    B, g1, d, V = w.B, w.gamma + 1, w.d, w.V

    W = (torch.randn(V, d, generator=g, device=device) * w.w_std).to(dt)
    h = torch.randn(B, g1, d, generator=g, device=device)
    if w.unit_rms:
        h = h / h.pow(2).mean(dim=-1, keepdim=True).sqrt()
    if w.near_dup_frac > 0:
        M = B * g1
        n_dup = max(1, round(w.near_dup_frac * M))
        perm = torch.randperm(M, generator=g, device=device)
        dst, src = perm[:n_dup], perm[n_dup:2 * n_dup]
        flat = h.reshape(M, d)
        rms = flat[src].pow(2).mean(dim=-1, keepdim=True).sqrt()
        noise = torch.randn(n_dup, d, generator=g, device=device)
        flat[dst] = flat[src] + 1e-3 * rms * noise
        h = flat.reshape(B, g1, d)
    hidden = h.to(dt)

    if w.sigma_hi is None:
        sigma = torch.full((B,), float(w.sigma), device=device)
    else:
        sigma = w.sigma + (w.sigma_hi - w.sigma) * torch.rand(B, generator=g, device=device)
    eps = torch.randn(B, w.gamma, d, generator=g, device=device)
    h_draft = hidden[:, :w.gamma].float() + sigma[:, None, None] * eps

    Wf = W.float()
    rows = h_draft.reshape(B * w.gamma, d)
    dl = torch.empty(B * w.gamma, V, dtype=dt, device=device)
    chunk = max(1, (1 << 28) // max(V, 1))
    for s in range(0, rows.shape[0], chunk):
        dl[s:s + chunk] = (rows[s:s + chunk] @ Wf.T).to(dt)
    del Wf
    draft_logits = dl.reshape(B, w.gamma, V)

    # The small model's own draws: inverse CDF of softmax(draft_logits / T).
    u = torch.rand(B, w.gamma, generator=g, device=device, dtype=torch.float64)
    tokens = torch.empty(B, w.gamma, dtype=torch.int32, device=device)
    for b in range(B):
        qd = torch.softmax(draft_logits[b].double() / w.temperature, dim=-1)
        cdf = torch.cumsum(qd, dim=-1)
        t = (u[b] * cdf[:, -1]).unsqueeze(-1)
        tokens[b] = torch.searchsorted(cdf, t, right=True).squeeze(-1).clamp_max(V - 1).int()

    return {
        "hidden": hidden.contiguous(),
        "W_lm": W.contiguous(),
        "draft_tokens": tokens.contiguous(),
        "draft_logits": draft_logits.contiguous(),
        "sigma": sigma.float(),
    }


@torch.no_grad()
def generate_tree(w: Workload, seed: int, device="cpu") -> dict:
    """Inputs of one tree verify step, as contiguous tensors on `device`.

    hidden [B, N, d], W_lm [V, d], draft_logits [B, N, V] (W (h + sigma eps)
    at every node), node_tokens [B, N] int32 with node n's token drawn from
    softmax(draft_logits[b, parent[n]] / T) (column 0 is 0), parent (tuple)
    and sigma [B].
    """
    assert w.tree is not None
    parent = tuple(int(x) for x in w.tree)
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    dt = _torch_dtype(w)
    B, N, d, V = w.B, len(parent), w.d, w.V
    W = (torch.randn(V, d, generator=g, device=device) * w.w_std).to(dt)
    h = torch.randn(B, N, d, generator=g, device=device)
    if w.unit_rms:
        h = h / h.pow(2).mean(dim=-1, keepdim=True).sqrt()
    hidden = h.to(dt)
    if w.sigma_hi is None:
        sigma = torch.full((B,), float(w.sigma), device=device)
    else:
        sigma = w.sigma + (w.sigma_hi - w.sigma) * torch.rand(B, generator=g, device=device)
    eps = torch.randn(B, N, d, generator=g, device=device)
    rows = (hidden.float() + sigma[:, None, None] * eps).reshape(B * N, d)
    Wf = W.float()
    dl = torch.empty(B * N, V, dtype=dt, device=device)
    chunk = max(1, (1 << 28) // max(V, 1))
    for s0 in range(0, rows.shape[0], chunk):
        dl[s0:s0 + chunk] = (rows[s0:s0 + chunk] @ Wf.T).to(dt)
    del Wf
    draft_logits = dl.reshape(B, N, V)
    # Every child of a node is an independent draw from that node's q.
    u = torch.rand(B, N, generator=g, device=device, dtype=torch.float64)
    tokens = torch.zeros(B, N, dtype=torch.int32, device=device)
    par = torch.tensor(parent[1:], dtype=torch.long, device=device)
    for b in range(B if N > 1 else 0):
        qd = torch.softmax(draft_logits[b].double() / w.temperature, dim=-1)
        cdf = torch.cumsum(qd, dim=-1)
        t = (u[b, 1:] * cdf[par, -1]).unsqueeze(-1)
        tokens[b, 1:] = torch.searchsorted(cdf[par], t, right=True).squeeze(-1).clamp_max(V - 1).int()
    return {
        "hidden": hidden.contiguous(),
        "W_lm": W.contiguous(),
        "node_tokens": tokens.contiguous(),
        "draft_logits": draft_logits.contiguous(),
        "parent": parent,
        "sigma": sigma.float(),
    }
