"""Speculative-decoding verify step on one GB300 (sm_103a).

The compute lives in libspecdec_verify.so (C ABI: include/specdec_verify.h);
this package only marshals torch tensors into that ABI. See ``verify`` for
the call a user makes.
"""
from __future__ import annotations

import torch

from . import _binding as _b
from ._binding import (SPECDEC_BF16, SPECDEC_FP32, SPECDEC_GREEDY, SPECDEC_MAX_GAMMA,
                       SPECDEC_SAMPLE, SpecdecError, status_string)

SAMPLE = SPECDEC_SAMPLE
GREEDY = SPECDEC_GREEDY

_DTYPES = {torch.bfloat16: SPECDEC_BF16, torch.float32: SPECDEC_FP32}


def _stream_ptr(stream) -> int:
    s = stream if stream is not None else torch.cuda.current_stream()
    return int(s.cuda_stream)


def _ptr(t) -> int:
    return 0 if t is None else int(t.data_ptr())


def _shape(hidden, W_lm):
    B, g1, d = hidden.shape
    V = W_lm.shape[0]
    return B, g1 - 1, d, V


def _check_inputs(hidden, W_lm, draft_tokens, draft_logits, mode, device_kind):
    if hidden.dtype not in _DTYPES or W_lm.dtype != hidden.dtype:
        raise TypeError("hidden and W_lm must both be bfloat16 or both float32")
    if draft_tokens.dtype != torch.int32:
        raise TypeError("draft_tokens must be int32")
    if mode == SAMPLE and (draft_logits is None or draft_logits.dtype != hidden.dtype):
        raise TypeError("sampling mode needs draft_logits in the dtype of hidden")
    for t in (hidden, W_lm, draft_tokens, draft_logits):
        if t is None:
            continue
        if not t.is_contiguous():
            raise ValueError("all tensors must be contiguous")
        if device_kind == "cuda" and not t.is_cuda:
            raise ValueError("specdec_verify takes CUDA tensors")


def workspace_bytes(B, gamma, d, V, dtype=torch.bfloat16, mode=SAMPLE, host=False) -> int:
    fn = _b.specdec_verify_host_workspace_size if host else _b.specdec_verify_workspace_size
    return fn(B, gamma, d, V, _DTYPES[dtype], mode)


def alloc_workspace(B, gamma, d, V, dtype=torch.bfloat16, mode=SAMPLE, host=False, device=None):
    n = workspace_bytes(B, gamma, d, V, dtype, mode, host)
    if n == 0:
        raise SpecdecError(_b.SPECDEC_ERR_UNSUPPORTED, "workspace_bytes")
    return torch.empty(n, dtype=torch.uint8, device=device or "cuda")


def verify(hidden, W_lm, draft_tokens, draft_logits, temperature=1.0, seed=0, mode=SAMPLE,
           out_tokens=None, n_accepted=None, workspace=None, stream=None, debug=None,
           events=None):
    """One verify step (see include/specdec_verify.h for the contract).

    hidden [B, gamma+1, d], W_lm [V, d] (bf16 or fp32), draft_tokens
    [B, gamma] int32, draft_logits [B, gamma, V] (None allowed in greedy
    mode). Returns (out_tokens [B, gamma+1] int32, n_accepted [B] int32).
    `debug` may be a dict of preallocated CUDA tensors with keys logits,
    lse_p, lse_q, p_x, q_x, argmax; `events` a (start, end) pair of
    torch.cuda.Event recorded around the LM-head kernel.
    """
    _check_inputs(hidden, W_lm, draft_tokens, draft_logits, mode, "cuda")
    B, gamma, d, V = _shape(hidden, W_lm)
    dev = hidden.device
    if out_tokens is None:
        out_tokens = torch.empty(B, gamma + 1, dtype=torch.int32, device=dev)
    if n_accepted is None:
        n_accepted = torch.empty(B, dtype=torch.int32, device=dev)
    if workspace is None:
        workspace = alloc_workspace(B, gamma, d, V, hidden.dtype, mode, device=dev)
    core = (_ptr(hidden), _ptr(W_lm), _ptr(draft_tokens), _ptr(draft_logits), B, gamma, d, V,
            _DTYPES[hidden.dtype], float(temperature), int(seed) & (2 ** 64 - 1), int(mode),
            _ptr(out_tokens), _ptr(n_accepted), _ptr(workspace), workspace.numel(),
            _stream_ptr(stream))
    if debug is not None:
        rc = _b.specdec_verify_debug(*core, *(_ptr(debug.get(k)) for k in
                                              ("logits", "lse_p", "lse_q", "p_x", "q_x", "argmax")))
    elif events is not None:
        rc = _b.specdec_verify_timed(*core, int(events[0].cuda_event), int(events[1].cuda_event))
    else:
        rc = _b.specdec_verify(*core)
    _b._check(rc, "specdec_verify")
    return out_tokens, n_accepted


def verify_host(hidden, W_lm, draft_tokens, draft_logits, temperature=1.0, seed=0, mode=SAMPLE,
                out_tokens=None, n_accepted=None, workspace=None, stream=None):
    """End-to-end verify step from host (ideally pinned) CPU tensors.

    W_lm and the workspace are CUDA tensors; the other inputs and both
    outputs live in host memory. Returns after the step's outputs are back.
    """
    _check_inputs(hidden, W_lm, draft_tokens, draft_logits, mode, "host")
    if not W_lm.is_cuda or hidden.is_cuda:
        raise ValueError("verify_host takes W_lm on the device and the step's tensors on the host")
    B, gamma, d, V = _shape(hidden, W_lm)
    if out_tokens is None:
        out_tokens = torch.empty(B, gamma + 1, dtype=torch.int32, pin_memory=True)
    if n_accepted is None:
        n_accepted = torch.empty(B, dtype=torch.int32, pin_memory=True)
    if workspace is None:
        workspace = alloc_workspace(B, gamma, d, V, hidden.dtype, mode, host=True,
                                    device=W_lm.device)
    rc = _b.specdec_verify_host(_ptr(hidden), _ptr(W_lm), _ptr(draft_tokens), _ptr(draft_logits),
                                B, gamma, d, V, _DTYPES[hidden.dtype], float(temperature),
                                int(seed) & (2 ** 64 - 1), int(mode), _ptr(out_tokens),
                                _ptr(n_accepted), _ptr(workspace), workspace.numel(),
                                _stream_ptr(stream))
    _b._check(rc, "specdec_verify_host")
    return out_tokens, n_accepted


def tree_workspace_bytes(B, n_nodes, d, V, dtype=torch.bfloat16, mode=SAMPLE) -> int:
    return _b.specdec_verify_tree_workspace_size(B, n_nodes, d, V, _DTYPES[dtype], mode)


def alloc_tree_workspace(B, n_nodes, d, V, dtype=torch.bfloat16, mode=SAMPLE, device=None):
    n = tree_workspace_bytes(B, n_nodes, d, V, dtype, mode)
    if n == 0:
        raise SpecdecError(_b.SPECDEC_ERR_UNSUPPORTED, "tree_workspace_bytes")
    return torch.empty(n, dtype=torch.uint8, device=device or "cuda")


def verify_tree(hidden, W_lm, parent, node_tokens, draft_logits, temperature=1.0, seed=0,
                mode=SAMPLE, out_tokens=None, out_nodes=None, n_accepted=None, workspace=None,
                stream=None, events=None):
    """Tree verification (see include/specdec_verify.h, specdec_verify_tree).

    hidden [B, N, d] bf16, W_lm [V, d] bf16, parent: N ints (parent[0] = -1,
    parent[n] < n), node_tokens [B, N] int32, draft_logits [B, N, V] bf16
    (None allowed in greedy mode). Returns (out_tokens [B, N], out_nodes
    [B, N], n_accepted [B]), all int32 on the device.
    """
    _check_inputs(hidden, W_lm, node_tokens, draft_logits, mode, "cuda")
    B, N, d = hidden.shape
    V = W_lm.shape[0]
    par = torch.as_tensor(list(parent), dtype=torch.int32).contiguous()
    if par.numel() != N:
        raise ValueError("parent must have one entry per node")
    dev = hidden.device
    if out_tokens is None:
        out_tokens = torch.empty(B, N, dtype=torch.int32, device=dev)
    if out_nodes is None:
        out_nodes = torch.empty(B, N, dtype=torch.int32, device=dev)
    if n_accepted is None:
        n_accepted = torch.empty(B, dtype=torch.int32, device=dev)
    if workspace is None:
        workspace = alloc_tree_workspace(B, N, d, V, hidden.dtype, mode, device=dev)
    args = (_ptr(hidden), _ptr(W_lm), _ptr(par), _ptr(node_tokens), _ptr(draft_logits), B, N, d,
            V, _DTYPES[hidden.dtype], float(temperature), int(seed) & (2 ** 64 - 1), int(mode),
            _ptr(out_tokens), _ptr(out_nodes), _ptr(n_accepted), _ptr(workspace),
            workspace.numel(), _stream_ptr(stream))
    if events is not None:
        rc = _b.specdec_verify_tree_timed(*args, int(events[0].cuda_event),
                                          int(events[1].cuda_event))
    else:
        rc = _b.specdec_verify_tree(*args)
    _b._check(rc, "specdec_verify_tree")
    return out_tokens, out_nodes, n_accepted


def attention_workspace_bytes(B, n_new, Hq, Hkv, D, Lmax) -> int:
    return _b.specdec_verify_attention_workspace_size(B, n_new, Hq, Hkv, D, Lmax)


def verify_attention(q, k_cache, v_cache, seq_lens, scale=0.0, out=None, workspace=None,
                     stream=None):
    """Verify-step attention for one layer (include/specdec_verify.h).

    q [B, n_new, Hq, D], k_cache / v_cache [B, Lmax, Hkv, D] (bf16, CUDA),
    seq_lens [B] int32 (CUDA). Returns out [B, n_new, Hq, D] fp32.
    """
    for t in (q, k_cache, v_cache):
        if t.dtype != torch.bfloat16 or not t.is_cuda or not t.is_contiguous():
            raise TypeError("q and the caches must be contiguous bfloat16 CUDA tensors")
    if seq_lens.dtype != torch.int32 or not seq_lens.is_cuda:
        raise TypeError("seq_lens must be an int32 CUDA tensor")
    B, n_new, Hq, D = q.shape
    Lmax, Hkv = k_cache.shape[1], k_cache.shape[2]
    if out is None:
        out = torch.empty(B, n_new, Hq, D, dtype=torch.float32, device=q.device)
    if workspace is None:
        n = attention_workspace_bytes(B, n_new, Hq, Hkv, D, Lmax)
        if n == 0:
            raise SpecdecError(_b.SPECDEC_ERR_UNSUPPORTED, "attention_workspace_bytes")
        workspace = torch.empty(n, dtype=torch.uint8, device=q.device)
    rc = _b.specdec_verify_attention(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(seq_lens), B,
                                     n_new, Hq, Hkv, D, Lmax, float(scale), _ptr(out),
                                     _ptr(workspace), workspace.numel(), _stream_ptr(stream))
    _b._check(rc, "specdec_verify_attention")
    return out


def cluster_head(hidden, cluster_emb, W_sorted, starts, token_of_row, top_k=1, max_cluster=None,
                 temperature=1.0, seed=0, position=0, mode=SAMPLE, logits_out=None,
                 workspace=None, stream=None):
    """The drafter's clustered LM head (include/specdec_verify.h).

    hidden [M, d], cluster_emb [n_c, d], W_sorted [V, d] (bf16, CUDA);
    starts [n_c + 1] and token_of_row [V] int32 CUDA tensors. Returns
    (tokens [M], clusters [M, top_k]) int32 on the device.
    """
    for t in (hidden, cluster_emb, W_sorted):
        if t.dtype != torch.bfloat16 or not t.is_cuda or not t.is_contiguous():
            raise TypeError("hidden, cluster_emb and W_sorted must be contiguous bf16 CUDA tensors")
    M, d = hidden.shape
    n_c, V = cluster_emb.shape[0], W_sorted.shape[0]
    if max_cluster is None:
        max_cluster = int((starts[1:] - starts[:-1]).max())
    dev = hidden.device
    tokens = torch.empty(M, dtype=torch.int32, device=dev)
    clusters = torch.empty(M, top_k, dtype=torch.int32, device=dev)
    if workspace is None:
        n = _b.specdec_cluster_head_workspace_size(M, n_c, top_k, max_cluster)
        if n == 0:
            raise SpecdecError(_b.SPECDEC_ERR_UNSUPPORTED, "cluster_head_workspace_size")
        workspace = torch.empty(n, dtype=torch.uint8, device=dev)
    rc = _b.specdec_cluster_head(_ptr(hidden), _ptr(cluster_emb), _ptr(W_sorted), _ptr(starts),
                                 _ptr(token_of_row), M, d, V, n_c, top_k, max_cluster,
                                 float(temperature), int(seed) & (2 ** 64 - 1), int(position),
                                 int(mode), _ptr(tokens), _ptr(clusters), _ptr(logits_out),
                                 _ptr(workspace), workspace.numel(), _stream_ptr(stream))
    _b._check(rc, "specdec_cluster_head")
    return tokens, clusters


class ClusterHeadStep:
    """The clustered LM head bound once to fixed device buffers, for a draft loop.

    Same contract as cluster_head(); the drafter refills `hidden` in place
    between calls and each call passes only the seed and the position.
    The results land in self.tokens [M] and self.clusters [M, top_k].
    """

    def __init__(self, hidden, cluster_emb, W_sorted, starts, token_of_row, top_k=1,
                 max_cluster=None, temperature=1.0, mode=SAMPLE, logits_out=None, workspace=None,
                 stream=None):
        for t in (hidden, cluster_emb, W_sorted):
            if t.dtype != torch.bfloat16 or not t.is_cuda or not t.is_contiguous():
                raise TypeError("hidden, cluster_emb and W_sorted must be contiguous bf16 CUDA tensors")
        M, d = hidden.shape
        n_c, V = cluster_emb.shape[0], W_sorted.shape[0]
        if max_cluster is None:
            max_cluster = int((starts[1:] - starts[:-1]).max())
        dev = hidden.device
        self.tokens = torch.empty(M, dtype=torch.int32, device=dev)
        self.clusters = torch.empty(M, top_k, dtype=torch.int32, device=dev)
        if workspace is None:
            n = _b.specdec_cluster_head_workspace_size(M, n_c, top_k, max_cluster)
            if n == 0:
                raise SpecdecError(_b.SPECDEC_ERR_UNSUPPORTED, "cluster_head_workspace_size")
            workspace = torch.empty(n, dtype=torch.uint8, device=dev)
        self.workspace = workspace
        self._keep = (hidden, cluster_emb, W_sorted, starts, token_of_row, logits_out)
        self._fn = _b.lib().specdec_cluster_head
        a = _b._SIGNATURES["specdec_cluster_head"][1]
        vals = [_ptr(hidden), _ptr(cluster_emb), _ptr(W_sorted), _ptr(starts), _ptr(token_of_row),
                M, d, V, n_c, top_k, max_cluster, float(temperature), 0, 0, int(mode),
                _ptr(self.tokens), _ptr(self.clusters), _ptr(logits_out), _ptr(workspace),
                workspace.numel(), _stream_ptr(stream)]
        self._args = [t(v) for t, v in zip(a, vals)]
        self._seed, self._position = self._args[12], self._args[13]

    def __call__(self, seed, position=0):
        self._seed.value = int(seed) & (2 ** 64 - 1)
        self._position.value = int(position)
        rc = self._fn(*self._args)
        if rc != 0:
            _b._check(rc, "specdec_cluster_head")
        return self.tokens, self.clusters


class HostStep:
    """A host-I/O verify step bound once to fixed buffers, for a decode loop.

    Same contract as verify_host(): hidden, draft_tokens and draft_logits
    are pinned CPU tensors that the caller refills in place before each
    call; out_tokens and n_accepted (pinned, allocated here if not given)
    receive the results. The argument checks and the marshalling happen
    once, here; each call passes only the new seed. Returns
    (out_tokens, n_accepted) after the step's results are back on the host.
    """

    def __init__(self, hidden, W_lm, draft_tokens, draft_logits, temperature=1.0, mode=SAMPLE,
                 out_tokens=None, n_accepted=None, workspace=None, stream=None):
        _check_inputs(hidden, W_lm, draft_tokens, draft_logits, mode, "host")
        if not W_lm.is_cuda or hidden.is_cuda:
            raise ValueError("HostStep takes W_lm on the device and the step's tensors on the host")
        B, gamma, d, V = _shape(hidden, W_lm)
        if out_tokens is None:
            out_tokens = torch.empty(B, gamma + 1, dtype=torch.int32, pin_memory=True)
        if n_accepted is None:
            n_accepted = torch.empty(B, dtype=torch.int32, pin_memory=True)
        if workspace is None:
            workspace = alloc_workspace(B, gamma, d, V, hidden.dtype, mode, host=True,
                                        device=W_lm.device)
        # keep every buffer alive for the lifetime of the step
        self._keep = (hidden, W_lm, draft_tokens, draft_logits, workspace)
        self.out_tokens, self.n_accepted = out_tokens, n_accepted
        self._fn = _b.lib().specdec_verify_host
        a = _b._SIGNATURES["specdec_verify_host"][1]
        vals = [_ptr(hidden), _ptr(W_lm), _ptr(draft_tokens), _ptr(draft_logits), B, gamma, d, V,
                _DTYPES[hidden.dtype], float(temperature), 0, int(mode), _ptr(out_tokens),
                _ptr(n_accepted), _ptr(workspace), workspace.numel(), _stream_ptr(stream)]
        self._args = [t(v) for t, v in zip(a, vals)]
        self._seed = self._args[10]

    def __call__(self, seed):
        self._seed.value = int(seed) & (2 ** 64 - 1)
        rc = self._fn(*self._args)
        if rc != 0:
            _b._check(rc, "specdec_verify_host")
        return self.out_tokens, self.n_accepted


class VocabShard:
    """One GPU's slice of a vocabulary-parallel LM head (include/specdec_verify.h,
    specdec_shard_*): rows [v_begin, v_begin + V_shard) of W_lm.

    A step is score() -> all-gather of the records -> accept() -> (sampling)
    all-gather of the sums -> draw() -> max-reduce of out_tokens;
    verify_vocab_parallel() runs it with torch.distributed collectives.
    """

    def __init__(self, W_shard, v_begin, V, B, gamma, mode=SAMPLE, temperature=1.0):
        if W_shard.dtype != torch.bfloat16 or not W_shard.is_cuda or not W_shard.is_contiguous():
            raise TypeError("W_shard must be a contiguous bf16 CUDA tensor")
        self.W, self.v_begin, self.V = W_shard, int(v_begin), int(V)
        self.V_shard, self.d = W_shard.shape
        self.B, self.gamma, self.mode, self.T = int(B), int(gamma), int(mode), float(temperature)
        dev = W_shard.device
        n = _b.specdec_shard_workspace_size(self.B, self.gamma, self.d, self.V_shard, self.mode)
        nr = _b.specdec_shard_record_bytes(self.B, self.gamma)
        if n == 0 or nr == 0:
            raise SpecdecError(_b.SPECDEC_ERR_UNSUPPORTED, "specdec_shard_workspace_size")
        self.workspace = torch.empty(n, dtype=torch.uint8, device=dev)
        self.records = torch.empty(nr, dtype=torch.uint8, device=dev)
        self.sums = torch.empty(self.B, 2, dtype=torch.float32, device=dev)

    def _shape(self):
        return (self.B, self.gamma, self.d, self.V_shard, self.v_begin, self.V)

    def score(self, hidden, draft_tokens, draft_logits_shard, stream=None):
        """LM head on the slice; returns this GPU's records (uint8 device tensor)."""
        rc = _b.specdec_shard_score(_ptr(hidden), _ptr(self.W), _ptr(draft_tokens),
                                    _ptr(draft_logits_shard), *self._shape(), self.T, self.mode,
                                    _ptr(self.records), _ptr(self.workspace),
                                    self.workspace.numel(), _stream_ptr(stream))
        _b._check(rc, "specdec_shard_score")
        return self.records

    def accept(self, all_records, n_shards, draft_tokens, draft_logits_shard, seed, out_tokens,
               n_accepted, stream=None):
        """Decides from the gathered records; returns this slice's sums [B, 2]."""
        rc = _b.specdec_shard_accept(_ptr(all_records), int(n_shards), _ptr(draft_tokens),
                                     _ptr(draft_logits_shard), *self._shape(), self.T,
                                     int(seed) & (2 ** 64 - 1), self.mode, _ptr(out_tokens),
                                     _ptr(n_accepted), _ptr(self.sums), _ptr(self.workspace),
                                     self.workspace.numel(), _stream_ptr(stream))
        _b._check(rc, "specdec_shard_accept")
        return self.sums

    def draw(self, all_sums, n_shards, shard, draft_logits_shard, seed, out_tokens, stream=None):
        """Writes the drawn token where this slice holds it, -1 elsewhere."""
        rc = _b.specdec_shard_draw(_ptr(all_sums), int(n_shards), int(shard),
                                   _ptr(draft_logits_shard), *self._shape(), self.T,
                                   int(seed) & (2 ** 64 - 1), self.mode, _ptr(out_tokens),
                                   _ptr(self.workspace), self.workspace.numel(),
                                   _stream_ptr(stream))
        _b._check(rc, "specdec_shard_draw")


def verify_vocab_parallel(shard, hidden, draft_tokens, draft_logits_shard, seed, group=None):
    """One vocabulary-parallel verify step on this rank's slice, with the
    three collectives over `group` (torch.distributed): all-gather of the
    records, all-gather of the slices' sums, max-reduce of the tokens.
    Returns (out_tokens [B, gamma+1], n_accepted [B]), identical on every rank."""
    import torch.distributed as dist
    G = dist.get_world_size(group)
    rank = dist.get_rank(group)
    B, g1 = shard.B, shard.gamma + 1
    dev = shard.records.device
    rec = shard.score(hidden, draft_tokens, draft_logits_shard)
    all_rec = torch.empty(G * rec.numel(), dtype=torch.uint8, device=dev)
    dist.all_gather_into_tensor(all_rec, rec, group=group)
    out = torch.empty(B, g1, dtype=torch.int32, device=dev)
    nacc = torch.empty(B, dtype=torch.int32, device=dev)
    sums = shard.accept(all_rec, G, draft_tokens, draft_logits_shard, seed, out, nacc)
    if shard.mode == SAMPLE:
        all_sums = torch.empty(G * B * 2, dtype=torch.float32, device=dev)
        dist.all_gather_into_tensor(all_sums, sums.reshape(-1), group=group)
        shard.draw(all_sums, G, rank, draft_logits_shard, seed, out)
        dist.all_reduce(out, op=dist.ReduceOp.MAX, group=group)
    return out, nacc


def read_status(workspace, stream=None) -> int:
    """The device status word of the last call that used `workspace`."""
    return _b.specdec_read_status(_ptr(workspace), _stream_ptr(stream))


def philox_uniforms(seed, B, n_pos, purpose, device="cuda", stream=None):
    """The library's r (purpose 0) or u (purpose 1) uniforms, [B, n_pos] fp32."""
    out = torch.empty(B, n_pos, dtype=torch.float32, device=device)
    rc = _b.specdec_philox_uniforms(int(seed) & (2 ** 64 - 1), B, n_pos, purpose, _ptr(out),
                                    _stream_ptr(stream))
    _b._check(rc, "specdec_philox_uniforms")
    return out


__all__ = ["verify", "verify_host", "alloc_workspace", "workspace_bytes", "read_status",
           "philox_uniforms", "status_string", "SpecdecError", "SAMPLE", "GREEDY", "HostStep",
           "verify_tree", "tree_workspace_bytes", "alloc_tree_workspace", "verify_attention",
           "attention_workspace_bytes", "cluster_head", "ClusterHeadStep", "VocabShard",
           "verify_vocab_parallel"]
