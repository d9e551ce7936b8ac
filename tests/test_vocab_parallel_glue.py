"""verify_vocab_parallel() on CPU ranks (gloo, world sizes 2 and 3).

The collectives of the vocabulary-parallel step run here exactly as under
NCCL: the shards are stand-ins whose calls check what the exchanges hand
them (records and sums concatenated in rank order, the caller's own rank
at the draw) and leave marks that show which slice produced each result.
The arithmetic of the three calls is covered on the GPU against the fp64
oracle (test_gpu_vocab_parallel.py).
"""
import os
import socket
import sys

import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
B, GAMMA, NREC = 5, 3, 48


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


class _StubShard:
    """Implements the three calls' contracts with marks instead of arithmetic."""

    def __init__(self, rank, world, mode):
        from target_model_verify_gb300 import SAMPLE
        self.rank, self.world, self.mode, self.SAMPLE = rank, world, mode, SAMPLE
        self.B, self.gamma = B, GAMMA
        self.records = torch.empty(NREC, dtype=torch.uint8)
        self.sums = torch.empty(B, 2, dtype=torch.float32)
        self.calls = []

    def score(self, hidden, draft_tokens, dl):
        self.calls.append("score")
        self.records.fill_(10 + self.rank)
        return self.records

    def accept(self, all_rec, G, draft_tokens, dl, seed, out, nacc):
        self.calls.append("accept")
        assert G == self.world and all_rec.numel() == G * NREC
        assert torch.equal(all_rec.view(G, NREC)[:, 0], torch.arange(10, 10 + G, dtype=torch.uint8))
        # every rank takes the same decisions from the same gathered records
        n = (draft_tokens.sum(dim=1) + int(all_rec.sum())) % (GAMMA + 1)
        nacc.copy_(n.to(torch.int32))
        for b in range(B):
            j = int(n[b])
            out[b, :j] = draft_tokens[b, :j]
            out[b, j:] = -1
            if self.mode != self.SAMPLE:
                out[b, j] = 1000 + b
        self.sums[:, 0] = 100.0 * self.rank + torch.arange(B)
        self.sums[:, 1] = -1.0
        return self.sums

    def draw(self, all_sums, G, shard, dl, seed, out):
        self.calls.append("draw")
        assert shard == self.rank
        s = all_sums.view(G, B, 2)
        for k in range(G):
            assert torch.equal(s[k, :, 0], 100.0 * k + torch.arange(B, dtype=torch.float32))
        for b in range(B):
            j = int((out[b] >= 0).sum())   # first position the accept left at -1
            owner = b % G
            out[b, j] = 2000 + 10 * b + owner if owner == self.rank else -1


def _worker(rank, world, port, mode, q):
    sys.path.insert(0, ROOT)
    import target_model_verify_gb300 as tv
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank,
                            world_size=world)
    try:
        sh = _StubShard(rank, world, mode)
        tok = torch.arange(B * GAMMA, dtype=torch.int32).view(B, GAMMA)
        out, nacc = tv.verify_vocab_parallel(sh, None, tok, None, 7)
        q.put((rank, out.tolist(), nacc.tolist(), sh.calls))
    finally:
        dist.destroy_process_group()


def _run(world, mode):
    port = _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, world, port, mode, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    return res


def _check(res, world, mode):
    from target_model_verify_gb300 import SAMPLE
    outs = [r[1] for r in res]
    naccs = [r[2] for r in res]
    assert all(o == outs[0] for o in outs) and all(n == naccs[0] for n in naccs)
    for rank, _, _, calls in res:
        assert calls == (["score", "accept", "draw"] if mode == SAMPLE else ["score", "accept"])
    tok = torch.arange(B * GAMMA).view(B, GAMMA)
    for b in range(B):
        j = naccs[0][b]
        row = outs[0][b]
        assert row[:j] == tok[b, :j].tolist()
        want = 2000 + 10 * b + b % world if mode == SAMPLE else 1000 + b
        assert row[j] == want
        assert row[j + 1:] == [-1] * (GAMMA - j)


def test_sampling_step_gathers_in_rank_order_and_keeps_the_owner_token():
    from target_model_verify_gb300 import SAMPLE
    for world in (2, 3):
        _check(_run(world, SAMPLE), world, SAMPLE)


def test_greedy_step_needs_one_exchange():
    from target_model_verify_gb300 import GREEDY
    _check(_run(2, GREEDY), 2, GREEDY)
