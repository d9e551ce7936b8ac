"""The multi-rank path of bench.py on CPU ranks (gloo, world size 2).

The verify step partitions over sequences, so ranks share nothing on the
data path: each draws its own batch, and the only cross-rank steps are the
barrier and the max-over-ranks reduction of the timed region. These run
here exactly as under torchrun on GPUs, with gloo in place of NCCL.
"""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    sys.path.insert(0, ROOT)
    import bench
    from target_model_verify_gb300 import workloads as wl
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank,
                            world_size=world)
    try:
        elapsed = [10.0, 12.5][rank]
        dist.barrier()
        mx = bench.reduce_max_ms(elapsed, world, "cpu")
        val = bench.whole_job_value(world, 100, mx)
        w = wl.get("tiny_fp32")
        inp = wl.generate(w, bench.rank_seed(7, rank), device="cpu")
        q.put((rank, mx, val, float(inp["hidden"].double().sum())))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_reduce_to_the_slowest_and_draw_their_own_batches():
    port = _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    (r0, mx0, v0, h0), (r1, mx1, v1, h1) = res
    assert (r0, r1) == (0, 1)
    assert mx0 == mx1 == 12.5                       # every rank sees the slowest time
    assert v0 == v1 == pytest.approx(2 * 100 / 12.5e-3)   # both ranks' steps / that time
    assert h0 != h1                                 # independent batches (weak scaling)


def test_reference_arm_under_torchrun_prints_once_from_rank_zero():
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes", "1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), "bench.py", "--impl",
           "reference", "--gpus", "2", "--workload", "tiny_fp32", "--steps", "3", "--warmup", "3"]
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="")
    out = subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [ln for ln in out.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, out.stdout
    rec = json.loads(lines[0])
    assert rec["impl"] == "reference"
    assert rec["n_gpus"] == 2
    assert rec["unit"] == "steps/s" and rec["value"] > 0
    # The keys of the benchmark line that the reference arm shares with the
    # library's arm, with the values this arm must carry.
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
                "cpu_baseline", "e2e"):
        assert key in rec, key
    assert (rec["steps"], rec["warmup"]) == (3, 3)
    assert rec["higher_is_better"] is True and rec["scaling"] == "weak"
    assert rec["vs_baseline"] is None and rec["dtype"] == "f64"
    assert rec["ms_per_step"] == pytest.approx(1e3 / rec["value"], rel=1e-6)
    assert rec["config"]["workload"] == "tiny_fp32"
    cpu = rec["cpu_baseline"]
    assert cpu["kind"] == "oracle" and cpu["cores"] >= 1 and cpu["value"] == rec["value"]
    assert isinstance(cpu["sample"], str) and cpu["sample"]
    assert rec["e2e"] == {"value": rec["value"], "unit": "steps/s", "h2d_bytes_per_step": 0,
                          "d2h_bytes_per_step": 0}
