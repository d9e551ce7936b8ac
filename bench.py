"""Benchmark of the speculative-decoding verify step on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
                    [--mode sample|greedy] [--impl ours|reference]

One step = one specdec_verify call: the LM head scores all gamma+1
positions of every sequence in one weight read, then the acceptance scan and
the residual / bonus draw run. Inputs are synthetic, seeded and resident in
HBM before the timed region; W_lm (1.05 GB for the default Llama-3-8B head)
is larger than L2, so no flush is needed between steps. Under torchrun each
rank runs an independent replica on its own GPU (weak scaling, no
collective on the data path); the step time is the maximum over ranks.

Prints one JSON line: steps/s (whole job), committed tokens/s, the LM-head
kernel's roofline fraction (CUDA events inside the timed steps), the fp64
oracle on the host cores as cpu_baseline, an end-to-end figure through the
host-pointer entry point, and the SM clocks sampled during the timed region.
--impl reference times the fp64 oracle itself on the host cores.
"""
from __future__ import annotations

import argparse
import datetime as _dt
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

from target_model_verify_gb300 import workloads as wl  # noqa: E402

METRIC = "verify steps/s and committed tokens/s at 1 GB300; % of HBM/tensor roofline"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
LMHEAD_SOURCES = ["target_model_verify_gb300/csrc/lmhead_tc.cu",
                  "target_model_verify_gb300/csrc/common.cuh"]
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "ncu_traffic.json")
CPU_BASELINE_SECONDS = 10.0
CLOCK_WINDOW_SECONDS = 1.5
REFERENCE_SECONDS_PER_RUN = 150.0


def parse_args(argv=None):
    ap = argparse.ArgumentParser(description="verify-step benchmark")
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=5000)
    ap.add_argument("--warmup", type=int, default=50)
    ap.add_argument("--workload", default="llama3_8b_head", choices=sorted(wl.WORKLOADS))
    ap.add_argument("--mode", default="sample", choices=["sample", "greedy"])
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--attention", default=None, metavar="B,L,N",
                    help="time verify-step attention for one Llama-3-8B-shaped layer (32 query, "
                         "8 KV heads, D 128): B sequences of L cached tokens, N new positions")
    ap.add_argument("--cluster-head", default=None, metavar="M,K",
                    help="time the drafter's clustered LM head at the Gemma-E2B shape "
                         "(V 262144, d 1536, 2048 clusters of 128): M rows, K kept clusters")
    ap.add_argument("--gamma-sweep", action="store_true",
                    help="Gemma-E2B head, gamma in {1,2,3,4,6,8}: mean tokens per step of 4000 "
                         "sequences with i.i.d. positions against (1 - a^(g+1)) / (1 - a)")
    ap.add_argument("--loop-c", type=float, default=None,
                    help="time the draft->verify loop with a synthetic drafter costing this "
                         "fraction of a target step per draft token (prints its own line)")
    ap.add_argument("--vocab-slices", default=None, metavar="G1,G2,...",
                    help="time one GPU's calls of the vocabulary-parallel step (specdec_shard_*) "
                         "with W_lm split into G slices, against the single-GPU step")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    return args


# --------------------------------------------------------------- helpers --

def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            return json.load(f), "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def lmhead_source_hash() -> str:
    h = hashlib.sha256()
    for rel in LMHEAD_SOURCES:
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def recorded_traffic(workload: str, mode: str):
    """DRAM bytes per LM-head launch from a committed ncu summary, if the
    kernel sources still match the ones it was captured from."""
    if not os.path.exists(TRAFFIC_FILE):
        return None
    with open(TRAFFIC_FILE) as f:
        rec = json.load(f)
    ent = rec.get(f"{workload}/{mode}")
    if not ent or ent.get("source_hash") != lmhead_source_hash():
        return None
    return ent.get("dram_bytes_per_launch")


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons (100 ms)."""
    FIELDS = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.proc = None
        self.lines = []
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100", "-i", str(gpu_index)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, ValueError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        self.lines = [ln for ln in out.splitlines() if ln.strip()]

    def summary(self, t0: float, t1: float, strict: bool = False):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        rows = []
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                ts = _dt.datetime.strptime(parts[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
                rows.append((ts, float(parts[1]), float(parts[2]), parts[5:9]))
            except ValueError:
                continue
        inside = [r for r in rows if t0 - 0.05 <= r[0] <= t1 + 0.05]
        if strict and not inside:
            return {"samples": 0}
        inside = inside or rows
        if not inside:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[k] for r in inside for k in range(4) if r[3][k] == "Active"})
        return {"sm_mhz": statistics.median(r[1] for r in inside),
                "sm_max_mhz": max(r[2] for r in inside), "reasons": reasons,
                "samples": len(inside)}


def host_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def _openblas_fns():
    """get/set functions of the OpenBLAS that NumPy loaded, or (None, None)."""
    import ctypes
    try:
        with open("/proc/self/maps") as f:
            paths = sorted({ln.split()[-1] for ln in f if "openblas" in ln.lower() and ".so" in ln})
    except OSError:
        return None, None
    for path in paths:
        try:
            lib = ctypes.CDLL(path)
        except OSError:
            continue
        for pre in ("scipy_openblas_", "openblas_", ""):
            for suf in ("64_", ""):
                g = getattr(lib, f"{pre}get_num_threads{suf}", None) if pre else None
                st = getattr(lib, f"{pre}set_num_threads{suf}", None) if pre else None
                if g is not None and st is not None:
                    g.restype = ctypes.c_int
                    st.argtypes = [ctypes.c_int]
                    return g, st
    return None, None


def blas_threads():
    """Threads NumPy's BLAS uses (None if it cannot be asked)."""
    get, _ = _openblas_fns()
    return int(get()) if get is not None else None


def time_oracle_one_thread(w, inp, mode, seconds: float):
    """time_oracle with NumPy's BLAS limited to one thread (restored after)."""
    get, set_ = _openblas_fns()
    if get is None:
        return None
    n0 = int(get())
    set_(1)
    try:
        return time_oracle(w, inp, mode, seconds)
    finally:
        set_(n0)


def bench_config(args, w, world) -> dict:
    """The `config` object, identical in both arms for the same workload."""
    return {"workload": args.workload, "B": w.B, "gamma": w.gamma, "d": w.d, "V": w.V,
            "mode": args.mode, "temperature": w.temperature,
            **({"tree_nodes": w.N, "tree_depth": tree_depth(w.tree)}
               if w.tree is not None else {}),
            "parallelism": "replicas" if world > 1 else "single GPU",
            "l2": "inputs larger than L2 (W_lm exceeds the 129 MB L2), no flush"}


# Workloads whose CPU baseline also reports the oracle on one thread: the
# small case and the single-sequence heads.
ONE_THREAD_WORKLOADS = ("tiny_fp32", "llama3_8b_head") + tuple(
    f"gemma_e2b_head_g{g}" for g in (1, 2, 3, 4, 6, 8))


def oracle_inputs(inp: dict, mode: int):
    h = inp["hidden"].float().cpu().double().numpy()
    W = inp["W_lm"].float().cpu().double().numpy()
    x = inp["node_tokens" if "node_tokens" in inp else "draft_tokens"].cpu().numpy().astype(np.int64)
    dl = inp["draft_logits"].float().cpu().double().numpy() if mode == wl.SAMPLE else None
    return h, W, x, dl


def oracle_step(w, h, W, x, dl, seed, mode):
    """One step of the fp64 oracle (chain or tree) on converted inputs."""
    if w.tree is not None:
        from oracle import tree as ot
        return ot.verify_tree(h, W, w.tree, x, dl, w.temperature, seed, mode)
    from oracle import verify as ov
    return ov.verify(h, W, x, dl, w.temperature, seed, mode)


def time_oracle(w, inp, mode, seconds: float, min_steps: int = 1):
    """Full oracle steps on the host cores until `seconds` have passed."""
    h, W, x, dl = oracle_inputs(inp, mode)
    n = 0
    t0 = time.perf_counter()
    while n < min_steps or time.perf_counter() - t0 < seconds:
        oracle_step(w, h, W, x, dl, 1000 + n, mode)
        n += 1
    return n / (time.perf_counter() - t0), n


# The library's launch plan for a chain step in sampling mode, by the
# number of (sequence, 4096-token chunk) pairs of the draw: up to 128 the
# acceptance test and the draw share one kernel; up to 608 the draw is one
# kernel after the acceptance kernel; beyond, chunk sums and draw are two.
SAMPLE_CHUNK = 4096
FUSED_ITEMS = 128
ONE_DRAW_KERNEL_ITEMS = 608


def kernels_per_step(w, mode) -> int:
    """Library kernels one step launches (see the plan above); for a tree,
    LM head and the tree walk; greedy: LM head and acceptance."""
    if w.tree is not None or mode != wl.SAMPLE:
        return 2
    items = w.B * -(-w.V // SAMPLE_CHUNK)
    if items <= FUSED_ITEMS:
        return 2
    return 3 if items <= ONE_DRAW_KERNEL_ITEMS else 4


# ------------------------------------------------------ multi-rank glue --
# One process per GPU, each verifying its own batch (independent sequences:
# no collective on the data path). These three are the only cross-rank
# steps, and run unchanged on CPU ranks over gloo.

def rank_seed(seed: int, rank: int) -> int:
    """Each rank draws its own synthetic batch."""
    return seed + rank


def reduce_max_ms(elapsed_ms: float, world: int, device) -> float:
    """The slowest rank's timed region (all ranks get it)."""
    t = torch.tensor([elapsed_ms], dtype=torch.float64, device=device)
    if world > 1:
        torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def whole_job_value(world: int, K: int, max_ms: float) -> float:
    """Steps of all ranks divided by the slowest rank's time."""
    return world * K / (max_ms / 1e3)


# ------------------------------------------------------------ our arm --

def run_ours(args, world, rank, local):
    import target_model_verify_gb300 as tv

    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=device)
    w = wl.get(args.workload)
    mode = wl.SAMPLE if args.mode == "sample" else wl.GREEDY
    is_tree = w.tree is not None
    gen = wl.generate_tree if is_tree else wl.generate
    inp = gen(w, rank_seed(args.seed, rank), device=device)
    dl = inp["draft_logits"] if mode == wl.SAMPLE else None
    if is_tree:
        ws = tv.alloc_tree_workspace(w.B, w.N, w.d, w.V, inp["hidden"].dtype, mode, device=device)
    else:
        ws = tv.alloc_workspace(w.B, w.gamma, w.d, w.V, inp["hidden"].dtype, mode, device=device)
    K, Wm = args.steps, args.warmup
    outs = torch.empty(K + Wm, w.B, w.N, dtype=torch.int32, device=device)
    nodes = torch.empty(K + Wm, w.B, w.N, dtype=torch.int32, device=device) if is_tree else None
    naccs = torch.empty(K + Wm, w.B, dtype=torch.int32, device=device)
    ev0 = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    ev1 = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    for e in ev0 + ev1:
        e.record()          # creates the underlying CUDA event
    torch.cuda.synchronize()

    def step(i, events=None):
        if is_tree:
            tv.verify_tree(inp["hidden"], inp["W_lm"], w.tree, inp["node_tokens"], dl,
                           w.temperature, args.seed * 1_000_003 + i, mode, out_tokens=outs[i],
                           out_nodes=nodes[i], n_accepted=naccs[i], workspace=ws, events=events)
        else:
            tv.verify(inp["hidden"], inp["W_lm"], inp["draft_tokens"], dl, w.temperature,
                      args.seed * 1_000_003 + i, mode, out_tokens=outs[i], n_accepted=naccs[i],
                      workspace=ws, events=events)

    sampler = ClockSampler(device.index) if rank == 0 else None
    time.sleep(0.6 if sampler else 0)
    for i in range(Wm):
        step(i)
    torch.cuda.synchronize()
    # Clock window: the same steps, untimed, for CLOCK_WINDOW_SECONDS right
    # before the timed region, so that the clock record holds enough
    # nvidia-smi samples (one per 100 ms) of this load even when the timed
    # region itself lasts a few milliseconds.
    t_clock0 = time.time()
    settle = 0
    while time.time() - t_clock0 < CLOCK_WINDOW_SECONDS:
        for _ in range(10):
            step(Wm - 1)
        settle += 10
        torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t_wall0 = time.time()
    start.record()
    for k in range(K):
        step(Wm + k)
    end.record()
    torch.cuda.synchronize()
    t_wall1 = time.time()
    if world > 1:
        torch.distributed.barrier()
    elapsed_ms = start.elapsed_time(end)
    # Second timed pass: the same K steps with events recorded around the
    # LM-head kernel (an event between two kernels stops the next one from
    # launching early, so the headline pass above runs without them).
    for k in range(K):
        step(Wm + k, (ev0[k], ev1[k]))
    torch.cuda.synchronize()
    lm_ms = [a.elapsed_time(b) for a, b in zip(ev0, ev1)]
    if sampler:
        time.sleep(0.2)
        sampler.stop()
    st = tv.read_status(ws)
    if st != 0:
        raise RuntimeError(f"device status {st}: {tv.status_string(st)}")

    max_ms = reduce_max_ms(elapsed_ms, world, device)
    nacc = naccs[Wm:].double()
    tokens_per_step = float((nacc + 1).sum(dim=1).mean().item())

    e2e = None
    if not args.no_e2e:
        e2e = run_e2e(tv, w, inp, mode, K, Wm, args, device)

    if rank != 0:
        if world > 1:
            torch.distributed.destroy_process_group()
        return

    peaks, peak_kind = load_peaks()
    steps_per_s = whole_job_value(world, K, max_ms)
    lm_avg_s = float(np.mean(lm_ms)) / 1e3
    step_s = max_ms / 1e3 / K
    bytes_alg = w.algorithmic_bytes(mode)
    n_tok = w.B * ((w.N - 1) if w.tree is not None else w.gamma)
    lm_bytes = bytes_alg - n_tok * 4                  # the LM-head kernel does not read the tokens
    t_hbm = bytes_alg / (peaks["hbm_gbs"] * 1e9)
    t_tc = w.flops() / (peaks["bf16_tflops"] * 1e12)
    tensor_bound = t_tc > t_hbm
    if tensor_bound:
        # The kernel is timed inside a step loop that runs for seconds: the
        # sustained (power-capped) GEMM rate is its ceiling; the burst rate
        # is kept beside it.
        achieved = w.flops() / lm_avg_s / 1e12
        sustained = peaks.get("bf16_tflops_sustained", peaks["bf16_tflops"])
        roof = {"bound": "tensor", "achieved": achieved, "peak": sustained,
                "unit": "TFLOP/s", "peak_kind": "sustained bf16 GEMM",
                "frac_of_burst": achieved / peaks["bf16_tflops"]}
    else:
        achieved = lm_bytes / lm_avg_s / 1e9
        roof = {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "peak_kind": "copy bandwidth"}
    roof["frac"] = roof["achieved"] / roof["peak"]
    roof["traffic"] = recorded_traffic(args.workload, args.mode)
    roof["kernel"] = "lmhead_tc_kernel"
    roof["kernel_us"] = lm_avg_s * 1e6
    roof["peak_source"] = f"{peak_kind} (MEASURED_PEAKS.json)" if peak_kind == "measured" \
        else "fallback"
    roof["algorithmic_bytes"] = lm_bytes

    cpu = None
    if world == 1 and not args.no_cpu_baseline:
        v, n = time_oracle(w, inp, mode, CPU_BASELINE_SECONDS)
        cpu = {"value": v, "unit": "steps/s", "cores": host_cores(), "kind": "oracle",
               "blas_threads": blas_threads(),
               "sample": f"{n} full {args.workload} steps (fp64 NumPy oracle, W converted "
                         f"to fp64 once outside the timing)"}
        if args.workload in ONE_THREAD_WORKLOADS:
            one = time_oracle_one_thread(w, inp, mode, CPU_BASELINE_SECONDS)
            if one is not None:
                cpu["one_thread"] = {"value": one[0], "unit": "steps/s", "steps": one[1]}

    clocks = None
    if sampler:
        clocks = sampler.summary(t_clock0, t_wall1)
        clocks["timed_region_samples"] = sampler.summary(t_wall0, t_wall1, strict=True).get("samples", 0)
        clocks["window"] = (f"{CLOCK_WINDOW_SECONDS:.1f} s of the same steps ({settle}, untimed) "
                            f"just before the timed region, and the timed region")
    line = {
        "metric": METRIC,
        "value": steps_per_s,
        "unit": "steps/s",
        "n_gpus": world,
        "steps": K,
        "warmup": Wm,
        "ms_per_step": max_ms / K,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16" if w.dtype == "bf16" else "f32",
        "data": "synthetic (seeded; random-init LM head)",
        "config": bench_config(args, w, world),
        "committed_tokens_per_s": steps_per_s * tokens_per_step,
        "mean_tokens_per_step": tokens_per_step,
        "step_roofline": {"time_us": max(t_hbm, t_tc) * 1e6, "frac": max(t_hbm, t_tc) / step_s,
                          "bound": "tensor" if tensor_bound else "hbm",
                          "frac_sustained": max(t_hbm, w.flops() / (peaks.get(
                              "bf16_tflops_sustained", peaks["bf16_tflops"]) * 1e12)) / step_s},
        "roofline": roof,
        "cpu_baseline": cpu,
        "e2e": e2e,
        "gpu_launches": K * kernels_per_step(w, mode),
        "clocks": clocks,
    }
    print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


def tree_depth(parent) -> int:
    depth = [0] * len(parent)
    for n in range(1, len(parent)):
        depth[n] = depth[parent[n]] + 1
    return max(depth)


def run_e2e_tree(tv, w, inp, mode, K, Wm, args, device):
    """Tree steps through the public API from pinned host tensors: copy the
    step's inputs in, verify, read the results back, every step."""
    host = {k: inp[k].cpu().pin_memory() for k in ("hidden", "node_tokens", "draft_logits")}
    dev = {k: torch.empty_like(v, device=device) for k, v in host.items()}
    out = torch.empty(w.B, w.N, dtype=torch.int32, pin_memory=True)
    nod = torch.empty(w.B, w.N, dtype=torch.int32, pin_memory=True)
    nacc = torch.empty(w.B, dtype=torch.int32, pin_memory=True)
    ws = tv.alloc_tree_workspace(w.B, w.N, w.d, w.V, inp["hidden"].dtype, mode, device=device)
    names = ("hidden", "node_tokens") + (("draft_logits",) if mode == wl.SAMPLE else ())

    def step(i):
        for k in names:
            dev[k].copy_(host[k], non_blocking=True)
        o, n, a = tv.verify_tree(dev["hidden"], inp["W_lm"], w.tree, dev["node_tokens"],
                                 dev["draft_logits"] if mode == wl.SAMPLE else None,
                                 w.temperature, i, mode, workspace=ws)
        out.copy_(o, non_blocking=True)
        nod.copy_(n, non_blocking=True)
        nacc.copy_(a, non_blocking=True)
        torch.cuda.current_stream().synchronize()

    for i in range(Wm):
        step(i)
    n = max(1, min(K, 2000))
    t0 = time.perf_counter()
    for i in range(n):
        step(Wm + i)
    dt = time.perf_counter() - t0
    h2d = sum(host[k].numel() * host[k].element_size() for k in names)
    d2h = out.numel() * 4 + nod.numel() * 4 + nacc.numel() * 4
    return {"value": n / dt, "unit": "steps/s", "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "steps": n}


def run_e2e(tv, w, inp, mode, K, Wm, args, device):
    """Same metric through the host-pointer entry point, copies included."""
    if w.tree is not None:
        return run_e2e_tree(tv, w, inp, mode, K, Wm, args, device)
    host = {k: v.cpu().pin_memory() for k, v in inp.items() if k != "W_lm"}
    hl = host["draft_logits"] if mode == wl.SAMPLE else None
    out = torch.empty(w.B, w.gamma + 1, dtype=torch.int32, pin_memory=True)
    nacc = torch.empty(w.B, dtype=torch.int32, pin_memory=True)
    ws = tv.alloc_workspace(w.B, w.gamma, w.d, w.V, inp["hidden"].dtype, mode, host=True,
                            device=device)

    # The decode-loop form of the host API: bound once, then one call per
    # step with the inputs re-read from the same pinned buffers.
    step = tv.HostStep(host["hidden"], inp["W_lm"], host["draft_tokens"], hl, w.temperature,
                       mode, out_tokens=out, n_accepted=nacc, workspace=ws)

    for i in range(Wm):
        step(i)
    n = max(1, min(K, 2000))
    t0 = time.perf_counter()
    for i in range(n):
        step(Wm + i)
    dt = time.perf_counter() - t0
    h2d = host["hidden"].numel() * host["hidden"].element_size() + host["draft_tokens"].numel() * 4
    if hl is not None:
        h2d += hl.numel() * hl.element_size()
    d2h = out.numel() * 4 + nacc.numel() * 4
    return {"value": n / dt, "unit": "steps/s", "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "steps": n}


# ---------------------------------------------------- reference arm --

def run_reference(args, world, rank, local):
    """The fp64 oracle on the host cores, on this arm's workload."""
    if rank != 0:
        return
    w = wl.get(args.workload)
    mode = wl.SAMPLE if args.mode == "sample" else wl.GREEDY
    device = "cuda" if torch.cuda.is_available() else "cpu"
    inp = (wl.generate_tree if w.tree is not None else wl.generate)(w, args.seed, device=device)
    h, W, x, dl = oracle_inputs(inp, mode)
    # One full step, to size the per-step sample so the run fits its time allowance.
    t0 = time.perf_counter()
    oracle_step(w, h, W, x, dl, 0, mode)
    t_full = time.perf_counter() - t0
    n_total = args.steps + args.warmup
    frac = min(1.0, REFERENCE_SECONDS_PER_RUN / max(n_total * t_full, 1e-9))
    Vs = max(1, int(w.V * frac))
    Ws = W[:Vs]
    xs = np.minimum(x, Vs - 1)
    dls = dl[..., :Vs] if dl is not None else None
    for i in range(args.warmup):
        oracle_step(w, h, Ws, xs, dls, i, mode)
    t0 = time.perf_counter()
    for k in range(args.steps):
        oracle_step(w, h, Ws, xs, dls, args.warmup + k, mode)
    dt = time.perf_counter() - t0
    scale = Vs / w.V
    value = args.steps * scale / dt
    sample = (f"each step runs the fp64 oracle on the first {Vs} of {w.V} vocabulary rows "
              f"(the oracle's cost is linear in V); value scaled by {Vs}/{w.V}")
    line = {
        "metric": METRIC, "value": value, "unit": "steps/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 / value,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f64", "data": "synthetic (seeded; random-init LM head)",
        "config": bench_config(args, w, world),
        "impl": "reference",
        "cpu_baseline": {"value": value, "unit": "steps/s", "cores": host_cores(),
                         "blas_threads": blas_threads(), "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": "steps/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def loop_measure(workload: str, c: float, K: int, Wm: int, seed: int = 0) -> dict:
    """The draft -> verify loop on one GPU, against its closed form.

    "推测解码", section 快多少: with acceptance rate alpha, gamma guesses per
    step and a draft step costing c target steps, a step costs gamma*c + 1
    target steps and writes (1 - alpha^(gamma+1)) / (1 - alpha) tokens on
    average. Here every position has the same p and q (one hidden row and
    one draft-logit row repeated), so acceptances are independent with alpha
    = sum_v min(p, q); the drafter is a GPU busy-wait of c target steps per
    guess, its guesses fresh draws from q every step; the target step is the
    LM head scoring one position (a greedy verify of one guess reads W once).

    Besides the page's closed form, the verify step's own cost is charged in
    a second one: the verify step timed alone (gamma + 1 positions, the
    acceptance scan and the draw) in units of the target step replaces the
    1 in gamma*c + 1.
    """
    import target_model_verify_gb300 as tv
    device = torch.device("cuda", 0)
    torch.cuda.set_device(device)
    w = wl.get(workload)
    if w.tree is not None:
        raise SystemExit("the loop timer runs the chain step")
    B, gamma, d, V, T = w.B, w.gamma, w.d, w.V, w.temperature
    base = wl.generate(w, seed, device=device)
    W = base["W_lm"]
    hidden = base["hidden"][:, :1].expand(B, gamma + 1, d).contiguous()
    dl = base["draft_logits"][:, :1].expand(B, gamma, V).contiguous()
    p = torch.softmax((hidden[:, 0].double() @ W.double().T) / T, dim=-1)
    q = torch.softmax(dl[:, 0].double() / T, dim=-1)
    alpha = float(torch.minimum(p, q).sum(dim=-1).mean())
    g = torch.Generator(device=device)
    g.manual_seed(seed + 17)
    draws = torch.multinomial(q.float(), (K + Wm) * gamma, replacement=True, generator=g)
    drafts = draws.view(B, K + Wm, gamma).transpose(0, 1).contiguous().int()
    ws = tv.alloc_workspace(B, gamma, d, V, W.dtype, wl.SAMPLE, device=device)
    out = torch.empty(B, gamma + 1, dtype=torch.int32, device=device)
    naccs = torch.empty(K + Wm, B, dtype=torch.int32, device=device)

    def timed(fn, n):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        for i in range(3):
            fn(i)
        torch.cuda.synchronize()
        e0.record()
        for i in range(n):
            fn(i)
        e1.record()
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) * 1e3 / n

    # one target step: the LM head reading W once for one position per sequence
    h1 = hidden[:, :2].contiguous()
    ws1 = tv.alloc_workspace(B, 1, d, V, W.dtype, wl.GREEDY, device=device)
    t_target = timed(lambda i: tv.verify(h1, W, drafts[0][:, :1].contiguous(), None, T, i,
                                         wl.GREEDY, workspace=ws1), 300)
    # the verify step alone, on the loop's own inputs
    t_verify = timed(lambda i: tv.verify(hidden, W, drafts[i % (K + Wm)], dl, T, i, wl.SAMPLE,
                                         out_tokens=out, n_accepted=naccs[0], workspace=ws), 300)
    # the drafter: a busy-wait calibrated in SM cycles
    calib = 2_000_000
    us_per_cycle = timed(lambda i: torch.cuda._sleep(calib), 20) / calib
    draft_cycles = max(1, int(c * t_target / us_per_cycle))
    t_draft = timed(lambda i: torch.cuda._sleep(draft_cycles), 200)

    def step(i):
        for _ in range(gamma):
            torch.cuda._sleep(draft_cycles)
        tv.verify(hidden, W, drafts[i], dl, T, seed * 1_000_003 + i, wl.SAMPLE,
                  out_tokens=out, n_accepted=naccs[i], workspace=ws)

    for i in range(Wm):
        step(i)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for k in range(K):
        step(Wm + k)
    e1.record()
    torch.cuda.synchronize()
    t_step = e0.elapsed_time(e1) * 1e3 / K
    n = (naccs[Wm:].double() + 1).flatten()
    tokens = float(n.mean())
    c_eff = t_draft / t_target
    tok_closed = (1 - alpha ** (gamma + 1)) / (1 - alpha)
    pk = [alpha ** k * (1 - alpha) for k in range(gamma)] + [alpha ** gamma]
    var = sum(pk[k] * (k + 1) ** 2 for k in range(gamma + 1)) - tok_closed ** 2
    sigma = (tokens - tok_closed) / math.sqrt(var / n.numel())
    return {
        "metric": "speculative decoding speed-up over one token per target step (draft->verify loop)",
        "value": tokens * t_target / t_step,
        "unit": "x",
        "closed_form": tok_closed / (gamma * c_eff + 1),
        "closed_form_with_verify_cost": tok_closed / (gamma * c_eff + t_verify / t_target),
        "speedup_at_closed_form_tokens": tok_closed * t_target / t_step,
        "tokens_per_step_law_sigma": sigma,
        "alpha": alpha, "gamma": gamma, "c": c_eff, "steps": K, "warmup": Wm,
        "tokens_per_step": tokens, "closed_form_tokens_per_step": tok_closed,
        "target_step_us": t_target, "draft_token_us": t_draft, "loop_step_us": t_step,
        "verify_us": t_verify, "verify_cost_target_steps": t_verify / t_target,
        "config": {"workload": workload, "B": B, "d": d, "V": V, "temperature": T},
    }


def run_loop(args):
    """Prints loop_measure's line for --loop-c."""
    print(json.dumps(loop_measure(args.workload, args.loop_c, args.steps, args.warmup,
                                  args.seed)), flush=True)


def run_gamma_sweep(args):
    """Mean tokens per verify step against the closed form of "推测解码",
    section 接受率 α, on the Gemma-E2B-shaped head: every position has the same
    target row p and draft row q, the guesses are fresh draws from q, so
    acceptances are independent with alpha = sum_v min(p, q) (computed here in
    fp64 from the same bf16 inputs)."""
    import target_model_verify_gb300 as tv
    device = torch.device("cuda", 0)
    torch.cuda.set_device(device)
    w = wl.get("gemma_e2b_head_g1")
    base = wl.generate(w, args.seed + 21, device=device)
    W = base["W_lm"]
    d, V = W.shape[1], W.shape[0]
    z = base["hidden"][0, 0].double() @ W.double().t()
    zq = base["draft_logits"][0, 0].double()
    p, q = torch.softmax(z, 0), torch.softmax(zq, 0)
    alpha = float(torch.minimum(p, q).sum())
    g = torch.Generator(device=device)
    g.manual_seed(args.seed + 40)
    B, calls = 500, 8
    for gamma in (1, 2, 3, 4, 6, 8):
        hidden = base["hidden"][:, :1].expand(B, gamma + 1, d).contiguous()
        dl = base["draft_logits"][:, :1].expand(B, gamma, V).contiguous()
        ws = tv.alloc_workspace(B, gamma, d, V, torch.bfloat16, wl.SAMPLE, device=device)
        n = []
        for c in range(calls):
            x = torch.multinomial(q.float(), B * gamma, replacement=True, generator=g)
            _, nacc = tv.verify(hidden, W, x.view(B, gamma).int(), dl, 1.0, 500 + c, wl.SAMPLE,
                                workspace=ws)
            n.append(nacc.double() + 1)
        n = torch.cat(n)
        cf = (1 - alpha ** (gamma + 1)) / (1 - alpha)
        print(json.dumps({"metric": "mean tokens per verify step (i.i.d. positions)",
                          "gamma": gamma, "alpha": alpha, "measured": float(n.mean()),
                          "stderr": float(n.std() / n.numel() ** 0.5), "closed_form": cf,
                          "sequences": n.numel(),
                          "config": {"workload": "gemma_e2b_head (d 1536, V 262144)",
                                     "T": 1.0}}), flush=True)
        del hidden, dl, ws


def run_cluster_head(args):
    """The drafter's clustered LM head ("多詞元預測視覺化指南", section
    高效嵌入器): cluster logits, the top-K clusters, their members' logits and
    the draft token, against the bytes of the full head."""
    import target_model_verify_gb300 as tv
    M, K = (int(x) for x in args.cluster_head.split(","))
    V, d, n_c = 262144, 1536, 2048
    device = torch.device("cuda", 0)
    torch.cuda.set_device(device)
    g = torch.Generator(device=device)
    g.manual_seed(args.seed)
    W = (torch.randn(V, d, generator=g, device=device) * 0.02).to(torch.bfloat16)
    size = V // n_c
    E = W.view(n_c, size, d).float().mean(1).to(torch.bfloat16)
    starts = torch.arange(0, V + 1, size, dtype=torch.int32, device=device)
    tor = torch.randperm(V, generator=g, device=device).int()
    h = torch.randn(M, d, generator=g, device=device)
    h = (h / h.pow(2).mean(-1, keepdim=True).sqrt() * 3.0).to(torch.bfloat16)
    head = tv.ClusterHeadStep(h, E, W, starts, tor, top_k=K, max_cluster=size)
    ws = head.workspace
    step = lambda i: head(seed=i, position=i)
    Kst, Wm = args.steps, args.warmup
    for i in range(Wm):
        step(i)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for i in range(Kst):
        step(Wm + i)
    e1.record()
    torch.cuda.synchronize()
    if tv.read_status(ws) != 0:
        raise RuntimeError("device status after the clustered head")
    us = e0.elapsed_time(e1) * 1e3 / Kst
    bytes_read = n_c * d * 2 + M * K * size * d * 2 + M * d * 2
    peaks, kind = load_peaks()
    cpu = None
    if not args.no_cpu_baseline:
        # The fp64 oracle on the same rows (the tables converted once,
        # outside the timing), for ~10 s.
        from oracle import cluster_head as och
        f64 = lambda t: t.float().cpu().double().numpy()
        hs, Es, Ws = f64(h), f64(E), f64(W)
        st_, tr_ = starts.cpu().numpy(), tor.cpu().numpy()
        n, t0 = 0, time.perf_counter()
        while n < 1 or time.perf_counter() - t0 < CPU_BASELINE_SECONDS:
            och.cluster_head(hs, Es, Ws, st_, tr_, K, 1.0, n, wl.SAMPLE)
            n += 1
        cpu = {"value": (time.perf_counter() - t0) / n * 1e6, "unit": "us",
               "cores": host_cores(), "kind": "oracle",
               "sample": f"{n} full calls of the fp64 NumPy oracle (tables converted to fp64 "
                         f"once outside the timing)"}
    line = {
        "metric": "drafter clustered LM head, one call", "value": us, "unit": "us",
        "higher_is_better": False, "steps": Kst, "warmup": Wm,
        "bytes_read": bytes_read, "full_head_bytes": V * d * 2,
        "achieved_gbs": bytes_read / (us * 1e-6) / 1e9,
        "roofline": {"bound": "hbm", "achieved": bytes_read / (us * 1e-6) / 1e9,
                     "peak": peaks["hbm_gbs"], "unit": "GB/s",
                     "frac": bytes_read / (us * 1e-6) / 1e9 / peaks["hbm_gbs"],
                     "algorithmic_bytes": bytes_read, "kernel": "cluster head (3 kernels with one kept cluster and up to 8 rows, else 4)",
                     "peak_source": f"{kind} (MEASURED_PEAKS.json)"},
        "cpu_baseline": cpu,
        "config": {"M": M, "top_k": K, "V": V, "d": d, "clusters": n_c, "cluster_size": size,
                   "mode": "sample", "l2": "cluster table and kept rows fit in L2 (latency-bound)"},
    }
    print(json.dumps(line), flush=True)


def run_attention(args):
    """Verify-step attention for one layer: one GPU, CUDA events, inputs far
    larger than L2 ("推测解码", section 几段话一起写: every sequence reads its
    own KV cache, 131 KB per token over Llama 3.1 8B's 32 layers)."""
    import target_model_verify_gb300 as tv
    B, L, n_new = (int(x) for x in args.attention.split(","))
    Hq, Hkv, D = 32, 8, 128
    device = torch.device("cuda", 0)
    torch.cuda.set_device(device)
    g = torch.Generator(device=device)
    g.manual_seed(args.seed)
    q = torch.randn(B, n_new, Hq, D, generator=g, device=device).to(torch.bfloat16)
    k = torch.randn(B, L, Hkv, D, generator=g, device=device).to(torch.bfloat16)
    v = torch.randn(B, L, Hkv, D, generator=g, device=device).to(torch.bfloat16)
    lens = torch.full((B,), L, dtype=torch.int32, device=device)
    out = torch.empty(B, n_new, Hq, D, dtype=torch.float32, device=device)
    ws = torch.empty(tv.attention_workspace_bytes(B, n_new, Hq, Hkv, D, L), dtype=torch.uint8,
                     device=device)
    K, Wm = args.steps, args.warmup
    for _ in range(Wm):
        tv.verify_attention(q, k, v, lens, out=out, workspace=ws)
    torch.cuda.synchronize()
    sampler = ClockSampler(0)
    time.sleep(0.6)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t_wall0 = time.time()
    e0.record()
    for _ in range(K):
        tv.verify_attention(q, k, v, lens, out=out, workspace=ws)
    e1.record()
    torch.cuda.synchronize()
    t_wall1 = time.time()
    time.sleep(0.2)
    sampler.stop()
    if tv.read_status(ws) != 0:
        raise RuntimeError("device status after attention")
    us = e0.elapsed_time(e1) * 1e3 / K
    cpu = None
    if not args.no_cpu_baseline:
        # The fp64 oracle on one sequence at a time (inputs converted once),
        # as many as ~10 s allow, scaled to calls of all B sequences.
        from oracle import attention as oa
        qs = q[:1].float().cpu().double().numpy()
        ks = k[:1].float().cpu().double().numpy()
        vs = v[:1].float().cpu().double().numpy()
        ls = lens[:1].cpu().numpy()
        n, t0 = 0, time.perf_counter()
        while n < 1 or time.perf_counter() - t0 < CPU_BASELINE_SECONDS:
            oa.verify_attention(qs, ks, vs, ls)
            n += 1
        per_seq = (time.perf_counter() - t0) / n
        cpu = {"value": per_seq * B * 1e6, "unit": "us", "cores": host_cores(), "kind": "oracle",
               "sample": f"{n} single-sequence calls of the fp64 NumPy oracle, scaled to B={B}"}
    kv_bytes = 2 * B * L * Hkv * D * 2
    bytes_alg = kv_bytes + q.numel() * 2 + out.numel() * 4
    peaks, kind = load_peaks()
    achieved = bytes_alg / (us * 1e-6) / 1e9
    line = {
        "metric": "verify-step attention, one Llama-3-8B-shaped layer", "value": us,
        "unit": "us", "higher_is_better": False, "steps": K, "warmup": Wm,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"],
                     "unit": "GB/s", "frac": achieved / peaks["hbm_gbs"],
                     "algorithmic_bytes": bytes_alg, "kernel": "attn_split_kernel",
                     "peak_source": f"{kind} (MEASURED_PEAKS.json)"},
        "cpu_baseline": cpu,
        "config": {"B": B, "cached_tokens": L, "new_positions": n_new, "Hq": Hq, "Hkv": Hkv,
                   "D": D, "l2": "KV cache larger than L2 per call" if kv_bytes > 129e6 else
                   "KV cache smaller than L2"},
        "clocks": sampler.summary(t_wall0, t_wall1),
    }
    print(json.dumps(line), flush=True)


def run_vocab_slices(args):
    """One GPU's share of the vocabulary-parallel step ("推测解码", section
    几段话一起写: the weight read is the cost, so a tensor-parallel target
    splits W_lm by vocabulary rows). For each G the workload's W_lm is cut
    into G slices; slice 0's three calls (score, accept, draw) are timed with
    CUDA events, each alone and the three back to back (slice_calls_us),
    the exchanges between them done once beforehand from all slices (on G
    GPUs they are collectives, not timed here: one GPU). L2 is flushed (by a
    512 MB read) before every timed step; the single-GPU step is timed the
    same way beside it."""
    import target_model_verify_gb300 as tv
    device = torch.device("cuda", 0)
    torch.cuda.set_device(device)
    w = wl.get(args.workload)
    if w.tree is not None:
        raise SystemExit("the vocabulary-parallel step runs the chain")
    mode = wl.SAMPLE if args.mode == "sample" else wl.GREEDY
    inp = wl.generate(w, args.seed, device=device)
    B, gamma, d, V, T = w.B, w.gamma, w.d, w.V, w.temperature
    W, x = inp["W_lm"], inp["draft_tokens"]
    # read (not written) between steps, so the L2 holds no dirty lines to
    # write back inside the timed calls
    flush = torch.ones(128 << 20, dtype=torch.float32, device=device)
    K, Wm = args.steps, args.warmup
    peaks, kind = load_peaks()

    def timed_calls(calls):
        """Mean µs of each call (events between the calls) and of the calls
        back to back (events around them only), over K flushed steps each.
        Means, not medians: the event clock ticks in ~2 µs steps here, and
        the mean of many ticks is unbiased where the median is not."""
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(len(calls) + 1)]
        times = []
        for it in range(Wm + K):
            flush.amax()
            ev[0].record()
            for i, fn in enumerate(calls):
                fn()
                ev[i + 1].record()
            torch.cuda.synchronize()
            if it >= Wm:
                times.append([ev[i].elapsed_time(ev[i + 1]) * 1e3 for i in range(len(calls))])
        whole = []
        for it in range(Wm + K):
            flush.amax()
            ev[0].record()
            for fn in calls:
                fn()
            ev[1].record()
            torch.cuda.synchronize()
            if it >= Wm:
                whole.append(ev[0].elapsed_time(ev[1]) * 1e3)
        return [float(np.mean([t[i] for t in times])) for i in range(len(calls))], \
            float(np.mean(whole))

    dl_full = inp["draft_logits"] if mode == wl.SAMPLE else None
    ws = tv.alloc_workspace(B, gamma, d, V, W.dtype, mode, device=device)
    _, single_us = timed_calls([lambda: tv.verify(inp["hidden"], W, x, dl_full, T, 1, mode,
                                                 workspace=ws)])
    for G in (int(g) for g in args.vocab_slices.split(",")):
        bounds = [V * g // G for g in range(G + 1)]
        shards, dls = [], []
        for g in range(G):
            v0, v1 = bounds[g], bounds[g + 1]
            shards.append(tv.VocabShard(W[v0:v1], v0, V, B, gamma, mode, T))
            dls.append(inp["draft_logits"][:, :, v0:v1].contiguous() if mode == wl.SAMPLE
                       else None)
        all_rec = torch.cat([sh.score(inp["hidden"], x, dls[g]).clone()
                             for g, sh in enumerate(shards)])
        out = torch.empty(B, gamma + 1, dtype=torch.int32, device=device)
        nacc = torch.empty(B, dtype=torch.int32, device=device)
        sums = [sh.accept(all_rec, G, x, dls[g], 1, out, nacc).clone().reshape(-1)
                for g, sh in enumerate(shards)]
        all_sums = torch.cat(sums)
        sh, dl0 = shards[0], dls[0]
        calls = [lambda: sh.score(inp["hidden"], x, dl0),
                 lambda: sh.accept(all_rec, G, x, dl0, 1, out, nacc)]
        if mode == wl.SAMPLE:
            calls.append(lambda: sh.draw(all_sums, G, 0, dl0, 1, out))
        us, whole_us = timed_calls(calls)
        torch.cuda.synchronize()
        if tv.read_status(sh.workspace) != 0:
            raise RuntimeError("device status after the slice's calls")
        Vs = bounds[1]
        score_bytes = Vs * d * 2 + B * (gamma + 1) * d * 2 + (B * gamma * Vs * 2 if mode == wl.SAMPLE
                                                              else 0)
        gbs = score_bytes / (us[0] * 1e-6) / 1e9
        print(json.dumps({
            "metric": "vocabulary-parallel verify step, one GPU's calls (collectives not included)",
            "slices": G, "V_shard": Vs, "mode": args.mode,
            "score_us": us[0], "accept_us": us[1], "draw_us": us[2] if len(us) > 2 else 0.0,
            "slice_calls_us": whole_us, "single_gpu_step_us": single_us,
            "ideal_slice_us": single_us / G,
            "score_roofline": {"achieved": gbs, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                               "frac": gbs / peaks["hbm_gbs"], "algorithmic_bytes": score_bytes,
                               "peak_source": f"{kind} (MEASURED_PEAKS.json)"},
            "steps": K, "warmup": Wm, "l2": "flushed before every step (512 MB read)",
            "config": {"workload": args.workload, "B": B, "gamma": gamma, "d": d, "V": V},
        }), flush=True)
        del shards, dls, all_rec, sums, all_sums


def main(argv=None):
    args = parse_args(argv)
    world, rank, local = dist_env()
    if args.gpus != world and world > 1:
        raise SystemExit(f"--gpus {args.gpus} but WORLD_SIZE={world}")
    if args.loop_c is not None:
        run_loop(args)
        return
    if args.attention is not None:
        run_attention(args)
        return
    if args.cluster_head is not None:
        run_cluster_head(args)
        return
    if args.gamma_sweep:
        run_gamma_sweep(args)
        return
    if args.vocab_slices is not None:
        run_vocab_slices(args)
        return
    if args.impl == "reference":
        run_reference(args, world, rank, local)
    else:
        run_ours(args, world, rank, local)


if __name__ == "__main__":
    main()
