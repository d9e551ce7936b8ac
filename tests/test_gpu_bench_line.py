"""The benchmark line of the library's arm, checked on the GPU.

One short run of bench.py at its default workload: the Llama-3-8B-shaped
head, B = 1, γ = 4, sampling. The test checks the keys the line must carry
and the arithmetic that ties them together. The byte counts are restated
here from the shapes. They are the step's inputs: W, the hidden rows and
the draft logits for the LM-head kernel, plus the draft tokens for the
end-to-end copies. So a line whose figures came from a different workload,
or from a kernel that skipped work, fails.
"""
import json
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
B, GAMMA, D, V = 1, 4, 4096, 128256
STEPS, WARMUP = 200, 5


@pytest.fixture(scope="module")
def line():
    cmd = [sys.executable, "bench.py", "--steps", str(STEPS), "--warmup", str(WARMUP),
           "--no-cpu-baseline"]
    out = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=900)
    assert out.returncode == 0, out.stderr[-3000:]
    lines = [ln for ln in out.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, out.stdout[-3000:]
    return json.loads(lines[0])


def test_bench_line_carries_the_contract_keys(line):
    r = line
    assert r["n_gpus"] == 1 and (r["steps"], r["warmup"]) == (STEPS, WARMUP)
    assert r["unit"] == "steps/s" and r["higher_is_better"] is True
    assert r["scaling"] == "weak" and r["vs_baseline"] is None
    assert r["dtype"] == "bf16" and r["data"].startswith("synthetic")
    assert r["config"]["workload"] == "llama3_8b_head"
    assert (r["config"]["B"], r["config"]["gamma"], r["config"]["d"], r["config"]["V"]) == \
        (B, GAMMA, D, V)
    assert r["cpu_baseline"] is None                     # skipped by --no-cpu-baseline
    for key in ("sm_mhz", "sm_max_mhz", "reasons"):
        assert key in r["clocks"], key


def test_bench_line_arithmetic(line):
    r = line
    M = B * (GAMMA + 1)
    assert r["value"] > 0
    assert r["ms_per_step"] == pytest.approx(1e3 / r["value"], rel=1e-9)
    assert 1.0 <= r["mean_tokens_per_step"] <= GAMMA + 1
    assert r["committed_tokens_per_s"] == pytest.approx(r["value"] * r["mean_tokens_per_step"],
                                                        rel=1e-9)
    # The LM-head kernel reads W, the hidden rows and the draft logits once.
    lm_bytes = V * D * 2 + M * D * 2 + B * GAMMA * V * 2
    roof = r["roofline"]
    assert roof["bound"] == "hbm" and roof["unit"] == "GB/s"
    assert roof["algorithmic_bytes"] == lm_bytes
    assert roof["achieved"] == pytest.approx(lm_bytes / (roof["kernel_us"] * 1e-6) / 1e9,
                                             rel=1e-9)
    assert roof["frac"] == pytest.approx(roof["achieved"] / roof["peak"], rel=1e-9)
    # A copy-bandwidth peak can be beaten a little, not by much; far below
    # it the kernel would not be streaming W.
    assert 0.5 < roof["frac"] < 1.15, roof
    # The LM head is part of the step. Its events sit between kernels, so its
    # time also holds the launch latency that back-to-back steps overlap
    # with the previous step's tail: a few percent of slack.
    assert roof["kernel_us"] < 1.03e3 * r["ms_per_step"]
    if roof["traffic"] is not None:
        assert roof["traffic"] >= 0.99 * lm_bytes
    assert 0.0 < r["step_roofline"]["frac"] <= 1.05
    # Two library kernels per step at B = 1: the LM head, then acceptance
    # with the draw.
    assert r["gpu_launches"] == 2 * STEPS


def test_bench_line_end_to_end_copies(line):
    r = line
    e2e = r["e2e"]
    assert e2e["unit"] == "steps/s" and e2e["value"] > 0
    # Host to device each step: hidden rows, draft tokens, draft logits;
    # device to host: the committed tokens and the accepted count.
    M = B * (GAMMA + 1)
    assert e2e["h2d_bytes_per_step"] == M * D * 2 + B * GAMMA * 4 + B * GAMMA * V * 2
    assert e2e["d2h_bytes_per_step"] == M * 4 + B * 4
    # Copies and a host round trip each step cannot beat the device-only rate.
    assert e2e["value"] <= 1.02 * r["value"]
