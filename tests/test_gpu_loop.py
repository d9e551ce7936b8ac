"""The draft -> verify loop on the GPU against the speed-up formula of
"推测解码", section 快多少: speed-up = (1 - a^(g+1)) / ((1 - a)(g c + 1)),
a the acceptance rate, g the guesses per step, c a draft step's cost in
target steps.

bench.loop_measure times the loop on the Llama-3-8B-shaped head (g = 4,
every position with the same p and q, so acceptances are independent with
a = sum_v min(p, q)): g busy-wait kernels of c target steps each, then one
verify step, against one target step (the LM head scoring one position).
The measured speed-up, with the sampled tokens per step replaced by their
closed form so that only the costs are compared, must lie between

  * the page's closed form, which charges the verify step as one target
    step (an upper bound: the verify step scores g + 1 positions and runs
    the acceptance scan and the draw after the LM head), and
  * the same form with the verify step charged at its own cost, timed
    alone on the same inputs (the loop's verify step is the same call).

Slack of 3 % on either side: the loop's kernels run back to back, so a
verify step's launch can overlap the last draft kernel's tail (a few us of
a ~200-300 us step), and the three costs are means of separately timed
runs, each good to about 1 %. The tokens per step must follow their law
within 5 standard errors.
"""
import pytest

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from target_model_verify_gb300 import build
    build.build()
    import target_model_verify_gb300  # noqa: F401  (fails loudly if the library is missing)


@pytest.mark.parametrize("c", [0.1, 0.25])
def test_loop_speedup_lies_between_the_closed_forms(c):
    import bench
    r = bench.loop_measure("llama3_8b_head", c, K=1000, Wm=20, seed=0)
    print(f"c={r['c']:.3f}: measured {r['value']:.3f}x (at closed-form tokens "
          f"{r['speedup_at_closed_form_tokens']:.3f}x), closed form {r['closed_form']:.3f}x, "
          f"with the verify cost ({r['verify_cost_target_steps']:.3f} target steps) "
          f"{r['closed_form_with_verify_cost']:.3f}x; tokens/step {r['tokens_per_step']:.3f} vs "
          f"{r['closed_form_tokens_per_step']:.3f} ({r['tokens_per_step_law_sigma']:+.2f} s.e.)")
    assert abs(r["c"] - c) < 0.25 * c, r["c"]
    assert 1.0 < r["verify_cost_target_steps"] < 1.5
    assert abs(r["tokens_per_step_law_sigma"]) < 5
    s = r["speedup_at_closed_form_tokens"]
    assert r["closed_form_with_verify_cost"] * 0.97 <= s <= r["closed_form"] * 1.03, r
