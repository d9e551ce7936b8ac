"""Closed forms printed on "推测解码" (world.lapla.si/zh/specdec).

Test infrastructure only (see the package docstring). These are the
acceptance-rate model of sections 接受率 α, 快多少 and 用的是闲着的算术:
with every position equally easy to guess (acceptance rate alpha), gamma
guesses give a geometric number of kept drafts, capped at gamma, plus the
one token the large model always writes.
"""
from __future__ import annotations


def acceptance_rate(p_row, q_row) -> float:
    """Probability one guess is kept: sum_v min(p_v, q_v) (section 接受率 α)."""
    return float(sum(min(a, b) for a, b in zip(p_row, q_row)))


def expected_tokens_per_step(alpha: float, gamma: int) -> float:
    """Mean tokens written per weight read: sum_{k=0..gamma} alpha^k.

    Equals (1 - alpha^(gamma+1)) / (1 - alpha) for alpha < 1.
    """
    return float(sum(alpha ** k for k in range(gamma + 1)))


def speedup(alpha: float, gamma: int, c: float) -> float:
    """Speed-up over one-token-per-read when a draft step costs c target steps.

    One step costs gamma*c + 1 target-step times and yields
    expected_tokens_per_step tokens (section 快多少).
    """
    return expected_tokens_per_step(alpha, gamma) / (gamma * c + 1.0)


def arithmetic_factor(alpha: float, gamma: int) -> float:
    """Target arithmetic per written token relative to plain decoding.

    Each step runs gamma + 1 target positions and writes
    expected_tokens_per_step tokens (section 用的是闲着的算术).
    """
    return (gamma + 1) / expected_tokens_per_step(alpha, gamma)
