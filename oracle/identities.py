"""ORACLE (test infrastructure only): the closed-form identities the model
cards use to reason about the drafter.

* Speculative throughput goes as a / (d + T), so the relative throughput of
  two drafters is (a1 / a2) * (d2 + T) / (d1 + T) -- "Kimi-K3-DSpark-NVFP4",
  "Considerations".
* Acceptance length is a prefix-run-length statistic: a block is accepted up
  to its first mismatch, so the expected accepted length is
  sum_k prod_{i<=k} s_i with s_i the agreement at position i given agreement
  before it -- "Kimi-K3-DSpark-NVFP4", "Why acceptance is so sensitive" and
  the drift tables in "Measurement".
"""
from __future__ import annotations

from typing import Sequence


def speculative_ratio(a1: float, a2: float, d1: float, d2: float, T: float) -> float:
    """Throughput of drafter 1 over drafter 2: (a1/a2) * (d2 + T) / (d1 + T)."""
    return (a1 / a2) * (d2 + T) / (d1 + T)


def draft_speed_limit(byte_ratio: float) -> float:
    """(d + T) / (r d + T) as d / T -> infinity: 1 / r."""
    return 1.0 / byte_ratio


def break_even_d_over_T(need: float, byte_ratio: float) -> float:
    """d / T at which (d + T) / (r d + T) reaches ``need``: d/T = (need - 1) / (1 - need r)."""
    return (need - 1.0) / (1.0 - need * byte_ratio)


def accepted_prefix(match: Sequence[bool]) -> int:
    """Number of leading positions that match (the accepted run)."""
    n = 0
    for m in match:
        if not m:
            break
        n += 1
    return n


def accepted_prefix_by_products(match: Sequence[bool]) -> int:
    """The same count written as sum_k prod_{i<=k} 1[match_i]."""
    total, run = 0, 1
    for m in match:
        run *= 1 if m else 0
        total += run
    return total


def expected_accept_length(conditional_agreement: Sequence[float]) -> float:
    """E[a] = sum_k prod_{i<=k} s_i."""
    total, run = 0.0, 1.0
    for s in conditional_agreement:
        run *= s
        total += run
    return total
