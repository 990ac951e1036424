"""Acceptance metrics derived from the R/I/D/A counters.

Definitions from "Structured output speculative decoding acceptance" (fanout.sh):
section "Name the three counters" -- R raw drafts, I grammar-invalidated drafts,
D = R - I eligible drafts, A drafts accepted by the target verifier; grammar
survival D/R, conditional target acceptance A/D (vLLM's draft_acceptance_rate),
end-to-end draft yield A/R. Section "Mean acceptance length uses another
denominator": mean acceptance length = 1 + A / (number of verification steps),
the 1 being the bonus (or recovered) token every step commits.
"""
from __future__ import annotations

from typing import Dict, Sequence


def _ratio(num: float, den: float) -> float:
    return float(num) / float(den) if den else float("nan")


def acceptance_rates(counters: Sequence[int]) -> Dict[str, float]:
    """counters = (R, I, D, A) -> the three ratios of the acceptance post."""
    R, I, D, A = (int(c) for c in counters)
    if D != R - I:
        raise ValueError(f"inconsistent counters: D={D} != R-I={R - I}")
    return {
        "grammar_survival": _ratio(D, R),
        "conditional_acceptance": _ratio(A, D),
        "end_to_end_yield": _ratio(A, R),
    }


def mean_acceptance_length(accepted: int, steps: int) -> float:
    """1 + A / steps (one verification step per request per call)."""
    return 1.0 + _ratio(accepted, steps)
