"""Expected number of distinct destination ranks per token.

TEST INFRASTRUCTURE ONLY (part of the oracle package).

DeepEP V2 deep-dive page ("DeepEP V2 深度深潜"), section 1.3 factor 1 and
section 2.2: with E experts spread evenly over G groups (ranks) and k experts
drawn uniformly without replacement per token, a group receives the token
unless all k experts avoid its E/G experts, which happens with probability
C(E - E/G, k) / C(E, k). Summing the hit probability over the G groups gives
the expectation; the page requires E % G == 0.

The variance is not on the page; it follows from the same counting. With
a = C(E-m, k)/C(E, k), b = C(E-2m, k)/C(E, k), m = E/G and p = 1 - a, two
distinct groups are both hit with probability 1 - 2a + b (inclusion-exclusion),
so Var(D) = G p (1 - p) + G (G - 1) ((1 - 2a + b) - p^2).
"""
from __future__ import annotations

from fractions import Fraction
from math import comb


def expected_topk_exact(num_experts: int, num_groups: int, num_topk: int) -> Fraction:
    if num_experts % num_groups != 0:
        raise ValueError("num_experts must be a multiple of num_groups")
    m = num_experts // num_groups
    miss = Fraction(comb(num_experts - m, num_topk), comb(num_experts, num_topk))
    return num_groups * (1 - miss)


def get_expected_topk(num_experts: int, num_groups: int, num_topk: int) -> float:
    return float(expected_topk_exact(num_experts, num_groups, num_topk))


def variance_topk_exact(num_experts: int, num_groups: int, num_topk: int) -> Fraction:
    if num_experts % num_groups != 0:
        raise ValueError("num_experts must be a multiple of num_groups")
    m = num_experts // num_groups
    total = comb(num_experts, num_topk)
    a = Fraction(comb(num_experts - m, num_topk), total)
    b = Fraction(comb(num_experts - 2 * m, num_topk), total) if num_experts - 2 * m >= 0 else Fraction(0)
    p = 1 - a
    both = 1 - 2 * a + b
    G = num_groups
    return G * p * (1 - p) + G * (G - 1) * (both - p * p)
