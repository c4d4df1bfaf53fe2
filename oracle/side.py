"""The pages' scheduling arithmetic, kept as oracle self-checks (test infrastructure only).

These steps are not on the GPU path (they split misses between a CPU and a
PCIe path, which this build does not have); they are restated because they
pin the reading of the pages' numbers.

  * Strata expert paths, "为什么 PCIe 份额从 0.49 调到 0.60？": the initial
    share is a base of 0.55 scaled by the link probe relative to 20 GB/s; the
    candidate share after measuring the CPU pool is P / (P + 1.85 * C).
  * FreeToken reading notes, section 3.2, equations (1)-(3): residual host
    bandwidth B_R = max(B_H - B_P, 0); fill and CPU times q*S/B_P and
    (m-q)*S/(B_H-B_P); balancing them gives q* = m * B_P / B_H, rounded, with
    at least one fill.
"""
from __future__ import annotations


def initial_share(probe_gbs: float, base: float = 0.55, reference_gbs: float = 20.0) -> float:
    return base * probe_gbs / reference_gbs


def candidate_share(pcie_rate: float, cpu_rate: float, coef: float = 1.85) -> float:
    return pcie_rate / (pcie_rate + coef * cpu_rate)


def residual_bandwidth(b_h: float, b_p: float) -> float:
    return max(b_h - b_p, 0.0)


def fill_time(q: int, size: float, b_p: float) -> float:
    return q * size / b_p


def cpu_time(m: int, q: int, size: float, b_h: float, b_p: float) -> float:
    return (m - q) * size / (b_h - b_p)


def q_star_fraction(b_p: float, b_h: float) -> float:
    return b_p / b_h


def q_star(m: int, b_p: float, b_h: float) -> int:
    if m <= 0:
        return 0
    return max(1, int(round(m * b_p / b_h)))
