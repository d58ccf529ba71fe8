"""Global-QSGD's performance model: when does quantising the allreduce speed training up?

Source: "Global-QSGD: Practical Floatless Quantization for Distributed Learning with Theoretical
Guarantees" (arXiv 2305.18627), performance-model section and the theta worked example of the
convergence section.  Pure arithmetic on the host; no GPU work.

Tree allreduce of S bytes over N workers (the section's model):
    T(S) = 2 log2(N) alpha + 2 log2(N) S / beta + log2(N) S / gamma
alpha: propagation delay (s); beta: link bandwidth (B/s); gamma: reduction speed (B/s).
With quantisation to S / rho bytes, a reduction speed gamma_hat = gamma / omega (omega >= 1: the
custom reduction is omega times slower than the native sum) and quantise + dequantise time
delta S:
    T_q(S) = 2 log2(N) alpha + 2 log2(N) S / (rho beta) + log2(N) omega S / (rho gamma) + delta S

Reading: the page writes the overhead as omega = gamma / gamma_hat and quotes omega_E = 1/79; the
quoted consequence ("a speed-up iff beta < 0.08 gamma") only follows with gamma / gamma_hat = 79,
i.e. the exponential scheme's custom reduction 79 times slower than the native sum, so omega here
is the slowdown factor (>= 1).  The equation of the speed-up condition is lost from the page; with
delta = 0, T_q < T reduces to
    (2 / beta)(1 - 1/rho) > (omega/rho - 1) / gamma,
always true when omega <= rho (standard dithering, omega = 1), otherwise true iff
    beta < 2 (1 - 1/rho) gamma / (omega/rho - 1).
"""
from __future__ import annotations

import math


def allreduce_time(n_workers: int, size_bytes: float, alpha: float, beta: float,
                   gamma: float) -> float:
    """Tree allreduce time of the uncompressed gradient (seconds)."""
    lg = math.log2(n_workers)
    return 2 * lg * alpha + 2 * lg * size_bytes / beta + lg * size_bytes / gamma


def quantized_allreduce_time(n_workers: int, size_bytes: float, alpha: float, beta: float,
                             gamma: float, rho: float, omega: float, delta: float = 0.0) -> float:
    """Tree allreduce time with Global-QSGD (seconds): S / rho bytes on the wire, a reduction
    omega times slower than the native one, and delta S for quantise + dequantise."""
    lg = math.log2(n_workers)
    s_hat = size_bytes / rho
    return (2 * lg * alpha + 2 * lg * s_hat / beta + lg * s_hat * omega / gamma
            + delta * size_bytes)


def speeds_up(beta: float, gamma: float, rho: float, omega: float) -> bool:
    """The speed-up condition with delta = 0 (independent of N, S and alpha)."""
    return (2.0 / beta) * (1.0 - 1.0 / rho) > (omega / rho - 1.0) / gamma


def max_link_bandwidth(gamma: float, rho: float, omega: float) -> float:
    """The largest link bandwidth beta at which quantising still pays (inf if always)."""
    if omega <= rho:
        return math.inf
    return 2.0 * (1.0 - 1.0 / rho) * gamma / (omega / rho - 1.0)


def compression_saving(bits_full: int = 32, bits_code: int = 8) -> float:
    """Fraction of communication saved by sending bits_code instead of bits_full per element."""
    return 1.0 - bits_code / bits_full


def iteration_factor(n_workers: int, dim: float, s: int) -> float:
    """Worst-case growth of the iteration count for Global-E_s as the theta worked example
    states it: 1 + n^1.17 (1/(8n) + sqrt(d) / (sqrt(n) 2^(s-1))).  The exponent 1.17 is as the
    page prints it (its derivation is not on the page)."""
    n = float(n_workers)
    return 1.0 + n ** 1.17 * (1.0 / (8.0 * n) + math.sqrt(dim) / (math.sqrt(n) * 2.0 ** (s - 1)))
