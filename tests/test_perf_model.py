"""The performance model against the numbers the pages print (tests/golden/performance_model.txt)."""
import math
import os

import pytest

from allreduce_compatible_gradient_gb300 import perf_model as pm

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "performance_model.txt")


def golden():
    g = {}
    for line in open(GOLDEN):
        line = line.strip()
        if line and not line.startswith("#"):
            k, v = line.split()
            g[k] = float(v)
    return g


def test_exponential_dithering_limit_is_point_08_gamma():
    g = golden()
    lim = pm.max_link_bandwidth(1.0, g["rho"], g["omega_exponential_slowdown"])
    assert lim == pytest.approx(g["beta_over_gamma_limit_exponential"], abs=5e-4)  # 1.5 / 18.75


def test_standard_dithering_always_speeds_up():
    g = golden()
    assert pm.max_link_bandwidth(1.0, g["rho"], g["omega_standard"]) == math.inf
    for beta in (1e6, 1e9, 1e12, 1e15):
        assert pm.speeds_up(beta, 2e12, g["rho"], g["omega_standard"])


def test_a100_links_satisfy_the_exponential_condition():
    g = golden()
    for beta in (g["beta_nvlink"], g["beta_pcie"]):
        assert pm.speeds_up(beta, g["gamma_a100"], g["rho"], g["omega_exponential_slowdown"])
    # a link faster than 0.08 gamma would not benefit
    assert not pm.speeds_up(0.1 * g["gamma_a100"], g["gamma_a100"], g["rho"],
                            g["omega_exponential_slowdown"])


def test_condition_agrees_with_the_time_model():
    for beta in (5.4e9, 53.9e9, 2e11, 5e11):
        for omega in (1, 4, 12.9, 79):
            t = pm.allreduce_time(16, 25e6, 5e-6, beta, 2e12)
            tq = pm.quantized_allreduce_time(16, 25e6, 5e-6, beta, 2e12, 4, omega)
            assert (tq < t) == pm.speeds_up(beta, 2e12, 4, omega)


def test_theta_worked_example():
    g = golden()
    s = 2 ** int(g["theta_level_bits"])  # 7 level bits: the level term vanishes
    f = pm.iteration_factor(int(g["theta_n"]), g["theta_d"], s)
    assert f - 1 == pytest.approx(g["theta_iteration_increase"], abs=0.005)
    assert pm.compression_saving(32, 8) == g["theta_comm_saving"]
