"""The stored offline profiles in ``workloads/demands.json`` are what the oracle
gives today.

S-HPLB profiles every head offline on calibration data (Italian summary,
"Profilatura Offline"; Chinese summary 2.1, "离线分析") and the plan is built
from that profile.  The calibrated tests and the bench read the stored copy,
so a silent change in the calibration oracle or in the seeded generator would
otherwise go unnoticed.  These tests re-run the oracle and compare: the whole
tiny workload and the lognormal workload, and a few heads (the densest, the
sparsest and the first and last) of each 8K-token calibration of the
Llama-3.1-8B-shaped workloads.
"""
import json
import os

import pytest

from oracle import make_demands, plan
from workloads import WORKLOADS

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
KEYS = ("k_uniform", "density", "demand", "budgets_maxmin")


@pytest.fixture(scope="module")
def stored():
    with open(os.path.join(ROOT, "workloads", "demands.json")) as f:
        return json.load(f)


@pytest.mark.parametrize("number", [1, 4])
def test_whole_profile_rederives(stored, number):
    got = make_demands.profile(number)
    for key in KEYS:
        assert got[key] == stored[str(number)][key], (number, key)
    assert got["mean_density_after_shift"] == pytest.approx(
        stored[str(number)]["mean_density_after_shift"], rel=1e-12)


@pytest.mark.parametrize("number", [2, 3])
def test_calibrated_heads_rederive(stored, number):
    prof = stored[str(number)]
    w = WORKLOADS[number]
    dens = prof["density"]
    heads = sorted({0, w.num_q_heads - 1, dens.index(max(dens)), dens.index(min(dens))})
    for h in heads:
        rho = round(float(make_demands._head_density((number, h))), 12)
        assert rho == dens[h], (number, h, rho, dens[h])
    # the rest of the profile follows from the densities by the plan's rules
    nb = w.nb
    assert prof["k_uniform"] == plan.budget_for_density(w.target_density, nb)
    assert prof["demand"] == [make_demands.calib.demand_for_density(r, nb) for r in dens]
    assert prof["budgets_maxmin"] == plan.maxmin_shift(prof["k_uniform"], prof["demand"],
                                                       make_demands.K_MIN, nb)
