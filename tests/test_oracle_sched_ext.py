"""Pins of the oracle's D-cut budget, static schedulers and STS calibration."""
import itertools

import numpy as np
import pytest

import oracle
import specsynth

RATIOS = [0.25, 0.5, 0.75, 1.0]


# ----------------------------------------------------------------- D-cut
def test_dcut_hand_trace():
    """B=2, gamma=2, survivals r0: [0.9, 0.45], r1: [0.6, 0.54]; B(gamma+1) = 6, so
    K = max(2, ceil(rho * 6)) = [2, 3, 5, 6] keep 0, 1, 3, 4 candidates and
    tau = [2, 2.9, 4.04, 4.49].  Costs [1, 1.4, 2.1, 2.3] give tau/C =
    [2, 2.071, 1.924, 1.952]: rho = 0.5 wins, keeping the 0.9 candidate."""
    conf = np.array([[0.9, 0.5], [0.6, 0.9]], np.float32)
    r = oracle.sched_dcut(conf, RATIOS, [1.0, 1.4, 2.1, 2.3])
    assert r["rc"] == 0 and r["choice"] == 1
    assert list(r["verify_len"]) == [1, 0]


def test_dcut_budget_lower_bound_keeps_every_anchor():
    """ceil(rho B (gamma+1)) below B is raised to B: every request keeps its
    bonus position and nothing else (AngelSpec eq. (22))."""
    conf = specsynth.make_confidences(8, 4, seed=9)
    r = oracle.sched_dcut(conf, [0.05], [1.0])
    assert (r["verify_len"] == 0).all()


def test_dcut_ties_go_to_the_first_ratio():
    """Confidences of 1 make tau(K) = K; costs equal to K tie every objective at
    exactly 1, and the first (smallest) ratio wins."""
    conf = np.ones((4, 3), np.float32)
    r = oracle.sched_dcut(conf, RATIOS, [4.0, 8.0, 12.0, 16.0])
    assert r["choice"] == 0 and (r["verify_len"] == 0).all()


def test_dcut_full_ratio_verifies_everything():
    conf = specsynth.make_confidences(8, 4, seed=9)
    r = oracle.sched_dcut(conf, [1.0], [3.0])
    assert (r["verify_len"] == 4).all()


def _brute_best_at(conf, N, min_len):
    """Largest progress over allocations in [min_len, gamma]^B with sum (l+1) = N."""
    B, gamma = conf.shape
    s = np.concatenate([np.ones((B, 1)), np.cumprod(conf.astype(np.float64), axis=1)], axis=1)
    prog = np.cumsum(s, axis=1)
    best, arg = -1.0, None
    for alloc in itertools.product(range(min_len, gamma + 1), repeat=B):
        if sum(a + 1 for a in alloc) != N:
            continue
        tau = sum(prog[b, alloc[b]] for b in range(B))
        if tau > best + 1e-12:
            best, arg = tau, alloc
    return best, arg


@pytest.mark.parametrize("min_len", [0, 1])
def test_dcut_matches_restricted_brute_force(min_len):
    """For every ratio, top-K selection gives the best allocation with exactly
    K_rho positions; the choice maximises progress / cost over the ratios."""
    rng = np.random.default_rng(4 + min_len)
    checked = 0
    for trial in range(300):
        B = int(rng.integers(1, 4))
        gamma = int(rng.integers(max(1, min_len), 4))
        conf = rng.uniform(0.05, 0.95, (B, gamma)).astype(np.float32)
        costs = list(np.sort(rng.uniform(1.0, 3.0, 4)))
        r = oracle.sched_dcut(conf, RATIOS, costs, min_len)
        assert r["rc"] == 0
        Nmax, N0 = B * (gamma + 1), B * (min_len + 1)
        objs = []
        for rho, cst in zip(RATIOS, costs):
            K = min(Nmax, max(N0, int(np.ceil(rho * Nmax))))
            tau, alloc = _brute_best_at(conf, K, min_len)
            objs.append((tau / cst, alloc))
        vals = np.array([o[0] for o in objs])
        order = np.sort(vals)
        if len(order) > 1 and order[-1] - order[-2] < 1e-9 * order[-1]:
            continue
        k = int(np.argmax(vals))
        checked += 1
        assert r["choice"] == k
        assert tuple(r["verify_len"]) == objs[k][1]
    assert checked > 200


# ------------------------------------------------- progress accuracy
def _exact_progress(conf, alloc):
    """tau of an allocation in exact rational arithmetic from the fp32 confidences."""
    from fractions import Fraction
    tau = Fraction(0)
    for b, ell in enumerate(alloc):
        s = Fraction(1)
        tau += s
        for k in range(ell):
            s *= Fraction(float(conf[b, k]))
            tau += s
    return tau


@pytest.mark.parametrize("cost_name", ["Bprime", "C"])
def test_objective_matches_exact_rational_progress(cost_name):
    """The reported best objective equals the exact tau / C of the chosen
    allocation to 1e-12 (relative): fp64 survival products plus survivals
    rounded to 2^-46 lose far less than that at these sizes."""
    from fractions import Fraction
    cost = specsynth.COST_TABLES[cost_name]
    rng = np.random.default_rng(12)
    for trial in range(60):
        B = int(rng.integers(1, 40))
        gamma = int(rng.integers(1, 9))
        conf = specsynth.make_confidences(B, gamma, seed=1300 + trial, mean=float(rng.uniform(-1, 3)))
        r = oracle.sched_exact(conf, cost, 0)
        alloc = r["verify_len"]
        N = int((alloc + 1).sum())
        exact = _exact_progress(conf, alloc) / Fraction(oracle.cost_at(N, cost))
        assert abs(Fraction(r["obj"]) - exact) <= Fraction(1, 10 ** 12) * exact, trial


# ---------------------------------------------------------- static modes
def test_threshold_zero_is_fixed_length():
    """'A threshold of zero recovers standard fixed-length verification.'"""
    conf = specsynth.make_confidences(16, 8, seed=1)
    assert (oracle.sched_threshold(conf, 0.0)["verify_len"] == 8).all()


def test_threshold_keeps_the_leading_run():
    conf = np.array([[0.9, 0.5, 0.95], [0.7, 0.7, 0.7], [0.2, 0.9, 0.9]], np.float32)
    assert list(oracle.sched_threshold(conf, 0.6)["verify_len"]) == [1, 3, 0]
    assert list(oracle.sched_threshold(conf, 0.6, min_len=1)["verify_len"]) == [1, 3, 1]
    assert (oracle.sched_threshold(conf, 1.5)["verify_len"] == 0).all()
    # a confidence equal to the threshold is kept
    assert list(oracle.sched_threshold(np.array([[0.5, 0.5, 0.25]], np.float32), 0.5)["verify_len"]) == [2]


def test_fixed_length_mode():
    conf = specsynth.make_confidences(16, 8, seed=1)
    assert (oracle.sched_threshold(conf, 0.0, max_len=3)["verify_len"] == 3).all()
    assert (oracle.sched_threshold(conf, 0.0, min_len=2, max_len=2)["verify_len"] == 2).all()


def test_threshold_is_monotone():
    conf = specsynth.make_confidences(64, 16, seed=2)
    prev = None
    for th in np.linspace(0, 1, 21):
        v = oracle.sched_threshold(conf, th)["verify_len"]
        if prev is not None:
            assert (v <= prev).all()
        prev = v


# -------------------------------------------------------------------- STS
def test_ece_closed_form():
    """Bins of width 1/15: 0.05 -> 0, 0.1 -> 1, 0.95 -> 14, 0.9 -> 13, so
    ECE = (0.05 + 0.1 + 0.05 + 0.9) / 4 = 0.275."""
    e = oracle.sts_ece([0.05, 0.1, 0.95, 0.9], [0, 0, 1, 0], 15)
    assert abs(e - 0.275) < 1e-15


def _labels(conf, rng, power):
    """Accept lengths when position k survives with probability c_k^power."""
    n, gamma = conf.shape
    acc = rng.random((n, gamma)) < conf.astype(np.float64) ** power
    first_rej = np.where(~acc, np.arange(gamma)[None, :], gamma).min(axis=1)
    return first_rej.astype(np.int32)


@pytest.mark.slow
@pytest.mark.parametrize("power,expect", [(1.0, 1.0), (2.0, 0.5), (0.5, 2.0)])
def test_sts_recovers_the_temperature(power, expect):
    """Survival c^power is c^(1/T) with T = 1/power: the fit finds it (on the
    0.1 grid) at every position."""
    rng = np.random.default_rng(7)
    conf = (1 / (1 + np.exp(-rng.normal(1.0, 1.0, (40000, 4))))).astype(np.float32)
    al = _labels(conf, rng, power)
    r = oracle.sts_fit(conf, al)
    assert r["rc"] == 0
    assert np.all(np.abs(r["T"] - expect) <= 0.15 * expect + 1e-9), r["T"]


def test_sts_temperatures_feed_the_schedulers():
    conf = specsynth.make_confidences(8, 6, seed=3)
    cost = ([0.0, 1000.0], [8.0, 28.0])
    ones = np.ones(6)
    assert (oracle.sched_exact(conf, cost, 0, sts_T=ones)["verify_len"]
            == oracle.sched_exact(conf, cost, 0)["verify_len"]).all()
    # T -> large pushes calibrated confidences to 1 (longer), T small to 0 (shorter)
    hot = oracle.sched_threshold(conf, 0.9, sts_T=np.full(6, 10.0))["verify_len"]
    cold = oracle.sched_threshold(conf, 0.9, sts_T=np.full(6, 0.1))["verify_len"]
    base = oracle.sched_threshold(conf, 0.9)["verify_len"]
    assert (hot >= base).all() and (cold <= base).all() and hot.sum() > cold.sum()
